"""The whole-output parity helpers (fullsize.py) on CPU: running the oracle
on all host cores, and cutting multi-token runs into pieces, give exactly the
oracle's single-call results."""
import numpy as np

import fullsize
import oracle
from paged_kv_cache_151_gb300 import workloads as wl


def test_decode_all_equals_one_thread():
    b = wl.random_batch(41, num_seqs=9, max_len=300, num_heads=8, num_kv_heads=2,
                        head_dim=64, dtype="bf16", device="cpu", new_in_pool=True,
                        keep_seq=False)
    ref = oracle.decode(b.q, b.k_cache, b.v_cache, b.block_tables, b.seq_lens, b.scale,
                        b.num_kv_heads, b.dtype, nthreads=1)
    got, _ = fullsize.decode_all(b)
    assert np.array_equal(got, ref)


def test_multi_all_pieces_equal_whole_sequences():
    """Rows cut into pieces of 5 (runs of 0..23 rows) reproduce the oracle's
    call over the whole runs bit for bit: each piece sees the positions its
    rows see in the whole run."""
    n = np.array([0, 1, 23, 5, 11, 6, 17])
    b = wl.multi_query_batch(42, num_seqs=len(n), min_ctx=0, max_ctx=70, n_new=n,
                             num_heads=8, num_kv_heads=2, head_dim=64, dtype="bf16",
                             device="cpu", keep_seq=False)
    ref = oracle.decode_multi(b.q, b.k_cache, b.v_cache, b.block_tables, b.seq_lens,
                              b.meta["query_start"], b.scale, b.num_kv_heads, b.dtype)
    got, _ = fullsize.multi_all(b, rows_per_piece=5)
    assert np.array_equal(got, ref)


def test_check_records_and_enforces_the_tolerance():
    ref = np.ones((2, 3, 4))
    n0 = len(fullsize.RESULTS)
    try:
        fullsize.check("within", ref + 1e-4, ref, "bf16")
        assert len(fullsize.RESULTS) == n0 + 1
        for gpu, dtype in ((ref + 0.1, "bf16"), (ref + 2e-4, "f32")):
            try:
                fullsize.check("too far", gpu, ref, dtype)
            except AssertionError:
                continue
            raise AssertionError(f"an error past the {dtype} tolerance passed")
    finally:
        del fullsize.RESULTS[n0:]
