"""Multi-token queries over the paged cache (pa_decode_multi): parity with the
fp64 oracle's causal multi-query attention, through the C ABI.

Tolerances as for decode with 16-bit caches: max |err| <= 2e-2 and relative
L2 error <= 5e-3 against the fp64 oracle, on the output as stored.
"""
import numpy as np
import pytest
import torch

import fullsize
import oracle
from paged_kv_cache_151_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

TOL_16_ABS = 2e-2
TOL_16_REL_L2 = 5e-3


def assert_close(gpu, ref, what=""):
    g = gpu.detach().double().cpu().numpy() if isinstance(gpu, torch.Tensor) else gpu
    ref = np.asarray(ref, dtype=np.float64)
    assert g.shape == ref.shape, (g.shape, ref.shape)
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    if not g.size:
        return
    err = np.abs(g - ref).max()
    rel = np.linalg.norm(g - ref) / max(np.linalg.norm(ref), 1e-30)
    assert err <= TOL_16_ABS, f"{what}: max abs err {err:.3g}"
    assert rel <= TOL_16_REL_L2, f"{what}: rel L2 err {rel:.3g}"


@pytest.fixture(autouse=True)
def _clean_error_word(cuda_lib):
    cuda_lib.pa_device_error(clear=True)
    yield
    flags = cuda_lib.pa_device_error(clear=True)
    assert flags == 0, f"device error word set: {flags:#x}"


def gpu_multi(pa, b, query_start=None, max_query_len=None, seq_lens=None,
              block_tables=None):
    qs = b.meta["query_start"] if query_start is None else query_start
    n = np.diff(qs)
    mq = int(n.max()) if max_query_len is None else max_query_len
    bt = torch.as_tensor(b.block_tables if block_tables is None else block_tables,
                         dtype=torch.int32, device="cuda").contiguous()
    sl = torch.as_tensor(b.seq_lens if seq_lens is None else seq_lens, dtype=torch.int32,
                         device="cuda").contiguous()
    qs_t = torch.as_tensor(qs, dtype=torch.int32, device="cuda").contiguous()
    out = torch.full_like(b.q, float("nan"))
    pa.pa_decode_multi(out, b.q, b.k_cache, b.v_cache, bt, sl, qs_t, mq, b.scale,
                       b.num_kv_heads)
    torch.cuda.synchronize()
    return out


def oracle_multi(b, query_start=None, seqs=None):
    """The oracle over all sequences, or over the subset ``seqs`` (then the
    rows come back in the subset's order)."""
    qs = b.meta["query_start"] if query_start is None else query_start
    q = b.q.cpu()
    if seqs is None:
        return oracle.decode_multi(q, b.k_cache.cpu(), b.v_cache.cpu(), b.block_tables,
                                   b.seq_lens, qs, b.scale, b.num_kv_heads, b.dtype)
    rows = np.concatenate([np.arange(qs[s], qs[s + 1]) for s in seqs])
    n = np.array([qs[s + 1] - qs[s] for s in seqs])
    sub_qs = np.zeros(len(seqs) + 1, dtype=np.int32)
    sub_qs[1:] = np.cumsum(n)
    ref = oracle.decode_multi(q[torch.from_numpy(rows)].contiguous(), b.k_cache.cpu(),
                              b.v_cache.cpu(), b.block_tables[seqs], b.seq_lens[seqs],
                              sub_qs, b.scale, b.num_kv_heads, b.dtype)
    return ref, rows


CASES = []
for dtype in ("bf16", "f16"):
    for D in (64, 128):
        for G, Hkv in ((1, 4), (2, 2), (4, 2), (8, 1)):
            CASES.append((dtype, D, G, Hkv))


@pytest.mark.parametrize("dtype,D,G,Hkv", CASES,
                         ids=[f"{c[0]}-d{c[1]}-g{c[2]}" for c in CASES])
def test_multi_parity_small(cuda_lib, dtype, D, G, Hkv):
    """1..20 new tokens over 0..300 cached ones: row tiles of 16 (token, head)
    pairs span several tokens, several tiles and ragged tails."""
    b = wl.multi_query_batch(500 + D + G, num_seqs=9, min_ctx=0, max_ctx=300,
                             n_new=(1, 20), num_heads=G * Hkv, num_kv_heads=Hkv,
                             head_dim=D, dtype=dtype, device="cuda", keep_seq=False)
    assert_close(gpu_multi(cuda_lib, b), oracle_multi(b), f"{dtype} d{D} g{G}")


@pytest.mark.parametrize("G", [1, 4, 8])
def test_multi_whole_sequence_is_new(cuda_lib, G):
    """n = seq_len: a first prefill chunk with nothing cached before it; row
    i sees exactly positions 0..i (the first row sees one token)."""
    Hkv = 2
    b = wl.multi_query_batch(520 + G, num_seqs=5, min_ctx=0, max_ctx=0, n_new=(1, 70),
                             num_heads=G * Hkv, num_kv_heads=Hkv, head_dim=128,
                             dtype="bf16", device="cuda", keep_seq=False)
    assert (np.diff(b.meta["query_start"]) == b.seq_lens).all()
    out = gpu_multi(cuda_lib, b)
    assert_close(out, oracle_multi(b), f"prefill g{G}")
    # the first row of every sequence sees only its own token: out = its V row
    qs = b.meta["query_start"]
    for s in range(b.num_seqs):
        blk = int(b.block_tables[s, 0])
        v0 = b.v_cache[blk, :, 0, :].repeat_interleave(G, dim=0)
        assert torch.equal(out[qs[s]], v0)


def test_multi_one_token_matches_decode(cuda_lib):
    """One query row per sequence is the decode step: same numbers as
    pa_decode within the 16-bit tolerance of each other's oracle."""
    b = wl.multi_query_batch(530, num_seqs=40, min_ctx=0, max_ctx=600, n_new=1,
                             num_heads=32, num_kv_heads=8, head_dim=128, dtype="bf16",
                             device="cuda", keep_seq=False)
    out = gpu_multi(cuda_lib, b)
    bt = torch.as_tensor(b.block_tables, device="cuda").contiguous()
    sl = torch.as_tensor(b.seq_lens, device="cuda").contiguous()
    dec = torch.full_like(b.q, float("nan"))
    cuda_lib.pa_decode(dec, b.q, b.k_cache, b.v_cache, bt, sl, b.scale, b.num_kv_heads)
    torch.cuda.synchronize()
    ref = oracle.decode(b.q.cpu(), b.k_cache.cpu(), b.v_cache.cpu(), b.block_tables,
                        b.seq_lens, b.scale, b.num_kv_heads, "bf16")
    assert_close(out, ref, "n=1 vs decode oracle")
    assert_close(dec, ref, "decode")
    assert_close(out, oracle_multi(b), "n=1 vs multi oracle")


def test_multi_sequences_without_rows(cuda_lib):
    """Sequences that run no token this step (n = 0) own no rows; the others
    are unaffected."""
    b = wl.multi_query_batch(540, num_seqs=12, min_ctx=1, max_ctx=200,
                             n_new=[3, 0, 5, 0, 0, 17, 1, 0, 2, 9, 0, 4], num_heads=16,
                             num_kv_heads=4, head_dim=128, dtype="bf16", device="cuda",
                             keep_seq=False)
    assert_close(gpu_multi(cuda_lib, b), oracle_multi(b), "with empty sequences")


def test_multi_larger_max_query_len_is_harmless(cuda_lib):
    b = wl.multi_query_batch(541, num_seqs=6, min_ctx=0, max_ctx=100, n_new=(1, 8),
                             num_heads=8, num_kv_heads=2, head_dim=64, dtype="f16",
                             device="cuda", keep_seq=False)
    a = gpu_multi(cuda_lib, b)
    c = gpu_multi(cuda_lib, b, max_query_len=64)
    assert_close(a, oracle_multi(b), "tight bound")
    assert_close(c, oracle_multi(b), "loose bound")


def test_multi_block_permutation_bit_identical(cuda_lib):
    b = wl.multi_query_batch(550, num_seqs=10, min_ctx=0, max_ctx=400, n_new=(1, 12),
                             num_heads=32, num_kv_heads=8, head_dim=128, dtype="bf16",
                             device="cuda", keep_seq=False)
    p = wl.permute_blocks(b, seed=9)
    p.meta["query_start"] = b.meta["query_start"]
    assert torch.equal(gpu_multi(cuda_lib, b), gpu_multi(cuda_lib, p))


def test_multi_invalid_row_range_is_flagged_and_skipped(cuda_lib):
    b = wl.multi_query_batch(560, num_seqs=4, min_ctx=5, max_ctx=60, n_new=[3, 1, 3, 2],
                             num_heads=8, num_kv_heads=2, head_dim=64, dtype="bf16",
                             device="cuda", keep_seq=False)
    qs = b.meta["query_start"]
    ref = oracle_multi(b)
    rows = lambda *ss: np.concatenate([np.arange(qs[s], qs[s + 1]) for s in ss])
    # sequences 0 and 2 have more rows than max_query_len allows
    out = gpu_multi(cuda_lib, b, max_query_len=2)
    assert cuda_lib.pa_device_error(clear=True) == cuda_lib.PA_DEVERR_SEQ_LEN
    assert torch.isnan(out[rows(0, 2)]).all()            # their rows are not written
    assert_close(out[rows(1, 3)], ref[rows(1, 3)], "other sequences unaffected")
    # sequence 2 has more new tokens than its seq_len
    sl = b.seq_lens.copy()
    sl[2] = 2
    out = gpu_multi(cuda_lib, b, seq_lens=sl)
    assert cuda_lib.pa_device_error(clear=True) == cuda_lib.PA_DEVERR_SEQ_LEN
    assert torch.isnan(out[rows(2)]).all()
    assert_close(out[rows(0, 1, 3)], ref[rows(0, 1, 3)], "other sequences unaffected")


def test_multi_padding_entries_never_read(cuda_lib):
    b = wl.multi_query_batch(570, num_seqs=7, min_ctx=0, max_ctx=150, n_new=(1, 9),
                             num_heads=16, num_kv_heads=4, head_dim=64, dtype="bf16",
                             device="cuda", keep_seq=False)
    bt = wl.tables_with_padding(b, b.block_tables.shape[1] + 6)
    assert_close(gpu_multi(cuda_lib, b, block_tables=bt), oracle_multi(b), "padded tables")


# ---------------------------------------------------------------------------
# sequences with 64 or more (token, head) rows: the prefill path (blocks of 64
# rows sharing one K/V ring), next to sequences on the other path
# ---------------------------------------------------------------------------

PREFILL_CASES = [(dt, D, G, Hkv) for dt in ("bf16", "f16") for D in (64, 128)
                 for G, Hkv in ((1, 4), (4, 2), (8, 1))]


@pytest.mark.parametrize("dtype,D,G,Hkv", PREFILL_CASES,
                         ids=[f"{c[0]}-d{c[1]}-g{c[2]}" for c in PREFILL_CASES])
def test_multi_prefill_path_parity(cuda_lib, dtype, D, G, Hkv):
    """Slices of 1..150 new tokens over 0..400 cached ones: with G heads per
    KV head, slices of 64/G tokens or more take the prefill path, the rest the
    persistent kernel; every row group, ragged tails of groups and blocks."""
    b = wl.multi_query_batch(600 + D + G, num_seqs=10, min_ctx=0, max_ctx=400,
                             n_new=[150, 1, 70, 3, 33, 64, 17, 2, 129, 8], num_heads=G * Hkv,
                             num_kv_heads=Hkv, head_dim=D, dtype=dtype, device="cuda",
                             keep_seq=False)
    assert_close(gpu_multi(cuda_lib, b), oracle_multi(b), f"{dtype} d{D} g{G}")


@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("f16", 64)])
def test_multi_prefill_fewer_rows_than_one_q_box(cuda_lib, dtype, D):
    """Multi-head attention (G = 1) with one 100-token chunk and two short
    runs: 103 query rows in all, fewer than the 128 tokens one Q copy of the
    prefill kernel spans; rows past the end of q are filled with zeros, never
    read."""
    b = wl.multi_query_batch(645 + D, num_seqs=3, min_ctx=10, max_ctx=120, n_new=[100, 1, 2],
                             num_heads=4, num_kv_heads=4, head_dim=D, dtype=dtype, device="cuda",
                             keep_seq=False)
    assert b.meta["query_start"][-1] == 103
    assert_close(gpu_multi(cuda_lib, b), oracle_multi(b), f"{dtype} d{D} 103 rows")


def test_multi_prefill_whole_prompt(cuda_lib):
    """A first chunk of 300 tokens with nothing cached: row i sees 0..i, the
    first row exactly its own V."""
    b = wl.multi_query_batch(640, num_seqs=3, min_ctx=0, max_ctx=0, n_new=[300, 97, 16],
                             num_heads=32, num_kv_heads=8, head_dim=128, dtype="bf16",
                             device="cuda", keep_seq=False)
    out = gpu_multi(cuda_lib, b)
    assert_close(out, oracle_multi(b), "whole prompt")
    qs = b.meta["query_start"]
    for s in range(b.num_seqs):
        blk = int(b.block_tables[s, 0])
        assert torch.equal(out[qs[s]], b.v_cache[blk, :, 0, :].repeat_interleave(4, dim=0))


def test_multi_prefill_block_permutation_bit_identical(cuda_lib):
    b = wl.multi_query_batch(650, num_seqs=4, min_ctx=10, max_ctx=300, n_new=(40, 120),
                             num_heads=16, num_kv_heads=4, head_dim=128, dtype="bf16",
                             device="cuda", keep_seq=False)
    p = wl.permute_blocks(b, seed=3)
    p.meta["query_start"] = b.meta["query_start"]
    assert torch.equal(gpu_multi(cuda_lib, b), gpu_multi(cuda_lib, p))


def test_multi_prefill_bad_block_is_flagged(cuda_lib):
    b = wl.multi_query_batch(660, num_seqs=2, min_ctx=20, max_ctx=60, n_new=[80, 5],
                             num_heads=8, num_kv_heads=2, head_dim=64, dtype="bf16",
                             device="cuda", keep_seq=False)
    bt = b.block_tables.copy()
    bt[0, 1] = b.num_blocks + 3
    gpu_multi(cuda_lib, b, block_tables=bt)
    assert cuda_lib.pa_device_error(clear=True) & cuda_lib.PA_DEVERR_BLOCK_ID


def test_multi_batch_larger_than_one_sort(cuda_lib):
    """More sequences than one thread block orders in shared memory: the batch
    runs as consecutive slices with absolute query rows."""
    b = wl.multi_query_batch(670, num_seqs=4500, min_ctx=0, max_ctx=30, n_new=(0, 3),
                             num_heads=8, num_kv_heads=2, head_dim=64, dtype="bf16",
                             device="cuda", keep_seq=False)
    assert_close(gpu_multi(cuda_lib, b), oracle_multi(b), "4500 seqs")


def test_multi_prefill_more_than_256_sequences(cuda_lib):
    """Long runs among more than 256 sequences: the prefill kernel lists their
    work items in sequence order (it sorts them by length only up to 256
    sequences); every long run and a few one-token rows against the oracle."""
    n = np.ones(300, dtype=np.int64)
    long_runs = [3, 77, 150, 255, 256, 299]
    n[long_runs] = [40, 25, 64, 17, 33, 90]          # 68..360 rows at G = 4
    b = wl.multi_query_batch(680, num_seqs=300, min_ctx=0, max_ctx=200, n_new=n,
                             num_heads=8, num_kv_heads=2, head_dim=64, dtype="bf16",
                             device="cuda", keep_seq=False)
    out = gpu_multi(cuda_lib, b)
    seqs = sorted(set(long_runs + [0, 100, 298]))
    ref, rows = oracle_multi(b, seqs=np.array(seqs))
    assert_close(out[torch.from_numpy(rows).cuda()], ref, "300 seqs")


@pytest.mark.parametrize("dtype,D,G,Hkv", [("bf16", 128, 4, 8), ("f16", 64, 2, 4)],
                         ids=["bf16-d128-g4", "f16-d64-g2"])
def test_multi_prefill_many_items_per_block(cuda_lib, dtype, D, G, Hkv):
    """More 128-row items than the persistent grid has blocks (two per SM), so
    every block runs several items in turn and the hand-over between items
    (the next item's Q, the step-indexed TMEM and shared-memory buffers) is
    exercised; lengths differ so that items of one block differ in steps."""
    rng = np.random.default_rng(690 + G)
    nseq = 48
    n = rng.integers(64 // G * 2, 64 // G * 5, size=nseq)     # 2..5 row groups of 64 rows
    b = wl.multi_query_batch(690 + D, num_seqs=nseq, min_ctx=0, max_ctx=300, n_new=n,
                             num_heads=G * Hkv, num_kv_heads=Hkv, head_dim=D, dtype=dtype,
                             device="cuda", keep_seq=False)
    items = int(sum((int(x) * G + 127) // 128 for x in n)) * Hkv
    assert items > 2 * torch.cuda.get_device_properties(0).multi_processor_count
    assert_close(gpu_multi(cuda_lib, b), oracle_multi(b), f"{dtype} d{D} g{G} {items} items")


# ---------------------------------------------------------------------------
# full-size workloads: every output element against the oracle (fullsize.py)
# ---------------------------------------------------------------------------

@pytest.mark.slow
def test_full_spec_verify(cuda_lib):
    b = wl.spec_verify(device="cuda")
    out = gpu_multi(cuda_lib, b)
    ref, t = fullsize.multi_all(b)
    fullsize.check("spec_verify: pa_decode_multi (4 rows/seq)", out, ref, b.dtype, t)


@pytest.mark.slow
def test_full_chunked_prefill_mix(cuda_lib):
    b = wl.chunked_prefill_mix(device="cuda")
    out = gpu_multi(cuda_lib, b)
    ref, t = fullsize.multi_all(b)
    fullsize.check("chunked_prefill_mix: pa_decode_multi", out, ref, b.dtype, t)
