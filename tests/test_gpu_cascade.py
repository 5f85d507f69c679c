"""Cascade decode over a shared prefix (pa_decode_cascade) through the C ABI.

A batch whose tables all begin with the same physical blocks is passed as
the prefix block list plus each sequence's own table; the result must equal
the fp64 oracle's decode over the whole tables (the prefix blocks followed by
the sequence's own), within the 16-bit tolerances: max |err| <= 2e-2 and
relative L2 error <= 5e-3.
"""
import math

import numpy as np
import pytest
import torch

import fullsize
import oracle
from paged_kv_cache_151_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

TOL_ABS = 2e-2
TOL_REL_L2 = 5e-3


def assert_close(gpu, ref, what=""):
    g = gpu.detach().double().cpu().numpy()
    ref = np.asarray(ref, dtype=np.float64)
    assert g.shape == ref.shape
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    err = np.abs(g - ref).max()
    rel = np.linalg.norm(g - ref) / max(np.linalg.norm(ref), 1e-30)
    assert err <= TOL_ABS, f"{what}: max abs err {err:.3g}"
    assert rel <= TOL_REL_L2, f"{what}: rel L2 err {rel:.3g}"


@pytest.fixture(autouse=True)
def _clean_error_word(cuda_lib):
    cuda_lib.pa_device_error(clear=True)
    yield
    flags = cuda_lib.pa_device_error(clear=True)
    assert flags == 0, f"device error word set: {flags:#x}"


def shared_batch(seed, *, num_seqs, prefix_blocks, own_lo, own_hi, num_heads, num_kv_heads,
                 head_dim, dtype, extra_blocks=8, device="cuda"):
    """Every table starts with the same `prefix_blocks` blocks, then
    own_lo..own_hi tokens of the sequence's own (the step's new token among
    them, already in the pool)."""
    rng = np.random.default_rng(seed)
    own = rng.integers(own_lo, own_hi, size=num_seqs, endpoint=True)
    own[0] = own_hi                                  # the longest first, for the table width
    L = 16 * prefix_blocks + own                     # tokens attended
    own_blocks = [math.ceil(int(x) / 16) for x in L]  # blocks of the whole sequence
    total = (prefix_blocks + sum(max(0, n - prefix_blocks) for n in own_blocks) +
             int((own == 0).sum()) + extra_blocks)
    fl = wl.FreeList(total, rng)
    prefix = fl.take(prefix_blocks)
    tables = [prefix + fl.take(max(0, n - prefix_blocks)) for n in own_blocks]
    # sequences whose own part is empty write their new token into the prefix's
    # last block: give them one more private block instead (keeps every
    # sequence's new token in its own blocks)
    for s in range(num_seqs):
        if own[s] == 0:
            tables[s] = tables[s] + fl.take(1)
    b = wl.build_batch("cascade", ctx_lens=np.maximum(L - 1, 0), num_heads=num_heads,
                       num_kv_heads=num_kv_heads, head_dim=head_dim, dtype=dtype,
                       num_blocks=total, tables=tables, seed=seed, device=device,
                       new_in_pool=True, kv_std=0.5, keep_seq=False)
    # attend over exactly L tokens (own == 0: the prefix alone)
    b.seq_lens[:] = L.astype(np.int32)
    return b


def run_cascade(pa, b, P):
    prefix, own_tab, own_len = wl.cascade_split(b, P)
    pt = torch.from_numpy(prefix).cuda()
    bt = torch.from_numpy(own_tab).cuda()
    sl = torch.from_numpy(own_len).cuda()
    nbytes = pa.pa_decode_cascade_workspace_size(b.num_seqs, b.num_heads, b.head_dim, P,
                                                 own_tab.shape[1])
    assert nbytes > 0
    ws = torch.full((nbytes,), 0xFF, dtype=torch.uint8, device="cuda")   # NaN partials
    out = torch.full_like(b.q, float("nan"))
    pa.pa_decode_cascade(out, b.q, b.k_cache, b.v_cache, pt, bt, sl, b.scale, b.num_kv_heads,
                         ws)
    torch.cuda.synchronize()
    return out


def oracle_whole_tables(b):
    return oracle.decode(b.q.cpu(), b.k_cache.cpu(), b.v_cache.cpu(), b.block_tables,
                         b.seq_lens, b.scale, b.num_kv_heads, b.dtype, nthreads=8)


CASES = [
    # dtype, D, G, Hkv, num_seqs, prefix blocks, own tokens lo..hi
    ("bf16", 128, 4, 2, 37, 20, 0, 70),      # one partial chunk (20 blocks), empty own parts
    ("f16", 64, 2, 4, 5, 1, 1, 40),          # one prefix block, one partial step
    ("bf16", 128, 8, 1, 64, 300, 0, 1100),   # 10 chunks (9 x 32 + 12), own parts over 3 partitions
    ("bf16", 64, 1, 4, 130, 17, 0, 3),       # 2 row groups (130 rows), one 17-block chunk
    ("f16", 128, 4, 8, 3, 64, 500, 520),     # few sequences, 8 KV heads, 2 chunks
]


@pytest.mark.parametrize("dtype,D,G,Hkv,B,P,lo,hi", CASES,
                         ids=[f"{c[0]}-d{c[1]}-g{c[2]}-b{c[4]}-p{c[5]}" for c in CASES])
def test_cascade_matches_oracle_over_whole_tables(cuda_lib, dtype, D, G, Hkv, B, P, lo, hi):
    b = shared_batch(1000 + P + B, num_seqs=B, prefix_blocks=P, own_lo=lo, own_hi=hi,
                     num_heads=G * Hkv, num_kv_heads=Hkv, head_dim=D, dtype=dtype)
    out = run_cascade(cuda_lib, b, P)
    assert_close(out, oracle_whole_tables(b), f"cascade {dtype} d{D} g{G} B{B} P{P}")


def test_cascade_equals_plain_decode_within_tolerance(cuda_lib):
    """The same batch through pa_decode (whole tables) and the cascade."""
    b = shared_batch(1101, num_seqs=48, prefix_blocks=40, own_lo=1, own_hi=300, num_heads=32,
                     num_kv_heads=8, head_dim=128, dtype="bf16")
    out = run_cascade(cuda_lib, b, 40)
    bt, sl, _ = b.torch_tables("cuda")
    ref = torch.empty_like(b.q)
    cuda_lib.pa_decode(ref, b.q, b.k_cache, b.v_cache, bt.contiguous(), sl.contiguous(),
                       b.scale, b.num_kv_heads)
    torch.cuda.synchronize()
    assert (out.float() - ref.float()).abs().max().item() <= TOL_ABS


def test_cascade_without_prefix_is_pa_decode(cuda_lib):
    b = wl.random_batch(1102, num_seqs=9, max_len=200, num_heads=16, num_kv_heads=4,
                        head_dim=128, dtype="bf16", device="cuda", new_in_pool=True,
                        keep_seq=False)
    bt, sl, _ = b.torch_tables("cuda")
    out = torch.full_like(b.q, float("nan"))
    ref = torch.full_like(b.q, float("nan"))
    empty = torch.zeros(0, dtype=torch.int32, device="cuda")
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    cuda_lib.pa_decode_cascade(out, b.q, b.k_cache, b.v_cache, empty, bt.contiguous(),
                               sl.contiguous(), b.scale, b.num_kv_heads, ws)
    cuda_lib.pa_decode(ref, b.q, b.k_cache, b.v_cache, bt.contiguous(), sl.contiguous(),
                       b.scale, b.num_kv_heads)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)


def test_cascade_bad_prefix_block_is_flagged(cuda_lib):
    b = shared_batch(1103, num_seqs=6, prefix_blocks=8, own_lo=1, own_hi=30, num_heads=8,
                     num_kv_heads=2, head_dim=64, dtype="bf16")
    prefix, own_tab, own_len = wl.cascade_split(b, 8)
    prefix = prefix.copy()
    prefix[3] = b.num_blocks + 7                     # outside the pool
    nbytes = cuda_lib.pa_decode_cascade_workspace_size(6, 8, 64, 8, own_tab.shape[1])
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    out = torch.empty_like(b.q)
    cuda_lib.pa_decode_cascade(out, b.q, b.k_cache, b.v_cache, torch.from_numpy(prefix).cuda(),
                               torch.from_numpy(own_tab).cuda(), torch.from_numpy(own_len).cuda(),
                               b.scale, b.num_kv_heads, ws)
    assert cuda_lib.pa_device_error(clear=True) & cuda_lib.PA_DEVERR_BLOCK_ID


@pytest.mark.slow
def test_full_shared_prefix_cascade(cuda_lib):
    """The 128-sequence, 2048-token shared-prefix workload in cascade form,
    every output element against the oracle over the whole tables."""
    b = wl.shared_prefix(device="cuda", new_in_pool=True)
    P = int(b.meta["prefix_tokens"]) // 16
    out = run_cascade(cuda_lib, b, P)
    ref, t = fullsize.decode_all(b)
    fullsize.check("shared_prefix: pa_decode_cascade", out, ref, b.dtype, t)


def test_cascade_batch_larger_than_one_sort(cuda_lib):
    """More sequences than the split-KV kernel orders in one block: its own
    blocks' pass runs as consecutive slices, each writing the partitions of
    its sequences; prefix rows span many row groups."""
    b = shared_batch(1104, num_seqs=5000, prefix_blocks=3, own_lo=0, own_hi=40, num_heads=8,
                     num_kv_heads=2, head_dim=64, dtype="bf16", extra_blocks=16)
    out = run_cascade(cuda_lib, b, 3)
    assert_close(out, oracle_whole_tables(b), "cascade 5000 sequences")


def test_cascade_driven_by_the_block_manager(cuda_lib):
    """Requests sharing a system prompt are admitted with prefix caching; the
    block manager reports the leading blocks the batch shares, the batch is
    decoded through the cascade and through pa_decode, and both match the
    oracle over the requests' own tables."""
    from paged_kv_cache_151_gb300 import blocks
    H, Hkv, D, BS = 16, 4, 128, 16
    rng = np.random.default_rng(1105)
    bm = blocks.BlockManager(4096, BS, prefix_caching=True)
    system = list(range(500000, 500000 + 5 * BS + 7))           # 5 full shared blocks + 7
    ids = list(range(24))
    for i in ids:
        own = (rng.integers(0, 30000, size=int(rng.integers(1, 90))) + 40000 * (i + 1)).tolist()
        assert bm.add_sequence(i, system + own) is not None
    P = bm.common_prefix(ids)
    assert P == 5
    width = max(len(bm.table(i)) for i in ids)
    tables, lens = bm.batch(ids, width)
    g = torch.Generator(device="cuda")
    g.manual_seed(1105)
    kc = (torch.randn((4096, Hkv, BS, D), generator=g, device="cuda") * 0.5).to(torch.bfloat16)
    vc = (torch.randn((4096, Hkv, BS, D), generator=g, device="cuda") * 0.5).to(torch.bfloat16)
    q = torch.randn((len(ids), H, D), generator=g, device="cuda").to(torch.bfloat16)
    scale = 1.0 / math.sqrt(D)
    ref = oracle.decode(q.cpu(), kc.cpu(), vc.cpu(), tables, lens, scale, Hkv, "bf16", nthreads=8)
    bt = torch.from_numpy(tables).cuda()
    sl = torch.from_numpy(lens).cuda()
    plain = torch.empty_like(q)
    cuda_lib.pa_decode(plain, q, kc, vc, bt, sl, scale, Hkv)
    prefix = torch.from_numpy(np.ascontiguousarray(tables[0, :P])).cuda()
    own_t = torch.from_numpy(np.ascontiguousarray(tables[:, P:])).cuda()
    own_l = torch.from_numpy((lens - BS * P).astype(np.int32)).cuda()
    ws = torch.empty(cuda_lib.pa_decode_cascade_workspace_size(len(ids), H, D, P, width - P),
                     dtype=torch.uint8, device="cuda")
    out = torch.full_like(q, float("nan"))
    cuda_lib.pa_decode_cascade(out, q, kc, vc, prefix, own_t, own_l, scale, Hkv, ws)
    torch.cuda.synchronize()
    assert_close(out, ref, "cascade from the block manager")
    assert_close(plain, ref, "pa_decode from the block manager")
