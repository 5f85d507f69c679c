"""Parity of the CUDA path (through the C ABI) with the fp64 CPU oracle.

Tolerances (against the fp64 oracle, on the output as stored):
  fp32 caches        max |err| <= 1e-4
  bf16 / f16 caches  max |err| <= 2e-2 and relative L2 error <= 5e-3
The cache write and every layout invariance are checked bit for bit.
"""
import math

import numpy as np
import pytest
import torch

import fullsize
import oracle
from paged_kv_cache_151_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

TOL_F32 = 1e-4
TOL_16_ABS = 2e-2
TOL_16_REL_L2 = 5e-3


def assert_close(gpu, ref, dtype, what=""):
    g = gpu.detach().double().cpu().numpy() if isinstance(gpu, torch.Tensor) else gpu
    ref = np.asarray(ref, dtype=np.float64)
    assert g.shape == ref.shape, (g.shape, ref.shape)
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    err = np.abs(g - ref).max() if g.size else 0.0
    if dtype == "f32":
        assert err <= TOL_F32, f"{what}: max abs err {err:.3g}"
    else:
        rel = np.linalg.norm(g - ref) / max(np.linalg.norm(ref), 1e-30)
        assert err <= TOL_16_ABS, f"{what}: max abs err {err:.3g}"
        assert rel <= TOL_16_REL_L2, f"{what}: rel L2 err {rel:.3g}"


def gpu_tables(b):
    bt, sl, sm = b.torch_tables("cuda")
    return bt.contiguous(), sl.contiguous(), sm.contiguous()


def gpu_decode(pa, b, splits=None, seq_lens=None, block_tables=None):
    bt, sl, _ = gpu_tables(b)
    if seq_lens is not None:
        sl = torch.as_tensor(seq_lens, dtype=torch.int32, device="cuda")
    if block_tables is not None:
        bt = torch.as_tensor(block_tables, dtype=torch.int32, device="cuda").contiguous()
    out = torch.full_like(b.q, float("nan"))
    if splits is None:
        pa.pa_decode(out, b.q, b.k_cache, b.v_cache, bt, sl, b.scale, b.num_kv_heads)
    else:
        pa.pa_decode_split(out, b.q, b.k_cache, b.v_cache, bt, sl, b.scale,
                           b.num_kv_heads, splits)
    torch.cuda.synchronize()
    return out


def gpu_partitioned(pa, b, partition_size, max_seq_len=None, seq_lens=None):
    bt, sl, _ = gpu_tables(b)
    if seq_lens is not None:
        sl = torch.as_tensor(seq_lens, dtype=torch.int32, device="cuda")
    msl = int(b.seq_lens.max()) if max_seq_len is None else max_seq_len
    nbytes = pa.pa_decode_partitioned_workspace_size(b.num_seqs, b.num_heads, b.head_dim,
                                                     msl, partition_size)
    ws = torch.full((nbytes,), 0xFF, dtype=torch.uint8, device="cuda")
    out = torch.full_like(b.q, float("nan"))
    pa.pa_decode_partitioned(out, b.q, b.k_cache, b.v_cache, bt, sl, b.scale,
                             b.num_kv_heads, partition_size, msl, ws)
    torch.cuda.synchronize()
    return out, ws, msl


def oracle_decode(b, seq_lens=None, k_cache=None, v_cache=None):
    return oracle.decode(b.q.cpu(), (b.k_cache if k_cache is None else k_cache).cpu(),
                         (b.v_cache if v_cache is None else v_cache).cpu(),
                         b.block_tables, b.seq_lens if seq_lens is None else seq_lens,
                         b.scale, b.num_kv_heads, b.dtype, nthreads=8)


@pytest.fixture(autouse=True)
def _clean_error_word(cuda_lib):
    cuda_lib.pa_device_error(clear=True)
    yield
    flags = cuda_lib.pa_device_error(clear=True)
    assert flags == 0, f"device error word set: {flags:#x}"


# ---------------------------------------------------------------------------
# reshape_and_cache: bit-exact
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype,H,Hkv,D", [("f32", 8, 2, 64), ("bf16", 32, 8, 128),
                                            ("f16", 16, 4, 64), ("bf16", 8, 8, 128)])
def test_reshape_and_cache_bit_exact(cuda_lib, dtype, H, Hkv, D):
    b = wl.random_batch(101, num_seqs=37, max_len=90, num_heads=H, num_kv_heads=Hkv,
                        head_dim=D, dtype=dtype, device="cuda", keep_seq=False)
    _, _, sm = gpu_tables(b)
    kc, vc = b.k_cache.clone(), b.v_cache.clone()
    cuda_lib.pa_reshape_and_cache(b.k_new, b.v_new, kc, vc, sm)
    torch.cuda.synchronize()
    rk, rv, bad = oracle.reshape_and_cache(b.k_new.cpu(), b.v_new.cpu(), b.k_cache.cpu(),
                                           b.v_cache.cpu(), b.slot_mapping, dtype)
    assert bad == 0
    as_bytes = lambda t: t.cpu().contiguous().view(torch.uint8).numpy()
    assert np.array_equal(as_bytes(kc), rk.view(np.uint8).reshape(as_bytes(kc).shape))
    assert np.array_equal(as_bytes(vc), rv.view(np.uint8).reshape(as_bytes(vc).shape))


def test_reshape_and_cache_tiny_config(cuda_lib):
    b = wl.tiny(device="cuda")
    _, _, sm = gpu_tables(b)
    kc, vc = b.k_cache.clone(), b.v_cache.clone()
    cuda_lib.pa_reshape_and_cache(b.k_new, b.v_new, kc, vc, sm)
    rk, rv, _ = oracle.reshape_and_cache(b.k_new.cpu(), b.v_new.cpu(), b.k_cache.cpu(),
                                         b.v_cache.cpu(), b.slot_mapping, "f32")
    assert np.array_equal(kc.cpu().numpy().view(np.uint32), rk.view(np.uint32))
    assert np.array_equal(vc.cpu().numpy().view(np.uint32), rv.view(np.uint32))
    # every canary outside the written slots is still NaN
    assert torch.isnan(kc).sum().item() == torch.isnan(b.k_cache).sum().item() - 4 * 2 * 64


def test_reshape_and_cache_strided_padding_and_bad_slot(cuda_lib):
    T, Hkv, D = 50, 4, 128
    b = wl.random_batch(102, num_seqs=T, max_len=40, num_heads=Hkv, num_kv_heads=Hkv,
                        head_dim=D, dtype="bf16", device="cuda")
    # k and v as slices of one fused [T, 3, Hkv, D] projection output
    qkv = torch.randn(T, 3, Hkv, D, device="cuda").to(torch.bfloat16)
    k, v = qkv[:, 1], qkv[:, 2]
    sm_np = b.slot_mapping.copy()
    sm_np[5] = -1                                  # padding token
    sm_np[7] = b.num_blocks * 16 + 3               # out of range: skipped, flagged
    sm = torch.from_numpy(sm_np).cuda()
    kc, vc = b.k_cache.clone(), b.v_cache.clone()
    cuda_lib.pa_reshape_and_cache(k, v, kc, vc, sm)
    flags = cuda_lib.pa_device_error(clear=True)
    assert flags == cuda_lib.PA_DEVERR_SLOT
    rk, rv, bad = oracle.reshape_and_cache(k.cpu().contiguous(), v.cpu().contiguous(),
                                           b.k_cache.cpu(), b.v_cache.cpu(), sm_np, "bf16")
    assert bad == 1
    as_u16 = lambda t: t.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(as_u16(kc), rk)
    assert np.array_equal(as_u16(vc), rv)


# ---------------------------------------------------------------------------
# decode parity on small cases
# ---------------------------------------------------------------------------

def test_tiny_config_before_and_after_write(cuda_lib):
    b = wl.tiny(device="cuda")
    bt, _, sm = gpu_tables(b)
    # before the write: attend over the L tokens already cached
    out = gpu_decode(cuda_lib, b, seq_lens=b.ctx_lens)
    assert_close(out, oracle_decode(b, seq_lens=b.ctx_lens), "f32", "tiny/before")
    # after the write: L + 1 tokens
    kc, vc = b.k_cache.clone(), b.v_cache.clone()
    cuda_lib.pa_reshape_and_cache(b.k_new, b.v_new, kc, vc, sm)
    out2 = torch.empty_like(b.q)
    cuda_lib.pa_decode(out2, b.q, kc, vc, bt, torch.from_numpy(b.seq_lens).cuda(),
                       b.scale, b.num_kv_heads)
    torch.cuda.synchronize()
    rk, rv, _ = oracle.reshape_and_cache(b.k_new.cpu(), b.v_new.cpu(), b.k_cache.cpu(),
                                         b.v_cache.cpu(), b.slot_mapping, "f32")
    ref = oracle.decode(b.q.cpu(), rk, rv, b.block_tables, b.seq_lens, b.scale,
                        b.num_kv_heads, "f32")
    assert_close(out2, ref, "f32", "tiny/after")


CASES = []
for dtype in ("f32", "bf16", "f16"):
    for D in (64, 128):
        for G, Hkv in ((1, 4), (2, 2), (4, 2), (8, 1)):
            CASES.append((dtype, D, G, Hkv))


@pytest.mark.parametrize("dtype,D,G,Hkv", CASES,
                         ids=[f"{c[0]}-d{c[1]}-g{c[2]}" for c in CASES])
def test_decode_parity_small(cuda_lib, dtype, D, G, Hkv):
    b = wl.random_batch(200 + D + G, num_seqs=9, max_len=300, num_heads=G * Hkv,
                        num_kv_heads=Hkv, head_dim=D, dtype=dtype, device="cuda",
                        new_in_pool=True, keep_seq=False, table_slack=2)
    ref = oracle_decode(b)
    for splits in (1, 2, 8):
        out = gpu_decode(cuda_lib, b, splits=splits)
        assert_close(out, ref, dtype, f"splits={splits}")
    assert_close(gpu_decode(cuda_lib, b), ref, dtype, "auto")


@pytest.mark.parametrize("splits", [1, 2, 4, 8])
def test_decode_ragged_lengths_every_remainder(cuda_lib, splits):
    """Lengths 1..80 cover every partial-block remainder and several warps."""
    L = np.arange(1, 81)
    Hkv, G, D = 2, 4, 128
    rng = np.random.default_rng(7)
    fl = wl.FreeList(int(sum(math.ceil(x / 16) for x in L)) + 4, rng)
    tables = [fl.allocate(int(x)) for x in L]
    b = wl.build_batch("ragged", ctx_lens=L - 1, num_heads=G * Hkv, num_kv_heads=Hkv,
                       head_dim=D, dtype="bf16", num_blocks=len(fl.free) + sum(map(len, tables)),
                       tables=tables, seed=8, device="cuda", new_in_pool=True, kv_std=0.5)
    out = gpu_decode(cuda_lib, b, splits=splits)
    assert_close(out, oracle_decode(b), "bf16", f"ragged splits={splits}")


def test_seq_len_one_returns_v_bit_exact(cuda_lib):
    b = wl.random_batch(301, num_seqs=6, max_len=0, num_heads=32, num_kv_heads=8,
                        head_dim=128, dtype="bf16", device="cuda", new_in_pool=True,
                        keep_seq=True)
    out = gpu_decode(cuda_lib, b)
    for s in range(b.num_seqs):
        v = b.seq_v[s][0]                                   # [Hkv, D]
        assert torch.equal(out[s], v.repeat_interleave(4, dim=0))


def test_seq_len_zero_gives_zeros(cuda_lib):
    b = wl.random_batch(302, num_seqs=5, max_len=40, num_heads=8, num_kv_heads=2,
                        head_dim=64, dtype="f32", device="cuda", new_in_pool=True)
    sl = b.seq_lens.copy()
    sl[[0, 3]] = 0
    for splits in (1, 4):
        out = gpu_decode(cuda_lib, b, splits=splits, seq_lens=sl)
        assert torch.equal(out[[0, 3]], torch.zeros_like(out[[0, 3]]))
        assert_close(out, oracle_decode(b, seq_lens=sl), "f32", "len0")
    out, _, _ = gpu_partitioned(cuda_lib, b, 32, seq_lens=sl)
    assert torch.equal(out[[0, 3]], torch.zeros_like(out[[0, 3]]))


def test_block_permutation_bit_identical(cuda_lib):
    b = wl.random_batch(303, num_seqs=12, max_len=400, num_heads=32, num_kv_heads=8,
                        head_dim=128, dtype="bf16", device="cuda", new_in_pool=True,
                        extra_blocks=64)
    p = wl.permute_blocks(b, seed=5)
    for splits in (1, 4):
        assert torch.equal(gpu_decode(cuda_lib, b, splits=splits),
                           gpu_decode(cuda_lib, p, splits=splits))
    assert torch.equal(gpu_partitioned(cuda_lib, b, 64)[0], gpu_partitioned(cuda_lib, p, 64)[0])


def test_shared_prefix_alias_bit_identical_to_private(cuda_lib):
    kw = dict(batch=10, prefix_blocks=20, lo=10, hi=90, device="cuda", new_in_pool=True)
    shared = wl.shared_prefix(**kw)
    private = wl.shared_prefix(private_prefix=True, **kw)
    a, p = gpu_decode(cuda_lib, shared), gpu_decode(cuda_lib, private)
    assert torch.equal(a, p)
    assert_close(a, oracle_decode(shared), "bf16", "shared prefix")


def test_padding_entries_never_read(cuda_lib):
    """Table entries past each sequence's last block hold an invalid id; any
    read of one would set the device error word (checked by the fixture)."""
    b = wl.random_batch(304, num_seqs=7, max_len=150, num_heads=16, num_kv_heads=4,
                        head_dim=64, dtype="bf16", device="cuda", new_in_pool=True,
                        table_slack=5)
    assert (b.block_tables == wl.PAD).any()
    ref = oracle_decode(b)
    for splits in (1, 2, 4, 8):
        assert_close(gpu_decode(cuda_lib, b, splits=splits), ref, "bf16", "pad")
    assert_close(gpu_partitioned(cuda_lib, b, 48)[0], ref, "bf16", "pad/part")


def test_bad_block_id_is_skipped_and_flagged(cuda_lib):
    b = wl.random_batch(305, num_seqs=4, max_len=60, num_heads=8, num_kv_heads=2,
                        head_dim=64, dtype="f32", device="cuda", new_in_pool=True)
    bt = b.block_tables.copy()
    bt[2, 0] = b.num_blocks + 5               # inside seq 2's range: out of the pool
    out = gpu_decode(cuda_lib, b, splits=1, block_tables=bt)
    assert cuda_lib.pa_device_error(clear=True) == cuda_lib.PA_DEVERR_BLOCK_ID
    ref = oracle_decode(b)
    keep = [0, 1, 3]
    assert_close(out[keep], ref[keep], "f32", "other sequences unaffected")


def test_seq_len_past_table_is_clamped_and_flagged(cuda_lib):
    b = wl.random_batch(306, num_seqs=3, max_len=30, num_heads=4, num_kv_heads=2,
                        head_dim=64, dtype="f32", device="cuda", new_in_pool=True)
    sl = b.seq_lens.copy()
    sl[1] = b.max_blocks * 16 + 100
    gpu_decode(cuda_lib, b, seq_lens=sl)
    assert cuda_lib.pa_device_error(clear=True) & cuda_lib.PA_DEVERR_SEQ_LEN


# ---------------------------------------------------------------------------
# split-KV partitions and the log-sum-exp merge
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("psize", [16, 64, 96, 512])
def test_partition_stats_and_merge(cuda_lib, psize):
    b = wl.random_batch(400 + psize, num_seqs=5, max_len=1500, num_heads=16,
                        num_kv_heads=2, head_dim=128, dtype="bf16", device="cuda",
                        new_in_pool=True, kv_std=0.5)
    out, ws, msl = gpu_partitioned(cuda_lib, b, psize)
    ref = oracle_decode(b)
    assert_close(out, ref, "bf16", f"partitioned p={psize}")
    o_p, m_p, l_p = cuda_lib.workspace_views(ws, b.num_seqs, b.num_heads, b.head_dim,
                                             msl, psize)
    pr = oracle.problem(b.q.cpu(), b.k_cache.cpu(), b.v_cache.cpu(), b.block_tables,
                        b.seq_lens, b.scale, b.num_kv_heads, "bf16")
    for s in range(b.num_seqs):
        for h in (0, 7, 15):
            m, l, o = oracle.partition_stats(s, h, psize, None, None, None, None, None,
                                             None, None, "bf16", problem=pr)
            n = m.shape[0]
            gm = m_p[s, h, :n].double().cpu().numpy()
            gl = l_p[s, h, :n].double().cpu().numpy()
            go = o_p[s, h, :n].double().cpu().numpy()
            np.testing.assert_allclose(gm, m, rtol=0, atol=2e-3)
            # l_p is relative to m_p: compare log-sum-exp = m + log l
            np.testing.assert_allclose(gm + np.log(gl), m + np.log(l), rtol=0, atol=2e-3)
            np.testing.assert_allclose(go, o, rtol=0, atol=2e-3)


def test_partitioned_f32_tight(cuda_lib):
    b = wl.random_batch(410, num_seqs=4, max_len=700, num_heads=8, num_kv_heads=2,
                        head_dim=64, dtype="f32", device="cuda", new_in_pool=True)
    out, _, _ = gpu_partitioned(cuda_lib, b, 128)
    assert_close(out, oracle_decode(b), "f32", "partitioned f32")


def test_partitioned_seq_len_past_max_is_flagged(cuda_lib):
    b = wl.random_batch(411, num_seqs=3, max_len=200, num_heads=8, num_kv_heads=2,
                        head_dim=64, dtype="f32", device="cuda", new_in_pool=True)
    gpu_partitioned(cuda_lib, b, 32, max_seq_len=int(b.seq_lens.max()) - 20)
    assert cuda_lib.pa_device_error(clear=True) & cuda_lib.PA_DEVERR_SEQ_LEN


# ---------------------------------------------------------------------------
# full-size workloads, in the launch configuration the benchmark times;
# every output element against the oracle (fullsize.py)
# ---------------------------------------------------------------------------

@pytest.mark.slow
def test_full_llama8b_uniform(cuda_lib):
    b = wl.llama8b_uniform(device="cuda", new_in_pool=True)
    out = gpu_decode(cuda_lib, b)
    ref, t = fullsize.decode_all(b)
    fullsize.check("llama8b_uniform: pa_decode", out, ref, "bf16", t)


@pytest.mark.slow
def test_full_serving_mix_step(cuda_lib):
    """The benchmark's step: cache write of one token per sequence, then decode."""
    b = wl.serving_mix(device="cuda")
    bt, sl, sm = gpu_tables(b)
    kc, vc = b.k_cache.clone(), b.v_cache.clone()
    cuda_lib.pa_reshape_and_cache(b.k_new, b.v_new, kc, vc, sm)
    out = torch.empty_like(b.q)
    cuda_lib.pa_decode(out, b.q, kc, vc, bt, sl, b.scale, b.num_kv_heads)
    torch.cuda.synchronize()
    # the write: bit-exact on the written rows, nothing else touched
    ref_k = b.k_cache.clone()
    slots = torch.from_numpy(b.slot_mapping).cuda()
    ref_k[slots // 16, :, slots % 16, :] = b.k_new
    assert torch.equal(kc.view(torch.int16), ref_k.view(torch.int16))
    b2 = wl.serving_mix(device="cuda", new_in_pool=True)
    assert torch.equal(kc.view(torch.int16), b2.k_cache.view(torch.int16))
    assert torch.equal(vc.view(torch.int16), b2.v_cache.view(torch.int16))
    ref, t = fullsize.decode_all(b2)
    fullsize.check("serving_mix: cache write + pa_decode", out, ref, "bf16", t)


@pytest.mark.slow
def test_full_shared_prefix(cuda_lib):
    shared = wl.shared_prefix(device="cuda", new_in_pool=True)
    out = gpu_decode(cuda_lib, shared)
    private = wl.shared_prefix(device="cuda", new_in_pool=True, private_prefix=True)
    # the oracle on the private-copy layout: the aliased output must equal it
    ref, t = fullsize.decode_all(private)
    fullsize.check("shared_prefix: pa_decode (aliased tables)", out, ref, "bf16", t)
    assert torch.equal(out, gpu_decode(cuda_lib, private))


@pytest.mark.slow
def test_full_long_context_partitioned(cuda_lib):
    b = wl.long_context(device="cuda", new_in_pool=True)
    out, _, _ = gpu_partitioned(cuda_lib, b, 512, max_seq_len=131072)
    ref, t = fullsize.decode_all(b)
    fullsize.check("long_context: pa_decode_partitioned 512", out, ref, "bf16", t)
    fullsize.check("long_context: pa_decode", gpu_decode(cuda_lib, b), ref, "bf16")


def test_decode_sees_the_cache_write_it_follows(cuda_lib):
    """The decode is launched to overlap the cache write before it (it sets up
    while the write finishes); every step writes a token whose key dominates
    the softmax, and the decode issued right after must already attend to it:
    the output is that token's value."""
    B, Hkv, G, D = 64, 8, 4, 128
    b = wl.random_batch(900, num_seqs=B, max_len=300, min_len=40, num_heads=G * Hkv,
                        num_kv_heads=Hkv, head_dim=D, dtype="bf16", device="cuda",
                        keep_seq=False, extra_blocks=B * 20 + 8)
    bt = [list(r[r != wl.PAD]) for r in b.block_tables]
    free = sorted(set(range(b.num_blocks)) - {x for r in bt for x in r})
    kc, vc = b.k_cache.clone(), b.v_cache.clone()
    lens = b.ctx_lens.astype(np.int64).copy()
    q = b.q
    for step in range(20):
        slots = []
        for s in range(B):
            if lens[s] // 16 >= len(bt[s]):
                bt[s].append(free.pop())
            slots.append(bt[s][lens[s] // 16] * 16 + lens[s] % 16)
        # the new key points along the mean query of each group, longer than
        # every earlier step's: it dominates the softmax
        qg = q.float().view(B, Hkv, G, D).mean(2)
        k_new = ((60.0 + 30.0 * step) * qg / qg.norm(dim=-1, keepdim=True)).to(
            torch.bfloat16).contiguous()
        v_new = torch.randn((B, Hkv, D), device="cuda").to(torch.bfloat16)
        lens += 1
        width = max(len(r) for r in bt)
        tab = np.full((B, width), wl.PAD, np.int32)
        for s in range(B):
            tab[s, :len(bt[s])] = bt[s]
        tab_t = torch.from_numpy(tab).cuda()
        sl_t = torch.from_numpy(lens.astype(np.int32)).cuda()
        sm_t = torch.tensor(slots, dtype=torch.int64, device="cuda")
        out = torch.empty_like(q)
        cuda_lib.pa_reshape_and_cache(k_new, v_new, kc, vc, sm_t)
        cuda_lib.pa_decode(out, q, kc, vc, tab_t, sl_t, b.scale, Hkv)
        torch.cuda.synchronize()
        want = v_new.float().repeat_interleave(G, dim=1)
        assert (out.float() - want).abs().max().item() < 0.1, f"step {step}"


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_decode_batch_larger_than_one_sort(cuda_lib, dtype):
    """More sequences than one thread block orders in shared memory: the batch
    runs as consecutive slices.  Checked against the oracle, whole-sequence and
    split-KV."""
    b = wl.random_batch(910, num_seqs=5000, max_len=40, num_heads=8, num_kv_heads=2,
                        head_dim=64, dtype=dtype, device="cuda", new_in_pool=True,
                        keep_seq=False)
    ref = oracle_decode(b)
    assert_close(gpu_decode(cuda_lib, b), ref, dtype, "5000 seqs")
    assert_close(gpu_partitioned(cuda_lib, b, 16)[0], ref, dtype, "5000 seqs split-KV")
