"""FP8 (E4M3) KV cache through the C ABI against the fp64 oracle.

The cache write is compared byte for byte (the quotient x / scale is taken in
binary32 on both sides and rounded once to E4M3).  Decode over E4M3 caches is
held to the 16-bit tolerance: the codes convert exactly, so the arithmetic
error is that of the bf16/f16 path -- max |err| <= 2e-2 and relative L2 error
<= 5e-3 against the oracle's fp64 attention over the dequantised values.
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
    g = gpu.detach().double().cpu().numpy() if isinstance(gpu, torch.Tensor) else gpu
    ref = np.asarray(ref, dtype=np.float64)
    assert g.shape == ref.shape, (g.shape, ref.shape)
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    if not g.size:
        return
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


def scales(b):
    return b.meta["k_scale"], b.meta["v_scale"]


def fp8_batch(seed, dtype="bf16", new_in_pool=True, **kw):
    b = wl.random_batch(seed, dtype=dtype, device="cuda", new_in_pool=new_in_pool,
                        keep_seq=False, **kw)
    return wl.with_fp8_pool(b, seed=seed)


def gpu_decode_fp8(pa, b, seq_lens=None, k_cache=None, v_cache=None):
    bt, sl, _ = b.torch_tables("cuda")
    if seq_lens is not None:
        sl = torch.as_tensor(seq_lens, dtype=torch.int32, device="cuda")
    ks, vs = scales(b)
    out = torch.full_like(b.q, float("nan"))
    pa.pa_decode_fp8(out, b.q, b.k_cache if k_cache is None else k_cache,
                     b.v_cache if v_cache is None else v_cache, ks, vs, bt.contiguous(),
                     sl.contiguous(), b.scale, b.num_kv_heads)
    torch.cuda.synchronize()
    return out


def gpu_partitioned_fp8(pa, b, psize, max_seq_len=None):
    bt, sl, _ = b.torch_tables("cuda")
    ks, vs = scales(b)
    msl = int(b.seq_lens.max()) if max_seq_len is None else max_seq_len
    ws = torch.full((pa.pa_decode_partitioned_workspace_size(b.num_seqs, b.num_heads,
                                                             b.head_dim, msl, psize),),
                    0xFF, dtype=torch.uint8, device="cuda")
    out = torch.full_like(b.q, float("nan"))
    pa.pa_decode_partitioned_fp8(out, b.q, b.k_cache, b.v_cache, ks, vs, bt, sl, b.scale,
                                 b.num_kv_heads, psize, msl, ws)
    torch.cuda.synchronize()
    return out


def oracle_fp8(b, seq_lens=None, k_cache=None, v_cache=None):
    ks, vs = scales(b)
    return oracle.decode(b.q.cpu(), (b.k_cache if k_cache is None else k_cache).cpu(),
                         (b.v_cache if v_cache is None else v_cache).cpu(), b.block_tables,
                         b.seq_lens if seq_lens is None else seq_lens, b.scale,
                         b.num_kv_heads, b.dtype, nthreads=8,
                         kv_scales=(ks.cpu(), vs.cpu()))


# ---------------------------------------------------------------------------
# the write: byte for byte
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype,Hkv,D", [("bf16", 8, 128), ("f16", 4, 64), ("f32", 2, 128),
                                         ("bf16", 2, 64)])
def test_reshape_and_cache_fp8_bit_exact(cuda_lib, dtype, Hkv, D):
    b = wl.random_batch(700 + D + Hkv, num_seqs=41, max_len=90, num_heads=Hkv,
                        num_kv_heads=Hkv, head_dim=D, dtype=dtype, device="cuda",
                        keep_seq=False, kv_std=1.0)
    b = wl.with_fp8_pool(b, seed=3)
    ks = torch.linspace(0.002, 0.02, Hkv, device="cuda")    # small scales: some saturate
    vs = torch.linspace(0.02, 0.003, Hkv, device="cuda")
    sm_np = b.slot_mapping.copy()
    sm_np[4] = -1                                          # padding
    sm = torch.from_numpy(sm_np).cuda()
    kc, vc = b.k_cache.clone(), b.v_cache.clone()
    cuda_lib.pa_reshape_and_cache_fp8(b.k_new, b.v_new, kc, vc, ks, vs, sm)
    torch.cuda.synchronize()
    rk, rv, bad = oracle.reshape_and_cache_fp8(b.k_new.cpu(), b.v_new.cpu(), b.k_cache.cpu(),
                                               b.v_cache.cpu(), sm_np, dtype, ks.cpu(),
                                               vs.cpu())
    assert bad == 0
    assert (rk == 0x7E).any() or (rk == 0xFE).any()        # saturation was exercised
    assert np.array_equal(kc.cpu().numpy(), rk)
    assert np.array_equal(vc.cpu().numpy(), rv)


def test_reshape_and_cache_fp8_strided_source_and_bad_slot(cuda_lib):
    T, Hkv, D = 30, 4, 128
    b = fp8_batch(710, num_seqs=T, max_len=40, num_heads=Hkv, num_kv_heads=Hkv, head_dim=D,
                  new_in_pool=False)
    qkv = torch.randn(T, 3, Hkv, D, device="cuda").to(torch.bfloat16)
    k, v = qkv[:, 1], qkv[:, 2]                            # token stride 3*Hkv*D
    ks, vs = scales(b)
    sm_np = b.slot_mapping.copy()
    sm_np[9] = b.num_blocks * 16 + 1                       # out of range: skipped, flagged
    sm = torch.from_numpy(sm_np).cuda()
    kc, vc = b.k_cache.clone(), b.v_cache.clone()
    cuda_lib.pa_reshape_and_cache_fp8(k, v, kc, vc, ks, vs, sm)
    assert cuda_lib.pa_device_error(clear=True) == cuda_lib.PA_DEVERR_SLOT
    rk, rv, bad = oracle.reshape_and_cache_fp8(k.cpu().contiguous(), v.cpu().contiguous(),
                                               b.k_cache.cpu(), b.v_cache.cpu(), sm_np,
                                               "bf16", ks.cpu(), vs.cpu())
    assert bad == 1
    assert np.array_equal(kc.cpu().numpy(), rk)
    assert np.array_equal(vc.cpu().numpy(), rv)


def test_reshape_and_cache_fp8_specials(cuda_lib):
    """inf saturates to +-448, NaN stays a NaN code, signed zeros keep their
    sign, values past 448 saturate (the oracle gives 0x7F for NaN; the other
    NaN code 0xFF is an equally valid answer, so only NaN-ness is checked)."""
    Hkv, D = 1, 64
    vals = torch.tensor([float("inf"), -float("inf"), float("nan"), -0.0, 0.0, 1e30, -1e30,
                         448.0, 464.0, -500.0, 2.0 ** -10, 3 * 2.0 ** -11], device="cuda")
    k = torch.zeros(1, Hkv, D, device="cuda")
    k[0, 0, :vals.numel()] = vals
    kc = torch.zeros(4, Hkv, 16, D, dtype=torch.uint8, device="cuda")
    vc = torch.zeros_like(kc)
    one = torch.ones(Hkv, device="cuda")
    sm = torch.tensor([17], dtype=torch.int64, device="cuda")      # block 1, row 1
    cuda_lib.pa_reshape_and_cache_fp8(k, k.clone(), kc, vc, one, one, sm)
    got = kc[1, 0, 1, :vals.numel()].cpu().numpy()
    ref = oracle.e4m3_encode(vals.cpu().numpy())
    nan = np.isnan(vals.cpu().numpy())
    assert ((got[nan] & 0x7F) == 0x7F).all()
    assert np.array_equal(got[~nan], ref[~nan])
    assert got[0] == 0x7E and got[1] == 0xFE and got[3] == 0x80 and got[4] == 0x00


# ---------------------------------------------------------------------------
# decode over E4M3 caches
# ---------------------------------------------------------------------------

CASES = []
for dtype in ("bf16", "f16"):
    for D in (64, 128):
        for G, Hkv in ((1, 4), (2, 2), (4, 2), (8, 1)):
            CASES.append((dtype, D, G, Hkv))


@pytest.mark.parametrize("dtype,D,G,Hkv", CASES,
                         ids=[f"{c[0]}-d{c[1]}-g{c[2]}" for c in CASES])
def test_decode_fp8_parity_small(cuda_lib, dtype, D, G, Hkv):
    b = fp8_batch(720 + D + G, dtype=dtype, num_seqs=9, max_len=300, num_heads=G * Hkv,
                  num_kv_heads=Hkv, head_dim=D, table_slack=2)
    ref = oracle_fp8(b)
    assert_close(gpu_decode_fp8(cuda_lib, b), ref, f"fp8 {dtype} d{D} g{G}")
    assert_close(gpu_partitioned_fp8(cuda_lib, b, 64), ref, f"fp8 part {dtype} d{D} g{G}")


def test_decode_fp8_ragged_lengths_every_remainder(cuda_lib):
    L = np.arange(1, 81)
    Hkv, G, D = 2, 4, 128
    rng = np.random.default_rng(7)
    fl = wl.FreeList(int(sum(math.ceil(x / 16) for x in L)) + 4, rng)
    tables = [fl.allocate(int(x)) for x in L]
    b = wl.build_batch("ragged", ctx_lens=L - 1, num_heads=G * Hkv, num_kv_heads=Hkv,
                       head_dim=D, dtype="bf16", num_blocks=len(fl.free) + sum(map(len, tables)),
                       tables=tables, seed=8, device="cuda", new_in_pool=True)
    b = wl.with_fp8_pool(b, seed=8)
    assert_close(gpu_decode_fp8(cuda_lib, b), oracle_fp8(b), "fp8 ragged")


def test_decode_fp8_seq_len_zero_and_one(cuda_lib):
    b = fp8_batch(730, num_seqs=6, max_len=40, num_heads=8, num_kv_heads=2, head_dim=128)
    sl = b.seq_lens.copy()
    sl[[0, 3]] = 0
    sl[[1, 4]] = 1
    out = gpu_decode_fp8(cuda_lib, b, seq_lens=sl)
    assert torch.equal(out[[0, 3]], torch.zeros_like(out[[0, 3]]))
    assert_close(out, oracle_fp8(b, seq_lens=sl), "fp8 len 0/1")


def test_decode_fp8_block_permutation_bit_identical(cuda_lib):
    b = fp8_batch(740, num_seqs=12, max_len=400, num_heads=32, num_kv_heads=8, head_dim=128,
                  extra_blocks=64)
    p = wl.permute_blocks(b, seed=5)
    assert torch.equal(gpu_decode_fp8(cuda_lib, b), gpu_decode_fp8(cuda_lib, p))


def test_decode_fp8_padding_entries_never_read(cuda_lib):
    b = fp8_batch(750, num_seqs=7, max_len=150, num_heads=16, num_kv_heads=4, head_dim=64,
                  table_slack=5)
    assert (b.block_tables == wl.PAD).any()
    assert_close(gpu_decode_fp8(cuda_lib, b), oracle_fp8(b), "fp8 pad")


def test_fp8_step_write_then_decode(cuda_lib):
    """One step: quantise and write the new token of every sequence, then
    decode over the written cache."""
    b = fp8_batch(760, num_seqs=20, max_len=200, num_heads=32, num_kv_heads=8, head_dim=128,
                  new_in_pool=False)
    bt, sl, sm = b.torch_tables("cuda")
    ks, vs = scales(b)
    kc, vc = b.k_cache.clone(), b.v_cache.clone()
    cuda_lib.pa_reshape_and_cache_fp8(b.k_new, b.v_new, kc, vc, ks, vs, sm)
    out = gpu_decode_fp8(cuda_lib, b, k_cache=kc, v_cache=vc)
    rk, rv, _ = oracle.reshape_and_cache_fp8(b.k_new.cpu(), b.v_new.cpu(), b.k_cache.cpu(),
                                             b.v_cache.cpu(), b.slot_mapping, "bf16",
                                             ks.cpu(), vs.cpu())
    assert np.array_equal(kc.cpu().numpy(), rk) and np.array_equal(vc.cpu().numpy(), rv)
    assert_close(out, oracle_fp8(b, k_cache=torch.from_numpy(rk), v_cache=torch.from_numpy(rv)),
                 "fp8 step")


def test_decode_fp8_batch_larger_than_one_sort(cuda_lib):
    b = fp8_batch(770, num_seqs=3500, max_len=40, num_heads=8, num_kv_heads=2, head_dim=128)
    ref = oracle_fp8(b)
    assert_close(gpu_decode_fp8(cuda_lib, b), ref, "3500 seqs")
    assert_close(gpu_partitioned_fp8(cuda_lib, b, 32), ref, "3500 seqs split-KV")


# ---------------------------------------------------------------------------
# full-size workloads: every output element against the oracle (fullsize.py)
# ---------------------------------------------------------------------------

@pytest.mark.slow
def test_full_serving_mix_fp8_step(cuda_lib):
    b = wl.serving_mix_fp8(device="cuda")
    bt, sl, sm = b.torch_tables("cuda")
    ks, vs = scales(b)
    kc, vc = b.k_cache.clone(), b.v_cache.clone()
    cuda_lib.pa_reshape_and_cache_fp8(b.k_new, b.v_new, kc, vc, ks, vs, sm)
    out = gpu_decode_fp8(cuda_lib, b, k_cache=kc, v_cache=vc)
    # the write: bit-exact on the whole pool (quotients in binary32)
    rk, rv, bad = oracle.reshape_and_cache_fp8(b.k_new.cpu(), b.v_new.cpu(), b.k_cache.cpu(),
                                               b.v_cache.cpu(), b.slot_mapping, b.dtype,
                                               ks.cpu(), vs.cpu())
    assert bad == 0
    assert np.array_equal(kc.cpu().numpy(), rk) and np.array_equal(vc.cpu().numpy(), rv)
    ref, t = fullsize.decode_all(b, k_cache=kc, v_cache=vc, kv_scales=(ks, vs))
    fullsize.check("serving_mix_fp8: cache write + pa_decode_fp8", out, ref, b.dtype, t)


@pytest.mark.slow
def test_full_long_context_fp8_partitioned(cuda_lib):
    b = wl.long_context_fp8(device="cuda", canary=False)
    out = gpu_partitioned_fp8(cuda_lib, b, 512, max_seq_len=131072)
    ref, t = fullsize.decode_all(b, kv_scales=scales(b))
    fullsize.check("long_context_fp8: pa_decode_partitioned_fp8", out, ref, b.dtype, t)
    fullsize.check("long_context_fp8: pa_decode_fp8", gpu_decode_fp8(cuda_lib, b), ref,
                   b.dtype)
