"""The allocation-free split-KV entry point.

Some callers cannot allocate device memory where they decode (a graph
capture in progress on another stream, an allocator that forbids growth after
warm-up, a plug-in whose host owns all memory).  pa_decode_partitioned_noalloc
serves them with a workspace compiled into the library.  This file runs last
(pytest collects it after every other test file) and checks, through the C
ABI, that two calls in a row give the same output as pa_decode_partitioned
with a caller workspace and match the fp64 oracle within the decode
tolerances, that the calls leave the device memory in use unchanged, and
that a problem too large for the built-in workspace is refused before
anything is launched.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_151_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

TOL_F32 = 1e-4                       # fp32 caches: max |err|
TOL_16_ABS, TOL_16_REL_L2 = 2e-2, 5e-3   # bf16 / f16 caches


def _assert_matches_oracle(b, out):
    ref = oracle.decode(b.q.cpu(), b.k_cache.cpu(), b.v_cache.cpu(), b.block_tables,
                        b.seq_lens, b.scale, b.num_kv_heads, b.dtype, nthreads=8)
    g = out.double().cpu().numpy()
    err = np.abs(g - ref).max()
    if b.dtype == "f32":
        assert err <= TOL_F32, err
    else:
        rel = np.linalg.norm(g - ref) / np.linalg.norm(ref)
        assert err <= TOL_16_ABS and rel <= TOL_16_REL_L2, (err, rel)


def _with_workspace(pa, b, bt, sl, psize, msl):
    nbytes = pa.pa_decode_partitioned_workspace_size(b.num_seqs, b.num_heads, b.head_dim,
                                                     msl, psize)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    out = torch.full_like(b.q, float("nan"))
    pa.pa_decode_partitioned(out, b.q, b.k_cache, b.v_cache, bt, sl, b.scale,
                             b.num_kv_heads, psize, msl, ws)
    return out


def _noalloc_via_abi(pa, b, bt, sl, psize, msl, out):
    """Call the entry point straight through ctypes (no Python wrapper)."""
    lib = pa.load()
    dt = {torch.float32: 0, torch.bfloat16: 1, torch.float16: 2}[b.q.dtype]
    return lib.pa_decode_partitioned_noalloc(
        out.data_ptr(), b.q.data_ptr(), b.k_cache.data_ptr(), b.v_cache.data_ptr(),
        bt.data_ptr(), sl.data_ptr(), b.num_seqs, b.num_heads, b.num_kv_heads, b.head_dim,
        b.num_blocks, 16, bt.shape[1], b.q.stride(0), ctypes.c_float(b.scale), dt, psize,
        msl, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("dtype,H,Hkv,D,psize", [("bf16", 32, 8, 128, 512),
                                                ("f32", 8, 2, 64, 64),
                                                ("f16", 16, 2, 128, 96)])
def test_noalloc_matches_workspace_call_twice(cuda_lib, dtype, H, Hkv, D, psize):
    pa = cuda_lib
    for seed in (501, 502):                     # two different problems, back to back
        b = wl.random_batch(seed, num_seqs=6, max_len=1200, num_heads=H, num_kv_heads=Hkv,
                            head_dim=D, dtype=dtype, device="cuda", new_in_pool=True,
                            keep_seq=False, kv_std=0.5)
        bt, sl, _ = b.torch_tables("cuda")
        msl = int(b.seq_lens.max())
        ref = _with_workspace(pa, b, bt, sl, psize, msl)
        outs = [torch.full_like(b.q, float("nan")) for _ in range(2)]
        torch.cuda.synchronize()
        for out in outs:                        # the second call reuses the same array
            rc = _noalloc_via_abi(pa, b, bt, sl, psize, msl, out)
            assert rc == 0, pa.pa_status_string(rc)
            torch.cuda.synchronize()
            assert torch.isfinite(out.float()).all()
            # same kernels and schedule as the workspace call: identical bits
            # (the tests' tolerances would also do)
            assert torch.equal(out, ref)
            _assert_matches_oracle(b, out)
    assert pa.pa_device_error(clear=True) == 0


def test_noalloc_allocates_nothing(cuda_lib):
    """Once the library's module is loaded (the first call), further calls
    change neither the device's free memory nor torch's allocations."""
    pa = cuda_lib
    b = wl.random_batch(504, num_seqs=8, max_len=2000, num_heads=32, num_kv_heads=8,
                        head_dim=128, dtype="bf16", device="cuda", new_in_pool=True,
                        keep_seq=False, kv_std=0.5)
    bt, sl, _ = b.torch_tables("cuda")
    msl = int(b.seq_lens.max())
    outs = [torch.empty_like(b.q) for _ in range(3)]
    assert _noalloc_via_abi(pa, b, bt, sl, 512, msl, outs[0]) == 0     # loads the module
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    torch0 = torch.cuda.memory_allocated()
    for out in outs[1:]:
        assert _noalloc_via_abi(pa, b, bt, sl, 512, msl, out) == 0
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    assert torch.cuda.memory_allocated() == torch0
    assert torch.equal(outs[1], outs[0]) and torch.equal(outs[2], outs[0])
    _assert_matches_oracle(b, outs[2])
    assert pa.pa_device_error(clear=True) == 0


def test_noalloc_rejects_problems_beyond_its_workspace(cuda_lib):
    pa = cuda_lib
    b = wl.random_batch(503, num_seqs=2, max_len=40, num_heads=64, num_kv_heads=8,
                        head_dim=128, dtype="bf16", device="cuda", new_in_pool=True,
                        keep_seq=False)
    bt, sl, _ = b.torch_tables("cuda")
    msl = 1 << 20                                # a bound far past the built-in array
    assert pa.pa_decode_partitioned_workspace_size(
        b.num_seqs, b.num_heads, b.head_dim, msl, 512) > pa.PA_NOALLOC_SCRATCH_BYTES
    out = torch.zeros_like(b.q)
    rc = _noalloc_via_abi(pa, b, bt, sl, 512, msl, out)
    assert rc == -3                              # PA_ERR_WORKSPACE, nothing launched
    torch.cuda.synchronize()
    assert torch.equal(out, torch.zeros_like(out))
