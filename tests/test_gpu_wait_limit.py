"""The kernels' bounded waits, exercised without a fault.

Every wait in a kernel (on an mbarrier phase) gives up after a 1 s wall-clock
limit, sets PA_DEVERR_TIMEOUT in the sticky device error word, waits (bounded)
for its own copies in flight and returns.  The test hook
pa_test_stall_next_decode makes the first copy of every warp of the next
decode call expect more bytes than it delivers, so the wait for it runs out:
the call must come back, report the timeout, and leave the context usable for
the next call, whose output must match the fp64 oracle.
"""
import time

import pytest
import torch

import oracle
from paged_kv_cache_151_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

PA_DEVERR_TIMEOUT = 0x8


def decode(pa, b):
    bt, sl, _ = b.torch_tables("cuda")
    out = torch.zeros_like(b.q)
    pa.pa_decode(out, b.q, b.k_cache, b.v_cache, bt.contiguous(), sl.contiguous(), b.scale,
                 b.num_kv_heads)
    return out


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_wait_limit_reports_timeout_and_context_survives(cuda_lib, dtype):
    pa = cuda_lib
    b = wl.random_batch(31, num_seqs=6, max_len=200, num_heads=8, num_kv_heads=2,
                        head_dim=128, dtype=dtype, device="cuda", new_in_pool=True,
                        keep_seq=False, table_slack=2)
    pa.pa_device_error(clear=True)

    pa.pa_test_stall_next_decode()
    t0 = time.perf_counter()
    decode(pa, b)
    flags = pa.pa_device_error(clear=True)          # synchronises
    waited = time.perf_counter() - t0
    assert flags & PA_DEVERR_TIMEOUT, f"flags {flags:#x}"
    assert waited < 30.0, f"the stalled call took {waited:.1f} s"

    # the hook is one-shot, and the context is usable: the next call is correct
    out = decode(pa, b)
    assert pa.pa_device_error(clear=True) == 0
    ref = oracle.decode(b.q.cpu(), b.k_cache.cpu(), b.v_cache.cpu(), b.block_tables,
                        b.seq_lens, b.scale, b.num_kv_heads, b.dtype, nthreads=8)
    g = out.double().cpu().numpy()
    err = abs(g - ref).max()
    assert err <= (1e-4 if dtype == "f32" else 2e-2), err
