"""Whole-output parity at full size: the fp64 oracle over every (sequence,
head) output of a workload, on all host cores, and the error figures of each
comparison, which ``conftest.py`` prints at the end of the run.

Tolerances, against the oracle on the output as stored:
  fp32 caches              max |err| <= 1e-4
  bf16 / f16 / E4M3 caches max |err| <= 2e-2 and relative L2 error <= 5e-3
(the relative L2 error is taken over the whole output tensor).
"""
from __future__ import annotations

import os
import time
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

import oracle

TOL_F32 = 1e-4
TOL_16_ABS = 2e-2
TOL_16_REL_L2 = 5e-3

# (name, elements compared, max |err|, relative L2 error, oracle seconds)
RESULTS: list[tuple[str, int, float, float, float]] = []


def host_threads() -> int:
    return max(1, os.cpu_count() or 1)


def check(name: str, gpu, ref, dtype: str, oracle_s: float = 0.0):
    """Assert the tolerance on every element and record the figures."""
    g = gpu.detach().double().cpu().numpy() if isinstance(gpu, torch.Tensor) else gpu
    ref = np.asarray(ref, dtype=np.float64)
    assert g.shape == ref.shape, (g.shape, ref.shape)
    assert np.isfinite(g).all(), f"{name}: non-finite output"
    err = float(np.abs(g - ref).max()) if g.size else 0.0
    rel = float(np.linalg.norm(g - ref) / max(np.linalg.norm(ref), 1e-30))
    RESULTS.append((name, int(g.size), err, rel, oracle_s))
    if dtype == "f32":
        assert err <= TOL_F32, f"{name}: max abs err {err:.3g}"
    else:
        assert err <= TOL_16_ABS, f"{name}: max abs err {err:.3g}"
        assert rel <= TOL_16_REL_L2, f"{name}: rel L2 err {rel:.3g}"


def decode_all(b, k_cache=None, v_cache=None, kv_scales=None):
    """oracle.decode of every (sequence, query head) of batch ``b``; returns
    (out [B, H, D] fp64, seconds)."""
    t0 = time.perf_counter()
    ks = None
    if kv_scales is not None:
        ks = (kv_scales[0].cpu(), kv_scales[1].cpu())
    ref = oracle.decode(b.q.cpu(), (b.k_cache if k_cache is None else k_cache).cpu(),
                        (b.v_cache if v_cache is None else v_cache).cpu(), b.block_tables,
                        b.seq_lens, b.scale, b.num_kv_heads, b.dtype,
                        nthreads=host_threads(), kv_scales=ks)
    return ref, time.perf_counter() - t0


def multi_all(b, rows_per_piece: int = 16):
    """oracle.decode_multi of every query row of batch ``b``; returns
    (out [T, H, D] fp64, seconds).

    The rows are cut into pieces of at most ``rows_per_piece`` consecutive
    rows of one sequence, decoded on all host cores.  A piece of rows
    a .. a+m-1 of a sequence with n new rows over seq_len L is passed as a
    sequence of its own with m rows over seq_len L - n + a + m: its row k then
    sees the first L - n + a + k + 1 positions, exactly what row a + k of the
    whole sequence sees, over the same block table."""
    t0 = time.perf_counter()
    qs = np.asarray(b.meta["query_start"], dtype=np.int64)
    L = np.asarray(b.seq_lens, dtype=np.int64)
    q = b.q.cpu().contiguous()
    kc, vc = b.k_cache.cpu(), b.v_cache.cpu()
    pieces = []                                   # (sequence, first row, rows)
    for s in range(len(L)):
        n = int(qs[s + 1] - qs[s])
        for a in range(0, n, rows_per_piece):
            pieces.append((s, a, min(rows_per_piece, n - a)))
    # a few sequences per oracle call, similar cost per call
    groups, cur, cost = [], [], 0
    budget = max(1, sum(m * int(L[s]) for s, _, m in pieces) // (4 * host_threads()))
    for pc in pieces:
        cur.append(pc)
        cost += pc[2] * int(L[pc[0]])
        if cost >= budget:
            groups.append(cur)
            cur, cost = [], 0
    if cur:
        groups.append(cur)
    out = np.zeros((q.shape[0],) + tuple(q.shape[1:]), dtype=np.float64)

    def run(group):
        seqs = np.array([s for s, _, _ in group])
        rows = np.concatenate([np.arange(qs[s] + a, qs[s] + a + m) for s, a, m in group])
        lens = np.array([L[s] - (qs[s + 1] - qs[s]) + a + m for s, a, m in group],
                        dtype=np.int32)
        sub_qs = np.zeros(len(group) + 1, dtype=np.int32)
        sub_qs[1:] = np.cumsum([m for _, _, m in group])
        r = oracle.decode_multi(q[torch.from_numpy(rows)].contiguous(), kc, vc,
                                b.block_tables[seqs], lens, sub_qs, b.scale,
                                b.num_kv_heads, b.dtype)
        out[rows] = r

    with ThreadPoolExecutor(host_threads()) as ex:
        list(ex.map(run, groups))
    return out, time.perf_counter() - t0
