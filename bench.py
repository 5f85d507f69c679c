#!/usr/bin/env python3
"""Benchmark of the paged decode hot path on GB300.

One step = one pass of the hot path over the serving-mix batch: the cache
write of one new token per sequence (pa_reshape_and_cache), then decode
attention over the paged context (pa_decode).  The batch: 256 sequences,
32 query / 8 KV heads x 128, bf16 cache in 16-token blocks, lengths lognormal
(median 350, sigma 1) clipped to [1, 4096], pool 1.2x the blocks needed.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Prints one JSON line (rank 0).  ``value`` is sequences per second over all
ranks with inputs resident in HBM (device time of K steps run back to back;
each streams far more than L2); ``e2e`` is the same metric with each step's inputs copied
from pinned host memory and its output copied back inside the timed region
(steps pipelined: the next step's inputs go in, and the last step's output
comes back, on their own streams while a step's kernels run).
``--impl reference`` times the fp64 CPU oracle on the host cores instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from paged_kv_cache_151_gb300 import workloads as wl  # noqa: E402

METRIC = "paged decode attention: seqs/sec and achieved KV HBM GB/s (% of GB300 peak)"
WORKLOAD = ("serving_mix: batch 256, 32 query / 8 KV heads x 128, bf16 KV cache, block 16, "
            "seq_lens lognormal(median 350, sigma 1.0) clipped to [1, 4096], pool 1.2x; "
            "step = reshape_and_cache of 1 token/seq + pa_decode")
FALLBACK_HBM_GBS = 6800.0


# ---------------------------------------------------------------------------
# byte accounting (what a call must touch at least)
# ---------------------------------------------------------------------------

def decode_bytes(b) -> dict:
    es = torch.tensor([], dtype=wl.DTYPES[b.dtype]).element_size()
    kv_es = 1 if b.meta.get("kv") == "e4m3" else es      # E4M3 caches: one byte
    L = b.seq_lens.astype(np.int64)
    kv = int(L.sum()) * 2 * b.num_kv_heads * b.head_dim * kv_es
    kv_full = int(np.ceil(L / 16).sum()) * 16 * 2 * b.num_kv_heads * b.head_dim * kv_es
    qo = 2 * b.num_seqs * b.num_heads * b.head_dim * es
    tab = int(np.ceil(L / 16).sum()) * 4 + 4 * b.num_seqs
    return {"kv": kv, "kv_full_blocks": kv_full, "total": kv + qo + tab}


def multi_bytes(b) -> dict:
    """Multi-token queries: every cached token's K and V read at least once,
    q and out once; flops of QK^T and PV over the causal positions."""
    es = torch.tensor([], dtype=wl.DTYPES[b.dtype]).element_size()
    L = b.seq_lens.astype(np.int64)
    n = np.diff(b.meta["query_start"]).astype(np.int64)
    kv = int(L.sum()) * 2 * b.num_kv_heads * b.head_dim * es
    T = int(n.sum())
    qo = 2 * T * b.num_heads * b.head_dim * es
    # row i of a sequence with n rows sees L - n + i + 1 positions
    seen = int(sum(int(n_s) * (int(L_s) - int(n_s)) + int(n_s) * (int(n_s) + 1) // 2
                   for L_s, n_s in zip(L, n)))
    flops = 4 * seen * b.num_heads * b.head_dim
    return {"kv": kv, "total": kv + qo, "rows": T, "flops": flops}


def cache_write_bytes(b) -> int:
    es = torch.tensor([], dtype=wl.DTYPES[b.dtype]).element_size()
    rows = b.num_seqs * b.num_kv_heads * b.head_dim * es
    return 2 * 2 * rows + 8 * b.num_seqs          # K and V, read + write, slots


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_digest(tu: str) -> str:
    """Hash of one kernel translation unit and every local header it
    includes, directly or through another header: a recorded DRAM figure
    stays valid while none of the sources it was compiled from changed."""
    csrc = os.path.join(ROOT, "paged_kv_cache_151_gb300", "csrc")
    inc = re.compile(rb'^\s*#\s*include\s+"([^"]+)"', re.M)
    seen, todo = set(), [os.path.normpath(os.path.join(csrc, tu))]
    while todo:
        p = todo.pop()
        if p in seen:
            continue
        seen.add(p)
        with open(p, "rb") as fh:
            for m in inc.finditer(fh.read()):
                todo.append(os.path.normpath(os.path.join(os.path.dirname(p), m.group(1).decode())))
    h = hashlib.sha256()
    for p in sorted(seen):
        with open(p, "rb") as fh:
            h.update(os.path.relpath(p, ROOT).encode() + fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(name: str):
    """DRAM bytes per launch of `name` from the committed ncu summary, if it
    was taken on the current sources of that kernel's translation unit;
    else None."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
        e = d[name]
        if e.get("kernel_src_sha") != kernel_source_digest(e["tu"]):
            return None
        return float(e["dram_bytes_per_launch"])
    except Exception:
        return None


def bench_config(b, world: int) -> dict:
    """The `config` of the bench line, the same for the GPU arm and the
    reference arm (which runs the same workload on the host)."""
    return {
        "workload": WORKLOAD,
        "global_batch": world * b.num_seqs,
        "tokens_attended": int(b.seq_lens.sum()),
        "num_blocks": int(b.num_blocks),
        "l2": "GPU arm: value = K steps back to back in one timed region, inputs larger "
              "than L2 (each step streams 617 MB of K/V; L2 flushed once before the region); "
              "kernel timings (decode_us, roofline): L2 flushed before each step (twice the "
              "L2 size written, then as much read, outside the events)",
        "parallelism": f"replicas x{world}" if world > 1 else "one replica",
    }


# ---------------------------------------------------------------------------
# ranks: every rank runs its own replica; time = max over ranks
# ---------------------------------------------------------------------------

def max_over_ranks(value: float, world: int, device=None) -> float:
    """The largest `value` over all ranks (identity for one rank)."""
    if world <= 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64,
                     device=device if device is not None else "cpu")
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def aggregate_rate(world: int, units_per_rank: int, steps: int, max_ms: float) -> float:
    """Whole-job units per second: all ranks' units over the slowest rank's time."""
    return world * units_per_rank * steps / (max_ms * 1e-3)


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.out.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4)
                          if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def make_flush(device):
    """L2 flush between timed calls: write a buffer of twice the L2 size,
    then read a second one, so that the lines left behind are clean and the
    next timed kernel does not pay for write-backs of the flush itself."""
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    n = max(2 * l2, 256 << 20)
    wbuf = torch.empty(n // 4, dtype=torch.int32, device=device)
    rbuf = torch.ones(n // 4, dtype=torch.int32, device=device)
    sink = torch.empty((), dtype=torch.int64, device=device)

    def flush():
        wbuf.fill_(1)
        torch.sum(rbuf, dim=0, dtype=torch.int64, out=sink)
    return flush, n


def time_calls(fn, iters, flush, stream):
    """Device time (ms) of each call, L2 flushed before each."""
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(iters)]
    for a, b in evs:
        flush()
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


def gpu_arm(args, rank, world, device):
    from paged_kv_cache_151_gb300 import pa

    torch.cuda.set_device(device)
    pa.load()
    stream = torch.cuda.current_stream()
    flush, flush_bytes = make_flush(device)

    b = wl.serving_mix(device=device, canary=False)
    bt, sl, sm = b.torch_tables(device)
    bt, sl, sm = bt.contiguous(), sl.contiguous(), sm.contiguous()
    kc, vc = b.k_cache, b.v_cache
    out = torch.empty_like(b.q)
    nbytes = decode_bytes(b)
    wbytes = cache_write_bytes(b)

    def step():
        pa.pa_reshape_and_cache(b.k_new, b.v_new, kc, vc, sm)
        pa.pa_decode(out, b.q, kc, vc, bt, sl, b.scale, b.num_kv_heads)

    for _ in range(args.warmup):
        flush()
        step()
    torch.cuda.synchronize()
    pa.pa_device_error(clear=True)

    # ---- the K timed steps ----
    # A step is the cache write followed by decode with nothing in between,
    # so the decode may set up while the write finishes (programmatic
    # dependent launch).  The K steps run back to back in one timed region:
    # each streams 617 MB of K/V, several times the L2, so no flush is needed
    # between them (L2 is flushed once before the region).  Each kernel's own
    # duration is then timed in a second pass over K steps with an event
    # between the two kernels and L2 flushed before each step.
    t_beg, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    evk = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    clocks = ClockSampler(torch.cuda.current_device())
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.2)
    flush()
    t_wall = time.perf_counter()
    t_beg.record(stream)
    for _ in range(args.steps):
        pa.pa_reshape_and_cache(b.k_new, b.v_new, kc, vc, sm)
        pa.pa_decode(out, b.q, kc, vc, bt, sl, b.scale, b.num_kv_heads)
    t_end.record(stream)
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall
    if world > 1:
        torch.distributed.barrier()
    for e0, e1, e2 in evk:
        flush()
        e0.record(stream)
        pa.pa_reshape_and_cache(b.k_new, b.v_new, kc, vc, sm)
        e1.record(stream)
        pa.pa_decode(out, b.q, kc, vc, bt, sl, b.scale, b.num_kv_heads)
        e2.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    write_ms = [e0.elapsed_time(e1) for e0, e1, _ in evk]
    dec_ms = [e1.elapsed_time(e2) for _, e1, e2 in evk]
    total_ms = max_over_ranks(float(t_beg.elapsed_time(t_end)), world, device)
    flags = pa.pa_device_error(clear=True)

    dec_mean = statistics.mean(dec_ms)
    achieved = nbytes["total"] / (dec_mean * 1e-3) / 1e9
    peak, peak_kind = measured_peak()

    # ---- end to end through the C ABI with host buffers ----
    e2e = e2e_arm(args, b, device, flush, pa)
    probe = read_probe(device) if world == 1 else None

    result = {
        "metric": METRIC,
        "value": aggregate_rate(world, b.num_seqs, args.steps, total_ms),
        "unit": "seqs/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": total_ms / args.steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded; no dataset)",
        "config": bench_config(b, world),
        "decode_kernel": "persistent (longest-first units, per-warp bulk-copy rings)",
        "l2_flush_bytes": flush_bytes,
        "kv_gbs": nbytes["kv"] / (dec_mean * 1e-3) / 1e9,
        "decode_us": dec_mean * 1e3,
        "decode_us_median": statistics.median(dec_ms) * 1e3,
        "cache_write_us": statistics.mean(write_ms) * 1e3,
        "cache_write_gbs": wbytes / (statistics.mean(write_ms) * 1e-3) / 1e9,
        "decode_bytes": nbytes,
        "roofline": {
            "kernel": "decode_persistent_kernel<bf16,128,4> (pa_decode)",
            "bound": "hbm",
            "achieved": achieved,
            "peak": peak,
            "peak_kind": peak_kind,
            "unit": "GB/s",
            "frac": achieved / peak,
            "frac_of_nominal_8tbs": achieved / 8000.0,
            "read_probe_gbs": probe["gbs"] if probe else None,
            "frac_of_read_probe": achieved / probe["gbs"] if probe else None,
            "traffic": recorded_traffic("decode_serving_mix"),
        },
        "e2e": e2e,
        "gpu_launches": 2 * args.steps,
        "kernel_timing": "decode_us / cache_write_us / roofline: the same K steps run again "
                         "with an event between the two kernels",
        "clocks": clk,
        "device_error_flags": flags,
        "wall_s_timed_region": t_wall,
    }
    if not args.no_extras and world == 1:
        result["long_context"] = long_context_arm(args, device, flush, pa)
        result["shared_prefix"] = shared_prefix_arm(args, device, flush, pa)
        result["paging_overhead"] = paging_overhead_arm(args, device, flush, pa)
        result["multi_query"] = multi_query_arm(args, device, flush, pa)
        result["fp8"] = fp8_arm(args, device, flush, pa)
        result["copy_blocks"] = copy_blocks_arm(args, device, flush, pa)
        result["block_manager"] = block_manager_arm(args)
        result["read_probe"] = probe
        result["launch_to_launch"] = launch_to_launch_arm(step)
    return result, b


def read_probe(device, gib: float = 2.0) -> dict:
    """Read-only bandwidth probe: a float32 sum over a buffer far larger than
    L2, best of 10 (the copy peak in MEASURED_PEAKS.json counts a read and a
    write; decode mostly reads)."""
    n = int(gib * (1 << 30)) // 4
    x = torch.ones(n, dtype=torch.float32, device=device)
    sink = torch.empty((), dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream()
    for _ in range(3):
        torch.sum(x, dim=0, out=sink)
    best = None
    for _ in range(10):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        torch.sum(x, dim=0, out=sink)
        e1.record(stream)
        torch.cuda.synchronize()
        t = e0.elapsed_time(e1)
        best = t if best is None else min(best, t)
    gbs = n * 4 / (best * 1e-3) / 1e9
    del x
    return {"gbs": gbs, "bytes": n * 4, "how": "torch.sum over a float32 buffer, best of 10"}


def launch_to_launch_arm(step, n: int = 50) -> dict:
    """The serving-mix step (cache write + decode) run n times back to back
    without L2 flushes: eagerly, each call going through the binding and the
    C ABI, and replayed from a CUDA graph captured from one step."""
    stream = torch.cuda.current_stream()

    def timed(fn):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / n * 1e3

    for _ in range(3):
        step()
    torch.cuda.synchronize()
    res = {"steps": n, "l2": "not flushed (steps back to back)", "eager_us_per_step": timed(step)}
    try:
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            step()
        stream.wait_stream(side)
        torch.cuda.synchronize()
        with torch.cuda.graph(g):
            step()
        g.replay()
        torch.cuda.synchronize()
        res["graph_us_per_step"] = timed(g.replay)
    except Exception as exc:                      # reported, not fatal
        res["graph_us_per_step"] = None
        res["graph_error"] = str(exc).splitlines()[0][:200]
    return res


def e2e_arm(args, b, device, flush, pa):
    """Same step, inputs from pinned host memory, output back to the host.

    A serving loop stages a step's inputs (q, the new K/V rows, slot_mapping,
    block_tables, seq_lens) in one pinned host buffer and sends them with one
    copy; the device buffer is viewed as the input tensors in place.  The
    loop is pipelined over two staging buffers and two output buffers: step
    i+1's inputs are copied in (one stream) and step i-1's output is read back
    (another stream) while step i's kernels run, each copy ordered by events
    against the kernels that use its buffers.  Every step carries its own
    host-to-device and device-to-host copy inside the timed region, which runs
    from the first copy in to the last copy out.  One step streams 617 MB of
    K/V, far more than L2, so the steps run back to back without a flush.
    Beside it: each step timed alone (copy in, kernels, copy out, L2 flushed
    before it), with one staged copy and with one copy per tensor."""
    comp = torch.cuda.current_stream()
    h = {
        "q": b.q.cpu().pin_memory(), "k_new": b.k_new.cpu().pin_memory(),
        "v_new": b.v_new.cpu().pin_memory(),
        "slot_mapping": torch.from_numpy(b.slot_mapping).pin_memory(),
        "block_tables": torch.from_numpy(b.block_tables).pin_memory(),
        "seq_lens": torch.from_numpy(b.seq_lens).pin_memory(),
    }
    # one staging buffer: each input at a 256-byte aligned offset
    offs, total = {}, 0
    for k, v in h.items():
        offs[k] = total
        total += (v.numel() * v.element_size() + 255) // 256 * 256
    stage_h = torch.empty(total, dtype=torch.uint8).pin_memory()
    stage_d = [torch.empty(total, dtype=torch.uint8, device=device) for _ in range(2)]
    views = [{}, {}]
    for k, v in h.items():
        n = v.numel() * v.element_size()
        stage_h[offs[k]:offs[k] + n].copy_(v.reshape(-1).view(torch.uint8))
        for s in range(2):
            views[s][k] = stage_d[s][offs[k]:offs[k] + n].view(v.dtype).view(v.shape)
    d = {k: torch.empty_like(v, device=device) for k, v in h.items()}
    out = [torch.empty_like(b.q) for _ in range(2)]
    out_h = [torch.empty(b.q.shape, dtype=b.q.dtype).pin_memory() for _ in range(2)]
    kc, vc = b.k_cache, b.v_cache
    cin, cout = torch.cuda.Stream(device=device), torch.cuda.Stream(device=device)

    def kernels(vw, o):
        pa.pa_reshape_and_cache(vw["k_new"], vw["v_new"], kc, vc, vw["slot_mapping"])
        pa.pa_decode(o, vw["q"], kc, vc, vw["block_tables"], vw["seq_lens"], b.scale,
                     b.num_kv_heads)

    def pipelined(n):
        """n steps; returns ms from the first copy in to the last copy out."""
        in_ev = [torch.cuda.Event() for _ in range(n)]
        done_ev = [torch.cuda.Event() for _ in range(n)]
        back_ev = [torch.cuda.Event() for _ in range(n)]
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        t0.record(cin)
        for i in range(n):
            s = i % 2
            if i >= 2:
                cin.wait_event(done_ev[i - 2])     # staging buffer s: step i-2 is done with it
            with torch.cuda.stream(cin):
                stage_d[s].copy_(stage_h, non_blocking=True)
            in_ev[i].record(cin)
            comp.wait_event(in_ev[i])
            if i >= 2:
                comp.wait_event(back_ev[i - 2])    # out[s] of step i-2 read back
            kernels(views[s], out[s])
            done_ev[i].record(comp)
            cout.wait_event(done_ev[i])
            with torch.cuda.stream(cout):
                out_h[s].copy_(out[s], non_blocking=True)
            back_ev[i].record(cout)
        t1.record(cout)
        torch.cuda.synchronize()
        return t0.elapsed_time(t1)

    def step():                                    # one copy in, one copy out
        stage_d[0].copy_(stage_h, non_blocking=True)
        kernels(views[0], out[0])
        out_h[0].copy_(out[0], non_blocking=True)

    def step_separate():                           # one copy per input tensor
        for k in h:
            d[k].copy_(h[k], non_blocking=True)
        kernels(d, out[0])
        out_h[0].copy_(out[0], non_blocking=True)

    n = max(10, args.steps // 4)
    res = {}
    for name, fn in (("separate", step_separate), ("staged", step)):
        for _ in range(args.warmup):
            flush()
            fn()
        torch.cuda.synchronize()
        res[name] = statistics.mean(time_calls(fn, n, flush, comp))
    npipe = max(200, args.steps)                   # a serving loop runs on: fill and drain amortised
    pipelined(max(3, args.warmup))
    pipe_ms = pipelined(npipe) / npipe
    torch.cuda.synchronize()
    for s in range(2):
        assert torch.equal(views[s]["q"], b.q) and torch.equal(
            views[s]["block_tables"].cpu(), torch.from_numpy(b.block_tables))
    assert torch.equal(out_h[0], out_h[1])         # every step computes the same output
    return {"value": b.num_seqs / (pipe_ms * 1e-3), "unit": "seqs/s",
            "h2d_bytes_per_step": int(total),
            "d2h_bytes_per_step": int(out_h[0].numel() * out_h[0].element_size()),
            "ms_per_step": pipe_ms, "steps": npipe,
            "inputs": "one pinned staging buffer, one host-to-device copy per step; "
                      "steps pipelined over two staging and two output buffers (copies on "
                      "their own streams); at least 200 steps, so the pipeline's fill and "
                      "drain are amortised as in a running serving loop; 617 MB of K/V per "
                      "step (> L2), no flush between steps",
            "serial": {"value": b.num_seqs / (res["staged"] * 1e-3), "ms_per_step": res["staged"],
                       "steps": n, "l2": "flushed before each step"},
            "separate_copies": {"value": b.num_seqs / (res["separate"] * 1e-3),
                                "ms_per_step": res["separate"],
                                "h2d_bytes_per_step": int(sum(v.numel() * v.element_size()
                                                              for v in h.values()))}}


def long_context_arm(args, device, flush, pa):
    """Split-KV decode on the long-context batch: 8 seqs x 32k..128k tokens,
    64 query / 8 KV heads x 128 bf16, 512-token partitions."""
    b = wl.long_context(device=device, canary=False)
    bt, sl, _ = b.torch_tables(device)
    msl = 131072
    ws = torch.empty(pa.pa_decode_partitioned_workspace_size(b.num_seqs, b.num_heads,
                                                             b.head_dim, msl, 512),
                     dtype=torch.uint8, device=device)
    out = torch.empty_like(b.q)

    def call():
        pa.pa_decode_partitioned(out, b.q, b.k_cache, b.v_cache, bt, sl, b.scale,
                                 b.num_kv_heads, 512, msl, ws)
    for _ in range(3):
        call()
    ms = time_calls(call, 20, flush, torch.cuda.current_stream())
    nb = decode_bytes(b)
    t = statistics.mean(ms) * 1e-3
    peak, kind = measured_peak()
    del b, ws
    torch.cuda.empty_cache()
    return {"workload": "long_context: batch 8, 64/8 x 128 bf16, seq_lens U[32768,131072], "
                        "1% keys x8, 512-token partitions (pa_decode_partitioned + merge)",
            "seqs_per_s": 8 / t, "us_per_call": t * 1e6, "kv_gbs": nb["kv"] / t / 1e9,
            "achieved_gbs": nb["total"] / t / 1e9, "frac_of_peak": nb["total"] / t / 1e9 / peak,
            "peak_kind": kind, "bytes": nb}


def shared_prefix_unique_bytes(b) -> int:
    """decode_bytes' total with the shared prefix's K/V counted once instead
    of once per sequence (every sequence's table starts with the same
    prefix_tokens / 16 physical blocks)."""
    es = torch.tensor([], dtype=wl.DTYPES[b.dtype]).element_size()
    per_tok = 2 * b.num_kv_heads * b.head_dim * es
    prefix = int(b.meta["prefix_tokens"])
    return decode_bytes(b)["total"] - (b.num_seqs - 1) * prefix * per_tok


def shared_prefix_arm(args, device, flush, pa):
    """pa_decode on the shared-prefix batch: 128 seqs whose tables start with
    the same 128 physical blocks (a 2048-token prefix), then 64..512 private
    tokens.  Logical bytes count every sequence's prefix; unique bytes count
    the prefix blocks once (the rest of a sequence's reads of them can hit
    L2).  No roofline gate: the logical rate may exceed HBM."""
    b = wl.shared_prefix(device=device, canary=False)
    bt, sl, _ = b.torch_tables(device)
    out = torch.empty_like(b.q)

    def call():
        pa.pa_decode(out, b.q, b.k_cache, b.v_cache, bt, sl, b.scale, b.num_kv_heads)
    for _ in range(3):
        call()
    ms = time_calls(call, 30, flush, torch.cuda.current_stream())
    # the same batch through the cascade entry point: the prefix blocks once,
    # each sequence's own table beside them
    P = int(b.meta["prefix_tokens"]) // 16
    prefix, own_tab, own_len = wl.cascade_split(b, P)
    pt = torch.from_numpy(prefix).to(device)
    ot = torch.from_numpy(own_tab).to(device)
    ol = torch.from_numpy(own_len).to(device)
    ws = torch.empty(pa.pa_decode_cascade_workspace_size(b.num_seqs, b.num_heads, b.head_dim, P,
                                                         own_tab.shape[1]),
                     dtype=torch.uint8, device=device)
    out_c = torch.empty_like(b.q)

    def call_c():
        pa.pa_decode_cascade(out_c, b.q, b.k_cache, b.v_cache, pt, ot, ol, b.scale,
                             b.num_kv_heads, ws)
    for _ in range(3):
        call_c()
    ms_c = time_calls(call_c, 30, flush, torch.cuda.current_stream())
    nb = decode_bytes(b)
    unique = shared_prefix_unique_bytes(b)
    t = statistics.median(ms) * 1e-3
    tc = statistics.median(ms_c) * 1e-3
    peak, kind = measured_peak()
    del b, ws
    torch.cuda.empty_cache()
    return {"workload": "shared_prefix: batch 128, 32/8 x 128 bf16, a 2048-token prefix in 128 "
                        "shared physical blocks + U[64,512] private tokens",
            "us_per_call": t * 1e6, "logical_gbs": nb["total"] / t / 1e9,
            "unique_gbs": unique / t / 1e9, "unique_frac_of_peak": unique / t / 1e9 / peak,
            "cascade": {"call": "pa_decode_cascade (prefix blocks once + own tables)",
                        "us_per_call": tc * 1e6, "unique_gbs": unique / tc / 1e9,
                        "unique_frac_of_peak": unique / tc / 1e9 / peak,
                        "speedup_over_pa_decode": t / tc},
            "peak_kind": kind, "bytes": {"logical": nb["total"], "unique": unique}}


def multi_query_arm(args, device, flush, pa):
    """pa_decode_multi on a speculative-verification step (256 seqs x 4 query
    rows, serving-mix lengths) and a chunked-prefill step (4 x 512-token
    chunks beside 124 one-token decodes)."""
    peak, kind = measured_peak()
    res = {}
    for name, make in (("spec_verify", wl.spec_verify), ("chunked_prefill", wl.chunked_prefill_mix)):
        b = make(device=device, canary=False)
        bt, sl, _ = b.torch_tables(device)
        qs = torch.from_numpy(b.meta["query_start"]).to(device)
        mq = int(np.diff(b.meta["query_start"]).max())
        out = torch.empty_like(b.q)

        def call():
            pa.pa_decode_multi(out, b.q, b.k_cache, b.v_cache, bt, sl, qs, mq, b.scale,
                               b.num_kv_heads)
        for _ in range(5):
            call()
        ms = time_calls(call, 40, flush, torch.cuda.current_stream())
        t = statistics.mean(ms) * 1e-3
        nb = multi_bytes(b)
        res[name] = {"workload": make.__doc__.split("\n\n")[0].replace("\n", " "),
                     "us_per_call": t * 1e6, "us_per_call_median": statistics.median(ms) * 1e3,
                     "calls": len(ms), "rows_per_s": nb["rows"] / t,
                     "kv_gbs": nb["kv"] / t / 1e9,
                     "achieved_gbs": nb["total"] / t / 1e9,
                     "frac_of_peak": nb["total"] / t / 1e9 / peak, "peak_kind": kind,
                     "attn_tflops": nb["flops"] / t / 1e12, "bytes": nb}
        del b, out
        torch.cuda.empty_cache()
    return res


def fp8_arm(args, device, flush, pa):
    """E4M3 caches: the serving-mix step (FP8 cache write of 256 tokens +
    pa_decode_fp8) and the long-context split-KV decode over E4M3."""
    peak, kind = measured_peak()
    res = {}
    b = wl.serving_mix_fp8(device=device, canary=False)
    bt, sl, sm = b.torch_tables(device)
    ks, vs = b.meta["k_scale"], b.meta["v_scale"]
    out = torch.empty_like(b.q)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(30)]
    for _ in range(3):
        pa.pa_reshape_and_cache_fp8(b.k_new, b.v_new, b.k_cache, b.v_cache, ks, vs, sm)
        pa.pa_decode_fp8(out, b.q, b.k_cache, b.v_cache, ks, vs, bt, sl, b.scale, b.num_kv_heads)
    stream = torch.cuda.current_stream()
    for e0, e1, e2 in ev:
        flush()
        e0.record(stream)
        pa.pa_reshape_and_cache_fp8(b.k_new, b.v_new, b.k_cache, b.v_cache, ks, vs, sm)
        e1.record(stream)
        pa.pa_decode_fp8(out, b.q, b.k_cache, b.v_cache, ks, vs, bt, sl, b.scale, b.num_kv_heads)
        e2.record(stream)
    torch.cuda.synchronize()
    dec = statistics.mean(e1.elapsed_time(e2) for _, e1, e2 in ev) * 1e-3
    wr = statistics.mean(e0.elapsed_time(e1) for e0, e1, _ in ev) * 1e-3
    step = statistics.mean(e0.elapsed_time(e2) for e0, _, e2 in ev) * 1e-3
    nb = decode_bytes(b)
    res["serving_mix_fp8"] = {
        "workload": "serving_mix over an E4M3 cache (per-KV-head scales): step = "
                    "pa_reshape_and_cache_fp8 of 256 tokens + pa_decode_fp8",
        "seqs_per_s": b.num_seqs / step, "step_us": step * 1e6, "decode_us": dec * 1e6,
        "cache_write_us": wr * 1e6, "kv_gbs": nb["kv"] / dec / 1e9,
        "achieved_gbs": nb["total"] / dec / 1e9, "frac_of_peak": nb["total"] / dec / 1e9 / peak,
        "peak_kind": kind, "bytes": nb}
    del b, out
    torch.cuda.empty_cache()

    b = wl.long_context_fp8(device=device, canary=False)
    bt, sl, _ = b.torch_tables(device)
    ks, vs = b.meta["k_scale"], b.meta["v_scale"]
    msl = 131072
    ws = torch.empty(pa.pa_decode_partitioned_workspace_size(b.num_seqs, b.num_heads,
                                                             b.head_dim, msl, 512),
                     dtype=torch.uint8, device=device)
    out = torch.empty_like(b.q)

    def call():
        pa.pa_decode_partitioned_fp8(out, b.q, b.k_cache, b.v_cache, ks, vs, bt, sl, b.scale,
                                     b.num_kv_heads, 512, msl, ws)
    for _ in range(3):
        call()
    t = statistics.mean(time_calls(call, 20, flush, stream)) * 1e-3
    nb = decode_bytes(b)
    res["long_context_fp8"] = {
        "workload": "long_context over an E4M3 cache: batch 8, 64/8 x 128, seq_lens "
                    "U[32768,131072], 512-token partitions (pa_decode_partitioned_fp8 + merge)",
        "seqs_per_s": b.num_seqs / t, "us_per_call": t * 1e6, "kv_gbs": nb["kv"] / t / 1e9,
        "achieved_gbs": nb["total"] / t / 1e9, "frac_of_peak": nb["total"] / t / 1e9 / peak,
        "peak_kind": kind, "bytes": nb}
    del b, ws, out
    torch.cuda.empty_cache()
    return res


def copy_blocks_arm(args, device, flush, pa):
    """Copy-on-write copies of one step: 256 (src, dst) pairs in K and V of
    32 Llama-3-8B-shaped layers (32 KiB blocks), one pa_copy_blocks call."""
    peak, kind = measured_peak()
    w = wl.cow_step(device=device, layers=32, num_blocks=2048, pairs=256, fill=False)
    m = torch.from_numpy(w["mapping"]).to(device)

    def call():
        pa.pa_copy_blocks(w["caches"], m)
    for _ in range(3):
        call()
    t = statistics.mean(time_calls(call, 30, flush, torch.cuda.current_stream())) * 1e-3
    moved = 2 * len(w["caches"]) * w["mapping"].shape[0] * w["block_bytes"]   # read + write
    del w, m
    torch.cuda.empty_cache()
    return {"workload": "cow_step: 256 block copies x K,V of 32 layers (bf16 8 x 16 x 128 "
                        "blocks, 32 KiB), one call",
            "us_per_call": t * 1e6, "bytes_read_plus_written": moved,
            "achieved_gbs": moved / t / 1e9, "frac_of_peak": moved / t / 1e9 / peak,
            "peak_kind": kind}


def block_manager_arm(args):
    """Host-side cost of the native block manager (no GPU work): the serving
    loop over 256 serving-mix requests with 64 new tokens each in a pool of
    60 % of their final size (so requests get preempted), and prefix-cached
    admissions of 2000-token chats sharing a 1500-token system prompt."""
    from paged_kv_cache_151_gb300 import blocks
    rng = np.random.default_rng(21)
    lens = wl.lognormal_lengths(rng, 256, hi=4096)
    new = 64
    pool = int(0.6 * sum(-(-(int(L) + new) // 16) for L in lens))
    loop = blocks.ServingLoop(blocks.BlockManager(pool, 16))
    for i, L in enumerate(lens):
        loop.submit(i, int(L), new)
    steps, tokens, preempts = 0, 0, 0
    t0 = time.perf_counter()
    more = True
    while more:
        more, steps, ev, wr = loop.step()
        tokens += len(wr)
        preempts += sum(e[1] == "preempt" for e in ev)
    t_loop = time.perf_counter() - t0
    bm = blocks.BlockManager(40000, 16, prefix_caching=True)
    system = np.arange(1500, dtype=np.int32)
    n_chats = 2000
    t0 = time.perf_counter()
    hits = 0
    for i in range(n_chats):
        toks = np.concatenate([system, np.arange(10**6 + 500 * i, 10**6 + 500 * (i + 1),
                                                 dtype=np.int32)])
        hits += bm.add_sequence(i, toks) or 0
        if i >= 16:
            bm.free_sequence(i - 16)
    t_add = time.perf_counter() - t0
    return {"workload": "serving loop: 256 serving-mix requests x 64 new tokens, pool 60% of "
                        f"their final blocks ({pool}); prefix cache: {n_chats} 2000-token chats "
                        "sharing a 1500-token prompt (16 live at a time)",
            "loop_steps": steps, "loop_tokens": tokens, "loop_preemptions": preempts,
            "loop_us_per_step": t_loop / max(steps, 1) * 1e6,
            "loop_tokens_per_s": tokens / t_loop,
            "prefix_adds_per_s": n_chats / t_add,
            "prefix_cached_tokens_per_add": hits / n_chats,
            "includes": "ctypes call overhead per operation"}


def paging_overhead_arm(args, device, flush, pa):
    """Decode time with a random block table over the same time with the
    same data in contiguous blocks (an identity table), batch 64 x 512..2048."""
    b = wl.llama8b_uniform(device=device, canary=False)
    nbk = [math.ceil(int(L) / 16) for L in b.seq_lens]
    ident = np.full_like(b.block_tables, wl.PAD)
    kc = torch.zeros_like(b.k_cache)
    vc = torch.zeros_like(b.v_cache)
    nxt = 0
    for s, n in enumerate(nbk):
        src = torch.from_numpy(b.block_tables[s, :n].astype(np.int64)).to(device)
        kc[nxt:nxt + n] = b.k_cache[src]
        vc[nxt:nxt + n] = b.v_cache[src]
        ident[s, :n] = np.arange(nxt, nxt + n)
        nxt += n
    out = torch.empty_like(b.q)
    sl = torch.from_numpy(b.seq_lens).to(device)
    bt_r = torch.from_numpy(b.block_tables).to(device)
    bt_i = torch.from_numpy(ident).to(device)
    res = {}
    for name, (bt, k, v) in {"random": (bt_r, b.k_cache, b.v_cache),
                             "identity": (bt_i, kc, vc)}.items():
        def call(bt=bt, k=k, v=v):
            pa.pa_decode(out, b.q, k, v, bt, sl, b.scale, b.num_kv_heads)
        for _ in range(3):
            call()
        res[name] = statistics.median(time_calls(call, 30, flush, torch.cuda.current_stream()))
    del b, kc, vc
    torch.cuda.empty_cache()
    return {"workload": "llama8b_uniform: batch 64, 32/8 x 128 bf16, seq_lens U[512,2048]",
            "random_table_us": res["random"] * 1e3, "identity_table_us": res["identity"] * 1e3,
            "overhead": res["random"] / res["identity"] - 1.0}


# ---------------------------------------------------------------------------
# the oracle on the host cores (CPU baseline / reference arm)
# ---------------------------------------------------------------------------

def oracle_step(b, threads: int):
    """One step of the hot path on the oracle: the cache write of the batch's
    new tokens, then decode of every (sequence, head) over the written
    caches, on `threads` host threads.  Returns the step's wall time (s)."""
    import oracle
    t0 = time.perf_counter()
    kc, vc, _ = oracle.reshape_and_cache(b.k_new, b.v_new, b.k_cache, b.v_cache,
                                         b.slot_mapping, b.dtype)
    oracle.decode(b.q, kc, vc, b.block_tables, b.seq_lens, b.scale, b.num_kv_heads,
                  b.dtype, nthreads=threads)
    return time.perf_counter() - t0


def host_serving_mix():
    """The serving-mix batch built on the host: the same seeded structure
    (lengths, tables, pool size) as the GPU arm's; values from the host's
    generator."""
    return wl.serving_mix(device="cpu", canary=False)


def cpu_baseline(budget_s: float):
    """The oracle on the host cores over the whole serving-mix batch: whole
    steps (cache write + decode of all 256 sequences) repeated for about
    `budget_s` seconds on all cores, and one whole step on one thread."""
    import oracle
    oracle.build()
    b = host_serving_mix()
    cores = os.cpu_count() or 1
    oracle_step(b, cores)                                  # first touch of the buffers
    times = []
    while sum(times) < budget_s or len(times) < 2:
        times.append(oracle_step(b, cores))
    t1 = oracle_step(b, 1)
    t = statistics.mean(times)
    return {"value": b.num_seqs / t, "unit": "seqs/s", "cores": cores, "kind": "oracle",
            "sample": f"the whole serving-mix batch ({b.num_seqs} sequences, "
                      f"{int(b.seq_lens.sum())} tokens): {len(times)} steps of fp64 cache "
                      f"write + decode with {cores} threads, {statistics.mean(times):.2f} s "
                      f"per step, no scaling",
            "ms_per_step": t * 1e3,
            "single_thread_value": b.num_seqs / t1,
            "single_thread_sample": f"one whole step on one thread ({t1:.2f} s)"}


def reference_arm(args):
    """The oracle as the reference implementation, on the host cores.  Each
    step is the whole serving-mix step: the cache write of 256 tokens, then
    decode of all 256 sequences, in fp64 on all host cores; nothing is
    sampled or scaled."""
    import oracle
    oracle.build()
    cores = os.cpu_count() or 1
    b = host_serving_mix()
    for _ in range(args.warmup):
        oracle_step(b, cores)
    times = [oracle_step(b, cores) for _ in range(args.steps)]
    t_step = statistics.mean(times)
    value = b.num_seqs / t_step
    sample = (f"the whole serving-mix batch every step ({b.num_seqs} sequences, "
              f"{int(b.seq_lens.sum())} tokens): fp64 oracle cache write + decode with "
              f"{cores} threads, {args.steps} timed steps after {args.warmup} warm-up")
    return {
        "impl": "reference",
        "metric": METRIC, "value": value, "unit": "seqs/s", "n_gpus": 0,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_step * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded; no dataset)",
        "config": bench_config(b, 1),
        "cpu_baseline": {"value": value, "unit": "seqs/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "seqs/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


# ---------------------------------------------------------------------------

def single_kernel(args, device):
    """Launch one kernel alone (for profilers): warm-up, then --steps launches
    timed with CUDA events, L2 flushed before each.  Prints a short JSON line
    (not a benchmark line)."""
    from paged_kv_cache_151_gb300 import pa
    torch.cuda.set_device(device)
    pa.load()
    flush, _ = make_flush(device)
    if args.only == "shared_prefix":
        b = wl.shared_prefix(device=device, canary=False)
        bt, sl, _ = b.torch_tables(device)
        out = torch.empty_like(b.q)

        def call():
            pa.pa_decode(out, b.q, b.k_cache, b.v_cache, bt, sl, b.scale, b.num_kv_heads)
    elif args.only == "cascade":
        b = wl.shared_prefix(device=device, canary=False)
        P = int(b.meta["prefix_tokens"]) // 16
        prefix, own_tab, own_len = wl.cascade_split(b, P)
        pt = torch.from_numpy(prefix).to(device)
        ot = torch.from_numpy(own_tab).to(device)
        ol = torch.from_numpy(own_len).to(device)
        ws = torch.empty(pa.pa_decode_cascade_workspace_size(
            b.num_seqs, b.num_heads, b.head_dim, P, own_tab.shape[1]), dtype=torch.uint8,
            device=device)
        out = torch.empty_like(b.q)

        def call():
            pa.pa_decode_cascade(out, b.q, b.k_cache, b.v_cache, pt, ot, ol, b.scale,
                                 b.num_kv_heads, ws)
    elif args.only == "partitioned":
        b = wl.long_context(device=device, canary=False)
        bt, sl, _ = b.torch_tables(device)
        msl = 131072
        ws = torch.empty(pa.pa_decode_partitioned_workspace_size(
            b.num_seqs, b.num_heads, b.head_dim, msl, 512), dtype=torch.uint8, device=device)
        out = torch.empty_like(b.q)

        def call():
            pa.pa_decode_partitioned(out, b.q, b.k_cache, b.v_cache, bt, sl, b.scale,
                                     b.num_kv_heads, 512, msl, ws)
    elif args.only in ("decode_fp8", "cache_write_fp8"):
        b = wl.serving_mix_fp8(device=device, canary=False)
        bt, sl, sm = b.torch_tables(device)
        ks, vs = b.meta["k_scale"], b.meta["v_scale"]
        out = torch.empty_like(b.q)
        if args.only == "decode_fp8":
            def call():
                pa.pa_decode_fp8(out, b.q, b.k_cache, b.v_cache, ks, vs, bt, sl, b.scale,
                                 b.num_kv_heads)
        else:
            def call():
                pa.pa_reshape_and_cache_fp8(b.k_new, b.v_new, b.k_cache, b.v_cache, ks, vs, sm)
    elif args.only == "partitioned_fp8":
        b = wl.long_context_fp8(device=device, canary=False)
        bt, sl, _ = b.torch_tables(device)
        ks, vs = b.meta["k_scale"], b.meta["v_scale"]
        msl = 131072
        ws = torch.empty(pa.pa_decode_partitioned_workspace_size(
            b.num_seqs, b.num_heads, b.head_dim, msl, 512), dtype=torch.uint8, device=device)
        out = torch.empty_like(b.q)

        def call():
            pa.pa_decode_partitioned_fp8(out, b.q, b.k_cache, b.v_cache, ks, vs, bt, sl,
                                         b.scale, b.num_kv_heads, 512, msl, ws)
    elif args.only == "copy_blocks":
        w = wl.cow_step(device=device, layers=32, num_blocks=2048, pairs=256, fill=False)
        m = torch.from_numpy(w["mapping"]).to(device)
        b = wl.serving_mix(device="cpu", canary=False)     # byte accounting only

        def call():
            pa.pa_copy_blocks(w["caches"], m)
    elif args.only in ("multi_spec", "multi_prefill"):
        b = (wl.spec_verify if args.only == "multi_spec" else wl.chunked_prefill_mix)(
            device=device, canary=False)
        bt, sl, _ = b.torch_tables(device)
        qs = torch.from_numpy(b.meta["query_start"]).to(device)
        mq = int(np.diff(b.meta["query_start"]).max())
        out = torch.empty_like(b.q)

        def call():
            pa.pa_decode_multi(out, b.q, b.k_cache, b.v_cache, bt, sl, qs, mq, b.scale,
                               b.num_kv_heads)
    else:
        b = wl.serving_mix(device=device, canary=False)
        bt, sl, sm = b.torch_tables(device)
        out = torch.empty_like(b.q)
        if args.only == "decode":
            def call():
                pa.pa_decode(out, b.q, b.k_cache, b.v_cache, bt, sl, b.scale, b.num_kv_heads)
        else:
            def call():
                pa.pa_reshape_and_cache(b.k_new, b.v_new, b.k_cache, b.v_cache, sm)
    for _ in range(args.warmup):
        flush()
        call()
    torch.cuda.synchronize()
    ms = time_calls(call, args.steps, flush, torch.cuda.current_stream())
    nb = multi_bytes(b) if args.only.startswith("multi") else decode_bytes(b)
    print(json.dumps({"only": args.only, "workload": b.name, "us": [m * 1e3 for m in ms],
                      "bytes": nb, "device_error_flags": pa.pa_device_error(clear=True)}))


def main():
    ap = argparse.ArgumentParser(description=__doc__,
                                 formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--cpu-budget", type=float, default=10.0,
                    help="seconds of oracle work for the CPU baseline")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the long-context, paging-overhead, multi-query, FP8 and "
                         "copy-on-write measurements")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", choices=["decode", "shared_prefix", "cascade", "partitioned",
                                       "cache_write",
                                       "multi_spec", "multi_prefill", "decode_fp8",
                                       "cache_write_fp8", "partitioned_fp8", "copy_blocks"],
                    help="launch one kernel alone (for profiling); prints timings only")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(reference_arm(args)), flush=True)
        return

    if args.only:
        single_kernel(args, torch.device("cuda", local))
        return

    if world > 1:
        torch.distributed.init_process_group(
            backend="nccl" if torch.cuda.is_available() else "gloo")
    device = torch.device("cuda", local)
    result, _ = gpu_arm(args, rank, world, device)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(args.cpu_budget)
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
