"""Multi-step traces: the native block manager and serving loop drive the GPU
path (cache write, copy-on-write copies, decode) step by step, and every
decode is checked against the oracle's attention over the same tokens laid
out contiguously -- so a wrong slot, table or copy anywhere in the host
bookkeeping shows up as wrong attention."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_151_gb300 import blocks

pytestmark = pytest.mark.gpu

H, HKV, D, BS = 8, 2, 64, 16
SCALE = 1.0 / np.sqrt(D)


@pytest.fixture(autouse=True)
def _clean_error_word(cuda_lib):
    cuda_lib.pa_device_error(clear=True)
    yield
    flags = cuda_lib.pa_device_error(clear=True)
    assert flags == 0, f"device error word set: {flags:#x}"


class Tokens:
    """Deterministic K, V and q of every (request, position)."""

    def __init__(self, rid, length, seed):
        g = torch.Generator(device="cuda")
        g.manual_seed(seed * 1000 + rid)
        self.k = (torch.randn((length, HKV, D), generator=g, device="cuda") * 0.5).to(torch.bfloat16)
        self.v = (torch.randn((length, HKV, D), generator=g, device="cuda") * 0.5).to(torch.bfloat16)
        self.q = torch.randn((length, H, D), generator=g, device="cuda").to(torch.bfloat16)

    def host(self):
        return self.k.cpu(), self.v.cpu(), self.q.cpu()


def contiguous_reference(toks, lens):
    """The oracle on a pool holding each sequence contiguously."""
    nbs = [-(-L // BS) for L in lens]
    width = max(nbs)
    kc = torch.zeros((sum(nbs), HKV, BS, D), dtype=torch.bfloat16)
    vc = torch.zeros_like(kc)
    tables = np.zeros((len(lens), width), np.int32)
    q = torch.zeros((len(lens), H, D), dtype=torch.bfloat16)
    base = 0
    for i, (t, L) in enumerate(zip(toks, lens)):
        k, v, qq = t.host()
        n = nbs[i]
        for cache, src in ((kc, k), (vc, v)):
            pad = torch.zeros((n * BS, HKV, D), dtype=torch.bfloat16)
            pad[:L] = src[:L]
            cache[base:base + n] = pad.view(n, BS, HKV, D).transpose(1, 2)
        tables[i, :n] = np.arange(base, base + n)
        q[i] = qq[L - 1]
        base += n
    return oracle.decode(q, kc, vc, tables, np.array(lens, np.int32), SCALE, HKV, "bf16")


def assert_close(out, ref, what):
    g = out.double().cpu().numpy()
    assert np.isfinite(g).all(), what
    assert np.abs(g - ref).max() <= 2e-2, what
    assert np.linalg.norm(g - ref) / np.linalg.norm(ref) <= 5e-3, what


def write(pa, kc, vc, rows_k, rows_v, slots):
    if not slots:
        return
    pa.pa_reshape_and_cache(torch.stack(rows_k).contiguous(), torch.stack(rows_v).contiguous(),
                            kc, vc, torch.tensor(slots, dtype=torch.int64, device="cuda"))


def decode(pa, bm, kc, vc, ids, toks, width):
    tables, lens = bm.batch(ids, width)
    q = torch.stack([toks[i].q[int(L) - 1] for i, L in zip(ids, lens)]).contiguous()
    out = torch.empty_like(q)
    pa.pa_decode(out, q, kc, vc, torch.from_numpy(tables).cuda(),
                 torch.from_numpy(lens).cuda(), SCALE, HKV)
    torch.cuda.synchronize()
    return out, lens


@pytest.mark.parametrize("seed,pool,n_req", [(1, 24, 6), (2, 40, 12), (3, 16, 5)])
def test_serving_loop_trace_on_the_gpu(cuda_lib, seed, pool, n_req):
    """The serving loop with preemption: admitted requests prefill their
    tokens, every running request writes one token per step, and each step's
    decode equals attention over the request's own tokens."""
    rng = np.random.default_rng(seed)
    reqs = []
    for i in range(n_req):
        tokens, new = int(rng.integers(1, 70)), int(rng.integers(1, 50))
        if -(-(tokens + new) // BS) <= pool:
            reqs.append((i, tokens, new))
    toks = {i: Tokens(i, t + n, seed) for i, t, n in reqs}
    bm = blocks.BlockManager(pool, BS, free_order=rng.permutation(pool))
    loop = blocks.ServingLoop(bm)
    for r in reqs:
        loop.submit(*r)
    kc = torch.full((pool, HKV, BS, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    vc = torch.full_like(kc, float("nan"))
    width = -(-max(t + n for _, t, n in reqs) // BS)
    more, checked, preempts = True, 0, 0
    while more:
        more, step, events, written = loop.step()
        preempts += sum(e[1] == "preempt" for e in events)
        alive = [e[2] for e in events if e[1] == "admit"]
        live = set()
        for i, _ in written:
            try:
                bm.seq_len(i)
                live.add(i)
            except KeyError:
                pass                              # finished or preempted this step
        rows_k, rows_v, slots = [], [], []
        # prefill of requests admitted in this iteration and still running
        for i in alive:
            if i not in live:
                continue
            table = bm.table(i)
            L = bm.seq_len(i) - 1                 # the tokens it was admitted with
            for p in range(L):
                rows_k.append(toks[i].k[p]); rows_v.append(toks[i].v[p])
                slots.append(table[p // BS] * BS + p % BS)
        # this step's token of every request still running
        for i, slot in written:
            if i in live:
                p = bm.seq_len(i) - 1
                rows_k.append(toks[i].k[p]); rows_v.append(toks[i].v[p])
                slots.append(slot)
        write(cuda_lib, kc, vc, rows_k, rows_v, slots)
        ids = [i for i, _ in written if i in live]
        if not ids:
            continue
        out, lens = decode(cuda_lib, bm, kc, vc, ids, toks, width)
        ref = contiguous_reference([toks[i] for i in ids], [int(L) for L in lens])
        assert_close(out, ref, f"step {step}")
        checked += len(ids)
    assert checked > 0


def test_parallel_sampling_with_copy_on_write_on_the_gpu(cuda_lib):
    """Four samples of one prompt share its blocks; each sample's first token
    lands in the shared partial block, so the manager moves it to a copy
    (executed by pa_copy_blocks) before the write.  Every sample then decodes
    its own continuation for several steps."""
    rng = np.random.default_rng(5)
    pool, prompt_len, n_samples, steps = 40, 37, 4, 30
    bm = blocks.BlockManager(pool, BS, free_order=rng.permutation(pool), prefix_caching=True)
    prompt = Tokens(0, prompt_len, 9)
    samples = {s: Tokens(100 + s, prompt_len + steps, 9) for s in range(n_samples)}
    for t in samples.values():                    # every sample starts with the prompt
        t.k[:prompt_len] = prompt.k
        t.v[:prompt_len] = prompt.v
    kc = torch.full((pool, HKV, BS, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    vc = torch.full_like(kc, float("nan"))
    assert bm.add_sequence(0, list(range(prompt_len))) == 0
    table = bm.table(0)
    write(cuda_lib, kc, vc, [prompt.k[p] for p in range(prompt_len)],
          [prompt.v[p] for p in range(prompt_len)],
          [table[p // BS] * BS + p % BS for p in range(prompt_len)])
    for s in range(1, n_samples):
        bm.fork(0, s)
    width = -(-(prompt_len + steps) // BS)
    copies_seen = 0
    for step in range(steps):
        copies, rows_k, rows_v, slots = [], [], [], []
        for s in range(n_samples):
            slot, copy = bm.append(s, 1000 * s + step)
            if copy is not None:
                copies.append(copy)
            p = bm.seq_len(s) - 1
            rows_k.append(samples[s].k[p]); rows_v.append(samples[s].v[p]); slots.append(slot)
        if copies:
            copies_seen += len(copies)
            cuda_lib.pa_copy_blocks([kc, vc], torch.tensor(copies, dtype=torch.int64,
                                                           device="cuda"))
        write(cuda_lib, kc, vc, rows_k, rows_v, slots)
        ids = list(range(n_samples))
        out, lens = decode(cuda_lib, bm, kc, vc, ids, samples, width)
        ref = contiguous_reference([samples[s] for s in ids], [int(L) for L in lens])
        assert_close(out, ref, f"step {step}")
    # samples 0..2 each copied the shared partial block; sample 3 kept the original
    assert copies_seen == n_samples - 1
    # the full prompt blocks stay shared by all four
    assert [bm.refcount(b) for b in bm.table(0)[:prompt_len // BS]] == [n_samples] * (prompt_len // BS)
