"""Copy-on-write block copies (pa_copy_blocks) through the C ABI: byte for
byte against the oracle, and a fork-then-diverge step end to end."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_151_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clean_error_word(cuda_lib):
    cuda_lib.pa_device_error(clear=True)
    yield
    flags = cuda_lib.pa_device_error(clear=True)
    assert flags == 0, f"device error word set: {flags:#x}"


def as_bytes(t):
    return t.contiguous().view(torch.uint8).cpu().numpy()


def run_and_compare(pa, caches, mapping, expect_bad=0):
    before = [c.clone() for c in caches]
    m = torch.from_numpy(np.ascontiguousarray(mapping, np.int64)).cuda()
    pa.pa_copy_blocks(caches, m)
    torch.cuda.synchronize()
    ref, bad = oracle.copy_blocks([c.cpu() for c in before], mapping)
    assert bad == expect_bad
    for c, r in zip(caches, ref):
        assert np.array_equal(as_bytes(c), r.reshape(-1).view(np.uint8).reshape(as_bytes(c).shape))


@pytest.mark.parametrize("layers,Hkv,D,dtype", [
    (1, 8, 128, torch.bfloat16),        # 32 KiB blocks: two 16 KiB pieces
    (3, 1, 64, torch.float16),          # 2 KiB blocks
    (2, 5, 128, torch.bfloat16),        # 20 KiB: one full piece and a ragged one
    (2, 4, 128, torch.uint8),           # E4M3 cache, 8 KiB blocks
    (1, 2, 64, torch.float32),
])
def test_copy_blocks_bit_exact(cuda_lib, layers, Hkv, D, dtype):
    N = 300
    g = torch.Generator(device="cuda")
    g.manual_seed(layers * 100 + Hkv * 10 + D)
    caches = []
    for _ in range(2 * layers):
        if dtype == torch.uint8:
            caches.append(torch.randint(0, 256, (N, Hkv, 16, D), generator=g, device="cuda",
                                        dtype=torch.uint8))
        else:
            caches.append(torch.randn((N, Hkv, 16, D), generator=g, device="cuda").to(dtype))
    run_and_compare(cuda_lib, caches, wl.cow_mapping(N, 97, seed=D + Hkv))


def test_copy_blocks_bad_pairs_are_skipped_and_flagged(cuda_lib):
    N = 40
    caches = [torch.randn((N, 2, 16, 64), device="cuda").to(torch.bfloat16) for _ in range(2)]
    m = wl.cow_mapping(N, 10, seed=3)
    m[2, 0] = N + 7
    m[5, 1] = -3
    run_and_compare(cuda_lib, caches, m, expect_bad=2)
    assert cuda_lib.pa_device_error(clear=True) == cuda_lib.PA_DEVERR_BLOCK_ID


def test_copy_blocks_empty_mapping_and_same_block(cuda_lib):
    caches = [torch.randn((8, 2, 16, 64), device="cuda") for _ in range(2)]
    before = [c.clone() for c in caches]
    cuda_lib.pa_copy_blocks(caches, torch.zeros((0, 2), dtype=torch.int64, device="cuda"))
    cuda_lib.pa_copy_blocks(caches, torch.tensor([[3, 3]], dtype=torch.int64, device="cuda"))
    torch.cuda.synchronize()
    assert all(torch.equal(a, b) for a, b in zip(caches, before))


def test_fork_copy_then_diverge_step(cuda_lib):
    """Parent and child share every block; the child's next token goes into a
    copy of the shared last block (copy_blocks), then each sequence writes its
    own token (reshape_and_cache) and decodes.  The parent reads exactly what
    it read before the child diverged; both match the oracle."""
    b = wl.random_batch(800, num_seqs=4, max_len=60, min_len=17, num_heads=32,
                        num_kv_heads=8, head_dim=128, dtype="bf16", device="cuda",
                        keep_seq=False, extra_blocks=8)
    # children: one per parent, sharing the parent's table up to its context
    bt = b.block_tables.copy()
    used = set(bt[bt != wl.PAD].tolist())
    fresh = [x for x in range(b.num_blocks) if x not in used]
    ctx = b.ctx_lens.astype(np.int64)
    pairs, child_tabs = [], []
    for s in range(b.num_seqs):
        lb = int(ctx[s]) // 16                     # block receiving the new token
        tab = bt[s].copy()
        if int(ctx[s]) % 16:                        # partly filled, shared: copy on write
            pairs.append([int(bt[s, lb]), fresh[0]])
            tab[lb] = fresh.pop(0)
        else:                                       # the new token opens a fresh block
            tab[lb] = fresh.pop(0)
        child_tabs.append(tab)
    mapping = np.array(pairs, np.int64).reshape(-1, 2)
    kc, vc = b.k_cache.clone(), b.v_cache.clone()
    cuda_lib.pa_copy_blocks([kc, vc], torch.from_numpy(mapping).cuda())
    # both write their token: parent at its slot, child at the same row of its block
    child_slots = np.array([child_tabs[s][int(ctx[s]) // 16] * 16 + int(ctx[s]) % 16
                            for s in range(b.num_seqs)], np.int64)
    k_child = torch.randn_like(b.k_new)
    v_child = torch.randn_like(b.v_new)
    k_all = torch.cat([b.k_new, k_child]).contiguous()
    v_all = torch.cat([b.v_new, v_child]).contiguous()
    slots = np.concatenate([b.slot_mapping, child_slots])
    cuda_lib.pa_reshape_and_cache(k_all, v_all, kc, vc, torch.from_numpy(slots).cuda())
    tables = np.concatenate([bt, np.stack(child_tabs)]).astype(np.int32)
    lens = np.concatenate([b.seq_lens, b.seq_lens]).astype(np.int32)
    q = torch.cat([b.q, b.q]).contiguous()
    out = torch.empty_like(q)
    cuda_lib.pa_decode(out, q, kc, vc, torch.from_numpy(tables).cuda(),
                       torch.from_numpy(lens).cuda(), b.scale, b.num_kv_heads)
    torch.cuda.synchronize()
    # oracle: copies, then the writes, then decode
    (rk, rv), bad = oracle.copy_blocks([b.k_cache.cpu(), b.v_cache.cpu()], mapping)
    assert bad == 0
    rk, rv, bad = oracle.reshape_and_cache(k_all.cpu(), v_all.cpu(), rk, rv, slots, "bf16")
    assert bad == 0
    assert np.array_equal(as_bytes(kc), rk.view(np.uint8).reshape(as_bytes(kc).shape))
    ref = oracle.decode(q.cpu(), rk, rv, tables, lens, b.scale, b.num_kv_heads, "bf16")
    g = out.double().cpu().numpy()
    assert np.abs(g - ref).max() <= 2e-2
    assert np.linalg.norm(g - ref) / np.linalg.norm(ref) <= 5e-3
    # the parent's blocks hold exactly what the parent alone would have written
    kp, vp = b.k_cache.clone(), b.v_cache.clone()
    cuda_lib.pa_reshape_and_cache(b.k_new, b.v_new, kp, vp,
                                  torch.from_numpy(b.slot_mapping).cuda())
    torch.cuda.synchronize()
    own = torch.from_numpy(np.unique(bt[bt != wl.PAD]).astype(np.int64)).cuda()
    assert torch.equal(kc[own].view(torch.int16), kp[own].view(torch.int16))
    assert torch.equal(vc[own].view(torch.int16), vp[own].view(torch.int16))


@pytest.mark.slow
def test_full_cow_step_all_layers(cuda_lib):
    """The measured workload: 256 copies in K and V of 32 layers."""
    w = wl.cow_step(device="cuda", layers=32, num_blocks=2048, pairs=256)
    before = [c[torch.from_numpy(w["mapping"][:, 0]).cuda()].clone() for c in w["caches"]]
    cuda_lib.pa_copy_blocks(w["caches"], torch.from_numpy(w["mapping"]).cuda())
    torch.cuda.synchronize()
    dst = torch.from_numpy(w["mapping"][:, 1]).cuda()
    for c, src_before in zip(w["caches"], before):
        assert torch.equal(c[dst].view(torch.int16), src_before.view(torch.int16))
