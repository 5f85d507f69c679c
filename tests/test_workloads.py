"""Host-side checks of the seeded input generators (no GPU, no oracle)."""
import math

import numpy as np
import torch

from paged_kv_cache_151_gb300 import workloads as wl


def _valid_rows(b):
    """(block, row) of every token a decode reads."""
    out = []
    for s in range(b.num_seqs):
        for t in range(int(b.seq_lens[s])):
            out.append((int(b.block_tables[s, t // 16]), t % 16))
    return out


def test_tiny_shape_and_tables():
    b = wl.tiny()
    assert list(b.ctx_lens) == [1, 7, 16, 33]
    assert list(b.seq_lens) == [2, 8, 17, 34]
    assert (b.num_heads, b.num_kv_heads, b.head_dim, b.num_blocks) == (8, 2, 64, 64)
    assert b.k_cache.shape == (64, 2, 16, 64) and b.k_cache.dtype == torch.float32
    # each table holds exactly the blocks needed for context + the new token
    for s, L in enumerate(b.ctx_lens):
        nb = math.ceil((int(L) + 1) / 16)
        assert (b.block_tables[s, :nb] != wl.PAD).all()
        assert (b.block_tables[s, nb:] == wl.PAD).all()
    used = b.block_tables[b.block_tables != wl.PAD]
    assert len(set(used.tolist())) == used.size          # no block handed out twice


def test_new_slot_follows_append_rule():
    """The new token at position L lands in a fresh block exactly when
    L % 16 == 0 ("vLLM: Architecture, PagedAttention & Internals",
    *The free list and the block table*, append_slot)."""
    b = wl.random_batch(3, num_seqs=40, max_len=70, num_heads=2, num_kv_heads=1,
                        head_dim=64, dtype="f32")
    for s in range(b.num_seqs):
        L = int(b.ctx_lens[s])
        blk, row = divmod(int(b.slot_mapping[s]), 16)
        assert row == L % 16
        assert blk == b.block_tables[s, L // 16]
        n_blocks = int((b.block_tables[s] != wl.PAD).sum())
        assert n_blocks == L // 16 + 1


def test_canaries_outside_context():
    b = wl.random_batch(4, num_seqs=6, max_len=50, num_heads=4, num_kv_heads=2,
                        head_dim=64, dtype="bf16")
    mask = torch.zeros(b.num_blocks, 16, dtype=torch.bool)
    for s in range(b.num_seqs):
        for t in range(int(b.ctx_lens[s])):
            mask[int(b.block_tables[s, t // 16]), t % 16] = True
    kc = b.k_cache.permute(0, 2, 1, 3)          # [N, 16, Hkv, D]
    assert not torch.isnan(kc[mask]).any()
    assert torch.isnan(kc[~mask]).all()          # new-token slots too, before the write


def test_new_in_pool_places_the_new_token():
    b = wl.random_batch(5, num_seqs=5, max_len=30, num_heads=4, num_kv_heads=2,
                        head_dim=64, dtype="f32", new_in_pool=True)
    for s in range(b.num_seqs):
        blk, row = divmod(int(b.slot_mapping[s]), 16)
        assert torch.equal(b.k_cache[blk, :, row], b.k_new[s])
        assert torch.equal(b.v_cache[blk, :, row], b.v_new[s])
        # and the contiguous ground truth agrees with the pool
        for t in range(int(b.seq_lens[s])):
            pb = int(b.block_tables[s, t // 16])
            assert torch.equal(b.k_cache[pb, :, t % 16], b.seq_k[s][t])


def test_permute_blocks_moves_data_with_tables():
    b = wl.random_batch(6, num_seqs=4, max_len=40, num_heads=2, num_kv_heads=2,
                        head_dim=64, dtype="f32", new_in_pool=True)
    p = wl.permute_blocks(b, seed=1)
    for s in range(b.num_seqs):
        for t in range(int(b.seq_lens[s])):
            a = b.k_cache[int(b.block_tables[s, t // 16]), :, t % 16]
            c = p.k_cache[int(p.block_tables[s, t // 16]), :, t % 16]
            assert torch.equal(a, c)
        assert p.slot_mapping[s] // 16 == p.block_tables[s, int(p.ctx_lens[s]) // 16]


def test_shared_prefix_structure():
    b = wl.shared_prefix(batch=6, prefix_blocks=4, lo=10, hi=30, keep_seq=True)
    assert (b.block_tables[:, :4] == b.block_tables[0, :4]).all()
    assert (b.seq_lens - 64 >= 10).all() and (b.seq_lens - 64 <= 30).all()
    tails = b.block_tables[:, 4:]
    t = tails[tails != wl.PAD]
    assert len(set(t.tolist())) == t.size
    assert not set(t.tolist()) & set(b.block_tables[0, :4].tolist())


def test_named_config_recipes():
    rng = np.random.default_rng(3)
    L = wl.lognormal_lengths(rng, 256)
    assert L.min() >= 1 and L.max() <= 4096
    assert 250 < np.median(L) < 450
    rng = np.random.default_rng(2)
    u = rng.integers(512, 2048, size=64, endpoint=True)
    assert u.min() >= 512 and u.max() <= 2048


def test_outlier_keys_fraction():
    b = wl.build_batch("o", ctx_lens=[4000], num_heads=8, num_kv_heads=8,
                       head_dim=64, dtype="f32", num_blocks=251,
                       tables=[list(range(251))], seed=9, kv_std=0.5,
                       outlier_frac=0.01, outlier_mult=8.0, keep_seq=True)
    norms = b.seq_k[0].norm(dim=-1)                    # [L, Hkv]
    frac = (norms > 2.0 * norms.median()).float().mean().item()
    assert 0.005 < frac < 0.02
