"""Pins of the fp64 oracle against facts that do not come from the oracle.

Each test ties the oracle to something independent of it: numbers printed on
the reference pages (``tests/golden/``), a library routine computing the same
quantity on non-paged data (torch's float64 scaled-dot-product attention and
logsumexp), closed forms and invariants of exact attention.  The last group
plants plausible mistakes in a copy of the oracle's source and checks that
the pins catch each one.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from paged_kv_cache_151_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "pages_sizing.json")


def golden():
    with open(GOLDEN) as f:
        return json.load(f)


# ---------------------------------------------------------------------------
# sizes printed on the pages
# ---------------------------------------------------------------------------

def test_kv_bytes_per_token_llama8b():
    g = golden()["kv_per_token_llama8b"]
    got = oracle.kv_bytes_per_token(g["num_layers"], g["num_kv_heads"],
                                    g["head_dim"], g["dtype_bytes"])
    assert got == g["kv_bytes_per_token"] == 128 * 1024


def test_conversation_size():
    g = golden()["conversation_2000_tokens"]
    per_tok = oracle.kv_bytes_per_token(32, 8, 128, 2)
    one = g["tokens"] * per_tok
    assert round(one / 2**20) == g["approx_mib"]
    assert round(g["conversations"] * one / 1e9) in (g["approx_gb_total"], 52)


def test_block_budget_exercise():
    g = golden()["block_budget_exercise"]
    bpb = oracle.bytes_per_block(g["block_size"], g["num_layers"],
                                 g["num_kv_heads"], g["head_dim"], g["dtype_bytes"])
    blocks = (g["pool_gib"] * 1024**3) // bpb
    assert blocks * g["block_size"] == g["token_slots"]


def test_worked_pool_example():
    g = golden()["worked_pool_example"]
    bs = g["block_size"]
    bpb = bs * g["kv_bytes_per_token"]
    assert bpb == g["bytes_per_block"]
    n = (g["pool_gib"] * 1024**3) // bpb
    assert n == g["num_blocks"]
    nb = oracle.blocks_for_tokens(g["short_request_tokens"], bs)
    assert nb == g["short_request_blocks"] and n // nb == g["short_requests_fit"]
    nb = oracle.blocks_for_tokens(g["reserved_tokens"], bs)
    assert nb == g["reserved_blocks"] and n // nb == g["reserved_requests_fit"]
    nb = oracle.blocks_for_tokens(g["long_chat_tokens"], bs)
    assert nb == g["long_chat_blocks"] and n // nb == g["long_chats_fit"]
    # only whole blocks of the shared prompt can be shared
    full = g["shared_prompt_tokens"] // bs
    assert full == g["shared_full_blocks"] and full * bs == g["shared_tokens_in_full_blocks"]
    priv = g["long_chat_tokens"] - full * bs
    assert priv == g["private_tokens_per_chat"]
    pb = oracle.blocks_for_tokens(priv, bs)
    assert pb == g["private_blocks_per_chat"]
    assert (n - full) // pb == g["shared_chats_fit"]


def test_waste_simulation_and_free_list():
    """The pages' waste simulation: sizes from the oracle, block tables from
    the generator's free list; both must reproduce the printed output."""
    g = golden()["waste_simulation"]
    per_tok = oracle.kv_bytes_per_token(32, 8, 128, 2)
    rng = np.random.default_rng(g["seed"])
    lengths = rng.integers(g["len_lo"], g["len_hi_exclusive"], size=g["num_requests"])
    used = int(lengths.sum())
    naive = g["max_len"] * len(lengths)
    paged = sum(oracle.blocks_for_tokens(int(n), g["block_size"]) * g["block_size"]
                for n in lengths)
    assert f"{naive * per_tok / 2**30:5.2f}".strip() == g["naive_reserved_gib"]
    assert f"{100 * (1 - used / naive):4.1f}".strip() == g["naive_waste_pct"]
    assert f"{paged * per_tok / 2**30:5.2f}".strip() == g["paged_reserved_gib"]
    assert f"{100 * (1 - used / paged):4.1f}".strip() == g["paged_waste_pct"]
    fl = wl.FreeList(g["pool_blocks"], rng)
    a = fl.allocate(g["table_a_tokens"], g["block_size"])
    assert a == g["table_a"]
    b = a[:g["table_b_shared_blocks"]] + fl.allocate(g["table_b_new_tokens"], g["block_size"])
    assert b == g["table_b"]
    ref = {blk: 1 for blk in a}
    for blk in a[:g["table_b_shared_blocks"]]:
        ref[blk] += 1
    assert {str(k): v for k, v in ref.items() if v > 1} == g["shared_refcounts"]


def test_startup_log_concurrency():
    g = golden()["startup_log_concurrency"]
    assert f"{g['kv_tokens'] / g['tokens_per_request']:.2f}" == g["concurrency"]


# ---------------------------------------------------------------------------
# decode attention against a library routine on non-paged data
# ---------------------------------------------------------------------------

def sdpa_reference(batch, s, scale=None):
    """torch float64 SDPA over the contiguous ground truth of sequence s
    (grouped-query attention through torch's own ``enable_gqa``)."""
    q = batch.q[s].double()[None, :, None, :]               # [1, H, 1, D]
    k = batch.seq_k[s].double().permute(1, 0, 2)[None]      # [1, Hkv, L, D]
    v = batch.seq_v[s].double().permute(1, 0, 2)[None]
    sc = batch.scale if scale is None else scale
    sc = float(np.float32(sc))        # the scale crosses the boundary as fp32
    o = F.scaled_dot_product_attention(q, k, v, scale=sc, enable_gqa=True)
    return o[0, :, 0, :].numpy()


def oracle_decode(batch, **kw):
    return oracle.decode(batch.q, batch.k_cache, batch.v_cache,
                         batch.block_tables, batch.seq_lens, batch.scale,
                         batch.num_kv_heads, batch.dtype, **kw)


CASES = [
    dict(dtype="f32", num_heads=8, num_kv_heads=2, head_dim=64),
    dict(dtype="bf16", num_heads=32, num_kv_heads=8, head_dim=128),
    dict(dtype="f16", num_heads=8, num_kv_heads=1, head_dim=128),
    dict(dtype="bf16", num_heads=16, num_kv_heads=2, head_dim=64),
    dict(dtype="f32", num_heads=4, num_kv_heads=4, head_dim=64),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c['dtype']}-{c['num_heads']}x{c['num_kv_heads']}x{c['head_dim']}")
def test_decode_matches_sdpa(case):
    b = wl.random_batch(11, num_seqs=5, max_len=70, new_in_pool=True, **case)
    out = oracle_decode(b)
    for s in range(b.num_seqs):
        np.testing.assert_allclose(out[s], sdpa_reference(b, s), rtol=0, atol=1e-12)


def test_tiny_config_matches_sdpa():
    b = wl.tiny(new_in_pool=True)
    out = oracle_decode(b, nthreads=3)
    for s in range(b.num_seqs):
        np.testing.assert_allclose(out[s], sdpa_reference(b, s), rtol=0, atol=1e-12)


def test_large_scores_stay_finite():
    """Keys scaled so that exp(z) overflows fp64 unless the maximum is
    subtracted first; SDPA handles the same data."""
    b = wl.random_batch(12, num_seqs=3, max_len=40, num_heads=4, num_kv_heads=2,
                        head_dim=64, dtype="f32", new_in_pool=True, kv_std=1.0)
    big = 400.0
    out = oracle.decode(b.q, b.k_cache * big, b.v_cache, b.block_tables,
                        b.seq_lens, b.scale, b.num_kv_heads, "f32")
    assert np.isfinite(out).all()
    for s in range(b.num_seqs):
        q = b.q[s].double()[None, :, None, :]
        k = (b.seq_k[s].double() * big).permute(1, 0, 2)[None]
        v = b.seq_v[s].double().permute(1, 0, 2)[None]
        ref = F.scaled_dot_product_attention(q, k, v, scale=float(np.float32(b.scale)),
                                             enable_gqa=True)
        np.testing.assert_allclose(out[s], ref[0, :, 0].numpy(), rtol=0, atol=1e-10)


def test_outlier_keys_long_context_shape():
    """The long-context workload's 1% x8 keys, at a small size, against SDPA."""
    b = wl.build_batch("outliers", ctx_lens=[300, 1000], num_heads=16,
                       num_kv_heads=2, head_dim=128, dtype="bf16", num_blocks=90,
                       tables=[list(range(0, 19)), list(range(19, 82))],
                       seed=5, kv_std=0.5, outlier_frac=0.01, outlier_mult=8.0,
                       keep_seq=True, new_in_pool=True)
    out = oracle_decode(b)
    for s in range(2):
        np.testing.assert_allclose(out[s], sdpa_reference(b, s), rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# closed forms and invariants
# ---------------------------------------------------------------------------

def test_seq_len_one_returns_v_exactly():
    b = wl.random_batch(13, num_seqs=4, max_len=0, num_heads=8, num_kv_heads=2,
                        head_dim=64, dtype="bf16", new_in_pool=True)
    assert (b.seq_lens == 1).all()
    out = oracle_decode(b)
    G = b.num_heads // b.num_kv_heads
    for s in range(b.num_seqs):
        for h in range(b.num_heads):
            v = b.seq_v[s][0, h // G].double().numpy()
            assert np.array_equal(out[s, h], v)


def test_seq_len_zero_gives_zeros():
    b = wl.random_batch(14, num_seqs=3, max_len=20, num_heads=4, num_kv_heads=2,
                        head_dim=64, dtype="f32", new_in_pool=True)
    sl = b.seq_lens.copy()
    sl[1] = 0
    out = oracle.decode(b.q, b.k_cache, b.v_cache, b.block_tables, sl, b.scale,
                        b.num_kv_heads, "f32")
    assert np.array_equal(out[1], np.zeros_like(out[1]))


def test_softmax_weights_sum_to_one():
    b = wl.random_batch(15, num_seqs=4, max_len=90, num_heads=8, num_kv_heads=2,
                        head_dim=128, dtype="bf16", new_in_pool=True)
    pr = oracle.problem(b.q, b.k_cache, b.v_cache, b.block_tables, b.seq_lens,
                        b.scale, b.num_kv_heads, "bf16")
    for s in range(b.num_seqs):
        for h in (0, 3, 7):
            out, w = oracle.decode_one(s, h, None, None, None, None, None, None,
                                       None, "bf16", problem=pr)
            assert w.shape[0] == b.seq_lens[s]
            assert (w >= 0).all()
            assert abs(w.sum() - 1.0) < 1e-12
            # the output is the weights applied to V
            v = b.seq_v[s][:, h // 4].double().numpy()
            np.testing.assert_allclose(out, w @ v, rtol=0, atol=1e-12)


def test_block_permutation_invariance():
    b = wl.random_batch(16, num_seqs=6, max_len=100, num_heads=8, num_kv_heads=2,
                        head_dim=64, dtype="bf16", new_in_pool=True, extra_blocks=20)
    p = wl.permute_blocks(b, seed=99)
    assert not np.array_equal(p.block_tables, b.block_tables)
    assert np.array_equal(oracle_decode(b), oracle_decode(p))


def test_shared_prefix_aliasing_equals_private_copies():
    kw = dict(batch=5, prefix_blocks=6, lo=3, hi=40)
    shared = wl.shared_prefix(new_in_pool=True, keep_seq=True, **kw)
    private = wl.shared_prefix(new_in_pool=True, private_prefix=True, **kw)
    # the shared layout really aliases: every table starts with the same blocks
    assert (shared.block_tables[:, :6] == shared.block_tables[0, :6]).all()
    assert len(set(private.block_tables[:, 0].tolist())) == 5
    a, p = oracle_decode(shared), oracle_decode(private)
    assert np.array_equal(a, p)
    for s in range(shared.num_seqs):
        np.testing.assert_allclose(a[s], sdpa_reference(shared, s), rtol=0, atol=1e-12)


def test_constant_v_and_zero_q():
    b = wl.random_batch(17, num_seqs=3, max_len=50, num_heads=4, num_kv_heads=2,
                        head_dim=64, dtype="f32", new_in_pool=True)
    row = torch.linspace(-2, 3, 64)
    vc = b.v_cache.clone()
    vc[:] = row
    out = oracle.decode(b.q, b.k_cache, vc, b.block_tables, b.seq_lens, b.scale,
                        b.num_kv_heads, "f32")
    np.testing.assert_allclose(out, np.broadcast_to(row.double().numpy(), out.shape),
                               rtol=0, atol=1e-12)
    out = oracle.decode(torch.zeros_like(b.q), b.k_cache, b.v_cache,
                        b.block_tables, b.seq_lens, b.scale, b.num_kv_heads, "f32")
    for s in range(b.num_seqs):
        mean = b.seq_v[s].double().mean(0).numpy()     # [Hkv, D]
        for h in range(b.num_heads):
            np.testing.assert_allclose(out[s, h], mean[h // 2], rtol=0, atol=1e-12)


def test_table_padding_is_never_read():
    b = wl.random_batch(18, num_seqs=4, max_len=60, num_heads=4, num_kv_heads=1,
                        head_dim=64, dtype="f32", new_in_pool=True, table_slack=3)
    assert (b.block_tables == wl.PAD).any()
    out = oracle_decode(b)
    assert np.isfinite(out).all()


# ---------------------------------------------------------------------------
# multi-token queries
# ---------------------------------------------------------------------------

def oracle_multi(b):
    return oracle.decode_multi(b.q, b.k_cache, b.v_cache, b.block_tables, b.seq_lens,
                               b.meta["query_start"], b.scale, b.num_kv_heads, b.dtype)


def test_multi_with_one_token_is_decode():
    b = wl.multi_query_batch(41, num_seqs=5, min_ctx=0, max_ctx=80, n_new=1, num_heads=8,
                             num_kv_heads=2, head_dim=64, dtype="bf16")
    out = oracle_multi(b)
    ref = oracle.decode(b.q, b.k_cache, b.v_cache, b.block_tables, b.seq_lens, b.scale,
                        b.num_kv_heads, "bf16")
    assert np.array_equal(out, ref)


def test_multi_token_i_is_decode_of_its_causal_prefix():
    b = wl.multi_query_batch(42, num_seqs=4, min_ctx=0, max_ctx=60, n_new=(1, 6),
                             num_heads=8, num_kv_heads=2, head_dim=64, dtype="f32")
    out = oracle_multi(b)
    qs, n = b.meta["query_start"], b.meta["n_new"]
    for s in range(b.num_seqs):
        for i in range(int(n[s])):
            tok = int(qs[s]) + i
            sl = b.seq_lens.copy()
            sl[s] = b.seq_lens[s] - n[s] + i + 1
            qb = torch.zeros((b.num_seqs, b.num_heads, b.head_dim))
            qb[s] = b.q[tok]
            ref = oracle.decode(qb, b.k_cache, b.v_cache, b.block_tables, sl, b.scale,
                                b.num_kv_heads, "f32")
            assert np.array_equal(out[tok], ref[s])


@pytest.mark.parametrize("dtype,H,Hkv,D", [("bf16", 32, 8, 128), ("f32", 8, 8, 64),
                                            ("f16", 16, 2, 64)])
def test_multi_matches_masked_sdpa(dtype, H, Hkv, D):
    b = wl.multi_query_batch(43, num_seqs=4, min_ctx=0, max_ctx=70, n_new=(1, 9),
                             num_heads=H, num_kv_heads=Hkv, head_dim=D, dtype=dtype)
    out = oracle_multi(b)
    qs, n = b.meta["query_start"], b.meta["n_new"]
    for s in range(b.num_seqs):
        L, ns = int(b.seq_lens[s]), int(n[s])
        q = b.q[int(qs[s]):int(qs[s]) + ns].double().permute(1, 0, 2)[None]  # [1,H,n,D]
        k = b.seq_k[s].double().permute(1, 0, 2)[None]                        # [1,Hkv,L,D]
        v = b.seq_v[s].double().permute(1, 0, 2)[None]
        pos_q = torch.arange(L - ns, L)[:, None]
        mask = torch.arange(L)[None, :] <= pos_q                              # [n, L]
        ref = F.scaled_dot_product_attention(q, k, v, attn_mask=mask,
                                             scale=float(np.float32(b.scale)),
                                             enable_gqa=True)[0].permute(1, 0, 2)
        np.testing.assert_allclose(out[int(qs[s]):int(qs[s]) + ns], ref.numpy(),
                                   rtol=0, atol=1e-12)


def test_multi_whole_sequence_new_is_causal_prefill():
    """All tokens new (a first prefill chunk): plain causal attention."""
    b = wl.multi_query_batch(44, num_seqs=2, min_ctx=0, max_ctx=0, n_new=(5, 20),
                             num_heads=4, num_kv_heads=2, head_dim=64, dtype="f32",
                             lens=[0, 0])
    out = oracle_multi(b)
    qs = b.meta["query_start"]
    for s in range(2):
        L = int(b.seq_lens[s])
        q = b.q[int(qs[s]):int(qs[s]) + L].double().permute(1, 0, 2)[None]
        k = b.seq_k[s].double().permute(1, 0, 2)[None]
        v = b.seq_v[s].double().permute(1, 0, 2)[None]
        ref = F.scaled_dot_product_attention(q, k, v, is_causal=True,
                                             scale=float(np.float32(b.scale)),
                                             enable_gqa=True)[0].permute(1, 0, 2)
        np.testing.assert_allclose(out[int(qs[s]):int(qs[s]) + L], ref.numpy(), rtol=0,
                                   atol=1e-12)


# ---------------------------------------------------------------------------
# split-KV partitions
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("psize", [16, 48, 64, 512])
def test_partition_stats_against_library(psize):
    b = wl.random_batch(19, num_seqs=3, max_len=300, num_heads=8, num_kv_heads=2,
                        head_dim=64, dtype="bf16", new_in_pool=True, kv_std=2.0)
    pr = oracle.problem(b.q, b.k_cache, b.v_cache, b.block_tables, b.seq_lens,
                        b.scale, b.num_kv_heads, "bf16")
    full = oracle_decode(b)
    for s in range(b.num_seqs):
        L = int(b.seq_lens[s])
        for h in (0, 5):
            m, l, o = oracle.partition_stats(s, h, psize, None, None, None, None,
                                             None, None, None, "bf16", problem=pr)
            assert m.shape[0] == math.ceil(L / psize)
            q = b.q[s, h].double()
            k = b.seq_k[s][:, h // 4].double()
            v = b.seq_v[s][:, h // 4].double()
            z = float(np.float32(b.scale)) * (k @ q)
            for p in range(m.shape[0]):
                sl = slice(p * psize, min(L, (p + 1) * psize))
                assert m[p] == pytest.approx(float(z[sl].max()), abs=1e-12)
                assert m[p] + math.log(l[p]) == pytest.approx(
                    float(torch.logsumexp(z[sl], 0)), abs=1e-12)
                ref = F.scaled_dot_product_attention(
                    q[None, None, None], k[sl][None, None], v[sl][None, None],
                    scale=float(np.float32(b.scale)))[0, 0, 0].numpy()
                np.testing.assert_allclose(o[p], ref, rtol=0, atol=1e-12)
            merged = oracle.lse_merge(m, l, o)
            np.testing.assert_allclose(merged, full[s, h], rtol=0, atol=1e-12)


def test_lse_merge_single_partition_is_identity():
    o = np.random.default_rng(0).normal(size=(1, 8))
    out = oracle.lse_merge(np.array([3.0]), np.array([7.0]), o)
    np.testing.assert_allclose(out, o[0], rtol=0, atol=1e-15)


# ---------------------------------------------------------------------------
# cache write against numpy's own indexing
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_reshape_and_cache_matches_index_assignment(dtype):
    b = wl.random_batch(20, num_seqs=9, max_len=40, num_heads=8, num_kv_heads=2,
                        head_dim=64, dtype=dtype)
    sm = b.slot_mapping.copy()
    sm[3] = -1                        # padding token: skipped
    kc, vc, bad = oracle.reshape_and_cache(b.k_new, b.v_new, b.k_cache,
                                           b.v_cache, sm, dtype)
    assert bad == 0
    for cache, new, got in ((b.k_cache, b.k_new, kc), (b.v_cache, b.v_new, vc)):
        ref = oracle._host(cache).copy()
        N, Hkv, bs, D = ref.shape
        tokview = ref.transpose(0, 2, 1, 3).reshape(N * bs, Hkv, D).copy()
        keep = sm >= 0
        tokview[sm[keep]] = oracle._host(new)[keep]
        ref = tokview.reshape(N, bs, Hkv, D).transpose(0, 2, 1, 3)
        assert np.array_equal(got.view(np.uint8), np.ascontiguousarray(ref).view(np.uint8))


def test_reshape_and_cache_rejects_out_of_range_slots():
    b = wl.random_batch(21, num_seqs=3, max_len=10, num_heads=2, num_kv_heads=2,
                        head_dim=64, dtype="f32")
    sm = b.slot_mapping.copy()
    sm[0] = b.num_blocks * b.block_size
    kc, vc, bad = oracle.reshape_and_cache(b.k_new, b.v_new, b.k_cache,
                                           b.v_cache, sm, "f32")
    assert bad == 1


# ---------------------------------------------------------------------------
# FP8 (E4M3) cache: the format against torch's float8_e4m3fn, the write
# against element-wise library conversion, the read against SDPA on the
# dequantised values
# ---------------------------------------------------------------------------

ALL_CODES = np.arange(256, dtype=np.uint8)


def torch_e4m3_values(codes) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(codes, np.uint8)).view(
        torch.float8_e4m3fn).double().numpy()


def torch_e4m3_codes(x) -> np.ndarray:
    """torch's round-to-nearest-even conversion (it does not saturate: only
    for magnitudes below 464)."""
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.float8_e4m3fn).view(
        torch.uint8).numpy()


def test_e4m3_decoding_of_every_code():
    got = oracle.e4m3_decode(ALL_CODES)
    ref = torch_e4m3_values(ALL_CODES)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(got[~np.isnan(got)], ref[~np.isnan(ref)])
    # the format's landmarks: largest finite, smallest normal and subnormal,
    # one, the two NaN codes
    assert got[0x7E] == 448.0 and got[0xFE] == -448.0
    assert got[0x08] == 2.0 ** -6 and got[0x01] == 2.0 ** -9
    assert got[0x38] == 1.0 and got[0xC0] == -2.0
    assert np.isnan(got[0x7F]) and np.isnan(got[0xFF])
    assert np.isnan(got).sum() == 2


def test_e4m3_encoding_round_to_nearest_even():
    vals = oracle.e4m3_decode(ALL_CODES)
    finite = np.sort(np.unique(vals[np.isfinite(vals)]))
    mids = (finite[:-1] + finite[1:]) / 2            # every tie between neighbours
    rng = np.random.default_rng(0)
    rand = rng.standard_normal(6000) * np.exp2(rng.integers(-14, 10, 6000))
    x = np.concatenate([finite, mids, np.nextafter(mids, 0), np.nextafter(mids, 1e9),
                        rand, -rand]).astype(np.float32)
    x = x[np.abs(x) < 464]
    assert np.array_equal(oracle.e4m3_encode(x), torch_e4m3_codes(x))
    # encode(decode(c)) == c for every finite code except -0 / +0 aliasing none
    fin = np.isfinite(vals)
    assert np.array_equal(oracle.e4m3_encode(vals[fin].astype(np.float32)), ALL_CODES[fin])


def test_e4m3_encoding_saturates_and_keeps_nan():
    big = np.array([448.5, 463.9, 464.0, 1e6, 3.4e38, np.inf], dtype=np.float32)
    assert (oracle.e4m3_encode(big) == 0x7E).all()
    assert (oracle.e4m3_encode(-big) == 0xFE).all()
    assert oracle.e4m3_encode(np.array([np.nan], np.float32))[0] == 0x7F
    assert oracle.e4m3_encode(np.array([-0.0, -1e-30, 1e-30], np.float32)).tolist() == \
        [0x80, 0x80, 0x00]


def fp8_scales(Hkv, seed):
    rng = np.random.default_rng(seed)
    return (rng.uniform(0.003, 0.02, Hkv).astype(np.float32),
            rng.uniform(0.003, 0.02, Hkv).astype(np.float32))


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
def test_reshape_and_cache_fp8_matches_elementwise_conversion(dtype):
    b = wl.random_batch(22, num_seqs=9, max_len=40, num_heads=8, num_kv_heads=4,
                        head_dim=64, dtype=dtype, kv_std=1.0)
    b = wl.with_fp8_pool(b, seed=1)
    ks, vs = fp8_scales(4, 2)
    sm = b.slot_mapping.copy()
    sm[2] = -1
    kc, vc, bad = oracle.reshape_and_cache_fp8(b.k_new, b.v_new, b.k_cache, b.v_cache, sm,
                                               dtype, ks, vs)
    assert bad == 0
    for pool, new, sc, got in ((b.k_cache, b.k_new, ks, kc), (b.v_cache, b.v_new, vs, vc)):
        q = new.float().numpy() / sc[None, :, None]          # binary32 quotients
        assert np.abs(q).max() > 448                          # some saturate
        q = np.clip(q, -448.0, 448.0)                         # saturation, then RNE
        ref = pool.numpy().copy()
        N, Hkv, bs, D = ref.shape
        tok = ref.transpose(0, 2, 1, 3).reshape(N * bs, Hkv, D).copy()
        keep = sm >= 0
        tok[sm[keep]] = torch_e4m3_codes(q[keep])
        ref = tok.reshape(N, bs, Hkv, D).transpose(0, 2, 1, 3)
        assert np.array_equal(got, ref)


def dequantised_sdpa(b, s, ks, vs):
    """SDPA of sequence s on K/V gathered by plain indexing and dequantised
    with torch's float8 conversion."""
    L = int(b.seq_lens[s])
    nb = -(-L // 16)
    blocks = torch.from_numpy(b.block_tables[s, :nb].astype(np.int64))
    def gather(pool, sc):
        c = pool[blocks].permute(0, 2, 1, 3).reshape(nb * 16, b.num_kv_heads, b.head_dim)[:L]
        v = c.contiguous().view(torch.float8_e4m3fn).double()
        return v * torch.from_numpy(sc).double().view(1, -1, 1)
    k, v = gather(b.k_cache, ks), gather(b.v_cache, vs)
    q = b.q[s].double()[None, :, None, :]
    out = F.scaled_dot_product_attention(q, k.permute(1, 0, 2)[None], v.permute(1, 0, 2)[None],
                                         scale=float(np.float32(b.scale)), enable_gqa=True)
    return out[0, :, 0, :].numpy()


@pytest.mark.parametrize("H,Hkv,D", [(32, 8, 128), (8, 8, 64), (16, 2, 64)])
def test_decode_fp8_matches_sdpa_on_dequantised_cache(H, Hkv, D):
    b = wl.random_batch(23 + H, num_seqs=5, max_len=90, num_heads=H, num_kv_heads=Hkv,
                        head_dim=D, dtype="bf16", new_in_pool=True)
    b = wl.with_fp8_pool(b, seed=3)
    ks, vs = b.meta["k_scale"].numpy(), b.meta["v_scale"].numpy()
    assert len(set(ks.tolist())) == Hkv                  # distinct per-head scales
    out = oracle.decode(b.q, b.k_cache, b.v_cache, b.block_tables, b.seq_lens, b.scale,
                        Hkv, "bf16", kv_scales=(ks, vs))
    for s in range(b.num_seqs):
        np.testing.assert_allclose(out[s], dequantised_sdpa(b, s, ks, vs), rtol=0, atol=1e-9)


def test_decode_fp8_with_power_of_two_scales_is_decode_of_the_values():
    """With scales 2^k the dequantised values are exact in f32: the FP8 read
    must give bit for bit what the f32 read of those values gives."""
    b = wl.random_batch(24, num_seqs=4, max_len=70, num_heads=8, num_kv_heads=2,
                        head_dim=64, dtype="f32", new_in_pool=True)
    b = wl.with_fp8_pool(b, seed=4)
    ks = np.array([2.0 ** -7, 2.0 ** -5], np.float32)
    vs = np.array([2.0 ** -6, 2.0 ** -8], np.float32)
    kf = (torch_e4m3_values(b.k_cache.numpy()) * ks[None, :, None, None]).astype(np.float32)
    vf = (torch_e4m3_values(b.v_cache.numpy()) * vs[None, :, None, None]).astype(np.float32)
    ref = oracle.decode(b.q, kf, vf, b.block_tables, b.seq_lens, b.scale, 2, "f32")
    got = oracle.decode(b.q, b.k_cache, b.v_cache, b.block_tables, b.seq_lens, b.scale, 2,
                        "f32", kv_scales=(ks, vs))
    assert np.array_equal(np.isnan(ref), np.isnan(got)) and not np.isnan(got).any()
    assert np.array_equal(ref, got)
    for s, h in ((0, 0), (3, 7)):
        one, _ = oracle.decode_one(s, h, b.q, b.k_cache, b.v_cache, b.block_tables,
                                   b.seq_lens, b.scale, 2, "f32", problem=oracle.problem(
                                       b.q, b.k_cache, b.v_cache, b.block_tables,
                                       b.seq_lens, b.scale, 2, "f32", kv_scales=(ks, vs)))
        assert np.array_equal(one, got[s, h])


# ---------------------------------------------------------------------------
# block copies for copy-on-write: numpy index assignment
# ---------------------------------------------------------------------------

def cow_mapping(num_blocks, n, seed):
    """n (src, dst) pairs with distinct dsts that are never a src (fresh blocks
    receiving copies of shared ones, as copy-on-write produces them)."""
    rng = np.random.default_rng(seed)
    ids = rng.permutation(num_blocks)
    dst = ids[:n]
    src = rng.choice(ids[n:], size=n)                   # a shared block may be copied twice
    return np.stack([src, dst], 1).astype(np.int64)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_copy_blocks_matches_index_assignment(dtype):
    b = wl.random_batch(25, num_seqs=6, max_len=80, num_heads=8, num_kv_heads=4,
                        head_dim=64, dtype=dtype, canary=False, new_in_pool=True,
                        extra_blocks=30)
    m = cow_mapping(b.num_blocks, 12, 1)
    layers = [b.k_cache, b.v_cache, b.k_cache * 2, b.v_cache * 3]
    got, bad = oracle.copy_blocks(layers, m)
    assert bad == 0
    for c, g in zip(layers, got):
        ref = oracle._host(c).copy()
        ref[m[:, 1]] = ref[m[:, 0]]
        assert np.array_equal(g.view(np.uint8), ref.view(np.uint8))


def test_copy_blocks_skips_out_of_range_pairs_and_keeps_the_rest():
    pool = np.arange(10 * 48, dtype=np.float32).reshape(10, 3, 16)
    m = np.array([[2, 7], [11, 3], [4, -1], [5, 5], [1, 8]], dtype=np.int64)
    (got,), bad = oracle.copy_blocks([pool], m)
    assert bad == 2
    ref = pool.copy()
    ref[7] = pool[2]
    ref[8] = pool[1]
    assert np.array_equal(got, ref)                       # src == dst is a no-op
    (same,), bad = oracle.copy_blocks([pool], np.zeros((0, 2), np.int64))
    assert bad == 0 and np.array_equal(same, pool)


def test_copy_on_write_fork_leaves_the_reader_unchanged():
    """A sequence forked from another shares its blocks; before the child
    appends into the shared last block, that block is copied to a fresh one
    and the child's table points at the copy.  The parent's attention is
    unchanged and the child's equals attention over the same data."""
    b = wl.random_batch(26, num_seqs=2, max_len=40, min_len=20, num_heads=8, num_kv_heads=2,
                        head_dim=64, dtype="f32", new_in_pool=True, extra_blocks=4)
    bt = b.block_tables.copy()
    L = int(b.seq_lens[0])
    nb = -(-L // 16)
    fresh = int(np.setdiff1d(np.arange(b.num_blocks), bt[bt != wl.PAD])[0])
    child = bt[0].copy()
    child[nb - 1] = fresh                                # the child's private copy
    (kc, vc), bad = oracle.copy_blocks([b.k_cache, b.v_cache],
                                       np.array([[bt[0, nb - 1], fresh]], np.int64))
    assert bad == 0
    tables = np.stack([bt[0], child])
    lens = np.array([L, L], np.int32)
    q = torch.stack([b.q[0], b.q[0]])
    out = oracle.decode(q, kc, vc, tables, lens, b.scale, 2, "f32")
    ref = oracle.decode(b.q[:1], b.k_cache, b.v_cache, bt[:1], lens[:1], b.scale, 2, "f32")
    assert np.array_equal(out[0], ref[0]) and np.array_equal(out[1], ref[0])


# ---------------------------------------------------------------------------
# planted mistakes: each must make at least one pin fail
# ---------------------------------------------------------------------------

MUTATIONS = {
    "gqa_map_modulo": ("const int32_t j = h / G;", "const int32_t j = h % a->num_kv_heads;"),
    "row_offset": ("int64_t base = ((pb * a->num_kv_heads + j) * bs + t % bs) * D;",
                   "int64_t base = ((pb * a->num_kv_heads + j) * bs + (t + 1) % bs) * D;"),
    "no_scale": ("z[t] = a->scale * acc;", "z[t] = acc;"),
    "no_max_subtract": ("for (int64_t t = 0; t < L; ++t) { z[t] = exp(z[t] - M); S += z[t]; }",
                        "for (int64_t t = 0; t < L; ++t) { z[t] = exp(z[t]); S += z[t]; }"),
    "drop_last_token": ("for (int64_t t = 0; t < L; ++t) {\n        double w = z[t] / S;",
                        "for (int64_t t = 0; t + 1 < L; ++t) {\n        double w = z[t] / S;"),
    "merge_sign": ("double c = l[p] * exp(m[p] - M);", "double c = l[p] * exp(M - m[p]);"),
    "table_row_stride": ("int64_t pb = a->block_tables[s * a->max_blocks + lb];",
                         "int64_t pb = a->block_tables[s + lb * a->num_seqs];"),
    "multi_causal_offset": ("const int64_t seen = L - n + i + 1;     /* causal prefix */",
                            "const int64_t seen = L - n + i;     /* causal prefix */"),
    "e4m3_bias": ("else v = ldexp((double)(8 + f), e - 10);", "else v = ldexp((double)(8 + f), e - 9);"),
    "e4m3_ties_away": ("if (rem > 0.5 || (rem == 0.5 && fmod(r, 2.0) != 0.0)) r += 1.0;",
                       "if (rem >= 0.5) r += 1.0;"),
    "fp8_write_multiplies": ("k_cache[dst + d] = (uint8_t)pa_ref_e4m3_from_float(xk / k_scale[j]);",
                             "k_cache[dst + d] = (uint8_t)pa_ref_e4m3_from_float(xk * k_scale[j]);"),
    "fp8_read_head_scale": ("const double vs = a->v_scale ? (double)a->v_scale[j] : 1.0;",
                            "const double vs = a->v_scale ? (double)a->v_scale[0] : 1.0;"),
    "copy_direction": ("memmove(base + dst * block_bytes, base + src * block_bytes,",
                       "memmove(base + src * block_bytes, base + dst * block_bytes,"),
}


def _pins_hold() -> bool:
    """A compact run of the pins above; False as soon as one fails."""
    try:
        b = wl.random_batch(31, num_seqs=4, max_len=60, num_heads=8,
                            num_kv_heads=2, head_dim=64, dtype="f32",
                            new_in_pool=True)
        out = oracle_decode(b)
        for s in range(b.num_seqs):
            if not np.allclose(out[s], sdpa_reference(b, s), rtol=0, atol=1e-9):
                return False
        big = oracle.decode(b.q, b.k_cache * 400.0, b.v_cache, b.block_tables,
                            b.seq_lens, b.scale, b.num_kv_heads, "f32")
        if not np.isfinite(big).all():
            return False
        m, l, o = oracle.partition_stats(1, 3, 16, b.q, b.k_cache, b.v_cache,
                                         b.block_tables, b.seq_lens, b.scale,
                                         b.num_kv_heads, "f32")
        if not np.allclose(oracle.lse_merge(m, l, o), out[1, 3], rtol=0, atol=1e-9):
            return False
        mb = wl.multi_query_batch(32, num_seqs=3, min_ctx=0, max_ctx=40, n_new=(2, 5),
                                  num_heads=4, num_kv_heads=2, head_dim=64, dtype="f32")
        mo = oracle.decode_multi(mb.q, mb.k_cache, mb.v_cache, mb.block_tables,
                                 mb.seq_lens, mb.meta["query_start"], mb.scale,
                                 mb.num_kv_heads, "f32")
        qs, n = mb.meta["query_start"], mb.meta["n_new"]
        for s in range(mb.num_seqs):
            L, ns = int(mb.seq_lens[s]), int(n[s])
            q = mb.q[int(qs[s]):int(qs[s]) + ns].double().permute(1, 0, 2)[None]
            k = mb.seq_k[s].double().permute(1, 0, 2)[None]
            v = mb.seq_v[s].double().permute(1, 0, 2)[None]
            mask = torch.arange(L)[None, :] <= torch.arange(L - ns, L)[:, None]
            ref = F.scaled_dot_product_attention(q, k, v, attn_mask=mask,
                                                 scale=float(np.float32(mb.scale)),
                                                 enable_gqa=True)[0].permute(1, 0, 2)
            if not np.allclose(mo[int(qs[s]):int(qs[s]) + ns], ref.numpy(), rtol=0,
                               atol=1e-9):
                return False
        # block copies
        pool = np.arange(6 * 32, dtype=np.float32).reshape(6, 2, 16)
        (cp,), nbad = oracle.copy_blocks([pool], np.array([[1, 4], [2, 5]], np.int64))
        ref = pool.copy()
        ref[[4, 5]] = pool[[1, 2]]
        if nbad != 0 or not np.array_equal(cp, ref):
            return False
        # FP8: every code's value, the ties of the encoder, the write and the read
        vals = oracle.e4m3_decode(ALL_CODES)
        ref = torch_e4m3_values(ALL_CODES)
        if not np.array_equal(vals[~np.isnan(ref)], ref[~np.isnan(ref)]):
            return False
        fin = np.sort(np.unique(vals[np.isfinite(vals)]))
        mids = ((fin[:-1] + fin[1:]) / 2).astype(np.float32)
        mids = mids[np.abs(mids) < 464]
        if not np.array_equal(oracle.e4m3_encode(mids), torch_e4m3_codes(mids)):
            return False
        fb = wl.with_fp8_pool(wl.random_batch(33, num_seqs=3, max_len=40, num_heads=4,
                                              num_kv_heads=2, head_dim=64, dtype="bf16",
                                              new_in_pool=True), seed=5)
        ks, vs = fb.meta["k_scale"].numpy(), fb.meta["v_scale"].numpy()
        kc, _, _ = oracle.reshape_and_cache_fp8(fb.k_new, fb.v_new, fb.k_cache, fb.v_cache,
                                                fb.slot_mapping, "bf16", ks, vs)
        sm = fb.slot_mapping
        want = torch_e4m3_codes(np.clip(fb.k_new.float().numpy() / ks[None, :, None],
                                        -448.0, 448.0))
        got = kc.transpose(0, 2, 1, 3).reshape(-1, 2, 64)[sm]
        if not np.array_equal(got, want):
            return False
        fo = oracle.decode(fb.q, fb.k_cache, fb.v_cache, fb.block_tables, fb.seq_lens,
                           fb.scale, 2, "bf16", kv_scales=(ks, vs))
        for s in range(fb.num_seqs):
            if not np.allclose(fo[s], dequantised_sdpa(fb, s, ks, vs), rtol=0, atol=1e-9):
                return False
    except ValueError:
        return False
    return True


def test_unmodified_oracle_passes_compact_pins():
    assert _pins_hold()


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, tmp_path):
    old, new = MUTATIONS[name]
    src = oracle.source_text()
    assert src.count(old) == 1, name
    lib = oracle.build_variant(src.replace(old, new), str(tmp_path))
    with oracle.use_library(lib):
        assert not _pins_hold(), f"planted mistake '{name}' was not caught"
