"""Seeded synthetic inputs for paged decode attention.

This module only *constructs inputs*: it draws values, hands out physical
blocks from a free list, lays prior context into a paged pool and writes the
slot mapping for each step's new token.  It computes no attention and is the
one module that both the CUDA path's tests and the fp64 oracle's tests share.

Layout (the pages leave it open; this is the reading used throughout):

* ``k_cache, v_cache``: ``[num_blocks, num_kv_heads, block_size, head_dim]``,
  contiguous, so one (physical block, KV head) tile is one contiguous run.
* ``q``: ``[num_seqs, num_heads, head_dim]``;
  ``k_new, v_new``: ``[num_tokens, num_kv_heads, head_dim]``.
* ``block_tables``: int32 ``[num_seqs, max_blocks]``; entries past a
  sequence's last block hold ``PAD`` and are never meant to be read.
* ``slot_mapping``: int64 ``[num_tokens]``, ``slot = block * block_size + row``
  ("vLLM: Architecture, PagedAttention & Internals", *The forward step in
  detail*).

The free-list allocator follows the pages' pattern (a seeded permutation of
the pool, blocks popped from its end, one block per ``block_size`` tokens;
"vLLM: High-Throughput Serving with PagedAttention" (lesson 13.15), *PagedAttention, the core idea*, ``paged_kv.py``), and
the five named workloads follow the configurations the build is measured on.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import List, Optional

import numpy as np
import torch

BLOCK_SIZE = 16
PAD = 2**31 - 1          # block-table padding: never a valid block id
DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}


class FreeList:
    """Free list of physical block ids: a seeded permutation, popped from the end."""

    def __init__(self, num_blocks: int, rng: np.random.Generator):
        self.free = list(rng.permutation(num_blocks))

    def take(self, n_blocks: int) -> List[int]:
        if n_blocks > len(self.free):
            raise ValueError("pool exhausted")
        return [int(self.free.pop()) for _ in range(n_blocks)]

    def allocate(self, n_tokens: int, block_size: int = BLOCK_SIZE) -> List[int]:
        return self.take(math.ceil(n_tokens / block_size))


@dataclass
class PagedBatch:
    """One decode step's inputs.

    ``ctx_lens[s]`` tokens are already in the pool at positions
    ``[0, ctx_lens[s])``; the step's new token of sequence ``s`` lands at
    position ``ctx_lens[s]`` through ``slot_mapping[s]``; decode then attends
    over ``seq_lens[s] = ctx_lens[s] + 1`` tokens.
    """

    name: str
    dtype: str
    num_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    scale: float
    ctx_lens: np.ndarray          # int32 [B]
    seq_lens: np.ndarray          # int32 [B]
    block_tables: np.ndarray      # int32 [B, max_blocks]
    slot_mapping: np.ndarray      # int64 [B]
    q: torch.Tensor
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    k_new: torch.Tensor
    v_new: torch.Tensor
    # contiguous ground truth per sequence ([seq_len, H_kv, D], context then
    # the new token); kept only for small batches
    seq_k: Optional[List[torch.Tensor]] = None
    seq_v: Optional[List[torch.Tensor]] = None
    meta: dict = field(default_factory=dict)

    @property
    def num_seqs(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def max_blocks(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def device(self) -> torch.device:
        return self.k_cache.device

    def torch_tables(self, device=None):
        device = self.device if device is None else device
        return (torch.from_numpy(self.block_tables).to(device),
                torch.from_numpy(self.seq_lens).to(device),
                torch.from_numpy(self.slot_mapping).to(device))


def _nan_or_zero(shape, dtype, device, canary: bool) -> torch.Tensor:
    if canary:
        return torch.full(shape, float("nan"), dtype=dtype, device=device)
    return torch.zeros(shape, dtype=dtype, device=device)


def _pad_tables(tables: List[List[int]], width: Optional[int] = None) -> np.ndarray:
    width = max([len(t) for t in tables] + [1]) if width is None else width
    out = np.full((len(tables), width), PAD, dtype=np.int32)
    for s, t in enumerate(tables):
        out[s, :len(t)] = t
    return out


def build_batch(name: str, *, ctx_lens, num_heads: int, num_kv_heads: int,
                head_dim: int, dtype: str, num_blocks: int, tables: List[List[int]],
                seed: int, scale: Optional[float] = None, device="cpu",
                canary: bool = True, keep_seq: bool = False,
                q_std: float = 1.0, kv_std: float = 1.0,
                outlier_frac: float = 0.0, outlier_mult: float = 1.0,
                table_width: Optional[int] = None,
                block_size: int = BLOCK_SIZE,
                new_in_pool: bool = False) -> PagedBatch:
    """Draw values and lay them out in a paged pool.

    ``tables[s]`` must hold at least ``ceil((ctx_lens[s] + 1) / block_size)``
    blocks (room for the new token).  Values are drawn in fp32 from a
    ``torch.Generator`` seeded with ``seed`` on ``device`` and rounded to the
    storage dtype (round-to-nearest-even).  With ``outlier_frac > 0`` each
    (token, KV head) key vector is multiplied by ``outlier_mult`` with that
    probability before rounding.  With ``new_in_pool=True`` the new token is
    also laid into its slot (the state after the step's cache write), so a
    decode can be checked on its own.
    """
    ctx_lens = np.asarray(ctx_lens, dtype=np.int64)
    B = len(ctx_lens)
    tdt = DTYPES[dtype]
    device = torch.device(device)
    for s in range(B):
        need = math.ceil((int(ctx_lens[s]) + 1) / block_size)
        if len(tables[s]) < need:
            raise ValueError(f"table of seq {s} too short")
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    H, Hkv, D = num_heads, num_kv_heads, head_dim
    if scale is None:
        scale = 1.0 / math.sqrt(D)

    q = (torch.randn((B, H, D), generator=gen, device=device) * q_std).to(tdt)
    n_ctx = int(ctx_lens.sum())
    k_ctx = torch.randn((n_ctx, Hkv, D), generator=gen, device=device) * kv_std
    v_ctx = torch.randn((n_ctx, Hkv, D), generator=gen, device=device) * kv_std
    k_new = torch.randn((B, Hkv, D), generator=gen, device=device) * kv_std
    v_new = torch.randn((B, Hkv, D), generator=gen, device=device) * kv_std
    if outlier_frac > 0.0:
        m_ctx = torch.rand((n_ctx, Hkv, 1), generator=gen, device=device) < outlier_frac
        m_new = torch.rand((B, Hkv, 1), generator=gen, device=device) < outlier_frac
        k_ctx = torch.where(m_ctx, k_ctx * outlier_mult, k_ctx)
        k_new = torch.where(m_new, k_new * outlier_mult, k_new)
    k_ctx, v_ctx = k_ctx.to(tdt), v_ctx.to(tdt)
    k_new, v_new = k_new.to(tdt), v_new.to(tdt)

    shape = (num_blocks, Hkv, block_size, D)
    k_cache = _nan_or_zero(shape, tdt, device, canary)
    v_cache = _nan_or_zero(shape, tdt, device, canary)

    # where every context token lives: (physical block, row)
    pb_idx = np.empty(n_ctx, dtype=np.int64)
    row_idx = np.empty(n_ctx, dtype=np.int64)
    slot_mapping = np.empty(B, dtype=np.int64)
    off = 0
    for s in range(B):
        L = int(ctx_lens[s])
        pos = np.arange(L)
        tab = np.asarray(tables[s], dtype=np.int64)
        pb_idx[off:off + L] = tab[pos // block_size]
        row_idx[off:off + L] = pos % block_size
        off += L
        slot_mapping[s] = tab[L // block_size] * block_size + L % block_size
    if n_ctx:
        pbt = torch.from_numpy(pb_idx).to(device)
        rwt = torch.from_numpy(row_idx).to(device)
        k_cache[pbt, :, rwt, :] = k_ctx
        v_cache[pbt, :, rwt, :] = v_ctx
    if new_in_pool:
        sl = torch.from_numpy(slot_mapping).to(device)
        k_cache[sl // block_size, :, sl % block_size, :] = k_new
        v_cache[sl // block_size, :, sl % block_size, :] = v_new

    seq_k = seq_v = None
    if keep_seq:
        seq_k, seq_v = [], []
        off = 0
        for s in range(B):
            L = int(ctx_lens[s])
            seq_k.append(torch.cat([k_ctx[off:off + L], k_new[s:s + 1]], 0))
            seq_v.append(torch.cat([v_ctx[off:off + L], v_new[s:s + 1]], 0))
            off += L

    return PagedBatch(
        name=name, dtype=dtype, num_heads=H, num_kv_heads=Hkv, head_dim=D,
        block_size=block_size, num_blocks=num_blocks, scale=float(scale),
        ctx_lens=ctx_lens.astype(np.int32),
        seq_lens=(ctx_lens + 1).astype(np.int32),
        block_tables=_pad_tables(tables, table_width),
        slot_mapping=slot_mapping, q=q, k_cache=k_cache, v_cache=v_cache,
        k_new=k_new, v_new=v_new, seq_k=seq_k, seq_v=seq_v)


# ---------------------------------------------------------------------------
# The five named workloads
# ---------------------------------------------------------------------------

def tiny(device="cpu", canary=True, keep_seq=True, new_in_pool=False) -> PagedBatch:
    """4 seqs holding {1, 7, 16, 33} tokens, 8/2 heads x 64, fp32 N(0,1),
    a 64-block pool handed out as a seeded permutation, scale 1/sqrt(64),
    then one new token per sequence written at its next position."""
    seed = 1
    rng = np.random.default_rng(seed)
    fl = FreeList(64, rng)
    ctx = [1, 7, 16, 33]
    tables = [fl.allocate(L + 1) for L in ctx]
    return build_batch("tiny", ctx_lens=ctx, num_heads=8, num_kv_heads=2,
                       head_dim=64, dtype="f32", num_blocks=64, tables=tables,
                       seed=seed, scale=1.0 / 8.0, device=device, canary=canary,
                       keep_seq=keep_seq, new_in_pool=new_in_pool)


def llama8b_uniform(device="cpu", canary=True, keep_seq=False, batch=64,
                    lo=512, hi=2048, num_blocks=16384, seed=2,
                    new_in_pool=False) -> PagedBatch:
    """Batch 64, 32/8 heads x 128, bf16, q ~ N(0,1), K/V ~ N(0,1)*0.5,
    seq_lens uniform in [512, 2048], tables drawn without replacement from a
    shuffled pool of 16384 blocks."""
    rng = np.random.default_rng(seed)
    seq_lens = rng.integers(lo, hi, size=batch, endpoint=True)
    fl = FreeList(num_blocks, rng)
    tables = [fl.allocate(int(L)) for L in seq_lens]
    return build_batch("llama8b_uniform", ctx_lens=seq_lens - 1, num_heads=32,
                       num_kv_heads=8, head_dim=128, dtype="bf16",
                       num_blocks=num_blocks, tables=tables, seed=seed,
                       device=device, canary=canary, keep_seq=keep_seq,
                       q_std=1.0, kv_std=0.5, new_in_pool=new_in_pool)


def lognormal_lengths(rng: np.random.Generator, batch: int, median=350.0,
                      sigma=1.0, lo=1, hi=4096) -> np.ndarray:
    x = rng.lognormal(mean=math.log(median), sigma=sigma, size=batch)
    return np.clip(np.round(x), lo, hi).astype(np.int64)


def serving_mix(device="cpu", canary=True, keep_seq=False, batch=256,
                seed=3, max_len=4096, new_in_pool=False) -> PagedBatch:
    """Batch 256, 32/8 x 128 bf16, seq_lens lognormal (median 350, sigma 1.0)
    clipped to [1, 4096], pool = ceil(1.2 x blocks needed); each step writes
    one new token per sequence (at position seq_len - 1) and then decodes.
    The block-table width covers the 4096-token maximum."""
    rng = np.random.default_rng(seed)
    seq_lens = lognormal_lengths(rng, batch, hi=max_len)
    need = int(sum(math.ceil(int(L) / BLOCK_SIZE) for L in seq_lens))
    num_blocks = math.ceil(1.2 * need)
    fl = FreeList(num_blocks, rng)
    tables = [fl.allocate(int(L)) for L in seq_lens]
    return build_batch("serving_mix", ctx_lens=seq_lens - 1, num_heads=32,
                       num_kv_heads=8, head_dim=128, dtype="bf16",
                       num_blocks=num_blocks, tables=tables, seed=seed,
                       device=device, canary=canary, keep_seq=keep_seq,
                       q_std=1.0, kv_std=0.5, new_in_pool=new_in_pool,
                       table_width=math.ceil(max_len / BLOCK_SIZE))


def shared_prefix(device="cpu", canary=True, keep_seq=False, batch=128,
                  prefix_blocks=128, lo=64, hi=512, seed=4,
                  private_prefix=False, new_in_pool=False) -> PagedBatch:
    """128 seqs whose tables all start with the same 128 physical blocks (a
    2048-token common prefix), each followed by 64..512 private tokens
    (uniform) in private blocks; 32/8 x 128 bf16.

    With ``private_prefix=True`` the same token data is laid out with a
    private copy of the prefix per sequence (the non-shared twin)."""
    rng = np.random.default_rng(seed)
    n_priv = rng.integers(lo, hi, size=batch, endpoint=True)
    prefix_tokens = prefix_blocks * BLOCK_SIZE
    seq_lens = prefix_tokens + n_priv
    priv_blocks = [math.ceil(int(n) / BLOCK_SIZE) for n in n_priv]
    extra = (batch - 1) * prefix_blocks if private_prefix else 0
    num_blocks = prefix_blocks + sum(priv_blocks) + 64 + extra
    fl = FreeList(num_blocks, rng)
    shared = fl.take(prefix_blocks)
    tables = [shared + fl.take(nb) for nb in priv_blocks]
    gen_seed = seed
    # Values: the shared prefix is one set of tokens for every sequence;
    # draw it once, then each sequence's private tail.
    return _build_shared(tables, shared, fl, seq_lens, prefix_tokens, gen_seed,
                         num_blocks, device, canary, keep_seq, private_prefix,
                         new_in_pool)


def _build_shared(tables, shared, fl, seq_lens, prefix_tokens, seed,
                  num_blocks, device, canary, keep_seq, private_prefix,
                  new_in_pool):
    B = len(tables)
    H, Hkv, D, bs = 32, 8, 128, BLOCK_SIZE
    tdt = torch.bfloat16
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    q = torch.randn((B, H, D), generator=gen, device=device).to(tdt)
    kp = (torch.randn((prefix_tokens, Hkv, D), generator=gen, device=device) * 0.5).to(tdt)
    vp = (torch.randn((prefix_tokens, Hkv, D), generator=gen, device=device) * 0.5).to(tdt)
    shape = (num_blocks, Hkv, bs, D)
    k_cache = _nan_or_zero(shape, tdt, device, canary)
    v_cache = _nan_or_zero(shape, tdt, device, canary)
    pos = np.arange(prefix_tokens)
    sh = np.asarray(shared, dtype=np.int64)
    pbt = torch.from_numpy(sh[pos // bs]).to(device)
    rwt = torch.from_numpy(pos % bs).to(device)
    k_cache[pbt, :, rwt, :] = kp
    v_cache[pbt, :, rwt, :] = vp
    if private_prefix:
        for s in range(1, B):
            copy = fl.take(len(shared))
            ct = torch.tensor(copy, dtype=torch.int64, device=device)
            k_cache[ct] = k_cache[torch.from_numpy(sh).to(device)]
            v_cache[ct] = v_cache[torch.from_numpy(sh).to(device)]
            tables[s] = copy + tables[s][len(shared):]
    ctx_lens = np.asarray(seq_lens, dtype=np.int64) - 1
    k_new_l, v_new_l, seq_k, seq_v = [], [], [], []
    slot_mapping = np.empty(B, dtype=np.int64)
    for s in range(B):
        L = int(ctx_lens[s])
        n_tail = L - prefix_tokens
        kt = (torch.randn((n_tail + 1, Hkv, D), generator=gen, device=device) * 0.5).to(tdt)
        vt = (torch.randn((n_tail + 1, Hkv, D), generator=gen, device=device) * 0.5).to(tdt)
        tab = np.asarray(tables[s], dtype=np.int64)
        p = np.arange(prefix_tokens, L)
        if n_tail:
            k_cache[torch.from_numpy(tab[p // bs]).to(device), :,
                    torch.from_numpy(p % bs).to(device), :] = kt[:n_tail]
            v_cache[torch.from_numpy(tab[p // bs]).to(device), :,
                    torch.from_numpy(p % bs).to(device), :] = vt[:n_tail]
        k_new_l.append(kt[n_tail:])
        v_new_l.append(vt[n_tail:])
        slot_mapping[s] = tab[L // bs] * bs + L % bs
        if new_in_pool:
            k_cache[int(tab[L // bs]), :, L % bs, :] = kt[n_tail]
            v_cache[int(tab[L // bs]), :, L % bs, :] = vt[n_tail]
        if keep_seq:
            seq_k.append(torch.cat([kp, kt], 0))
            seq_v.append(torch.cat([vp, vt], 0))
    return PagedBatch(
        name="shared_prefix" + ("_private" if private_prefix else ""),
        dtype="bf16", num_heads=H, num_kv_heads=Hkv, head_dim=D,
        block_size=bs, num_blocks=num_blocks, scale=1.0 / math.sqrt(D),
        ctx_lens=ctx_lens.astype(np.int32),
        seq_lens=(ctx_lens + 1).astype(np.int32),
        block_tables=_pad_tables(tables), slot_mapping=slot_mapping, q=q,
        k_cache=k_cache, v_cache=v_cache, k_new=torch.cat(k_new_l, 0),
        v_new=torch.cat(v_new_l, 0), seq_k=seq_k if keep_seq else None,
        seq_v=seq_v if keep_seq else None,
        meta={"shared_blocks": list(shared), "prefix_tokens": prefix_tokens})


def cascade_split(b: PagedBatch, prefix_blocks: int):
    """The cascade layout of a batch whose tables all begin with the same
    ``prefix_blocks`` physical blocks: (prefix block ids int32 [P], each
    sequence's own table int32 [B, W - P] (padded), own lengths int32 [B] =
    seq_lens - 16 P).  Raises ValueError if the tables do not share those
    leading blocks or a sequence is shorter than the prefix."""
    P = int(prefix_blocks)
    bt = np.asarray(b.block_tables)
    if P <= 0 or P > bt.shape[1]:
        raise ValueError("prefix_blocks out of range")
    prefix = bt[0, :P]
    if not (bt[:, :P] == prefix[None, :]).all():
        raise ValueError("the tables do not share their first prefix_blocks entries")
    own = np.asarray(b.seq_lens, dtype=np.int64) - BLOCK_SIZE * P
    if (own < 0).any():
        raise ValueError("a sequence is shorter than the prefix")
    rest = bt[:, P:] if bt.shape[1] > P else np.full((bt.shape[0], 1), PAD, np.int32)
    return (np.ascontiguousarray(prefix, dtype=np.int32),
            np.ascontiguousarray(rest, dtype=np.int32), own.astype(np.int32))


def long_context(device="cpu", canary=True, keep_seq=False, batch=8,
                 lo=32768, hi=131072, seed=5, slack=1.02,
                 new_in_pool=False) -> PagedBatch:
    """Batch 8, 64/8 heads x 128 (GQA 8), bf16, seq_lens uniform in
    [32768, 131072], K/V ~ N(0,1)*0.5 with 1% of the (token, KV head) key
    vectors scaled by 8; split into 512-token partitions by the caller."""
    rng = np.random.default_rng(seed)
    seq_lens = rng.integers(lo, hi, size=batch, endpoint=True)
    need = int(sum(math.ceil(int(L) / BLOCK_SIZE) for L in seq_lens))
    num_blocks = math.ceil(slack * need)
    fl = FreeList(num_blocks, rng)
    tables = [fl.allocate(int(L)) for L in seq_lens]
    return build_batch("long_context", ctx_lens=seq_lens - 1, num_heads=64,
                       num_kv_heads=8, head_dim=128, dtype="bf16",
                       num_blocks=num_blocks, tables=tables, seed=seed,
                       device=device, canary=canary, keep_seq=keep_seq,
                       q_std=1.0, kv_std=0.5, outlier_frac=0.01,
                       outlier_mult=8.0, new_in_pool=new_in_pool)


def random_batch(seed: int, *, num_seqs: int, max_len: int, num_heads: int,
                 num_kv_heads: int, head_dim: int, dtype: str, device="cpu",
                 canary=True, keep_seq=True, min_len: int = 0,
                 extra_blocks: int = 8, table_slack: int = 0,
                 kv_std: float = 1.0, new_in_pool=False) -> PagedBatch:
    """A small random batch: context lengths uniform in [min_len, max_len]
    (0 allowed: the sequence then attends over its new token only)."""
    rng = np.random.default_rng(seed)
    ctx = rng.integers(min_len, max_len, size=num_seqs, endpoint=True)
    need = sum(math.ceil((int(L) + 1) / BLOCK_SIZE) for L in ctx)
    num_blocks = need + extra_blocks
    fl = FreeList(num_blocks, rng)
    tables = [fl.allocate(int(L) + 1) for L in ctx]
    width = max(len(t) for t in tables) + table_slack
    return build_batch(f"random{seed}", ctx_lens=ctx, num_heads=num_heads,
                       num_kv_heads=num_kv_heads, head_dim=head_dim,
                       dtype=dtype, num_blocks=num_blocks, tables=tables,
                       seed=seed, device=device, canary=canary,
                       keep_seq=keep_seq, kv_std=kv_std, table_width=width,
                       new_in_pool=new_in_pool)


def multi_query_batch(seed: int, *, num_seqs: int, min_ctx: int, max_ctx: int,
                      n_new, num_heads: int, num_kv_heads: int, head_dim: int,
                      dtype: str, device="cpu", canary=True, keep_seq=True,
                      kv_std: float = 1.0, lens=None, table_width=None) -> PagedBatch:
    """Several new query tokens per sequence (a prefill chunk, or the k+1
    positions of a speculative step), already written to the cache.

    Sequence s holds ``seq_lens[s] = ctx + n_s`` tokens in the pool; its n_s
    query tokens (positions seq_len - n_s .. seq_len - 1) are rows
    ``query_start[s] .. query_start[s+1]`` of ``q`` ([T, H, D]), kept in
    ``meta["query_start"]``.  ``n_new`` is an int or an inclusive (lo, hi)
    range or one count per sequence; ``lens`` optionally fixes the context
    lengths."""
    rng = np.random.default_rng(seed)
    if lens is None:
        ctx = rng.integers(min_ctx, max_ctx, size=num_seqs, endpoint=True)
    else:
        ctx = np.asarray(lens, dtype=np.int64)
    if isinstance(n_new, int):
        n = np.full(num_seqs, n_new, dtype=np.int64)
    elif isinstance(n_new, tuple):
        n = rng.integers(n_new[0], n_new[1], size=num_seqs, endpoint=True)
    else:
        n = np.asarray(n_new, dtype=np.int64)
    total = ctx + n
    # every sequence gets at least one block (an empty one holds no tokens)
    need = sum(math.ceil(max(int(L), 1) / BLOCK_SIZE) for L in total)
    fl = FreeList(need + 8, rng)
    tables = [fl.allocate(max(int(L), 1)) for L in total]
    b = build_batch(f"multi{seed}", ctx_lens=np.maximum(total - 1, 0), num_heads=num_heads,
                    num_kv_heads=num_kv_heads, head_dim=head_dim, dtype=dtype,
                    num_blocks=need + 8, tables=tables, seed=seed, device=device,
                    canary=canary, keep_seq=keep_seq, kv_std=kv_std, new_in_pool=True,
                    table_width=table_width)
    qs = np.zeros(num_seqs + 1, dtype=np.int32)
    qs[1:] = np.cumsum(n)
    gen = torch.Generator(device=torch.device(device))
    gen.manual_seed(int(seed) + 7919)
    T = int(qs[-1])
    q = torch.randn((T, num_heads, head_dim), generator=gen,
                    device=torch.device(device)).to(DTYPES[dtype])
    b = replace(b, q=q, seq_lens=total.astype(np.int32), name=f"multi{seed}")
    b.meta["query_start"] = qs
    b.meta["n_new"] = n.astype(np.int32)
    return b


def spec_verify(device="cpu", canary=True, batch=256, k=3, seed=11,
                max_len=4096) -> PagedBatch:
    """Speculative-decoding verification step: 256 sequences with the
    serving-mix context lengths (lognormal, median 350, sigma 1.0, clipped to
    [1, 4096]), each scoring k = 3 drafted tokens plus the next one (k + 1 = 4
    query rows), 32/8 heads x 128, bf16, K/V ~ N(0,1)*0.5."""
    rng = np.random.default_rng(seed)
    ctx = lognormal_lengths(rng, batch, hi=max_len)
    b = multi_query_batch(seed, num_seqs=batch, min_ctx=0, max_ctx=0, n_new=k + 1,
                          num_heads=32, num_kv_heads=8, head_dim=128, dtype="bf16",
                          device=device, canary=canary, keep_seq=False, kv_std=0.5,
                          lens=ctx, table_width=math.ceil((max_len + k + 1) / BLOCK_SIZE))
    return replace(b, name="spec_verify")


def chunked_prefill_mix(device="cpu", canary=True, batch=128, chunks=4, chunk=512,
                        seed=12, max_len=4096) -> PagedBatch:
    """One mixed step of chunked prefill: ``chunks`` sequences each run a
    ``chunk``-token slice of their prompt on top of 0..3072 earlier prompt
    tokens, next to batch - chunks one-token decodes with serving-mix
    lengths; 32/8 heads x 128, bf16, K/V ~ N(0,1)*0.5."""
    rng = np.random.default_rng(seed)
    ctx = lognormal_lengths(rng, batch, hi=max_len - 1)
    ctx[:chunks] = rng.integers(0, 3072, size=chunks, endpoint=True)
    n = np.ones(batch, dtype=np.int64)
    n[:chunks] = chunk
    b = multi_query_batch(seed, num_seqs=batch, min_ctx=0, max_ctx=0, n_new=n,
                          num_heads=32, num_kv_heads=8, head_dim=128, dtype="bf16",
                          device=device, canary=canary, keep_seq=False, kv_std=0.5,
                          lens=ctx, table_width=math.ceil((max_len + chunk) / BLOCK_SIZE))
    return replace(b, name="chunked_prefill_mix")


# ---------------------------------------------------------------------------
# Copy-on-write
# ---------------------------------------------------------------------------

def cow_mapping(num_blocks: int, pairs: int, seed: int) -> np.ndarray:
    """int64 [pairs, 2] (src, dst): distinct fresh destinations that are never
    a source, sources drawn from the other blocks (a shared block may be
    copied more than once), as copy-on-write produces them."""
    rng = np.random.default_rng(seed)
    ids = rng.permutation(num_blocks)
    dst = ids[:pairs]
    src = rng.choice(ids[pairs:], size=pairs)
    return np.stack([src, dst], 1).astype(np.int64)


def cow_step(device="cpu", layers=32, num_blocks=2048, pairs=256, seed=14,
             fill=True) -> dict:
    """One step's copy-on-write copies for a Llama-3-8B-shaped cache: K and V
    of ``layers`` layers, each [num_blocks, 8, 16, 128] bf16 (32 KiB per
    block), and ``pairs`` (src, dst) copies -- e.g. 256 parallel-sampling
    children each diverging inside their shared last block.  ``fill`` draws
    N(0, 0.5^2) contents (else zeros)."""
    gen = torch.Generator(device=torch.device(device))
    gen.manual_seed(int(seed))
    shape = (num_blocks, 8, BLOCK_SIZE, 128)
    caches = []
    for _ in range(2 * layers):
        if fill:
            caches.append((torch.randn(shape, generator=gen, device=torch.device(device))
                           * 0.5).to(torch.bfloat16))
        else:
            caches.append(torch.zeros(shape, dtype=torch.bfloat16, device=torch.device(device)))
    return {"caches": caches, "mapping": cow_mapping(num_blocks, pairs, seed),
            "block_bytes": 8 * BLOCK_SIZE * 128 * 2, "layers": layers}


# ---------------------------------------------------------------------------
# FP8 (E4M3) pools
# ---------------------------------------------------------------------------

FP8_NAN = 0x7F            # an E4M3 NaN code: the canary of unreferenced FP8 slots


def with_fp8_pool(batch: PagedBatch, seed: int, kv_std: float = 0.5) -> PagedBatch:
    """The same tables, queries and new rows over a pool of E4M3 codes.

    Per KV head j a K scale and a V scale are drawn as ``4 * kv_std / 448``
    times U[0.75, 1.25]; every pool element that holds a token gets the code
    of a N(0, (kv_std / scale_j)^2) draw clamped to [-448, 448] (so real
    values are about N(0, kv_std^2) and the largest ones saturate), and slots
    left as canaries in ``batch`` hold the NaN code.  Codes are uint8 tensors
    [N, H_kv, bs, D]; the scales are float32 [H_kv] in ``meta["k_scale"]`` and
    ``meta["v_scale"]``.  ``q``, ``k_new`` and ``v_new`` keep their 16-bit (or
    f32) values: the step's cache write quantises them."""
    device = batch.device
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed) + 104729)
    Hkv = batch.num_kv_heads
    base = 4.0 * kv_std / 448.0
    scales = []
    for _ in range(2):
        u = torch.rand((Hkv,), generator=gen, device=device) * 0.5 + 0.75
        scales.append((u * base).float())
    pools = []
    for cache, sc in ((batch.k_cache, scales[0]), (batch.v_cache, scales[1])):
        z = torch.randn(cache.shape, generator=gen, device=device)
        z = (z * (kv_std / sc).view(1, Hkv, 1, 1)).clamp_(-448.0, 448.0)
        codes = z.to(torch.float8_e4m3fn).view(torch.uint8)
        codes = torch.where(torch.isnan(cache), torch.full_like(codes, FP8_NAN), codes)
        pools.append(codes.contiguous())
    meta = dict(batch.meta)
    meta["kv"] = "e4m3"
    meta["k_scale"] = scales[0].contiguous()
    meta["v_scale"] = scales[1].contiguous()
    return replace(batch, k_cache=pools[0], v_cache=pools[1], seq_k=None, seq_v=None,
                   name=batch.name + "_fp8", meta=meta)


def serving_mix_fp8(device="cpu", canary=True, new_in_pool=False) -> PagedBatch:
    """The serving mix (batch 256, lognormal lengths, 32/8 x 128, bf16 q and
    new rows) over an E4M3 pool with per-KV-head scales."""
    return with_fp8_pool(serving_mix(device=device, canary=canary, new_in_pool=new_in_pool),
                         seed=13)


def long_context_fp8(device="cpu", canary=True) -> PagedBatch:
    """The long-context batch (8 seqs x 32k..128k tokens, 64/8 x 128, bf16 q)
    over an E4M3 pool with per-KV-head scales."""
    return with_fp8_pool(long_context(device=device, canary=canary), seed=15)


# ---------------------------------------------------------------------------
# Layout transforms used by the invariance tests
# ---------------------------------------------------------------------------

def permute_blocks(batch: PagedBatch, seed: int) -> PagedBatch:
    """The same logical data with every physical block moved: block ``b``
    goes to ``perm[b]``; tables and slot mapping are remapped to match."""
    rng = np.random.default_rng(seed)
    perm = rng.permutation(batch.num_blocks)
    inv = np.argsort(perm)
    dev = batch.device
    inv_t = torch.from_numpy(inv).to(dev)
    k_cache = batch.k_cache[inv_t].contiguous()
    v_cache = batch.v_cache[inv_t].contiguous()
    bt = batch.block_tables.copy()
    valid = bt != PAD
    bt[valid] = perm[bt[valid]].astype(np.int32)
    sm = batch.slot_mapping.copy()
    ok = sm >= 0
    sm[ok] = perm[sm[ok] // batch.block_size] * batch.block_size + sm[ok] % batch.block_size
    return replace(batch, k_cache=k_cache, v_cache=v_cache, block_tables=bt,
                   slot_mapping=sm, name=batch.name + "_perm")


def tables_with_padding(batch: PagedBatch, width: int, pad=PAD) -> np.ndarray:
    """Re-pad the block tables to ``width`` columns filled with ``pad``."""
    out = np.full((batch.num_seqs, width), pad, dtype=np.int32)
    for s in range(batch.num_seqs):
        nb = math.ceil(int(batch.seq_lens[s]) / batch.block_size)
        out[s, :nb] = batch.block_tables[s, :nb]
    return out


CONFIGS = {
    "tiny": tiny,
    "llama8b_uniform": llama8b_uniform,
    "serving_mix": serving_mix,
    "shared_prefix": shared_prefix,
    "long_context": long_context,
}
