"""Reference block manager and toy serving loop -- TEST INFRASTRUCTURE ONLY.

Plain Python written from the pages, used to pin the native block manager of
the package (``csrc/pa_blocks.cpp``) operation by operation.  It shares no
code with it.

What it follows:

* "vLLM: Architecture, PagedAttention & Internals", *The free list and the
  block table*: a free list of physical block ids (``pop()`` takes from its
  end), per-block reference counts, ``allocate`` of ceil(n / block_size)
  blocks, ``append_slot`` that takes a new block only when the token about
  to be written starts one (position % block_size == 0), ``free`` that
  returns a block when its last owner releases it.
* same page, *Copy-on-write for shared blocks*: appending into a shared
  (refcount > 1) partially filled block first moves the writer to a fresh
  block and emits a (src, dst) copy.
* same page, *Prefix caching: reuse KV across requests*: a full block is
  identified by everything before it plus its own tokens (and an extra key
  such as an adapter id or cache salt); a new request reuses its leading
  blocks while they match and allocates the rest; blocks no sequence
  references stay cached until evicted, least recently freed first and, for
  one sequence, leaves before roots.
* "vLLM: High-Throughput Serving with PagedAttention" (lesson 13.15),
  *Practice: try it yourself*: the toy serving loop (admit while the head of
  the queue fits, one token per running request per step, preempt the newest
  request when a block is needed and the pool is empty).

Readings where the pages leave a choice (stated once here, and kept by the
native manager):

* Freed blocks go to the FRONT of the free list (the end is popped), the
  blocks of one sequence in reverse order: never-used blocks are handed out
  first, then the least recently freed, and a sequence's last block before
  its first.  (The page's simplified class appends freed blocks to the end;
  with cached blocks in the list that would evict the newest first.)
* A prompt's full blocks are committed (made matchable) when the request is
  added; decode commits a block when its last slot is written.  A block whose
  identity is already cached stays private.
* ``num_cached`` of a new request counts the tokens of its matched blocks.
"""
from __future__ import annotations

import math


class BlockManager:
    def __init__(self, num_blocks: int, block_size: int = 16, free_order=None,
                 prefix_caching: bool = False):
        self.block_size = block_size
        self.num_blocks = num_blocks
        self.free = list(range(num_blocks)) if free_order is None else [int(b) for b in free_order]
        if sorted(self.free) != list(range(num_blocks)):
            raise ValueError("free_order must be a permutation of the block ids")
        self.ref = [0] * num_blocks
        self.prefix_caching = prefix_caching
        self.key_of = [None] * num_blocks       # identity of a committed block
        self.cached = {}                        # identity -> block
        self.seqs = {}                          # seq id -> dict(table, tokens, extra)

    # ---- allocation primitives ------------------------------------------
    def num_free(self) -> int:
        return len(self.free)

    def _pop(self) -> int:
        blk = self.free.pop()
        key = self.key_of[blk]
        if key is not None:                      # evict: its contents are overwritten
            del self.cached[key]
            self.key_of[blk] = None
        self.ref[blk] = 1
        return blk

    def _release(self, table):
        for blk in reversed(table):              # leaves first, so they are evicted first
            self.ref[blk] -= 1
            if self.ref[blk] == 0:
                self.free.insert(0, blk)

    def blocks_for(self, n_tokens: int) -> int:
        return math.ceil(n_tokens / self.block_size)

    def can_allocate(self, n_tokens: int) -> bool:
        return len(self.free) >= self.blocks_for(n_tokens)

    def _key(self, tokens, i, extra):
        """Identity of full block i of a token sequence: all tokens up to its
        end, and the extra key."""
        return (extra, tuple(tokens[:(i + 1) * self.block_size]))

    # ---- sequences --------------------------------------------------------
    def add_sequence(self, seq_id, tokens, extra=0):
        """Blocks for a prompt; returns the number of tokens whose blocks were
        found cached, or None if the pool cannot hold it (nothing changes)."""
        if seq_id in self.seqs:
            raise ValueError("sequence exists")
        tokens = list(tokens)
        n = len(tokens)
        nb = self.blocks_for(n)
        full = n // self.block_size
        hits = []
        if self.prefix_caching:
            for i in range(full):
                blk = self.cached.get(self._key(tokens, i, extra))
                if blk is None:
                    break
                hits.append(blk)
        # blocks the hits take out of the free list do not count as free
        revived = sum(1 for b in hits if self.ref[b] == 0)
        if len(self.free) - revived < nb - len(hits):
            return None
        table = []
        for blk in hits:
            if self.ref[blk] == 0:
                self.free.remove(blk)
            self.ref[blk] += 1
            table.append(blk)
        for i in range(len(hits), nb):
            blk = self._pop()
            table.append(blk)
            if self.prefix_caching and i < full:
                self._commit(blk, self._key(tokens, i, extra))
        self.seqs[seq_id] = {"table": table, "tokens": tokens, "extra": extra}
        return len(hits) * self.block_size

    def _commit(self, blk, key):
        if key not in self.cached:
            self.cached[key] = blk
            self.key_of[blk] = key

    def fork(self, parent, child):
        p = self.seqs[parent]
        if child in self.seqs:
            raise ValueError("sequence exists")
        for blk in p["table"]:
            self.ref[blk] += 1
        self.seqs[child] = {"table": list(p["table"]), "tokens": list(p["tokens"]),
                            "extra": p["extra"]}

    def append(self, seq_id, token):
        """Slot of the next token, with the copy-on-write copy it needs:
        returns (slot, (src, dst) or None), or None when no block is free
        (nothing changes)."""
        s = self.seqs[seq_id]
        table, tokens = s["table"], s["tokens"]
        pos = len(tokens)
        copy = None
        if pos % self.block_size == 0:           # the token starts a new block
            if not self.free:
                return None
            table.append(self._pop())
        else:
            last = table[-1]
            if self.ref[last] > 1:               # shared: copy before writing
                if not self.free:
                    return None
                new = self._pop()
                self.ref[last] -= 1
                table[-1] = new
                copy = (last, new)
        tokens.append(int(token))
        blk = table[pos // self.block_size]
        if self.prefix_caching and len(tokens) % self.block_size == 0:
            self._commit(blk, self._key(tokens, len(tokens) // self.block_size - 1,
                                        s["extra"]))
        return blk * self.block_size + pos % self.block_size, copy

    def free_sequence(self, seq_id):
        s = self.seqs.pop(seq_id)
        self._release(s["table"])

    def table(self, seq_id):
        return list(self.seqs[seq_id]["table"])

    def seq_len(self, seq_id) -> int:
        return len(self.seqs[seq_id]["tokens"])


class Request:
    """A request of the toy loop: its name, the tokens it holds, the output
    tokens it still has to write."""

    def __init__(self, name, tokens, left):
        self.name, self.tokens, self.left = name, int(tokens), int(left)


def serving_loop(requests, pool_blocks, block_size=16):
    """The pages' toy serving loop run on a BlockManager of ``pool_blocks``
    blocks.  ``requests``: (name, tokens held, output tokens to write), all
    queued at step 0.  Each iteration admits queued requests in order while
    the first one's blocks fit, then advances the step and lets every running
    request (in admission order) write one token; a request that needs a
    block when none is free first preempts the most recently admitted running
    request, which returns to the front of the queue with the tokens it
    holds (to be prefilled again).  Returns the events as (step, what, name,
    tokens, free blocks after the event) and the final step."""
    bm = BlockManager(pool_blocks, block_size)
    queue = [Request(*r) for r in requests]
    running = []
    events = []
    step = 0

    def admit_ready():
        while queue and bm.can_allocate(queue[0].tokens):
            r = queue.pop(0)
            bm.add_sequence(r.name, [0] * r.tokens)
            running.append(r)
            events.append((step, "admit", r.name, r.tokens, bm.num_free()))

    def preempt_newest():
        victim = running.pop()
        bm.free_sequence(victim.name)
        queue.insert(0, victim)
        events.append((step, "preempt", victim.name, victim.tokens, bm.num_free()))
        return victim

    while queue or running:
        admit_ready()
        if not running:
            raise ValueError("the first queued request cannot fit into the pool")
        step += 1
        for r in list(running):
            if r not in running:                  # preempted earlier in this step
                continue
            while bm.append(r.name, 0) is None:   # no block for the next token
                if preempt_newest() is r:
                    break
            if r not in running:
                continue
            r.tokens += 1
            r.left -= 1
            if r.left == 0:
                running.remove(r)
                bm.free_sequence(r.name)
                events.append((step, "finish", r.name, r.tokens, bm.num_free()))
    return events, step
