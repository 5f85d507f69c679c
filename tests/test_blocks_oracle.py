"""Pins of the reference block manager and serving loop (oracle/block_manager.py)
against numbers and traces printed on the pages, and against properties the
pages state."""
import json
import os

import numpy as np
import pytest

from oracle import block_manager as obm

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def pages_free_list():
    """The free list of paged_kv.py: default_rng(7), 40 request lengths drawn
    first, then a permutation of 64 block ids."""
    g = golden("pages_sizing.json")["waste_simulation"]
    rng = np.random.default_rng(g["seed"])
    rng.integers(g["len_lo"], g["len_hi_exclusive"], size=g["num_requests"])
    return rng.permutation(g["pool_blocks"]), g


def test_tables_of_the_paged_kv_example_by_prefix_caching():
    order, g = pages_free_list()
    bm = obm.BlockManager(64, 16, free_order=order, prefix_caching=True)
    prompt = list(range(1000, 1000 + g["table_a_tokens"]))
    assert bm.add_sequence("A", prompt) == 0
    assert bm.table("A") == g["table_a"]
    # B has the same 32-token system prompt, then 20 tokens of its own
    b_tokens = prompt[:16 * g["table_b_shared_blocks"]] + list(range(5000, 5000 +
                                                                  g["table_b_new_tokens"]))
    assert bm.add_sequence("B", b_tokens) == 32
    assert bm.table("B") == g["table_b"]
    shared = {blk: bm.ref[blk] for blk in range(64) if bm.ref[blk] > 1}
    assert shared == {int(k): v for k, v in g["shared_refcounts"].items()}


def test_worked_example_capacities():
    g = golden("pages_sizing.json")["worked_pool_example"]
    n = g["num_blocks"]

    def fill(make, prefix_caching=False):
        bm = obm.BlockManager(n, 16, prefix_caching=prefix_caching)
        count = 0
        while bm.add_sequence(count, make(count)) is not None:
            count += 1
        return count

    assert fill(lambda i: [0] * g["short_request_tokens"]) == g["short_requests_fit"]
    assert fill(lambda i: [0] * g["reserved_tokens"]) == g["reserved_requests_fit"]
    assert fill(lambda i: [0] * g["long_chat_tokens"]) == g["long_chats_fit"]
    system = list(range(g["shared_prompt_tokens"]))
    own = g["long_chat_tokens"] - g["shared_prompt_tokens"]

    def chat(i):                              # shared policy text, then the chat's own tokens
        return system + [100000 + i * own + k for k in range(own)]
    assert fill(chat, prefix_caching=True) == g["shared_chats_fit"]

    def named_first(i):                        # the customer's name before the policy text
        return [200000 + i] + system + [100000 + i * own + k for k in range(own - 1)]
    assert fill(named_first, prefix_caching=True) == g["long_chats_fit"]


def test_cached_system_prompt_prefills_only_the_new_tokens():
    """A 4000-token cached prompt and 50 new tokens: about 80x less prefill."""
    bm = obm.BlockManager(1000, 16, prefix_caching=True)
    system = list(range(4000))
    bm.add_sequence("first", system)
    cached = bm.add_sequence("second", system + list(range(9000, 9050)))
    assert cached == 4000
    assert round((4000 + 50) / (4050 - cached)) in (80, 81)


def test_prefixes_diverging_at_token_5_share_nothing():
    bm = obm.BlockManager(100, 16, prefix_caching=True)
    base = list(range(64))
    bm.add_sequence(0, base)
    other = list(base)
    other[5] = -1
    assert bm.add_sequence(1, other) == 0
    assert bm.add_sequence(2, base) == 64                     # identical: every block
    assert bm.add_sequence(3, base[:40] + [7] * 24) == 32     # equal through token 39
    assert bm.add_sequence(4, base[:15]) == 0                 # only full blocks match
    assert bm.add_sequence(5, base, extra=3) == 0             # another adapter / salt
    assert bm.add_sequence(6, base[16:32]) == 0               # same tokens, other position


def test_append_slot_takes_a_block_only_at_block_starts():
    bm = obm.BlockManager(20, 16)
    bm.add_sequence(0, [])
    grown = []
    for pos in range(100):
        before = len(bm.table(0))
        slot, copy = bm.append(0, pos)
        assert copy is None
        if len(bm.table(0)) != before:
            grown.append(pos)
        assert slot == bm.table(0)[pos // 16] * 16 + pos % 16
    assert grown == [0, 16, 32, 48, 64, 80, 96]
    assert bm.num_free() == 20 - 7


def test_copy_on_write_of_a_shared_partial_block():
    bm = obm.BlockManager(10, 16, free_order=list(range(10)))
    bm.add_sequence("p", list(range(20)))                    # blocks 9, 8
    bm.fork("p", "c")
    assert [bm.ref[b] for b in (9, 8)] == [2, 2]
    slot, copy = bm.append("c", 99)                          # writes into shared block 8
    assert copy == (8, 7) and bm.table("c") == [9, 7] and bm.table("p") == [9, 8]
    assert (bm.ref[8], bm.ref[7], bm.ref[9]) == (1, 1, 2)
    assert slot == 7 * 16 + 4
    slot, copy = bm.append("p", 98)                          # parent's block is its own now
    assert copy is None and slot == 8 * 16 + 4


def test_release_keeps_cached_blocks_and_evicts_leaves_first():
    bm = obm.BlockManager(6, 4, free_order=[5, 4, 3, 2, 1, 0], prefix_caching=True)
    bm.add_sequence("a", list(range(12)))                    # blocks 0, 1, 2
    bm.free_sequence("a")
    assert bm.free == [0, 1, 2, 5, 4, 3]                     # root 0 in front, leaf 2 last
    assert bm.add_sequence("b", list(range(8))) == 8         # revives 0 and 1
    bm.add_sequence("c", [50] * 4)                           # never-used block 3 first
    assert bm.table("c") == [3]
    bm.add_sequence("d", [60] * 8)                           # then 4, 5
    bm.add_sequence("e", [70] * 4)                           # now evict: leaf 2 goes
    assert bm.table("e") == [2]
    assert bm.add_sequence("f", list(range(12))) is None     # pool empty


def test_serving_loop_trace_printed_on_the_page():
    g = golden("serving_loop.json")
    events, last = obm.serving_loop([tuple(r) for r in g["requests"]], g["pool_blocks"],
                                    g["block_size"])
    assert [list(e) for e in events] == g["events"]
    assert last == g["all_done_at_step"]


# planted mistakes in a copy of the reference: each must fail a pin above
MUTATIONS = {
    "new_block_every_step": ("if pos % self.block_size == 0:           # the token starts a new block",
                             "if True:"),
    "free_to_the_end": ("self.free.insert(0, blk)", "self.free.append(blk)"),
    "roots_before_leaves": ("for blk in reversed(table):", "for blk in table:"),
    "key_without_prefix": ("return (extra, tuple(tokens[:(i + 1) * self.block_size]))",
                           "return (extra, tuple(tokens[i * self.block_size:(i + 1) * self.block_size]))"),
    "no_copy_on_write": ("if self.ref[last] > 1:", "if False:"),
    "preempt_oldest": ("victim = running.pop()", "victim = running.pop(0)"),
}


def _pins_hold(mod) -> bool:
    global obm
    saved = obm
    obm = mod
    try:
        for fn in (test_tables_of_the_paged_kv_example_by_prefix_caching,
                   test_cached_system_prompt_prefills_only_the_new_tokens,
                   test_prefixes_diverging_at_token_5_share_nothing,
                   test_append_slot_takes_a_block_only_at_block_starts,
                   test_copy_on_write_of_a_shared_partial_block,
                   test_release_keeps_cached_blocks_and_evicts_leaves_first,
                   test_serving_loop_trace_printed_on_the_page):
            try:
                fn()
            except (AssertionError, ValueError, KeyError, IndexError, TypeError):
                return False
        return True
    finally:
        obm = saved


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name):
    import types
    old, new = MUTATIONS[name]
    src = open(obm.__file__).read()
    assert src.count(old) == 1, name
    mod = types.ModuleType("variant")
    exec(compile(src.replace(old, new), "variant", "exec"), mod.__dict__)
    assert not _pins_hold(mod), f"planted mistake '{name}' was not caught"


def test_unmodified_reference_passes_the_compact_pins():
    assert _pins_hold(obm)
