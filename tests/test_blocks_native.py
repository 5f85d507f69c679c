"""The native block manager and serving loop (include/pa_blocks.h) against the
reference in oracle/block_manager.py: identical decisions -- block tables,
slots, copy-on-write copies, cache hits, free counts, reference counts, loop
events -- on the pages' examples and on random operation sequences.  Host
code only: no GPU."""
import json
import os

import numpy as np
import pytest

from oracle import block_manager as obm
from paged_kv_cache_151_gb300 import blocks
from paged_kv_cache_151_gb300 import build as pabuild

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module", autouse=True)
def _library():
    pabuild.build()


def same_state(nat, ref, live, num_blocks):
    assert nat.num_free() == ref.num_free()
    for sid in live:
        assert nat.table(sid) == ref.table(sid), sid
        assert nat.seq_len(sid) == ref.seq_len(sid)
    assert [nat.refcount(b) for b in range(num_blocks)] == ref.ref


def test_paged_kv_example_tables():
    g = json.load(open(os.path.join(GOLDEN, "pages_sizing.json")))["waste_simulation"]
    rng = np.random.default_rng(g["seed"])
    rng.integers(g["len_lo"], g["len_hi_exclusive"], size=g["num_requests"])
    order = rng.permutation(g["pool_blocks"])
    bm = blocks.BlockManager(64, 16, free_order=order, prefix_caching=True)
    prompt = list(range(1000, 1040))
    assert bm.add_sequence(0, prompt) == 0
    assert bm.table(0) == g["table_a"]
    assert bm.add_sequence(1, prompt[:32] + list(range(5000, 5020))) == 32
    assert bm.table(1) == g["table_b"]
    assert {b: bm.refcount(b) for b in range(64) if bm.refcount(b) > 1} == \
        {int(k): v for k, v in g["shared_refcounts"].items()}


def test_serving_loop_trace_printed_on_the_page():
    g = json.load(open(os.path.join(GOLDEN, "serving_loop.json")))
    names = [r[0] for r in g["requests"]]
    loop = blocks.ServingLoop(blocks.BlockManager(g["pool_blocks"], g["block_size"]))
    for i, (_, tokens, new) in enumerate(g["requests"]):
        loop.submit(i, tokens, new)
    events, more, step = [], True, 0
    while more:
        more, step, ev, _ = loop.step()
        events += [[e[0], e[1], names[e[2]], e[3], e[4]] for e in ev]
    assert events == g["events"]
    assert step == g["all_done_at_step"]


@pytest.mark.parametrize("seed", range(12))
def test_random_operations_match_the_reference(seed):
    rng = np.random.default_rng(seed)
    prefix_caching = bool(seed % 2)
    bs = int(rng.choice([2, 4, 16]))
    nb = int(rng.integers(8, 40))
    order = rng.permutation(nb)
    nat = blocks.BlockManager(nb, bs, free_order=order, prefix_caching=prefix_caching)
    ref = obm.BlockManager(nb, bs, free_order=order, prefix_caching=prefix_caching)
    # a few shared prompt stems so prefix caching finds hits
    stems = [rng.integers(0, 5, size=int(rng.integers(0, 4 * bs))).tolist() for _ in range(3)]
    live, next_id = [], 0
    for _ in range(400):
        op = rng.choice(["add", "add", "append", "append", "append", "fork", "free"])
        if op == "add" or not live:
            stem = stems[int(rng.integers(0, 3))]
            toks = stem + rng.integers(0, 3, size=int(rng.integers(0, 3 * bs))).tolist()
            extra = int(rng.integers(0, 2))
            a = nat.add_sequence(next_id, toks, extra)
            b = ref.add_sequence(next_id, toks, extra)
            assert a == b
            if a is not None:
                live.append(next_id)
            next_id += 1
        elif op == "append":
            sid = live[int(rng.integers(0, len(live)))]
            tok = int(rng.integers(0, 3))
            assert nat.append(sid, tok) == ref.append(sid, tok)
        elif op == "fork":
            sid = live[int(rng.integers(0, len(live)))]
            nat.fork(sid, next_id)
            ref.fork(sid, next_id)
            live.append(next_id)
            next_id += 1
        else:
            sid = live.pop(int(rng.integers(0, len(live))))
            nat.free_sequence(sid)
            ref.free_sequence(sid)
        same_state(nat, ref, live, nb)


@pytest.mark.parametrize("seed", range(6))
def test_random_serving_loops_match_the_reference(seed):
    rng = np.random.default_rng(100 + seed)
    bs = 16
    pool = int(rng.integers(10, 40))
    reqs = [(i, int(rng.integers(1, 6 * bs)), int(rng.integers(1, 60)))
            for i in range(int(rng.integers(2, 12)))]
    reqs = [r for r in reqs if -(-r[1] // bs) + -(-r[2] // bs) + 1 <= pool]
    ref_events, ref_last = obm.serving_loop(reqs, pool, bs)
    loop = blocks.ServingLoop(blocks.BlockManager(pool, bs))
    for r in reqs:
        loop.submit(*r)
    events, more, step = [], True, 0
    while more:
        more, step, ev, _ = loop.step()
        events += ev
    assert events == [tuple(e) for e in ref_events]
    assert step == ref_last


def test_batch_export_and_errors():
    bm = blocks.BlockManager(16, 4)
    bm.add_sequence(7, [1] * 9)
    bm.add_sequence(8, [1] * 2)
    tables, lens = bm.batch([8, 7], width=5, pad=-1)
    assert tables.tolist() == [bm.table(8) + [-1] * 4, bm.table(7) + [-1] * 2]
    assert lens.tolist() == [2, 9]
    with pytest.raises(Exception):
        bm.batch([7], width=2)                 # table wider than the batch
    with pytest.raises(Exception):
        bm.add_sequence(7, [0])                # duplicate id
    with pytest.raises(Exception):
        bm.append(99, 0)                       # unknown id
    assert bm.add_sequence(9, [0] * 100) is None
    loop = blocks.ServingLoop(blocks.BlockManager(2, 16))
    loop.submit(0, 100, 5)                     # can never fit
    with pytest.raises(Exception):
        loop.step()


def brute_common_prefix(bm, ids, bs):
    """The leading blocks all of `ids` share, each full in all of them, from
    their exported tables and lengths (position by position)."""
    tabs = [bm.table(i) for i in ids]
    full = min(bm.seq_len(i) // bs for i in ids)
    p = 0
    while p < full and all(p < len(t) and t[p] == tabs[0][p] for t in tabs):
        p += 1
    return p


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_common_prefix_matches_brute_force(seed):
    """Prompts sharing 0..3 blocks of a system prompt (prefix caching), forks
    sharing a partial last block, appends; random subsets of the live
    sequences against a position-by-position count."""
    rng = np.random.default_rng(seed)
    bs = 16
    bm = blocks.BlockManager(4000, bs, prefix_caching=True)
    system = list(range(100000, 100000 + 3 * bs + 5))
    live = []
    for i in range(40):
        cut = int(rng.integers(0, len(system) + 1))
        own = (rng.integers(0, 1000, size=int(rng.integers(1, 60))) + 1000 * i).tolist()
        assert bm.add_sequence(i, system[:cut] + own) is not None
        live.append(i)
    for i in range(40, 50):
        parent = int(rng.choice(live))
        bm.fork(parent, i)
        live.append(i)
    for _ in range(200):
        sid = int(rng.choice(live))
        bm.append(sid, int(rng.integers(0, 50000)))
    assert bm.common_prefix([]) == 0
    for _ in range(300):
        k = int(rng.integers(1, 8))
        ids = [int(x) for x in rng.choice(live, size=k, replace=False)]
        assert bm.common_prefix(ids) == brute_common_prefix(bm, ids, bs), ids
    # everything that shares the whole system prompt's three full blocks
    whole = [i for i in live if bm.seq_len(i) >= 3 * bs and
             bm.table(i)[:3] == bm.table(live[0])[:3]]
    if len(whole) > 1:
        assert bm.common_prefix(whole) == brute_common_prefix(bm, whole, bs)
    with pytest.raises(KeyError):
        bm.common_prefix([0, 12345])
