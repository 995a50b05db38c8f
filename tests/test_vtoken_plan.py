"""The repacking planner: the library's host planner (pkv_vtoken_plan)
against the independent Python model (oracle/vtoken_plan.py), and both
against the page's example and the invariants repacking must keep.  No GPU."""
import os

import numpy as np
import pytest

import oracle.vtoken_plan as model

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def random_tables(rng, S, bs, NB, keep_frac, shared=0):
    """Token tables of S sequences over private blocks (a few shared ones
    first when `shared` > 0), thinned by a random deletion."""
    perm = list(rng.permutation(np.arange(1, NB)))
    shared_blocks = [perm.pop() for _ in range(shared)]
    tabs = []
    for s in range(S):
        n = int(rng.integers(0, 12 * bs))
        nb = -(-n // bs)
        blocks = (shared_blocks if s < 2 else []) + [perm.pop() for _ in range(nb)]
        sl = [b * bs + o for b in blocks for o in range(bs)][: n + (len(shared_blocks) * bs if s < 2 else 0)]
        keep = rng.random(len(sl)) < keep_frac
        tabs.append([x for x, k in zip(sl, keep) if k or (shared and x // bs in shared_blocks)])
    MT = max(max((len(t) for t in tabs), default=1), 1)
    slots = np.zeros((S, MT), np.int32)
    nt = np.zeros(S, np.int32)
    for s, t in enumerate(tabs):
        slots[s, : len(t)] = t
        nt[s] = len(t)
    return slots, nt, set(shared_blocks)


def check_invariants(plan_fn, apply_fn, slots, nt, bs, NB, shared=frozenset()):
    moves, freed = plan_fn(slots, nt, bs, NB)
    after = apply_fn(slots, moves)
    live = [int(x) for s in range(len(nt)) for x in after[s, : nt[s]]]
    for s in range(len(nt)):
        assert len(set(after[s, : nt[s]].tolist())) == nt[s], "two live tokens of a sequence in one slot"
    priv = [x for x in live if x // bs not in shared]
    assert len(priv) == len(set(priv)), "two sequences in one private slot"
    assert not {x // bs for x in live} & set(freed), "a released block still holds a live token"
    assert not set(freed) & shared, "a shared block was released"
    for s, t, src, dst in moves:
        assert src // bs not in shared and dst // bs not in shared
    for s in range(len(nt)):
        priv = [int(x) for x in after[s, : nt[s]] if int(x) // bs not in shared]
        assert len({x // bs for x in priv}) == -(-len(priv) // bs), "not compacted"
    # planning again finds nothing to do
    m2, f2 = plan_fn(after, nt, bs, NB)
    assert not m2 and not f2
    return moves, freed


def pages_example(plan_fn):
    rows = [ln.split() for ln in open(os.path.join(GOLDEN, "vtoken_repack_example.txt"), encoding="utf-8")
            if ln.strip() and not ln.startswith("#")]
    kv = {r[0]: r[1:] for r in rows if r[0] in ("bs", "NB", "slots", "freed")}
    slots = np.array([[int(x) for x in kv["slots"]]], np.int32)
    moves, freed = plan_fn(slots, np.array([slots.shape[1]], np.int32), int(kv["bs"][0]), int(kv["NB"][0]))
    assert [tuple(m) for m in moves] == [tuple(int(x) for x in r[1:]) for r in rows if r[0] == "move"]
    assert list(freed) == [int(x) for x in kv["freed"]]


def hole_order_case(plan_fn):
    """bs 4: blocks 1 and 2 hold 3 live tokens each, block 3 holds 2.  Eight
    tokens need two blocks: 1 and 2 stay (most live, lower id first); block
    3's tokens fill the free slots lowest first (7, then 11); block 3 goes."""
    slots = np.array([[4, 5, 6, 8, 9, 10, 12, 13]], np.int32)
    moves, freed = plan_fn(slots, np.array([8], np.int32), 4, 4)
    assert [tuple(m) for m in moves] == [(0, 6, 12, 7), (0, 7, 13, 11)]
    assert list(freed) == [3]


def sparse_shared_case(plan_fn, apply_fn):
    """Block 1 is shared by both sequences, each keeping a few of its tokens
    after its own deletions: it is neither emptied nor released, and neither
    sequence moves into or out of it."""
    bs = 4
    slots = np.array([[4, 6, 8, 13, 0], [5, 6, 7, 16, 18]], np.int32)
    nt = np.array([4, 5], np.int32)
    moves, freed = check_invariants(plan_fn, apply_fn, slots, nt, bs, 8, frozenset({1}))
    assert 1 not in freed


def model_pins(mod):
    """Every pin of the planner, run against a planner module."""
    pages_example(mod.plan)
    hole_order_case(mod.plan)
    sparse_shared_case(mod.plan, mod.apply)
    rng = np.random.default_rng(11)
    for shared in (0, 2):
        for keep in (0.2, 0.5, 0.9):
            slots, nt, sh = random_tables(rng, 6, 16, 200, keep, shared)
            check_invariants(mod.plan, mod.apply, slots, nt, 16, 200, sh)


def test_model_pins():
    model_pins(model)


def test_model_rejects_bad_tables():
    with pytest.raises(ValueError):
        model.plan(np.array([[3, 3]], np.int32), np.array([2]), 16, 4)
    with pytest.raises(ValueError):
        model.plan(np.array([[99]], np.int32), np.array([1]), 16, 4)


# ---- the library's planner (C++, pkv_vtoken_plan) against the model

@pytest.fixture(scope="module")
def pkv():
    import __graft_entry__
    __graft_entry__.build()
    import paged_kv_cache_44_gb300 as P
    return P


def _lib_plan(pkv):
    def plan_fn(slots, nt, bs, NB):
        m, f = pkv.vtoken_plan(slots, nt, bs, NB)
        return [tuple(int(x) for x in r) for r in m], [int(x) for x in f]
    return plan_fn


def test_library_planner_pins(pkv):
    fn = _lib_plan(pkv)
    pages_example(fn)
    hole_order_case(fn)
    sparse_shared_case(fn, model.apply)


@pytest.mark.parametrize("seed", range(8))
def test_library_planner_matches_model(pkv, seed):
    rng = np.random.default_rng(100 + seed)
    bs = int(rng.choice([4, 16, 32]))
    slots, nt, sh = random_tables(rng, int(rng.integers(1, 9)), bs, 400, float(rng.uniform(0.05, 1.0)),
                                  int(rng.integers(0, 3)))
    want = model.plan(slots, nt, bs, 400)
    got = _lib_plan(pkv)(slots, nt, bs, 400)
    assert got[0] == [tuple(m) for m in want[0]] and got[1] == want[1]


def test_library_planner_rejects(pkv):
    with pytest.raises(pkv.PkvError):
        pkv.vtoken_plan(np.array([[3, 3]], np.int32), np.array([2], np.int32), 16, 4)
    with pytest.raises(pkv.PkvError):
        pkv.vtoken_plan(np.array([[99]], np.int32), np.array([1], np.int32), 16, 4)
