"""Host block manager (pkv_pool_* in the C ABI) against the pages and against
an independent Python model of the same policy (oracle/block_pool.py).
These tests need no GPU."""
import os

import numpy as np
import pytest

from oracle.block_pool import BlockPoolModel

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module")
def pkv():
    import __graft_entry__
    __graft_entry__.build()
    import paged_kv_cache_44_gb300 as P
    return P


def _golden_lru():
    rows = [ln.split() for ln in open(os.path.join(GOLDEN, "prefix_cache_lru.txt"), encoding="utf-8")
            if ln.strip() and not ln.startswith("#")]
    bs, usable, docs, ntok = map(int, rows[0])
    passes = [(int(r[0]), r[1], int(r[2])) for r in rows[1:]]
    return bs, usable, docs, ntok, passes


def _run_lru(pool, docs, ntok, passes, seed=0):
    rng = np.random.default_rng(seed)
    # documents of random tokens: no two share a prefix
    texts = [rng.integers(1, 150_000, ntok, dtype=np.int32) for _ in range(docs)]
    sid = 0
    hits = []
    for _, order, _ in passes:
        idx = range(docs) if order == "forward" else reversed(range(docs))
        total = 0
        for d in idx:
            got = pool.add_sequence(sid, texts[d])
            assert got is not None
            total += got
            pool.free_sequence(sid)
            sid += 1
        hits.append(total)
    return hits


def test_pages_lru_experiment_library(pkv):
    bs, usable, docs, ntok, passes = _golden_lru()
    pool = pkv.BlockPool(usable + 1, bs, prefix_caching=True)
    assert pool.num_free() == usable
    assert _run_lru(pool, docs, ntok, passes) == [p[2] for p in passes]


def test_pages_lru_experiment_model():
    bs, usable, docs, ntok, passes = _golden_lru()
    pool = BlockPoolModel(usable + 1, bs, prefix_caching=True)
    assert _run_lru(pool, docs, ntok, passes) == [p[2] for p in passes]


def test_capacity_null_block(pkv):
    """21,520 tokens are 1,345 blocks of 16, of which 1,344 are usable
    (first page, section 4): a pool of 1,345 blocks holds 21,504 tokens, not
    21,520."""
    pool = pkv.BlockPool(1345, 16)
    assert pool.num_free() == 1344
    assert pool.add_sequence(1, np.arange(21520) % 1000 + 1) is None
    assert pool.num_free() == 1344                      # nothing changed
    assert pool.add_sequence(2, np.arange(21504) % 1000 + 1) == 0
    assert pool.num_free() == 0
    table, n = pool.block_table(2)
    assert n == 21504 and len(table) == 1344 and 0 not in table


def test_pages_block_table_diagram(pkv):
    """First page, section 4 diagram: request A holds 38 tokens in 3 blocks,
    the last 6/16 full; request B has the same first block of tokens and
    shares that physical block (reference count 2)."""
    rng = np.random.default_rng(3)
    a = rng.integers(1, 30000, 38, dtype=np.int32)
    b = np.concatenate([a[:16], rng.integers(1, 30000, 10, dtype=np.int32)])
    for pool in (pkv.BlockPool(20, 16), BlockPoolModel(20, 16)):
        assert pool.add_sequence(0, a) == 0
        assert pool.add_sequence(1, b) == 16
        ta = list(pool.block_table(0)[0] if hasattr(pool, "close") else pool.block_table(0))
        tb = list(pool.block_table(1)[0] if hasattr(pool, "close") else pool.block_table(1))
        assert len(ta) == 3 and len(tb) == 2 and ta[0] == tb[0] and ta[1:] != tb[1:]
        assert pool.ref_count(ta[0]) == 2 if hasattr(pool, "ref_count") else pool.ref[ta[0]] == 2
        assert 38 - 2 * 16 == 6                          # tokens in A's last block


def _full_hit_recomputes_last_token(pool):
    """First page, section 5: even when every block of a prompt is cached,
    the last token is computed again (its logits are needed), so a prompt of
    exactly two blocks reuses one block, not two."""
    toks = list(range(1, 33))                       # 32 tokens = 2 full blocks of 16
    assert pool.add_sequence(0, toks) == 0
    pool.free_sequence(0)
    return pool.add_sequence(1, toks) == 16


def test_last_token_always_recomputed(pkv):
    assert _full_hit_recomputes_last_token(pkv.BlockPool(10, 16))
    assert _full_hit_recomputes_last_token(BlockPoolModel(10, 16))


def test_fork_then_append_copies_on_write(pkv):
    pool = pkv.BlockPool(10, 16)
    assert pool.add_sequence(7, np.arange(1, 21, dtype=np.int32)) == 0     # 20 tokens: 16 + 4
    t7, _ = pool.block_table(7)
    pool.fork(7, 8)
    assert pool.ref_count(int(t7[1])) == 2
    slot, src, dst = pool.append_token(8, 99)                                # child writes first
    assert src == t7[1] and dst not in t7 and slot == dst * 16 + 4
    t8, n8 = pool.block_table(8)
    assert t8[0] == t7[0] and t8[1] == dst and n8 == 21
    assert pool.ref_count(int(t7[1])) == 1 and pool.ref_count(int(t7[0])) == 2
    slot, src, dst2 = pool.append_token(7, 5)                               # parent: no longer shared
    assert src == -1 and dst2 == -1 and slot == t7[1] * 16 + 4
    pool.free_sequence(7)
    pool.free_sequence(8)
    assert pool.num_free() == 9


def test_extra_key_separates_caches(pkv):
    """Section 5's extra keys (LoRA id, cache salt): the same tokens under
    another key find nothing; back under the first key they hit again.  49
    tokens give 3 full blocks, all reusable (the 49th token is recomputed)."""
    toks = np.arange(1, 50, dtype=np.int32)
    pool = pkv.BlockPool(20, 16)
    assert pool.add_sequence(0, toks) == 0
    pool.free_sequence(0)
    pool.set_extra_key(1234)
    assert pool.add_sequence(1, toks) == 0
    pool.free_sequence(1)
    pool.set_extra_key(0)
    assert pool.add_sequence(2, toks) == 48
    pool.free_sequence(2)
    model = BlockPoolModel(20, 16)
    assert model.add_sequence(0, list(toks)) == 0
    model.free_sequence(0)
    assert model.add_sequence(1, list(toks)) == 48


def test_no_caching_never_hits(pkv):
    pool = pkv.BlockPool(50, 16, prefix_caching=False)
    t = np.arange(1, 100, dtype=np.int32)
    assert pool.add_sequence(0, t) == 0
    pool.free_sequence(0)
    assert pool.add_sequence(1, t) == 0
    assert pool.num_cached() == 0


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("caching", [True, False])
def test_library_matches_model_on_random_operations(pkv, seed, caching):
    """Differential check: the same random sequence of operations on the C++
    manager and on the Python model gives the same tables, slots, copy pairs,
    cache hits and free counts at every step."""
    rng = np.random.default_rng(seed)
    NB, bs = int(rng.integers(8, 80)), int(rng.choice([4, 16]))
    lib_pool = pkv.BlockPool(NB, bs, prefix_caching=caching)
    model = BlockPoolModel(NB, bs, prefix_caching=caching)
    prefixes = [rng.integers(1, 9, int(rng.integers(1, 3 * bs)), dtype=np.int32) for _ in range(4)]
    live, next_id = [], 0
    for _ in range(400):
        op = rng.random()
        if op < 0.35 or not live:
            p = prefixes[int(rng.integers(0, len(prefixes)))]
            toks = np.concatenate([p, rng.integers(1, 9, int(rng.integers(0, 2 * bs)), dtype=np.int32)])
            a, b = lib_pool.add_sequence(next_id, toks), model.add_sequence(next_id, list(toks))
            assert a == b
            if a is not None:
                live.append(next_id)
            next_id += 1
        elif op < 0.75:
            sid = live[int(rng.integers(0, len(live)))]
            tok = int(rng.integers(1, 9))
            assert lib_pool.append_token(sid, tok) == model.append_token(sid, tok)
        elif op < 0.85:
            parent = live[int(rng.integers(0, len(live)))]
            lib_pool.fork(parent, next_id)
            model.fork(parent, next_id)
            live.append(next_id)
            next_id += 1
        else:
            sid = live.pop(int(rng.integers(0, len(live))))
            lib_pool.free_sequence(sid)
            model.free_sequence(sid)
        assert lib_pool.num_free() == model.num_free()
        assert lib_pool.num_cached() == model.num_cached()
        for sid in live:
            t, n = lib_pool.block_table(sid)
            assert list(t) == model.block_table(sid) and n == len(model.seqs[sid]["tokens"])
    for b in range(NB):
        assert lib_pool.ref_count(b) == model.ref[b]


def test_block_table_padding_and_errors(pkv):
    pool = pkv.BlockPool(10, 16)
    pool.add_sequence(3, np.arange(1, 40, dtype=np.int32))
    t, n = pool.block_table(3, max_blocks=6)
    assert n == 39 and list(t[3:]) == [0, 0, 0] and 0 not in t[:3]
    with pytest.raises(pkv.PkvError):
        pool.add_sequence(3, np.arange(1, 5, dtype=np.int32))        # duplicate id
    with pytest.raises(pkv.PkvError):
        pool.free_sequence(99)
    with pytest.raises(pkv.PkvError):
        pool.block_table(3, max_blocks=2)                          # too small


def test_batched_step_matches_single_appends(pkv):
    """pkv_pool_append_tokens gives the same slots and copy pairs as one
    append per sequence (the model), and the batched tables the same rows."""
    rng = np.random.default_rng(5)
    pool, model = pkv.BlockPool(64, 16), BlockPoolModel(64, 16)
    for sid in range(5):
        toks = rng.integers(1, 50, int(rng.integers(1, 40)), dtype=np.int32)
        assert pool.add_sequence(sid, toks) == model.add_sequence(sid, list(toks))
    pool.fork(2, 5)
    model.fork(2, 5)
    ids = np.array([5, 0, 2, 1, 4, 3], np.int64)
    for _ in range(30):
        toks = rng.integers(1, 50, ids.size, dtype=np.int32)
        slots, pairs = pool.append_tokens(ids, toks)
        want = [model.append_token(int(i), int(t)) for i, t in zip(ids, toks)]
        assert list(slots) == [w[0] for w in want]
        assert [tuple(p) for p in pairs] == [(w[1], w[2]) for w in want if w[1] >= 0]
    tabs, cl = pool.block_tables(ids, 8)
    for row, sid, n in zip(tabs, ids, cl):
        t = model.block_table(int(sid))
        assert list(row[: len(t)]) == t and (row[len(t):] == 0).all() and n == len(model.seqs[int(sid)]["tokens"])


def test_batched_step_rejects_without_changing(pkv):
    pool = pkv.BlockPool(4, 4)                       # 3 usable blocks
    pool.add_sequence(0, np.arange(1, 5, dtype=np.int32))      # 1 full block
    pool.add_sequence(1, np.arange(1, 9, dtype=np.int32) + 10)  # 2 full blocks
    free = pool.num_free()
    assert free == 0
    assert pool.append_tokens(np.array([0, 1]), np.array([3, 3])) is None    # needs 2 new blocks
    assert pool.num_free() == free and pool.block_table(0)[1] == 4 and pool.block_table(1)[1] == 8
    with pytest.raises(pkv.PkvError):
        pool.append_tokens(np.array([0, 0]), np.array([1, 2]))               # an id twice
    with pytest.raises(pkv.PkvError):
        pool.append_tokens(np.array([7]), np.array([1]))                     # unknown id
