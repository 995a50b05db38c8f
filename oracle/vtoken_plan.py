"""Repacking plan for token tables -- TEST INFRASTRUCTURE ONLY.

An independent Python statement of the policy the library's host planner
(``pkv_vtoken_plan`` in the C ABI) follows, for differential tests.  Nothing
in the product imports this module.

"LLM推論の「見えないメモリ問題」を解く … vToken", section on asynchronous
repacking: when a deletion policy leaves a block with few surviving tokens,
those tokens move to free space in other blocks and the emptied block is
released at once; the token table is rewritten so the logical order of the
sequence does not change.

Policy, per sequence, over the blocks only that sequence uses (a block that
several sequences reference stays where it is and lends no free slots):
the sequence needs k = ceil(live tokens in its private blocks / bs) blocks;
it keeps the k private blocks with the most live tokens (lower block id
first on ties); its tokens in the other private blocks move, in logical
order, to the free slots of the kept blocks, lowest slot first; the other
private blocks are then empty and are released.
"""
from __future__ import annotations

from collections import Counter, defaultdict
from typing import List, Tuple

import numpy as np


def plan(token_slots: np.ndarray, num_tokens: np.ndarray, bs: int, NB: int) -> Tuple[List[tuple], List[int]]:
    """Returns (moves, freed): moves are (sequence, logical index, src slot,
    dst slot) in sequence then index order; freed are block ids, ascending
    within each sequence, sequences in order."""
    S = len(num_tokens)
    users = defaultdict(set)
    for s in range(S):
        for t in range(int(num_tokens[s])):
            slot = int(token_slots[s, t])
            if not 0 <= slot < NB * bs:
                raise ValueError("slot out of range")
            users[slot // bs].add(s)
    for s in range(S):
        sl = [int(token_slots[s, t]) for t in range(int(num_tokens[s]))]
        if len(sl) != len(set(sl)):
            raise ValueError("two live tokens of one sequence in one slot")
    moves, freed = [], []
    for s in range(S):
        n = int(num_tokens[s])
        slots = [int(token_slots[s, t]) for t in range(n)]
        count = Counter(sl // bs for sl in slots if len(users[sl // bs]) == 1)
        if not count:
            continue
        k = -(-sum(count.values()) // bs)
        if len(count) <= k:
            continue
        order = sorted(count, key=lambda b: (-count[b], b))
        keep, drop = set(order[:k]), set(order[k:])
        used = set(slots)
        holes = [b * bs + o for b in sorted(keep) for o in range(bs) if b * bs + o not in used]
        hi = 0
        for t, sl in enumerate(slots):
            if sl // bs in drop:
                moves.append((s, t, sl, holes[hi]))
                hi += 1
        freed.extend(sorted(drop))
    return moves, freed


def apply(token_slots: np.ndarray, moves) -> np.ndarray:
    """The token table after the moves (a copy)."""
    out = token_slots.copy()
    for s, t, src, dst in moves:
        assert out[s, t] == src
        out[s, t] = dst
    return out
