"""Plain model of the host block manager -- TEST INFRASTRUCTURE ONLY.

Only the tests use it.  It shares no code with the library's C++ manager: it
keeps the same policy with Python lists and dicts, and it identifies a
cached block by the exact token prefix it ends (a tuple), where the library
uses a 64-bit hash chain.

The policy follows "LLM推論の基礎とvLLMの内部":
  section 4 -- blocks of `block_size` tokens, handed out one at a time; a
    block table per sequence; block 0 reserved as the null block; a free
    queue; reference counts and copy-on-write for shared blocks;
  section 5 -- only full blocks are cached, keyed by their whole prefix
    (parent, own tokens, extra key); a prompt's cached prefix is reused in
    whole blocks but the last prompt token is always recomputed; a finished
    sequence returns its blocks last-first, and the queue is reused from
    its front (least recently freed first);
and, where the pages are silent, a free block with no cached contents is
handed out before any cached block.
"""
from __future__ import annotations

from typing import Dict, List, Optional, Tuple


class BlockPoolModel:
    def __init__(self, num_blocks: int, block_size: int, prefix_caching: bool = True, extra_key: int = 0):
        assert num_blocks >= 2 and block_size >= 1
        self.bs = block_size
        self.caching = prefix_caching
        self.extra_key = extra_key
        self.ref = [0] * num_blocks
        self.queue: List[int] = list(range(1, num_blocks))   # front (index 0) is reused first
        self.key_of: Dict[int, tuple] = {}                  # cached block -> its prefix key
        self.block_of: Dict[tuple, int] = {}                 # prefix key -> cached block
        self.seqs: Dict[int, dict] = {}

    # -- helpers
    def _key(self, tokens: List[int], j: int) -> tuple:
        """Identity of full block j: every token up to its end, and the extra key."""
        return (self.extra_key, tuple(tokens[: (j + 1) * self.bs]))

    def _take(self) -> int:
        b = self.queue.pop(0)
        if b in self.key_of:
            k = self.key_of.pop(b)
            if self.block_of.get(k) == b:
                del self.block_of[k]
        self.ref[b] = 1
        return b

    def _release(self, b: int) -> None:
        self.ref[b] -= 1
        if self.ref[b] == 0:
            if b in self.key_of:
                self.queue.append(b)          # cached: kept as long as possible
            else:
                self.queue.insert(0, b)       # nothing worth keeping: reused first

    def _cache(self, seq: dict, j: int) -> None:
        if not self.caching:
            return
        b = seq["table"][j]
        k = self._key(seq["tokens"], j)
        if b in self.key_of or k in self.block_of:
            return
        self.key_of[b] = k
        self.block_of[k] = b

    # -- operations
    def num_free(self) -> int:
        return len(self.queue)

    def num_cached(self) -> int:
        return len(self.block_of)

    def add_sequence(self, sid: int, tokens: List[int]) -> Optional[int]:
        """Returns the number of cached prompt tokens, or None if the pool
        has too few free blocks (then nothing changes)."""
        assert sid not in self.seqs and len(tokens) >= 1
        n = len(tokens)
        nblk = -(-n // self.bs)
        hits = []
        if self.caching:
            while (len(hits) < n // self.bs and (len(hits) + 1) * self.bs <= n - 1
                   and self._key(tokens, len(hits)) in self.block_of):
                hits.append(self.block_of[self._key(tokens, len(hits))])
        held = sum(1 for b in hits if self.ref[b] == 0)
        if nblk - len(hits) > len(self.queue) - held:
            return None
        seq = {"table": [], "tokens": list(tokens)}
        for b in hits:
            if self.ref[b] == 0:
                self.queue.remove(b)
            self.ref[b] += 1
            seq["table"].append(b)
        while len(seq["table"]) < nblk:
            seq["table"].append(self._take())
        for j in range(n // self.bs):
            self._cache(seq, j)
        self.seqs[sid] = seq
        return len(hits) * self.bs

    def append_token(self, sid: int, token: int) -> Optional[Tuple[int, int, int]]:
        """Returns (slot, cow_src, cow_dst) -- cow_* are -1 without a copy --
        or None if a needed block is not available."""
        seq = self.seqs[sid]
        pos = len(seq["tokens"])
        src = dst = -1
        if pos % self.bs == 0:
            if not self.queue:
                return None
            seq["table"].append(self._take())
        elif self.ref[seq["table"][-1]] > 1:
            if not self.queue:
                return None
            src = seq["table"][-1]
            dst = self._take()
            self._release(src)
            seq["table"][-1] = dst
        seq["tokens"].append(token)
        if len(seq["tokens"]) % self.bs == 0:
            self._cache(seq, len(seq["tokens"]) // self.bs - 1)
        return seq["table"][-1] * self.bs + pos % self.bs, src, dst

    def fork(self, parent: int, child: int) -> None:
        assert child not in self.seqs
        p = self.seqs[parent]
        for b in p["table"]:
            self.ref[b] += 1
        self.seqs[child] = {"table": list(p["table"]), "tokens": list(p["tokens"])}

    def free_sequence(self, sid: int) -> None:
        for b in reversed(self.seqs.pop(sid)["table"]):
            self._release(b)

    def block_table(self, sid: int) -> List[int]:
        return list(self.seqs[sid]["table"])
