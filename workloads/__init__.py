"""Seeded synthetic inputs for paged KV-cache decode.

This module builds the *inputs* both the CUDA path and the CPU oracle consume:
sequence lengths, block tables, slot mappings, copy-on-write pairs and
normally distributed values.  It holds none of the method's arithmetic (no
attention, no quantisation, no reading of K/V through a table); the only
index arithmetic is the allocator's bookkeeping that names the slot of each
new token (block id * block_size + offset).  Random numbers come only from
here.

Shapes follow the pages' models ("LLM推論の基礎とvLLMの内部", section 2,
table of Qwen2.5 1.5B / 7B / 72B: layers, K/V heads, head dim 128), the
block size 16 of section 4, and the "100 requests with the same system
prompt" sharing example of "vLLM 内部構造 (2) — PagedAttention", section
"共有".

Value recipe: N(0, 1) draws in float32.  A bf16 input is the float32 draw
with its low 16 bits dropped (round toward zero), which is a way of drawing
bf16 values, not a rounding the method performs.  fp8 caches receive the
float32 draws through the write call of each side, with per-tensor scale
amax / 448.

Physical block 0 is never handed out: it is the reserved "null block" of the
vLLM block pool (first page, section 4), and block-table padding points at
it.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional

import numpy as np

NULL_BLOCK = 0
E4M3_MAX = 448.0

DT_F32, DT_BF16, DT_E4M3 = "f32", "bf16", "e4m3"


@dataclasses.dataclass
class Workload:
    """One decode step's structure (no K/V values)."""
    name: str
    seed: int
    S: int
    Hq: int
    Hkv: int
    d: int
    bs: int
    NB: int
    q_dtype: str
    cache_dtype: str
    context_lens: np.ndarray          # int32 [S]: tokens attended by decode (incl. the new one)
    block_tables: np.ndarray          # int32 [S, MB]; padding = NULL_BLOCK
    slot_mapping: np.ndarray          # int64 [S]: slot of each sequence's new token
    cow_pairs: np.ndarray             # int64 [P, 2]: (src in use, dst free)
    partition_size: int               # 0 = library default
    shared_prefix_blocks: int = 0     # logical blocks shared by the first `shared_seqs`
    shared_seqs: int = 0
    layers_for_bytes: int = 1

    @property
    def g(self) -> int:
        return self.Hq // self.Hkv

    @property
    def MB(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens.max()) if self.S else 0

    @property
    def scale(self) -> float:
        return float(np.float32(1.0) / np.sqrt(np.float32(self.d)))

    def blocks_in_use(self) -> np.ndarray:
        """Sorted unique physical blocks the decode reads."""
        ids = [self.block_tables[s, : -(-int(n) // self.bs)] for s, n in enumerate(self.context_lens)]
        return np.unique(np.concatenate(ids)) if ids else np.zeros(0, np.int32)


def _rng(seed: int, tag: str) -> np.random.Generator:
    return np.random.default_rng([seed, sum(ord(c) << (8 * (i % 4)) for i, c in enumerate(tag))])


# ----------------------------------------------------------------- lengths

def _lengths(name: str, rng: np.random.Generator, S: int) -> np.ndarray:
    if name == "tiny":
        return np.array([1, 15, 16, 37], np.int64) + 1          # one written token each
    if name == "qwen2.5-1.5b":
        return rng.integers(512, 4096, size=S, endpoint=True)
    if name == "qwen2.5-7b-prefix":
        n = np.rint(rng.lognormal(mean=math.log(1024.0), sigma=1.0, size=S))
        n = np.clip(n, 1, 8192).astype(np.int64)
        n[:100] = np.maximum(n[:100], 1025)                      # private tail after the prefix
        return n
    if name == "qwen2.5-72b-long":
        return np.full(S, 32768, np.int64)
    if name.startswith("fp8"):
        return rng.integers(256, 16384, size=S, endpoint=True)
    if name == "qwen2.5-7b-chunked":
        p = min(S, CHUNKED_PROMPTS)
        chunk_end = CHUNK_TOKENS * rng.integers(1, 8192 // CHUNK_TOKENS, size=p, endpoint=True)
        dec = np.clip(np.rint(rng.lognormal(mean=math.log(1024.0), sigma=1.0, size=S - p)), 1, 8192)
        return np.concatenate([chunk_end, dec]).astype(np.int64)
    if name == "qwen2.5-72b-spec":
        return np.full(S, 32768, np.int64)
    raise KeyError(name)


def query_lens(w: "Workload") -> np.ndarray:
    """Queries per sequence: the chunk of the chunked workload's prompts,
    the speculative tokens of the verification workload, else one."""
    if w.name == "qwen2.5-7b-chunked":
        q = np.ones(w.S, np.int64)
        q[: min(w.S, CHUNKED_PROMPTS)] = CHUNK_TOKENS
        return np.minimum(q, w.context_lens).astype(np.int32)
    if w.name == "qwen2.5-72b-spec":
        return np.minimum(SPEC_QUERIES, w.context_lens).astype(np.int32)
    return np.minimum(1, w.context_lens).astype(np.int32)


def query_start(qlens: np.ndarray) -> np.ndarray:
    """Offsets of each sequence's queries in the packed query array [S + 1]."""
    return np.concatenate([[0], np.cumsum(np.asarray(qlens, np.int64))]).astype(np.int32)


SHAPES: Dict[str, dict] = {
    # 1 layer, GQA group 2, fp32 everything
    "tiny": dict(S=4, Hq=4, Hkv=2, d=64, bs=16, q_dtype=DT_F32, cache_dtype=DT_F32,
                 partition_size=0, NB=16, seed=1),
    # Qwen2.5-1.5B: 12 query heads, 2 K/V heads
    "qwen2.5-1.5b": dict(S=64, Hq=12, Hkv=2, d=128, bs=16, q_dtype=DT_BF16,
                         cache_dtype=DT_BF16, partition_size=0, seed=2),
    # Qwen2.5-7B: 28 query heads, 4 K/V heads; 100 sequences share a 1024-token prefix
    "qwen2.5-7b-prefix": dict(S=256, Hq=28, Hkv=4, d=128, bs=16, q_dtype=DT_BF16,
                              cache_dtype=DT_BF16, partition_size=0, seed=3,
                              shared_seqs=100, shared_tokens=1024),
    # Qwen2.5-72B: 64 query heads, 8 K/V heads, 32K context, 512-token partitions
    "qwen2.5-72b-long": dict(S=32, Hq=64, Hkv=8, d=128, bs=16, q_dtype=DT_BF16,
                             cache_dtype=DT_BF16, partition_size=512, seed=4),
    # fp8 E4M3 KV with per-tensor scales, block size 16 or 32
    "fp8-bs16": dict(S=128, Hq=28, Hkv=4, d=128, bs=16, q_dtype=DT_BF16,
                     cache_dtype=DT_E4M3, partition_size=0, seed=5),
    "fp8-bs32": dict(S=128, Hq=28, Hkv=4, d=128, bs=32, q_dtype=DT_BF16,
                     cache_dtype=DT_E4M3, partition_size=0, seed=5),
    # Several queries per sequence.  Chunked prefill next to decodes
    # ("LLM推論の基礎とvLLMの内部", section 6: running requests first, then
    # prompts cut to the rest of the step's token budget, which section 7's
    # table puts at 16384 tokens on cards with >= 160 GiB): 16 prompts each
    # computing a 512-token chunk that ends at a multiple of 512 up to 8,192,
    # beside 48 decoding sequences (one query each) -- 8,240 query tokens.
    "qwen2.5-7b-chunked": dict(S=64, Hq=28, Hkv=4, d=128, bs=16, q_dtype=DT_BF16,
                               cache_dtype=DT_BF16, partition_size=0, seed=6),
    # Speculative verification at long context (same page, section 3: a
    # request's tokens to compute include its speculative ones): the
    # accepted token plus 4 proposed ones, 5 queries per sequence.
    "qwen2.5-72b-spec": dict(S=32, Hq=64, Hkv=8, d=128, bs=16, q_dtype=DT_BF16,
                             cache_dtype=DT_BF16, partition_size=0, seed=8),
}

CHUNK_TOKENS = 512          # prefill chunk of the chunked workload
CHUNKED_PROMPTS = 16        # sequences of that workload computing a chunk
SPEC_QUERIES = 5            # 1 accepted + 4 proposed tokens

COW_PAIRS = 64


def make(name: str, *, seed: Optional[int] = None, S: Optional[int] = None,
         lengths: Optional[np.ndarray] = None, cow_pairs: int = COW_PAIRS,
         spare_blocks: int = 0, shared_seqs: Optional[int] = None) -> Workload:
    """Build the structure of workload `name` (see SHAPES).

    Blocks are handed out from a seeded random permutation of the pool's
    non-null blocks, in logical order (sequence 0's blocks first).  Shared
    prefix blocks are allocated once and referenced by every sharer.  The
    pool has exactly the blocks in use, plus `cow_pairs` free blocks used as
    copy-on-write destinations, plus `spare_blocks`, plus the null block
    (the tiny case uses a fixed pool of 16).  `shared_seqs` overrides how
    many leading sequences share the prefix (for prefix workloads)."""
    cfg = dict(SHAPES[name])
    seed = cfg.pop("seed") if seed is None else seed
    cfg.pop("seed", None)
    cfg_shared = cfg.pop("shared_seqs", 0)
    shared_seqs = cfg_shared if shared_seqs is None else shared_seqs
    shared_tokens = cfg.pop("shared_tokens", 0)
    fixed_nb = cfg.pop("NB", None)
    if S is not None:
        cfg["S"] = S
    S_ = cfg["S"]
    bs = cfg["bs"]
    rng = _rng(seed, "structure:" + name)
    ctx = np.asarray(lengths if lengths is not None else _lengths(name, rng, S_), np.int64)
    assert ctx.shape == (S_,)
    nblk = -(-ctx // bs)
    shared_seqs = min(shared_seqs, S_)
    pre = shared_tokens // bs if shared_seqs else 0
    if pre:
        assert (ctx[:shared_seqs] > shared_tokens).all()
    needed = int(nblk.sum()) - (shared_seqs - 1) * pre if pre else int(nblk.sum())
    NB = fixed_nb if fixed_nb is not None else needed + cow_pairs + spare_blocks + 1
    assert NB - 1 >= needed + (cow_pairs if fixed_nb is None else 0), "pool too small"
    perm = rng.permutation(np.arange(1, NB, dtype=np.int64))
    MB = int(nblk.max()) if S_ else 1
    tables = np.full((S_, max(MB, 1)), NULL_BLOCK, np.int32)
    nxt = 0
    prefix_ids = None
    if pre:
        prefix_ids = perm[nxt: nxt + pre]
        nxt += pre
    for s in range(S_):
        j0 = 0
        if pre and s < shared_seqs:
            tables[s, :pre] = prefix_ids
            j0 = pre
        k = int(nblk[s]) - j0
        tables[s, j0: j0 + k] = perm[nxt: nxt + k]
        nxt += k
    free = perm[nxt:]
    # the new token of each sequence sits at position ctx-1
    pos = ctx - 1
    slots = np.where(ctx > 0,
                     tables[np.arange(S_), np.maximum(pos, 0) // bs].astype(np.int64) * bs + pos % bs,
                     -1).astype(np.int64)
    in_use = np.unique(tables[tables != NULL_BLOCK]) if S_ else np.zeros(0, np.int64)
    P = min(cow_pairs, len(free), len(in_use))
    src = rng.choice(in_use, size=P, replace=False) if P else np.zeros(0, np.int64)
    dst = rng.choice(free, size=P, replace=False) if P else np.zeros(0, np.int64)
    cow = np.stack([src, dst], axis=1).astype(np.int64) if P else np.zeros((0, 2), np.int64)
    return Workload(name=name, seed=seed, NB=int(NB), context_lens=ctx.astype(np.int32),
                    block_tables=tables, slot_mapping=slots, cow_pairs=cow,
                    shared_prefix_blocks=pre, shared_seqs=shared_seqs if pre else 0, **cfg)


# ------------------------------------------------------------------ values

def host_normal(seed: int, tag: str, shape) -> np.ndarray:
    """float32 N(0, 1) draws, one stream per (seed, tag)."""
    return _rng(seed, tag).standard_normal(size=shape, dtype=np.float32)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Draw bf16 values from float32 draws: keep the upper 16 bits."""
    return (np.ascontiguousarray(x, np.float32).view(np.uint32) >> 16).astype(np.uint16)


def bf16_bits_to_float32(h: np.ndarray) -> np.ndarray:
    return (np.asarray(h, np.uint16).astype(np.uint32) << 16).view(np.float32)


def e4m3_scale(values: np.ndarray) -> float:
    """Per-tensor fp8 scale amax / 448, as float32."""
    amax = np.float32(np.abs(values).max()) if values.size else np.float32(1.0)
    return float(amax / np.float32(E4M3_MAX))


@dataclasses.dataclass
class HostValues:
    """Host-side values of one workload (float32 draws).

    k_pool/v_pool hold the draws of the blocks listed in `blocks`
    ([len(blocks), bs, Hkv, d]); query is [S, Hq, d]; new_k/new_v are the
    step's new tokens [S, Hkv, d]."""
    blocks: np.ndarray
    k_pool: np.ndarray
    v_pool: np.ndarray
    query: np.ndarray
    new_k: np.ndarray
    new_v: np.ndarray
    k_scale: float = 1.0
    v_scale: float = 1.0


def host_values(w: Workload, blocks: Optional[np.ndarray] = None) -> HostValues:
    """Draw values for `blocks` (default: every block of the pool)."""
    blocks = np.arange(w.NB, dtype=np.int64) if blocks is None else np.asarray(blocks, np.int64)
    shp = (len(blocks), w.bs, w.Hkv, w.d)
    k = host_normal(w.seed, "k-pool:%d" % len(blocks), shp)
    v = host_normal(w.seed, "v-pool:%d" % len(blocks), shp)
    q = host_normal(w.seed, "query", (w.S, w.Hq, w.d))
    nk = host_normal(w.seed, "new-k", (w.S, w.Hkv, w.d))
    nv = host_normal(w.seed, "new-v", (w.S, w.Hkv, w.d))
    hv = HostValues(blocks=blocks, k_pool=k, v_pool=v, query=q, new_k=nk, new_v=nv)
    if w.cache_dtype == DT_E4M3:
        hv.k_scale = e4m3_scale(k)
        hv.v_scale = e4m3_scale(v)
    return hv


def sample_sequences(w: Workload, count: int, seed_tag: str = "sample") -> np.ndarray:
    """Sequences whose outputs a sampled check recomputes: the shortest, the
    longest, a sharer of the prefix when there is one, and random others."""
    rng = _rng(w.seed, seed_tag)
    pick: List[int] = [int(np.argmin(w.context_lens)), int(np.argmax(w.context_lens))]
    if w.shared_seqs:
        pick.append(int(rng.integers(0, w.shared_seqs)))
    rest = [s for s in rng.permutation(w.S) if s not in pick]
    pick += [int(s) for s in rest[: max(0, count - len(pick))]]
    return np.array(sorted(set(pick))[:max(count, 1)], np.int64)


def sub_workload(w: Workload, seqs: np.ndarray) -> Workload:
    """The same workload restricted to `seqs`, with the blocks they read
    renumbered densely (block 0 stays the null block).  Returns a Workload
    whose `NB` covers just those blocks; `renumber` maps old -> new ids."""
    seqs = np.asarray(seqs, np.int64)
    ctx = w.context_lens[seqs]
    tabs = w.block_tables[seqs]
    nblk = -(-ctx.astype(np.int64) // w.bs)
    MB = max(int(nblk.max()) if len(seqs) else 1, 1)
    used = np.unique(np.concatenate([tabs[i, : nblk[i]] for i in range(len(seqs))] + [np.zeros(1, np.int32)]))
    newid = {int(b): i for i, b in enumerate(used)}
    t2 = np.zeros((len(seqs), MB), np.int32)
    for i in range(len(seqs)):
        t2[i, : nblk[i]] = [newid[int(b)] for b in tabs[i, : nblk[i]]]
    pos = ctx.astype(np.int64) - 1
    slots = np.where(ctx > 0, t2[np.arange(len(seqs)), np.maximum(pos, 0) // w.bs].astype(np.int64)
                     * w.bs + pos % w.bs, -1).astype(np.int64)
    sw = dataclasses.replace(w, S=len(seqs), NB=len(used), context_lens=ctx.copy(),
                             block_tables=t2, slot_mapping=slots,
                             cow_pairs=np.zeros((0, 2), np.int64))
    sw.renumber = used  # type: ignore[attr-defined]
    return sw


# ------------------------------------------------------ device-side draws

def device_normal(seed: int, tag: int, numel: int, device="cuda"):
    """float32 N(0, 1) draws from torch's seeded generator on `device`
    (used where host draws of several GB would take too long)."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1000003 + tag)
    return torch.randn(numel, generator=g, device=device, dtype=torch.float32)


def device_bf16_from_draws(x):
    """bf16 values from float32 draws on the device: keep the upper 16 bits
    (the same drawing recipe as bf16_bits)."""
    import torch
    return (x.view(torch.int32) >> 16).to(torch.int16).view(torch.bfloat16)


def device_pool_chunks(seed: int, which: int, numel: int, device="cuda", chunk: int = 1 << 26):
    """Yield (offset, float32 draws) covering `numel` pool elements."""
    for i, c0 in enumerate(range(0, numel, chunk)):
        n = min(chunk, numel - c0)
        yield c0, device_normal(seed, which * 100000 + i, n, device)


# ------------------------------------------------------------- token tables

def token_tables(w: Workload, keep_frac: float, seed_tag: str = "deletion"):
    """Token tables after a deletion policy thinned each sequence of `w`: every
    token survives with probability keep_frac (at least one per non-empty
    sequence).  Returns (token_slots int32 [S, MT], num_tokens int32 [S]): the
    survivors' slots (block * bs + offset, from the block table) in logical
    order, and their counts."""
    rng = _rng(w.seed, seed_tag)
    MT = max(int(w.context_lens.max()) if w.S else 1, 1)
    slots = np.zeros((w.S, MT), np.int32)
    nt = np.zeros(w.S, np.int32)
    for s in range(w.S):
        n = int(w.context_lens[s])
        keep = rng.random(n) < keep_frac
        if n and not keep.any():
            keep[int(rng.integers(0, n))] = True
        t = np.nonzero(keep)[0]
        slots[s, : t.size] = w.block_tables[s, t // w.bs].astype(np.int64) * w.bs + t % w.bs
        nt[s] = t.size
    return slots, nt
