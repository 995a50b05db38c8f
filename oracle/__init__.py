"""CPU oracle for paged KV-cache decode attention -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU
baseline leg may import this package.  The product library never does, and
this package never imports the product: the two share no code.

The arithmetic lives in ``pkv_oracle.c`` (plain C, fp64 accumulation); this
module compiles it with gcc and marshals numpy arrays into it.  Arrays carry
raw element bits: fp32 as ``float32``, bf16 as ``uint16`` (the upper half of a
binary32) and fp8 E4M3 as ``uint8`` codes.

What each function computes, and the pages it follows:

* ``paged_kv_write``  -- reshape_and_cache: each new token's K/V goes to the
  slot its slot mapping names ("LLM推論の基礎とvLLMの内部", section 4:
  physical blocks are handed out one at a time as tokens arrive).
* ``paged_attention_decode`` -- gather every cached token of a sequence
  through its block table, then textbook softmax attention in fp64
  (same page, section 4; "vLLM 内部構造 (2) — PagedAttention", section
  "ブロックテーブル").
* ``copy_blocks`` -- copy-on-write duplication of physical blocks (first page,
  section 4: shared blocks carry a reference count and are copied on write).
* ``kv_bytes_per_token`` / ``blocks_for_tokens`` -- the size formula of the
  first page, section 2, and ceil(n / block_size).
* ``paged_attention_prefill`` -- several queries per sequence, causal (first
  page, sections 3 and 6).
* ``token_attention_decode`` / ``repack_tokens`` -- decode through a token
  table and the repacking that moves live tokens ("LLM推論の「見えないメモリ
  問題」を解く … vToken", token-level virtualisation and asynchronous
  repacking).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

F32, BF16, E4M3 = 0, 1, 2

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkv_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile ``pkv_oracle.c`` into ``liboracle.so`` next to it (gcc, no
    floating-point contraction so that x86 and Arm give identical bits)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + ".tmp%d" % os.getpid()
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
                           "-fPIC", "-shared", "-pthread", "-o", tmp, _SRC, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        c_p, c_i, c_f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        lib.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_to_double.restype = ctypes.c_double
        lib.oracle_e4m3_from_float.argtypes = [c_f]
        lib.oracle_e4m3_from_float.restype = ctypes.c_uint8
        lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_double.restype = ctypes.c_double
        lib.oracle_bf16_from_double.argtypes = [ctypes.c_double]
        lib.oracle_bf16_from_double.restype = ctypes.c_uint16
        lib.oracle_paged_kv_write.argtypes = [c_p, c_p, c_i, c_p, c_p, c_i, c_p, c_i, c_i,
                                              c_i, c_i, c_i, c_f, c_f]
        lib.oracle_paged_kv_write.restype = c_i
        lib.oracle_paged_attention_decode.argtypes = [c_p, c_p, c_i, c_p, c_p, c_i, c_p, c_i,
                                                      c_p, c_i, c_i, c_i, c_i, c_i, c_i, c_f,
                                                      c_f, c_f, c_i, c_i]
        lib.oracle_paged_attention_decode.restype = c_i
        lib.oracle_paged_attention_prefill.argtypes = [c_p, c_p, c_i, c_p, c_p, c_i, c_p, c_i, c_p, c_p,
                                                       c_i, c_i, c_i, c_i, c_i, c_i, c_f, c_f, c_f, c_i]
        lib.oracle_paged_attention_prefill.restype = c_i
        lib.oracle_copy_blocks.argtypes = [ctypes.POINTER(c_p), ctypes.POINTER(c_p), c_i, c_p,
                                           c_i, c_i, ctypes.c_size_t]
        lib.oracle_copy_blocks.restype = c_i
        lib.oracle_token_attention_decode.argtypes = [c_p, c_p, c_i, c_p, c_p, c_i, c_p, c_i, c_p, c_i, c_i, c_i,
                                                      c_i, c_i, c_i, c_f, c_f, c_f, c_i]
        lib.oracle_token_attention_decode.restype = c_i
        lib.oracle_repack_tokens.argtypes = [ctypes.POINTER(c_p), ctypes.POINTER(c_p), c_i, c_p, c_i, c_i, c_p, c_i,
                                             c_i, c_i, ctypes.c_size_t]
        lib.oracle_repack_tokens.restype = c_i
        lib.oracle_kv_bytes_per_token.argtypes = [c_i, c_i, c_i, c_i]
        lib.oracle_kv_bytes_per_token.restype = ctypes.c_longlong
        lib.oracle_blocks_for_tokens.argtypes = [ctypes.c_longlong, c_i]
        lib.oracle_blocks_for_tokens.restype = ctypes.c_longlong
        _lib = lib
        return lib


_NP_OF = {F32: np.float32, BF16: np.uint16, E4M3: np.uint8}


def _check(a: np.ndarray, dt: int, name: str) -> np.ndarray:
    if a.dtype != _NP_OF[dt]:
        raise TypeError(f"{name}: expected {np.dtype(_NP_OF[dt])} for dtype code {dt}, got {a.dtype}")
    if not a.flags.c_contiguous:
        raise ValueError(f"{name} must be C-contiguous")
    return a


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


# ----------------------------------------------------------------- formats

def e4m3_to_float64(codes) -> np.ndarray:
    lib = _load()
    c = np.asarray(codes, dtype=np.uint8)
    return np.array([lib.oracle_e4m3_to_double(int(v)) for v in c.ravel()],
                    dtype=np.float64).reshape(c.shape)


def e4m3_from_float32(x) -> np.ndarray:
    lib = _load()
    a = np.asarray(x, dtype=np.float32)
    return np.array([lib.oracle_e4m3_from_float(float(v)) for v in a.ravel()],
                    dtype=np.uint8).reshape(a.shape)


def bf16_from_float64(x) -> np.ndarray:
    lib = _load()
    a = np.asarray(x, dtype=np.float64)
    return np.array([lib.oracle_bf16_from_double(float(v)) for v in a.ravel()],
                    dtype=np.uint16).reshape(a.shape)


def bf16_to_float64(h) -> np.ndarray:
    lib = _load()
    a = np.asarray(h, dtype=np.uint16)
    return np.array([lib.oracle_bf16_to_double(int(v)) for v in a.ravel()],
                    dtype=np.float64).reshape(a.shape)


# ---------------------------------------------------------- the three calls

def paged_kv_write(key, value, in_dt, key_cache, value_cache, cache_dt, slot_mapping,
                   block_size, k_scale=1.0, v_scale=1.0) -> int:
    """In place on ``key_cache``/``value_cache`` ([NB, bs, Hkv, d])."""
    lib = _load()
    key = _check(np.ascontiguousarray(key), in_dt, "key")
    value = _check(np.ascontiguousarray(value), in_dt, "value")
    _check(key_cache, cache_dt, "key_cache")
    _check(value_cache, cache_dt, "value_cache")
    slots = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    T, Hkv, d = key.shape
    NB, bs = key_cache.shape[0], key_cache.shape[1]
    assert bs == block_size and key_cache.shape[2:] == (Hkv, d)
    return lib.oracle_paged_kv_write(_ptr(key), _ptr(value), in_dt, _ptr(key_cache),
                                     _ptr(value_cache), cache_dt, _ptr(slots), T, NB, bs,
                                     Hkv, d, float(k_scale), float(v_scale))


def paged_attention_decode(query, q_dt, key_cache, value_cache, cache_dt, block_tables,
                           context_lens, scale, k_scale=1.0, v_scale=1.0, partition=0,
                           threads=None) -> np.ndarray:
    """Returns the fp64 output [S, Hq, d]."""
    lib = _load()
    query = _check(np.ascontiguousarray(query), q_dt, "query")
    _check(key_cache, cache_dt, "key_cache")
    _check(value_cache, cache_dt, "value_cache")
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    S, Hq, d = query.shape
    NB, bs, Hkv, d2 = key_cache.shape
    assert d2 == d and bt.shape[0] == S and cl.shape == (S,)
    MB = bt.shape[1] if bt.ndim == 2 else 0
    out = np.zeros((S, Hq, d), dtype=np.float64)
    if threads is None:
        threads = os.cpu_count() or 1
    rc = lib.oracle_paged_attention_decode(_ptr(out), _ptr(query), q_dt, _ptr(key_cache),
                                           _ptr(value_cache), cache_dt, _ptr(bt), MB, _ptr(cl),
                                           S, Hq, Hkv, d, bs, NB, float(scale), float(k_scale),
                                           float(v_scale), int(partition), int(threads))
    if rc != 0:
        raise ValueError(f"oracle decode failed with code {rc}")
    return out


def paged_attention_prefill(query, q_dt, key_cache, value_cache, cache_dt, block_tables, context_lens,
                            query_start, scale, k_scale=1.0, v_scale=1.0, threads=None) -> np.ndarray:
    """Several query tokens per sequence, causal: the fp64 output [T, Hq, d].
    query [T, Hq, d] packs every sequence's queries; query_start [S + 1]."""
    lib = _load()
    query = _check(np.ascontiguousarray(query), q_dt, "query")
    _check(key_cache, cache_dt, "key_cache")
    _check(value_cache, cache_dt, "value_cache")
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    qs = np.ascontiguousarray(query_start, dtype=np.int32)
    T, Hq, d = query.shape
    NB, bs, Hkv, d2 = key_cache.shape
    S = cl.shape[0]
    assert d2 == d and qs.shape == (S + 1,) and qs[-1] == T and bt.shape[0] == S
    out = np.zeros((T, Hq, d), dtype=np.float64)
    if threads is None:
        threads = os.cpu_count() or 1
    rc = lib.oracle_paged_attention_prefill(_ptr(out), _ptr(query), q_dt, _ptr(key_cache), _ptr(value_cache),
                                            cache_dt, _ptr(bt), bt.shape[1], _ptr(cl), _ptr(qs), S, Hq, Hkv, d,
                                            bs, NB, float(scale), float(k_scale), float(v_scale), int(threads))
    if rc != 0:
        raise ValueError(f"oracle prefill failed with code {rc}")
    return out


def copy_blocks(key_caches, value_caches, block_mapping) -> int:
    """In place on every layer's caches (lists of arrays [NB, bs, Hkv, d])."""
    lib = _load()
    L = len(key_caches)
    bm = np.ascontiguousarray(block_mapping, dtype=np.int64).reshape(-1, 2)
    NB = key_caches[0].shape[0]
    block_bytes = key_caches[0][0].nbytes
    for a in list(key_caches) + list(value_caches):
        assert a.flags.c_contiguous and a.shape[0] == NB and a[0].nbytes == block_bytes
    kp = (ctypes.c_void_p * L)(*[_ptr(a) for a in key_caches])
    vp = (ctypes.c_void_p * L)(*[_ptr(a) for a in value_caches])
    return lib.oracle_copy_blocks(kp, vp, L, _ptr(bm), bm.shape[0], NB, block_bytes)


# ------------------------------------------------------------- token table

def token_attention_decode(query, q_dt, key_cache, value_cache, cache_dt, token_slots, num_tokens, scale,
                           k_scale=1.0, v_scale=1.0, threads=None) -> np.ndarray:
    """Decode through a token table: token_slots [S, MT] int32 lists each
    sequence's live tokens in logical order as slots (block * bs + offset);
    num_tokens [S].  Returns the fp64 output [S, Hq, d]."""
    lib = _load()
    query = _check(np.ascontiguousarray(query), q_dt, "query")
    _check(key_cache, cache_dt, "key_cache")
    _check(value_cache, cache_dt, "value_cache")
    ts = np.ascontiguousarray(token_slots, dtype=np.int32)
    nt = np.ascontiguousarray(num_tokens, dtype=np.int32)
    S, Hq, d = query.shape
    NB, bs, Hkv, d2 = key_cache.shape
    assert d2 == d and ts.shape[0] == S and nt.shape == (S,)
    out = np.zeros((S, Hq, d), dtype=np.float64)
    if threads is None:
        threads = os.cpu_count() or 1
    rc = lib.oracle_token_attention_decode(_ptr(out), _ptr(query), q_dt, _ptr(key_cache), _ptr(value_cache),
                                           cache_dt, _ptr(ts), ts.shape[1], _ptr(nt), S, Hq, Hkv, d, bs, NB,
                                           float(scale), float(k_scale), float(v_scale), int(threads))
    if rc != 0:
        raise ValueError(f"oracle token decode failed with code {rc}")
    return out


def repack_tokens(key_caches, value_caches, token_slots, moves) -> int:
    """Apply moves [M, 4] = (sequence, logical index, src slot, dst slot) in
    place: every layer's K/V row of the token is copied and the table entry
    rewritten.  Returns 0, or -1 if a move was skipped."""
    lib = _load()
    assert token_slots.dtype == np.int32 and token_slots.flags.c_contiguous
    L = len(key_caches)
    mv = np.ascontiguousarray(moves, dtype=np.int64).reshape(-1, 4)
    NB, bs = key_caches[0].shape[0], key_caches[0].shape[1]
    token_bytes = key_caches[0][0, 0].nbytes
    for a in list(key_caches) + list(value_caches):
        assert a.flags.c_contiguous and a.shape[:2] == (NB, bs)
    kp = (ctypes.c_void_p * L)(*[_ptr(a) for a in key_caches])
    vp = (ctypes.c_void_p * L)(*[_ptr(a) for a in value_caches])
    return lib.oracle_repack_tokens(kp, vp, L, _ptr(token_slots), token_slots.shape[1], token_slots.shape[0],
                                    _ptr(mv), mv.shape[0], NB, bs, token_bytes)


# --------------------------------------------------------- byte accounting

def kv_bytes_per_token(num_layers: int, num_kv_heads: int, head_dim: int, elem_bytes: int) -> int:
    return int(_load().oracle_kv_bytes_per_token(num_layers, num_kv_heads, head_dim, elem_bytes))


def blocks_for_tokens(n: int, block_size: int) -> int:
    return int(_load().oracle_blocks_for_tokens(n, block_size))
