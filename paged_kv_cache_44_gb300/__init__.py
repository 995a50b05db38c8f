"""Paged KV-cache decode attention for GB300 (sm_103a): Python binding.

A thin ctypes layer over ``libpkv.so`` (declared in ``include/pkv.h``).  It
only marshals arguments: torch tensors become device pointers and sizes, the
current torch stream becomes the launch stream, and a non-zero status
becomes a :class:`PkvError`.  Every step of the computation runs in the
library's CUDA kernels; there is no other implementation to fall back on.

The three calls (vLLM-style PagedAttention, "LLM推論の基礎とvLLMの内部",
section 4):

* :func:`paged_kv_write` -- store each new token's K/V into its slot;
* :func:`paged_attention_decode` -- one query token per sequence against the
  paged K/V pool, through block tables;
* :func:`copy_blocks` -- copy-on-write duplication of shared blocks.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import numpy as np
import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
# PKV_LIBRARY may name another build of the same library (e.g. a tuning variant)
LIB_PATH = os.environ.get("PKV_LIBRARY") or os.path.join(_PKG, "libpkv.so")

F32, BF16, FP8_E4M3 = 0, 1, 2
KERNELS = {"auto": 0, "cuda_cores": 1, "tensor_cores": 2}
STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported dtype or shape",
          3: "workspace missing or too small", 4: "CUDA launch failed"}

EXPORTED = ("pkv_paged_kv_write", "pkv_decode_workspace_size", "pkv_decode_partition_size",
            "pkv_decode_launch_partition_size",
            "pkv_paged_attention_decode", "pkv_paged_attention_decode_ex", "pkv_copy_blocks",
            "pkv_status_string", "pkv_version", "pkv_paged_attention_decode_static",
            "pkv_pool_create", "pkv_pool_destroy", "pkv_pool_set_extra_key", "pkv_pool_num_free_blocks",
            "pkv_pool_num_cached_blocks", "pkv_pool_block_ref_count", "pkv_pool_add_sequence",
            "pkv_pool_append_token", "pkv_pool_fork", "pkv_pool_free_sequence", "pkv_pool_block_table",
            "pkv_pool_append_tokens", "pkv_pool_block_tables", "pkv_prefill_workspace_size",
            "pkv_paged_attention_prefill", "pkv_paged_attention_prefill_ex", "pkv_token_attention_decode",
            "pkv_repack_tokens", "pkv_vtoken_plan", "pkv_paged_kv_write_decode")
STATIC_SCRATCH_BYTES = 32 << 20


class PkvError(RuntimeError):
    def __init__(self, call: str, status: int):
        super().__init__(f"{call} failed: {STATUS.get(status, status)} (status {status})")
        self.status = status


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is not built. Build it with "
            "`python -c 'import __graft_entry__ as g; g.build()'` or "
            "`python paged_kv_cache_44_gb300/_build.py` (needs nvcc for sm_103a).")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.pkv_paged_kv_write.argtypes = [vp, vp, i32, vp, vp, i32, vp, i32, i32, i32, i32, i32, f32, f32, vp, vp]
    lib.pkv_paged_kv_write.restype = i32
    lib.pkv_decode_workspace_size.argtypes = [i32] * 7
    lib.pkv_decode_workspace_size.restype = sz
    lib.pkv_decode_partition_size.argtypes = [i32] * 7
    lib.pkv_decode_partition_size.restype = i32
    lib.pkv_decode_launch_partition_size.argtypes = [i32] * 11
    lib.pkv_decode_launch_partition_size.restype = i32
    dec = [vp, vp, i32, vp, vp, i32, vp, i32, vp, i32, i32, i32, i32, i32, i32, i32, f32, f32, f32, i32,
           vp, sz, vp, vp]
    lib.pkv_paged_attention_decode.argtypes = dec
    lib.pkv_paged_attention_decode.restype = i32
    lib.pkv_paged_attention_decode_ex.argtypes = dec + [i32]
    lib.pkv_paged_attention_decode_ex.restype = i32
    lib.pkv_paged_attention_decode_static.argtypes = dec[:20] + [vp, vp]
    lib.pkv_paged_attention_decode_static.restype = i32
    lib.pkv_copy_blocks.argtypes = [ctypes.POINTER(vp), ctypes.POINTER(vp), i32, vp, i32, i32, sz, vp, vp]
    lib.pkv_copy_blocks.restype = i32
    i64, pi32, pi64 = ctypes.c_int64, ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int64)
    lib.pkv_pool_create.argtypes = [i32, i32, i32, ctypes.POINTER(vp)]
    lib.pkv_pool_create.restype = i32
    lib.pkv_pool_destroy.argtypes = [vp]
    lib.pkv_pool_destroy.restype = None
    lib.pkv_pool_set_extra_key.argtypes = [vp, ctypes.c_uint64]
    lib.pkv_pool_set_extra_key.restype = i32
    lib.pkv_pool_num_free_blocks.argtypes = [vp]
    lib.pkv_pool_num_free_blocks.restype = i32
    lib.pkv_pool_num_cached_blocks.argtypes = [vp]
    lib.pkv_pool_num_cached_blocks.restype = i32
    lib.pkv_pool_block_ref_count.argtypes = [vp, i32]
    lib.pkv_pool_block_ref_count.restype = i32
    lib.pkv_pool_add_sequence.argtypes = [vp, i64, pi32, i32, pi32]
    lib.pkv_pool_add_sequence.restype = i32
    lib.pkv_pool_append_token.argtypes = [vp, i64, ctypes.c_int32, pi64, pi64, pi64]
    lib.pkv_pool_append_token.restype = i32
    lib.pkv_pool_fork.argtypes = [vp, i64, i64]
    lib.pkv_pool_fork.restype = i32
    lib.pkv_pool_free_sequence.argtypes = [vp, i64]
    lib.pkv_pool_free_sequence.restype = i32
    lib.pkv_pool_block_table.argtypes = [vp, i64, pi32, i32, pi32, pi32]
    lib.pkv_pool_block_table.restype = i32
    lib.pkv_pool_append_tokens.argtypes = [vp, pi64, pi32, i32, pi64, pi64, pi32]
    lib.pkv_pool_append_tokens.restype = i32
    lib.pkv_pool_block_tables.argtypes = [vp, pi64, i32, pi32, i32, pi32]
    lib.pkv_pool_block_tables.restype = i32
    lib.pkv_prefill_workspace_size.argtypes = [i32] * 9
    lib.pkv_prefill_workspace_size.restype = sz
    lib.pkv_paged_attention_prefill.argtypes = [vp, vp, i32, vp, vp, i32, vp, i32, vp, vp, i32, i32, i32, i32,
                                                i32, i32, i32, i32, i32, f32, i32, vp, sz, vp, vp]
    lib.pkv_paged_attention_prefill.restype = i32
    lib.pkv_paged_attention_prefill_ex.argtypes = lib.pkv_paged_attention_prefill.argtypes + [i32]
    lib.pkv_paged_attention_prefill_ex.restype = i32
    lib.pkv_paged_kv_write_decode.argtypes = [vp, vp, i32, vp, vp, i32, vp, vp, i32, vp, vp, i32, vp, i32, i32, i32,
                                              i32, i32, i32, i32, f32, f32, f32, i32, vp, sz, vp, vp]
    lib.pkv_paged_kv_write_decode.restype = i32
    lib.pkv_token_attention_decode.argtypes = dec
    lib.pkv_token_attention_decode.restype = i32
    lib.pkv_repack_tokens.argtypes = [ctypes.POINTER(vp), ctypes.POINTER(vp), i32, vp, i32, i32, vp, i32, i32, i32,
                                      sz, vp, vp]
    lib.pkv_repack_tokens.restype = i32
    lib.pkv_vtoken_plan.argtypes = [pi32, i32, pi32, i32, i32, i32, pi64, i64, pi64, pi32, i64, pi64]
    lib.pkv_vtoken_plan.restype = i32
    lib.pkv_status_string.argtypes = [i32]
    lib.pkv_status_string.restype = ctypes.c_char_p
    lib.pkv_version.argtypes = []
    lib.pkv_version.restype = ctypes.c_char_p
    return lib


lib = _load()


def version() -> str:
    return lib.pkv_version().decode()


def dtype_code(t: torch.dtype) -> int:
    if t == torch.float32:
        return F32
    if t == torch.bfloat16:
        return BF16
    if t in (torch.float8_e4m3fn, torch.uint8):
        return FP8_E4M3
    raise TypeError(f"unsupported dtype {t}")


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("pkv calls take CUDA tensors")
    if not t.is_contiguous():
        raise ValueError("pkv calls take contiguous tensors")
    return t.data_ptr()


def _check(call: str, st: int) -> None:
    if st != 0:
        raise PkvError(call, st)


def paged_kv_write(key: torch.Tensor, value: torch.Tensor, key_cache: torch.Tensor, value_cache: torch.Tensor,
                   slot_mapping: torch.Tensor, k_scale: float = 1.0, v_scale: float = 1.0,
                   err_word: Optional[torch.Tensor] = None, stream=None) -> None:
    """key/value [T, Hkv, d] (fp32|bf16); caches [NB, bs, Hkv, d] (fp32|bf16|e4m3);
    slot_mapping int64 [T] (negative = skip)."""
    T, Hkv, d = key.shape
    NB, bs = key_cache.shape[0], key_cache.shape[1]
    if tuple(key_cache.shape[2:]) != (Hkv, d) or value.shape != key.shape or value_cache.shape != key_cache.shape:
        raise ValueError("shape mismatch between tokens and caches")
    if slot_mapping.dtype != torch.int64 or slot_mapping.numel() != T:
        raise ValueError("slot_mapping must be int64 [T]")
    _check("paged_kv_write", lib.pkv_paged_kv_write(
        _ptr(key), _ptr(value), dtype_code(key.dtype), _ptr(key_cache), _ptr(value_cache),
        dtype_code(key_cache.dtype), _ptr(slot_mapping), T, NB, bs, Hkv, d, float(k_scale), float(v_scale),
        _ptr(err_word), _stream(stream)))


def decode_partition_size(S: int, Hq: int, Hkv: int, d: int, bs: int, max_context_len: int,
                          partition_size: int = 0) -> int:
    return int(lib.pkv_decode_partition_size(S, Hq, Hkv, d, bs, max_context_len, partition_size))


def decode_launch_partition_size(S: int, Hq: int, Hkv: int, d: int, bs: int, NB: int, max_context_len: int,
                                 partition_size: int, q_dtype: torch.dtype, cache_dtype: torch.dtype,
                                 kernel: str = "auto") -> int:
    return int(lib.pkv_decode_launch_partition_size(S, Hq, Hkv, d, bs, NB, max_context_len, partition_size,
                                                    dtype_code(q_dtype), dtype_code(cache_dtype),
                                                    KERNELS[kernel]))


def decode_workspace_size(S: int, Hq: int, Hkv: int, d: int, bs: int, max_context_len: int,
                          partition_size: int = 0) -> int:
    return int(lib.pkv_decode_workspace_size(S, Hq, Hkv, d, bs, max_context_len, partition_size))


def make_workspace(S: int, Hq: int, Hkv: int, d: int, bs: int, max_context_len: int, partition_size: int = 0,
                   device=None) -> torch.Tensor:
    """A zero-filled workspace of the size the decode needs (the decode
    leaves its header zero, so the tensor can be reused call after call)."""
    n = decode_workspace_size(S, Hq, Hkv, d, bs, max_context_len, partition_size)
    return torch.zeros(max(n, 16), dtype=torch.uint8, device=device or "cuda")


def paged_attention_decode(out: torch.Tensor, query: torch.Tensor, key_cache: torch.Tensor,
                           value_cache: torch.Tensor, block_tables: torch.Tensor, context_lens: torch.Tensor,
                           max_context_len: int, scale: float, k_scale: float = 1.0,
                           v_scale: float = 1.0, partition_size: int = 0,
                           workspace: Optional[torch.Tensor] = None, err_word: Optional[torch.Tensor] = None,
                           stream=None, kernel: str = "auto") -> torch.Tensor:
    """out/query [S, Hq, d]; caches [NB, bs, Hkv, d]; block_tables int32 [S, MB];
    context_lens int32 [S]; max_context_len (host) >= every context length."""
    S, Hq, d = query.shape
    NB, bs, Hkv, d2 = key_cache.shape
    if d2 != d or out.shape != query.shape or out.dtype != query.dtype or value_cache.shape != key_cache.shape:
        raise ValueError("shape or dtype mismatch")
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32 or block_tables.dim() != 2:
        raise ValueError("block_tables and context_lens must be int32")
    MB = block_tables.shape[1]
    if workspace is None:          # convenience: a fresh one per call (pass one in to avoid the allocation)
        workspace = make_workspace(S, Hq, Hkv, d, bs, max_context_len, partition_size, device=query.device)
    ws_ptr, ws_bytes = _ptr(workspace), workspace.numel() * workspace.element_size()
    _check("paged_attention_decode", lib.pkv_paged_attention_decode_ex(
        _ptr(out), _ptr(query), dtype_code(query.dtype), _ptr(key_cache), _ptr(value_cache),
        dtype_code(key_cache.dtype), _ptr(block_tables), MB, _ptr(context_lens), S, int(max_context_len),
        Hq, Hkv, d, bs, NB, float(scale), float(k_scale), float(v_scale), int(partition_size),
        ws_ptr, ws_bytes, _ptr(err_word), _stream(stream), KERNELS[kernel]))
    return out


def paged_attention_decode_static(out: torch.Tensor, query: torch.Tensor, key_cache: torch.Tensor,
                                  value_cache: torch.Tensor, block_tables: torch.Tensor, context_lens: torch.Tensor,
                                  max_context_len: int, scale: float, k_scale: float = 1.0,
                                  v_scale: float = 1.0, partition_size: int = 0,
                                  err_word: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """paged_attention_decode without a workspace: the library's fixed device
    scratch (STATIC_SCRATCH_BYTES per GPU) stands in for it, so nothing is
    allocated.  Calls that may overlap on the GPU must not use it together."""
    S, Hq, d = query.shape
    NB, bs, Hkv, d2 = key_cache.shape
    if d2 != d or out.shape != query.shape or out.dtype != query.dtype or value_cache.shape != key_cache.shape:
        raise ValueError("shape or dtype mismatch")
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32 or block_tables.dim() != 2:
        raise ValueError("block_tables and context_lens must be int32")
    _check("paged_attention_decode_static", lib.pkv_paged_attention_decode_static(
        _ptr(out), _ptr(query), dtype_code(query.dtype), _ptr(key_cache), _ptr(value_cache),
        dtype_code(key_cache.dtype), _ptr(block_tables), block_tables.shape[1], _ptr(context_lens), S,
        int(max_context_len), Hq, Hkv, d, bs, NB, float(scale), float(k_scale), float(v_scale),
        int(partition_size), _ptr(err_word), _stream(stream)))
    return out


PREFILL_KERNELS = {"auto": 0, "mma_sync": 1, "tcgen05": 2, "tcgen05_2tile": 3}


def prefill_workspace_size(S: int, num_query_tokens: int, max_query_len: int, Hq: int, Hkv: int, d: int,
                           bs: int, max_context_len: int, partition_size: int = 0) -> int:
    return int(lib.pkv_prefill_workspace_size(S, num_query_tokens, max_query_len, Hq, Hkv, d, bs, max_context_len,
                                              partition_size))


def paged_attention_prefill(out: torch.Tensor, query: torch.Tensor, key_cache: torch.Tensor,
                            value_cache: torch.Tensor, block_tables: torch.Tensor, context_lens: torch.Tensor,
                            query_start: torch.Tensor, max_query_len: int, max_context_len: int,
                            scale: float, partition_size: int = 0,
                            workspace: Optional[torch.Tensor] = None, err_word: Optional[torch.Tensor] = None,
                            stream=None, kernel: str = "auto") -> torch.Tensor:
    """Several query tokens per sequence, causal.  query/out [T, Hq, d];
    query_start int32 [S+1] (device); caches [NB, bs, Hkv, d].  kernel:
    "auto", "tcgen05" (tensor-memory accumulators, one 128-row tile per
    unit), "tcgen05_2tile" (two tiles per unit) or "mma_sync"."""
    if kernel not in PREFILL_KERNELS:
        raise ValueError(f"kernel must be one of {sorted(PREFILL_KERNELS)}")
    T, Hq, d = query.shape
    NB, bs, Hkv, d2 = key_cache.shape
    S = context_lens.numel()
    if d2 != d or out.shape != query.shape or out.dtype != query.dtype or query_start.numel() != S + 1:
        raise ValueError("shape or dtype mismatch")
    if query_start.dtype != torch.int32 or context_lens.dtype != torch.int32 or block_tables.dtype != torch.int32:
        raise ValueError("query_start, context_lens and block_tables must be int32")
    if workspace is None:
        n = prefill_workspace_size(S, T, max_query_len, Hq, Hkv, d, bs, max_context_len, partition_size)
        workspace = torch.zeros(max(n, 256), dtype=torch.uint8, device=query.device)
    _check("paged_attention_prefill", lib.pkv_paged_attention_prefill_ex(
        _ptr(out), _ptr(query), dtype_code(query.dtype), _ptr(key_cache), _ptr(value_cache),
        dtype_code(key_cache.dtype), _ptr(block_tables), block_tables.shape[1], _ptr(context_lens),
        _ptr(query_start), S, T, int(max_query_len), int(max_context_len), Hq, Hkv, d, bs, NB, float(scale),
        int(partition_size), _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(err_word),
        _stream(stream), PREFILL_KERNELS[kernel]))
    return out


def copy_blocks(key_caches: Sequence[torch.Tensor], value_caches: Sequence[torch.Tensor],
                block_mapping: torch.Tensor, err_word: Optional[torch.Tensor] = None, stream=None) -> None:
    """For every layer: block dst of each cache becomes a copy of block src,
    for every (src, dst) row of block_mapping (int64 [P, 2])."""
    L = len(key_caches)
    if len(value_caches) != L or L == 0:
        raise ValueError("need the same, non-zero number of key and value caches")
    NB = key_caches[0].shape[0]
    block_bytes = key_caches[0][0].numel() * key_caches[0].element_size()
    for t in list(key_caches) + list(value_caches):
        if t.shape != key_caches[0].shape or t.dtype != key_caches[0].dtype:
            raise ValueError("all caches must share shape and dtype")
    if block_mapping.dtype != torch.int64:
        raise ValueError("block_mapping must be int64 [P, 2]")
    P = block_mapping.numel() // 2
    kp = (ctypes.c_void_p * L)(*[_ptr(t) for t in key_caches])
    vp = (ctypes.c_void_p * L)(*[_ptr(t) for t in value_caches])
    _check("copy_blocks", lib.pkv_copy_blocks(kp, vp, L, _ptr(block_mapping), P, NB, block_bytes,
                                              _ptr(err_word), _stream(stream)))


def paged_kv_write_decode(out: torch.Tensor, query: torch.Tensor, key: torch.Tensor, value: torch.Tensor,
                          key_cache: torch.Tensor, value_cache: torch.Tensor, slot_mapping: torch.Tensor,
                          block_tables: torch.Tensor, context_lens: torch.Tensor, max_context_len: int,
                          scale: float, k_scale: float = 1.0, v_scale: float = 1.0,
                          partition_size: int = 0, workspace: Optional[torch.Tensor] = None,
                          err_word: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """paged_kv_write of each sequence's new token (key/value [S, Hkv, d],
    slot_mapping int64 [S]: the slot of its last position) and the decode, in
    one launch.  Same results as the two calls."""
    S, Hq, d = query.shape
    NB, bs, Hkv, d2 = key_cache.shape
    if d2 != d or out.shape != query.shape or out.dtype != query.dtype or value_cache.shape != key_cache.shape:
        raise ValueError("shape or dtype mismatch")
    if key.shape != (S, Hkv, d) or value.shape != key.shape or key.dtype != value.dtype:
        raise ValueError("key/value must be [S, Hkv, d] of one dtype")
    if slot_mapping.dtype != torch.int64 or slot_mapping.numel() != S:
        raise ValueError("slot_mapping must be int64 [S]")
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32 or block_tables.dim() != 2:
        raise ValueError("block_tables and context_lens must be int32")
    if workspace is None:
        workspace = make_workspace(S, Hq, Hkv, d, bs, max_context_len, partition_size, device=query.device)
    ws_ptr, ws_bytes = _ptr(workspace), workspace.numel() * workspace.element_size()
    _check("paged_kv_write_decode", lib.pkv_paged_kv_write_decode(
        _ptr(out), _ptr(query), dtype_code(query.dtype), _ptr(key), _ptr(value), dtype_code(key.dtype),
        _ptr(key_cache), _ptr(value_cache), dtype_code(key_cache.dtype), _ptr(slot_mapping), _ptr(block_tables),
        block_tables.shape[1], _ptr(context_lens), S, int(max_context_len), Hq, Hkv, d, bs, NB, float(scale),
        float(k_scale), float(v_scale), int(partition_size), ws_ptr, ws_bytes, _ptr(err_word), _stream(stream)))
    return out


def token_attention_decode(out: torch.Tensor, query: torch.Tensor, key_cache: torch.Tensor,
                           value_cache: torch.Tensor, token_slots: torch.Tensor, num_tokens: torch.Tensor,
                           max_tokens: int, scale: float, k_scale: float = 1.0, v_scale: float = 1.0,
                           partition_size: int = 0, workspace: Optional[torch.Tensor] = None,
                           err_word: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Decode through a token table: token_slots int32 [S, MT] lists each
    sequence's live tokens as slots (block * bs + offset) in logical order;
    num_tokens int32 [S]; max_tokens (host) >= every count."""
    S, Hq, d = query.shape
    NB, bs, Hkv, d2 = key_cache.shape
    if d2 != d or out.shape != query.shape or out.dtype != query.dtype or value_cache.shape != key_cache.shape:
        raise ValueError("shape or dtype mismatch")
    if token_slots.dtype != torch.int32 or num_tokens.dtype != torch.int32 or token_slots.dim() != 2:
        raise ValueError("token_slots and num_tokens must be int32")
    if workspace is None:
        workspace = make_workspace(S, Hq, Hkv, d, bs, max_tokens, partition_size, device=query.device)
    ws_ptr, ws_bytes = _ptr(workspace), workspace.numel() * workspace.element_size()
    _check("token_attention_decode", lib.pkv_token_attention_decode(
        _ptr(out), _ptr(query), dtype_code(query.dtype), _ptr(key_cache), _ptr(value_cache),
        dtype_code(key_cache.dtype), _ptr(token_slots), token_slots.shape[1], _ptr(num_tokens), S,
        int(max_tokens), Hq, Hkv, d, bs, NB, float(scale), float(k_scale), float(v_scale), int(partition_size),
        ws_ptr, ws_bytes, _ptr(err_word), _stream(stream)))
    return out


def repack_tokens(key_caches: Sequence[torch.Tensor], value_caches: Sequence[torch.Tensor],
                  token_slots: torch.Tensor, moves: torch.Tensor, err_word: Optional[torch.Tensor] = None,
                  stream=None) -> None:
    """Move live tokens: moves int64 [M, 4] = (sequence, logical index, src
    slot, dst slot); every layer's K/V row is copied and token_slots (int32
    [S, MT], device) rewritten."""
    L = len(key_caches)
    if len(value_caches) != L or L == 0:
        raise ValueError("need the same, non-zero number of key and value caches")
    NB, bs = key_caches[0].shape[0], key_caches[0].shape[1]
    token_bytes = key_caches[0][0, 0].numel() * key_caches[0].element_size()
    for t in list(key_caches) + list(value_caches):
        if t.shape != key_caches[0].shape or t.dtype != key_caches[0].dtype:
            raise ValueError("all caches must share shape and dtype")
    if moves.dtype != torch.int64 or token_slots.dtype != torch.int32 or token_slots.dim() != 2:
        raise ValueError("moves must be int64 [M, 4], token_slots int32 [S, MT]")
    kp = (ctypes.c_void_p * L)(*[_ptr(t) for t in key_caches])
    vp = (ctypes.c_void_p * L)(*[_ptr(t) for t in value_caches])
    _check("repack_tokens", lib.pkv_repack_tokens(kp, vp, L, _ptr(token_slots), token_slots.shape[1],
                                                  token_slots.shape[0], _ptr(moves), moves.numel() // 4, NB, bs,
                                                  token_bytes, _ptr(err_word), _stream(stream)))


def vtoken_plan(token_slots: np.ndarray, num_tokens: np.ndarray, block_size: int, num_blocks: int):
    """Host repacking plan (pkv_vtoken_plan): returns (moves int64 [M, 4],
    freed int32 [F]) for host token tables."""
    ts = np.ascontiguousarray(token_slots, dtype=np.int32)
    nt = np.ascontiguousarray(num_tokens, dtype=np.int32)
    S, MT = ts.shape
    nm, nf = ctypes.c_int64(0), ctypes.c_int64(0)
    cap_m, cap_f = max(int(nt.sum()), 1), max(num_blocks, 1)
    moves = np.zeros((cap_m, 4), np.int64)
    freed = np.zeros(cap_f, np.int32)
    as32 = lambda a: a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))  # noqa: E731
    as64 = lambda a: a.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))  # noqa: E731
    _check("vtoken_plan", lib.pkv_vtoken_plan(as32(ts), MT, as32(nt), S, block_size, num_blocks, as64(moves), cap_m,
                                              ctypes.byref(nm), as32(freed), cap_f, ctypes.byref(nf)))
    return moves[: nm.value].copy(), freed[: nf.value].copy()


class BlockPool:
    """Host block manager (pkv_pool_* in include/pkv.h): block tables, slots
    and copy-on-write pairs for the device calls.  Block 0 is the null block."""

    def __init__(self, num_blocks: int, block_size: int, prefix_caching: bool = True, extra_key: int = 0):
        h = ctypes.c_void_p()
        _check("pkv_pool_create", lib.pkv_pool_create(num_blocks, block_size, int(prefix_caching), ctypes.byref(h)))
        self._h = h
        self.block_size = block_size
        if extra_key:
            self.set_extra_key(extra_key)

    def set_extra_key(self, extra_key: int) -> None:
        """Key mixed into later block hashes: blocks cached under one key are
        never reused under another."""
        _check("pkv_pool_set_extra_key", lib.pkv_pool_set_extra_key(self._h, extra_key))

    def close(self) -> None:
        if self._h:
            lib.pkv_pool_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def num_free(self) -> int:
        return lib.pkv_pool_num_free_blocks(self._h)

    def num_cached(self) -> int:
        return lib.pkv_pool_num_cached_blocks(self._h)

    def ref_count(self, block: int) -> int:
        return lib.pkv_pool_block_ref_count(self._h, block)

    def add_sequence(self, seq_id: int, tokens) -> Optional[int]:
        """Cached prompt tokens, or None when the pool has too few free blocks."""
        import numpy as np
        t = np.ascontiguousarray(tokens, dtype=np.int32)
        got = ctypes.c_int32(0)
        st = lib.pkv_pool_add_sequence(self._h, seq_id, t.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                                       t.size, ctypes.byref(got))
        if st == 3:
            return None
        _check("pkv_pool_add_sequence", st)
        return got.value

    def append_token(self, seq_id: int, token: int):
        """(slot, cow_src, cow_dst) -- cow_* = -1 without a copy -- or None when no block is free."""
        slot, src, dst = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
        st = lib.pkv_pool_append_token(self._h, seq_id, token, ctypes.byref(slot), ctypes.byref(src),
                                       ctypes.byref(dst))
        if st == 3:
            return None
        _check("pkv_pool_append_token", st)
        return slot.value, src.value, dst.value

    def append_tokens(self, seq_ids, tokens):
        """One step for many sequences: (slot_mapping int64 [n], copy pairs
        int64 [c, 2]) -- the inputs of paged_kv_write and copy_blocks -- or
        None when the pool cannot cover the step."""
        import numpy as np
        ids = np.ascontiguousarray(seq_ids, dtype=np.int64)
        tok = np.ascontiguousarray(tokens, dtype=np.int32)
        n = ids.size
        slots = np.zeros(n, np.int64)
        pairs = np.zeros((max(n, 1), 2), np.int64)
        nc = ctypes.c_int32(0)
        P64, P32 = ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int32)
        st = lib.pkv_pool_append_tokens(self._h, ids.ctypes.data_as(P64), tok.ctypes.data_as(P32), n,
                                        slots.ctypes.data_as(P64), pairs.ctypes.data_as(P64), ctypes.byref(nc))
        if st == 3:
            return None
        _check("pkv_pool_append_tokens", st)
        return slots, pairs[: nc.value]

    def block_tables(self, seq_ids, max_blocks: int):
        """(tables int32 [n, max_blocks], context_lens int32 [n]) for the decode."""
        import numpy as np
        ids = np.ascontiguousarray(seq_ids, dtype=np.int64)
        tabs = np.zeros((ids.size, max_blocks), np.int32)
        cl = np.zeros(ids.size, np.int32)
        P64, P32 = ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int32)
        _check("pkv_pool_block_tables", lib.pkv_pool_block_tables(
            self._h, ids.ctypes.data_as(P64), ids.size, tabs.ctypes.data_as(P32), max_blocks,
            cl.ctypes.data_as(P32)))
        return tabs, cl

    def fork(self, parent_id: int, child_id: int) -> None:
        _check("pkv_pool_fork", lib.pkv_pool_fork(self._h, parent_id, child_id))

    def free_sequence(self, seq_id: int) -> None:
        _check("pkv_pool_free_sequence", lib.pkv_pool_free_sequence(self._h, seq_id))

    def block_table(self, seq_id: int, max_blocks: Optional[int] = None):
        """(table as int32 numpy array padded with 0 to max_blocks, number of tokens)."""
        import numpy as np
        nb, nt = ctypes.c_int32(), ctypes.c_int32()
        _check("pkv_pool_block_table", lib.pkv_pool_block_table(self._h, seq_id, None, 0, ctypes.byref(nb),
                                                                 ctypes.byref(nt)))
        m = nb.value if max_blocks is None else max_blocks
        out = np.zeros(max(m, 1), dtype=np.int32)
        _check("pkv_pool_block_table", lib.pkv_pool_block_table(
            self._h, seq_id, out.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), out.size, None, None))
        return out[:m] if m else out[:0], nt.value
