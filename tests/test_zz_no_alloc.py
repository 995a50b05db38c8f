"""The decode entry point that allocates nothing.

pkv_paged_attention_decode_static serves callers that cannot allocate device
memory where they decode (an engine that reserved all of its memory up
front, a latency-critical loop that must not wait on the allocator, a caller
that holds raw pointers but no allocator).  It uses the library's fixed
device scratch instead of a caller-provided workspace.  These tests call it
through the C ABI and check:

* two calls in a row give exactly the allocating entry point's output (same
  kernels, same partition plan, same merge order: bit for bit), and that
  output is within the cache dtype's tolerance of the CPU oracle;
* a later call with other sizes, made after split calls left partition
  results in the shared scratch, is again exact: stale scratch contents
  never leak into a result;
* sizes whose scratch would exceed the fixed maximum are refused.

The file is named so that pytest collects it last.
"""
import dataclasses

import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import paged_kv_cache_44_gb300 as pkv
    from tests.gpu_cases import assert_close, build_case, oracle_decode


def _static_call(c, out, partition_size):
    w = c.w
    return pkv.lib.pkv_paged_attention_decode_static(
        out.data_ptr(), c.q.data_ptr(), pkv.dtype_code(c.q.dtype), c.k_cache.data_ptr(), c.v_cache.data_ptr(),
        pkv.dtype_code(c.k_cache.dtype), c.block_tables.data_ptr(), c.block_tables.shape[1],
        c.context_lens.data_ptr(), w.S, w.max_context_len, w.Hq, w.Hkv, w.d, w.bs, w.NB, w.scale,
        c.k_scale, c.v_scale, partition_size, None, torch.cuda.current_stream().cuda_stream)


def _allocating_call(c, partition_size):
    w = c.w
    ref = torch.empty_like(c.q)
    ws = pkv.make_workspace(w.S, w.Hq, w.Hkv, w.d, w.bs, w.max_context_len, partition_size)
    pkv.paged_attention_decode(ref, c.q, c.k_cache, c.v_cache, c.block_tables, c.context_lens,
                               w.max_context_len, scale=w.scale, k_scale=c.k_scale, v_scale=c.v_scale,
                               partition_size=partition_size, workspace=ws)
    torch.cuda.synchronize()
    return ref


def _case(name, lengths):
    lens = np.array(lengths)
    w = W.make(name, S=len(lens), lengths=np.maximum(lens, 1))
    if (lens == 0).any():
        w = dataclasses.replace(w, context_lens=lens.astype(np.int32))
    return build_case(w)


CASES = [
    ("qwen2.5-72b-long", [32768, 20000, 1, 777], 512),      # split-K: the scratch holds partition triples
    ("fp8-bs16", [16384, 300, 5000, 0], 256),
    ("qwen2.5-1.5b", [4096, 17, 2049, 512], -1),            # no split: only the work counter is used
]


@pytest.mark.parametrize("name,lengths,partition", CASES, ids=[c[0] for c in CASES])
def test_static_scratch_decode_matches_allocating_entry(name, lengths, partition):
    c = _case(name, lengths)
    w = c.w
    need = pkv.decode_workspace_size(w.S, w.Hq, w.Hkv, w.d, w.bs, w.max_context_len, partition)
    assert 0 < need <= pkv.STATIC_SCRATCH_BYTES
    ref = _allocating_call(c, partition)
    assert_close(ref, oracle_decode(c), w.cache_dtype, "allocating entry point")
    for call in range(2):
        out = torch.full_like(c.q, float("nan"))
        assert _static_call(c, out, partition) == 0
        torch.cuda.synchronize()
        assert torch.equal(out, ref), f"static-scratch call {call + 1} differs from the allocating entry point"


def test_stale_scratch_does_not_leak_into_a_later_call():
    """Split calls fill the scratch with partition results; a call with
    other sizes and another partition plan then reads only what it wrote."""
    big = _case("qwen2.5-72b-long", [32768, 9000, 4100, 300])
    small = _case("qwen2.5-1.5b", [1, 700, 1500, 3000, 64, 2049])
    for c, P in ((big, 256), (big, 512), (small, 0), (small, 128), (small, 512), (big, 512)):
        ref = _allocating_call(c, P)
        out = torch.full_like(c.q, float("nan"))
        assert _static_call(c, out, P) == 0
        torch.cuda.synchronize()
        assert torch.equal(out, ref), f"{c.w.name} P={P}"
    assert_close(out, oracle_decode(big), big.w.cache_dtype, "after other calls")


def test_static_scratch_rejects_sizes_beyond_its_maximum():
    w = W.make("qwen2.5-72b-long", S=2)
    c = build_case(w, sample=1)
    need = pkv.decode_workspace_size(w.S, w.Hq, w.Hkv, w.d, w.bs, w.max_context_len, 16)
    assert need > pkv.STATIC_SCRATCH_BYTES
    out = torch.empty_like(c.q)
    assert _static_call(c, out, 16) == 3          # PKV_ERR_WORKSPACE, nothing enqueued
