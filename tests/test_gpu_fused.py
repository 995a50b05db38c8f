"""Fused write + decode (pkv_paged_kv_write_decode) against the two calls it
replaces, and against the oracle."""
import dataclasses

import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import paged_kv_cache_44_gb300 as pkv
    from tests.gpu_cases import assert_close, build_case, gpu_decode, gpu_write, oracle_decode, oracle_write


def _clone(c):
    return dataclasses.replace(c, k_cache=c.k_cache.clone(), v_cache=c.v_cache.clone())


def _fused(c, P, slot_mapping=None):
    w = c.w
    out = torch.empty_like(c.q)
    ws = pkv.make_workspace(w.S, w.Hq, w.Hkv, w.d, w.bs, w.max_context_len, P)
    pkv.paged_kv_write_decode(out, c.q, c.new_k, c.new_v, c.k_cache, c.v_cache,
                              c.slot_mapping if slot_mapping is None else slot_mapping, c.block_tables,
                              c.context_lens, w.max_context_len, scale=w.scale, k_scale=c.k_scale,
                              v_scale=c.v_scale, partition_size=P, workspace=ws)
    return out


CONFIGS = [
    # (workload, cache, q/in dtype, d, bs)
    ("qwen2.5-1.5b", W.DT_BF16, W.DT_BF16, 128, 16),
    ("qwen2.5-1.5b", W.DT_BF16, W.DT_BF16, 64, 32),
    ("fp8-bs16", W.DT_E4M3, W.DT_BF16, 128, 16),
    ("fp8-bs32", W.DT_E4M3, W.DT_F32, 128, 32),
    ("fp8-bs16", W.DT_E4M3, W.DT_F32, 64, 16),
]


@pytest.mark.parametrize("cfg", CONFIGS, ids=[f"{c[0]}-{c[1]}-{c[2]}-d{c[3]}-bs{c[4]}" for c in CONFIGS])
# 128: partial partitions cut into 32-token chunks; with an E4M3 cache the
# longer sequences' last full partition too
@pytest.mark.parametrize("P", [-1, 0, 64, 128])
def test_fused_equals_write_then_decode(cfg, P):
    name, cache, qdt, d, bs = cfg
    lens = np.array([1, 16, 17, 100, 513, 1000, 2049])
    w = W.make(name, S=len(lens), lengths=lens, seed=31)
    assert w.bs == bs or name.startswith("qwen")
    if w.bs != bs:                      # the tables are built for the workload's block size
        w = W.make("fp8-bs32" if bs == 32 else "fp8-bs16", S=len(lens), lengths=lens, seed=31)
    w = dataclasses.replace(w, d=d, cache_dtype=cache, q_dtype=qdt)
    c = build_case(w)
    if P > 0 and P % w.bs:
        P = 2 * w.bs
    a = _clone(c)
    gpu_write(a)
    out_a = gpu_decode(a, partition_size=P, kernel="tensor_cores")
    b = _clone(c)
    out_b = _fused(b, P)
    torch.cuda.synchronize()
    assert torch.equal(out_a, out_b)
    assert torch.equal(a.k_cache, b.k_cache) and torch.equal(a.v_cache, b.v_cache)
    oracle_write(c)
    assert_close(out_b, oracle_decode(c), cache, f"fused P={P}")


def test_fused_skips_negative_slots():
    lens = np.array([5, 40, 300, 77])
    w = W.make("qwen2.5-1.5b", S=len(lens), lengths=lens, seed=32)
    c = build_case(w)
    sm = c.slot_mapping.clone()
    sm[1] = -1
    sm[3] = -1
    a = _clone(c)
    pkv.paged_kv_write(a.new_k, a.new_v, a.k_cache, a.v_cache, sm, a.k_scale, a.v_scale)
    out_a = gpu_decode(a, partition_size=0, kernel="tensor_cores")
    b = _clone(c)
    out_b = _fused(b, 0, sm)
    torch.cuda.synchronize()
    assert torch.equal(out_a, out_b)
    assert torch.equal(a.k_cache, b.k_cache) and torch.equal(a.v_cache, b.v_cache)


@pytest.mark.parametrize("name,sample", [("qwen2.5-72b-long", 3), ("fp8-bs16", 4)])
def test_fused_full_size(name, sample):
    """At full size, in the launch configuration of the benchmark: the fused
    call equals the two calls bit for bit (output and caches)."""
    w = W.make(name)
    c = build_case(w, sample=sample)
    a = _clone(c)
    gpu_write(a)
    out_a = gpu_decode(a, kernel="tensor_cores")
    out_b = _fused(c, w.partition_size)
    torch.cuda.synchronize()
    assert torch.equal(out_a, out_b)
    assert torch.equal(a.k_cache, c.k_cache) and torch.equal(a.v_cache, c.v_cache)
