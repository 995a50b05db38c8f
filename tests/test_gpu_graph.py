"""A whole decode step -- paged_kv_write, paged_attention_decode (split, with
its merge pass), copy_blocks -- recorded into a CUDA graph and replayed.
The calls allocate nothing and never synchronise the host, so capture
works; replays must equal eager execution bit for bit, and must read the
inputs' current contents ("vToken" page, section on CUDA Graph: addresses
are fixed at capture, contents are not)."""
import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import paged_kv_cache_44_gb300 as pkv
    from tests.gpu_cases import assert_close, build_case, oracle_decode


@pytest.mark.parametrize("name,partition", [("qwen2.5-1.5b", 512), ("fp8-bs16", 256)])
def test_step_in_cuda_graph(name, partition):
    w = W.make(name, S=6, lengths=np.array([1, 17, 600, 1500, 2048, 3000]), cow_pairs=8)
    c = build_case(w)
    out = torch.empty_like(c.q)
    ws = pkv.make_workspace(w.S, w.Hq, w.Hkv, w.d, w.bs, w.max_context_len, partition)

    def step():
        pkv.paged_kv_write(c.new_k, c.new_v, c.k_cache, c.v_cache, c.slot_mapping, c.k_scale, c.v_scale)
        pkv.paged_attention_decode(out, c.q, c.k_cache, c.v_cache, c.block_tables, c.context_lens,
                                   w.max_context_len, scale=w.scale, k_scale=c.k_scale, v_scale=c.v_scale,
                                   partition_size=partition, workspace=ws)
        pkv.copy_blocks([c.k_cache], [c.v_cache], c.cow)

    step()                                    # eager, also sets the kernels' shared-memory opt-in
    torch.cuda.synchronize()
    eager = out.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, eager)
    # new query contents, same buffers: the replay must see them
    q2 = W.host_normal(w.seed + 1, "query-2", (w.S, w.Hq, w.d))
    c.q.copy_(torch.from_numpy(W.bf16_bits(q2).view(np.int16)).view(torch.bfloat16))
    c.o_q = W.bf16_bits(q2)
    g.replay()
    torch.cuda.synchronize()
    from tests.gpu_cases import oracle_write
    oracle_write(c)
    assert_close(out, oracle_decode(c), w.cache_dtype, "graph replay with new queries")
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert_close(out, oracle_decode(c), w.cache_dtype, "repeated replays")
