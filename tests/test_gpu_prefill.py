"""Paged attention for several query tokens per sequence (chunked prefill,
speculative-decoding verification) through the C ABI, against the oracle."""
import dataclasses

import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import oracle as O
    import paged_kv_cache_44_gb300 as pkv
    from tests.gpu_cases import assert_close, to_device


def _case(name, lens, qlens, Hq=None, Hkv=None, d=None, seed=7):
    w = W.make(name, S=len(lens), lengths=np.array(lens), seed=seed)
    if Hq is not None:
        w = dataclasses.replace(w, Hq=Hq, Hkv=Hkv, d=d)
    hv = W.host_values(w)
    qs = np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)
    q32 = W.host_normal(seed, "prefill-query", (int(qs[-1]), w.Hq, w.d))
    return w, hv, qs, q32


KERNELS = ["tcgen05", "tcgen05_2tile", "mma_sync"]


def _run(w, hv, qs, q32, partition, dev="cuda", query_start=None, err=None, max_query_len=None, kernel="auto"):
    kc = to_device(hv.k_pool, W.DT_BF16, dev)
    vc = to_device(hv.v_pool, W.DT_BF16, dev)
    q = to_device(q32, W.DT_BF16, dev)
    out = torch.full_like(q, float("nan"))
    qs_dev = torch.from_numpy(qs if query_start is None else query_start).to(dev)
    mq = int(np.diff(qs).max()) if max_query_len is None else max_query_len
    pkv.paged_attention_prefill(out, q, kc, vc, torch.from_numpy(w.block_tables).to(dev),
                                torch.from_numpy(w.context_lens).to(dev), qs_dev, mq,
                                w.max_context_len, scale=w.scale, partition_size=partition, err_word=err,
                                kernel=kernel)
    return out


def _ref(w, hv, qs, q32):
    return O.paged_attention_prefill(W.bf16_bits(q32), O.BF16, W.bf16_bits(hv.k_pool), W.bf16_bits(hv.v_pool),
                                     O.BF16, w.block_tables, w.context_lens, qs, w.scale)


CASES = [
    # (workload for bs, lens, qlens, Hq, Hkv, d)
    ("qwen2.5-1.5b", [1, 17, 40, 300, 64, 1000], [1, 17, 5, 128, 0, 33], 8, 2, 128),
    ("qwen2.5-1.5b", [2048, 100, 513], [7, 100, 1], 28, 4, 128),
    ("qwen2.5-1.5b", [77, 500], [77, 250], 8, 8, 64),
    ("fp8-bs32", [33, 700, 64], [16, 65, 64], 16, 2, 128),
    ("fp8-bs32", [1500, 31], [4, 31], 8, 1, 64),
]


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("case", CASES, ids=[f"{c[0]}-g{c[3] // c[4]}-d{c[5]}" for c in CASES])
@pytest.mark.parametrize("partition", [-1, 0, 64])
def test_prefill_matches_oracle(case, partition, kernel):
    name, lens, qlens, Hq, Hkv, d = case
    w, hv, qs, q32 = _case(name, lens, qlens, Hq, Hkv, d)
    if partition > 0 and partition % w.bs:
        partition = 2 * w.bs
    out = _run(w, hv, qs, q32, partition, kernel=kernel)
    assert_close(out, _ref(w, hv, qs, q32), W.DT_BF16, f"prefill {kernel} P={partition}")


@pytest.mark.parametrize("kernel", KERNELS)
def test_prefill_wide_groups_and_tile_edges(kernel):
    """Rows that cross 128-row tiles mid-query (g = 12, 40 and 64 heads per
    K/V head), a query count that is not a multiple of anything, and
    sequences whose key range ends inside a block."""
    for (Hq, Hkv, lens, qlens) in ((24, 2, [300, 77, 1200], [23, 77, 130]),
                                   (40, 1, [129, 64], [7, 64]),
                                   (64, 1, [513, 1000], [3, 2])):
        w, hv, qs, q32 = _case("qwen2.5-1.5b", lens, qlens, Hq, Hkv, 128, seed=Hq)
        for partition in (-1, 96):
            out = _run(w, hv, qs, q32, partition, kernel=kernel)
            assert_close(out, _ref(w, hv, qs, q32), W.DT_BF16, f"g={Hq // Hkv} P={partition} {kernel}")


@pytest.mark.parametrize("kernel", KERNELS)
def test_prefill_bad_block_id_reported(kernel):
    """A block-table entry outside the pool: that block is skipped (its keys
    count as absent) and error word 1 is reported; nothing faults."""
    w, hv, qs, q32 = _case("qwen2.5-1.5b", [40, 50], [8, 8], 8, 2, 128)
    bt = w.block_tables.copy()
    bt[1, 1] = w.NB + 5
    w2 = dataclasses.replace(w, block_tables=bt)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = _run(w2, hv, qs, q32, -1, err=err, kernel=kernel)
    torch.cuda.synchronize()
    assert int(err.item()) == 1
    assert_close(out[:8], _ref(w, hv, qs, q32)[:8], W.DT_BF16, "the sequence with a valid table")
    assert torch.isfinite(out.float()).all()


@pytest.mark.parametrize("kernel", KERNELS)
def test_prefill_graph_replay_reuses_workspace(kernel):
    """The call is capturable and its scheduling counters reset themselves:
    several replays of one captured call give identical outputs."""
    w, hv, qs, q32 = _case("qwen2.5-1.5b", [600, 1500, 90], [40, 100, 90], 12, 2, 128)
    out = _run(w, hv, qs, q32, 128, kernel=kernel)
    ref = out.clone()
    kc = to_device(hv.k_pool, W.DT_BF16)
    vc = to_device(hv.v_pool, W.DT_BF16)
    q = to_device(q32, W.DT_BF16)
    o2 = torch.empty_like(q)
    bt, cl, qd = (torch.from_numpy(a).cuda() for a in (w.block_tables, w.context_lens, qs))
    mq = int(np.diff(qs).max())
    n = pkv.prefill_workspace_size(w.S, q.shape[0], mq, w.Hq, w.Hkv, w.d, w.bs, w.max_context_len, 128)
    ws = torch.zeros(max(n, 256), dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        pkv.paged_attention_prefill(o2, q, kc, vc, bt, cl, qd, mq, w.max_context_len, scale=w.scale,
                                    partition_size=128, workspace=ws, stream=s, kernel=kernel)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        pkv.paged_attention_prefill(o2, q, kc, vc, bt, cl, qd, mq, w.max_context_len, scale=w.scale,
                                    partition_size=128, workspace=ws, stream=s, kernel=kernel)
    for _ in range(3):
        o2.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(o2, ref)


@pytest.mark.parametrize("kernel", KERNELS)
def test_prefill_one_query_equals_decode(kernel):
    w, hv, qs, q32 = _case("qwen2.5-1.5b", [5, 200, 1025], [1, 1, 1], 12, 2, 128)
    out = _run(w, hv, qs, q32, 0, kernel=kernel)
    q = to_device(q32, W.DT_BF16, "cuda")
    dec = torch.empty_like(q)
    ws = pkv.make_workspace(w.S, w.Hq, w.Hkv, w.d, w.bs, w.max_context_len, -1)
    pkv.paged_attention_decode(dec, q, to_device(hv.k_pool, W.DT_BF16, "cuda"),
                               to_device(hv.v_pool, W.DT_BF16, "cuda"), torch.from_numpy(w.block_tables).cuda(),
                               torch.from_numpy(w.context_lens).cuda(), w.max_context_len, scale=w.scale,
                               partition_size=-1, workspace=ws)
    ref = _ref(w, hv, qs, q32)
    assert_close(out, ref, W.DT_BF16, "prefill q_len=1")
    assert_close(dec, ref, W.DT_BF16, "decode")


@pytest.mark.parametrize("kernel", KERNELS)
def test_prefill_chunked_long_prompt(kernel):
    """A Qwen2.5-7B-shaped batch: 8 sequences with 512-token chunks at the
    end of 1,024 .. 4,096-token contexts, and 24 decoding sequences (one
    query) next to them, as one call."""
    rng = np.random.default_rng(12)
    lens = list(rng.integers(1024, 4097, 8)) + list(rng.integers(16, 3000, 24))
    qlens = [512] * 8 + [1] * 24
    w, hv, qs, q32 = _case("qwen2.5-1.5b", lens, qlens, 28, 4, 128, seed=13)
    out = _run(w, hv, qs, q32, 0, kernel=kernel)
    assert_close(out, _ref(w, hv, qs, q32), W.DT_BF16, f"mixed chunk + decode batch {kernel}")


@pytest.mark.parametrize("kernel", KERNELS)
def test_prefill_bad_query_count_reported(kernel):
    w, hv, qs, q32 = _case("qwen2.5-1.5b", [20, 30], [4, 4], 8, 2, 128)
    bad = np.array([0, 4, 40], np.int32)            # second sequence: 36 queries > 30 tokens
    q32 = W.host_normal(7, "prefill-query-bad", (40, w.Hq, w.d))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = _run(w, hv, bad, q32, -1, query_start=bad, err=err, max_query_len=4, kernel=kernel)   # host's view
    torch.cuda.synchronize()
    assert int(err.item()) == 6
    ref = O.paged_attention_prefill(W.bf16_bits(q32[:4]), O.BF16, W.bf16_bits(hv.k_pool), W.bf16_bits(hv.v_pool),
                                    O.BF16, w.block_tables[:1], w.context_lens[:1], np.array([0, 4], np.int32),
                                    w.scale)
    assert_close(out[:4], ref, W.DT_BF16, "valid sequence of a batch with a bad one")


@pytest.mark.parametrize("kernel", KERNELS)
def test_prefill_queries_outside_the_batch_are_skipped(kernel):
    """query_start naming rows past T, or more queries than max_query_len
    covers: skipped and reported, nothing written out of bounds."""
    w, hv, qs, q32 = _case("qwen2.5-1.5b", [20, 30, 25], [4, 4, 4], 8, 2, 128)
    cases = [(bad, mq, part) for bad, mq in ((np.array([0, 4, 8, 40], np.int32), 4),
                                             (np.array([0, 4, 12, 12], np.int32), 4)) for part in (-1, 16)]
    for bad, mq, part in cases:
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        out = _run(w, hv, qs, q32, part, query_start=bad, err=err, max_query_len=mq, kernel=kernel)
        torch.cuda.synchronize()
        assert int(err.item()) == 6
        ref = _ref(w, hv, qs, q32)
        assert_close(out[:4], ref[:4], W.DT_BF16, "the valid first sequence")


FULL = [("qwen2.5-7b-chunked", 4, 6), ("qwen2.5-72b-spec", 3, 5)]


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("name,nseq,nq", FULL, ids=[f[0] for f in FULL])
def test_full_size_query_chunks(name, nseq, nq, kernel):
    """The query-chunk workloads at full size, in the launch configuration
    the benchmark times (default partitioning).  Sampled sequences hold host
    draws; for each, a few of its queries (first, last, random) are
    recomputed by the oracle as one-query sequences ending at the query's
    position, which is the causal rule itself.  Every output is finite and
    bounded by max |V| (a convex combination)."""
    from tests.gpu_cases import build_case
    w = W.make(name)
    c = build_case(w, sample=nseq)
    qlens = W.query_lens(w)
    qs = W.query_start(qlens)
    T = int(qs[-1])
    q32 = W.host_normal(w.seed, "chunk-query", (T, w.Hq, w.d))
    q = to_device(q32, W.DT_BF16)
    out = torch.empty_like(q)
    P = 0
    wsb = pkv.prefill_workspace_size(w.S, T, int(qlens.max()), w.Hq, w.Hkv, w.d, w.bs, w.max_context_len, P)
    wsp = torch.zeros(wsb, dtype=torch.uint8, device="cuda")
    pkv.paged_attention_prefill(out, q, c.k_cache, c.v_cache, c.block_tables, c.context_lens,
                                torch.from_numpy(qs).cuda(), int(qlens.max()), w.max_context_len, scale=w.scale,
                                partition_size=P, workspace=wsp, kernel=kernel)
    torch.cuda.synchronize()
    rng = np.random.default_rng(5)
    rows, tabs, lens = [], [], []
    for j, s in enumerate(c.seqs):
        ql, n = int(qlens[s]), int(w.context_lens[s])
        pick = sorted({0, ql - 1} | set(rng.integers(0, ql, max(0, nq - 2)).tolist()))
        for i in pick:
            rows.append(int(qs[s]) + i)
            tabs.append(c.ow.block_tables[j])
            lens.append(n - ql + i + 1)
    rows_a = np.array(rows)
    ref = O.paged_attention_prefill(W.bf16_bits(q32[rows_a]), O.BF16, c.o_k, c.o_v, O.BF16, np.stack(tabs),
                                    np.array(lens, np.int32), np.arange(len(rows) + 1, dtype=np.int32), w.scale)
    assert_close(out[torch.from_numpy(rows_a).cuda()], ref, W.DT_BF16, f"{name} {kernel} sampled queries")
    of = out.float()
    assert torch.isfinite(of).all()
    assert float(of.abs().max()) <= float(c.v_cache.float().abs().max()) * 1.01 + 1e-3


@pytest.mark.parametrize("kernel", KERNELS)
def test_prefill_growing_logits_rescale(kernel):
    """Keys whose scale grows along the sequence (token t scaled by
    1 + t / 40): each 128-token stage's largest logit exceeds the previous
    ones by far more than 2^8, so the kernels must rescale the running
    output many times; the softmax itself is unchanged by that."""
    w, hv, qs, q32 = _case("qwen2.5-1.5b", [1100, 700, 260], [300, 5, 260], 8, 2, 128, seed=9)
    for s in range(w.S):
        n = int(w.context_lens[s])
        for t in range(n):
            b = int(w.block_tables[s, t // w.bs])
            hv.k_pool[b, t % w.bs] *= np.float32(1.0 + t / 40.0)
    for partition in (-1, 256):
        out = _run(w, hv, qs, q32, partition, kernel=kernel)
        assert_close(out, _ref(w, hv, qs, q32), W.DT_BF16, f"growing logits {kernel} P={partition}")
