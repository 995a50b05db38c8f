"""The benchmark's algorithmic byte counts (the numerator of every roofline
fraction it reports) against closed forms written from the workload shapes:
the per-token K/V size 2 * Hkv * d * b of one layer ("LLM推論の基礎とvLLMの
内部", section 2, with L = 1), the query and output once, one 4-byte table
entry per block read and one length per sequence."""
import numpy as np

import bench
import workloads as W


def test_72b_long_decode_bytes():
    w = W.make("qwen2.5-72b-long")
    S, Hq, Hkv, d, n, bs = 32, 64, 8, 128, 32768, 16
    per_token = 2 * Hkv * d * 2                                   # K and V, bf16
    assert per_token == 4096
    kv = S * n * per_token                                        # 4 GiB
    assert kv == 4 * 2**30
    want = kv + 2 * S * Hq * d * 2 + S * (n // bs) * 4 + S * 4
    assert bench.decode_bytes(w) == want == 4_296_278_144


def test_shared_prefix_counted_once():
    w = W.make("qwen2.5-7b-prefix")
    assert w.shared_seqs == 100
    prefix_tokens = 64 * w.bs                                     # 64 shared blocks
    assert int(w.context_lens[:100].min()) > prefix_tokens       # every sharer reads the whole prefix
    per_token = 2 * w.Hkv * w.d * 2
    logical = bench.decode_bytes(w, unique=False)
    assert logical - bench.decode_bytes(w) == (w.shared_seqs - 1) * prefix_tokens * per_token
    kv_logical = int(w.context_lens.astype(np.int64).sum()) * per_token
    blocks = int((-(-w.context_lens.astype(np.int64) // w.bs)).sum())
    assert logical == kv_logical + 2 * w.S * w.Hq * w.d * 2 + blocks * 4 + w.S * 4


def test_fp8_step_write_and_copy_bytes():
    w = W.make("fp8-bs16")
    # one new token per sequence: bf16 K and V read, E4M3 codes written, an 8-byte slot each
    assert bench.write_bytes(w) == w.S * w.Hkv * w.d * 2 * (2 + 1) + w.S * 8
    # 64 copy-on-write pairs: each K and V block (bs * Hkv * d codes) read and written, a 16-byte pair
    blk = w.bs * w.Hkv * w.d * 1
    assert len(w.cow_pairs) == 64
    assert bench.copy_bytes(w) == 64 * (2 * 2 * blk + 16)
