"""GPU parity: the CUDA path through the C ABI against the CPU oracle, on the
same seeded inputs.  Write and copy must match bit for bit; decode must stay
within the tolerance of its cache dtype (fp32 1e-5; bf16 2e-2 abs + 1e-2
rel; fp8 5e-2 against the oracle fed the same dequantised values)."""
import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import oracle as O
    import paged_kv_cache_44_gb300 as pkv
    from tests.gpu_cases import (ODT, assert_close, build_case, gpu_decode, gpu_write, oracle_decode,
                                 oracle_write, tolerance)

KERNELS = ["cuda_cores", "tensor_cores"]


def _kernels_for(w):
    """Kernels that apply to this workload (PKV_TEST_KERNELS narrows the list)."""
    import os
    ks = ["cuda_cores"]
    if w.cache_dtype == W.DT_E4M3 or (w.cache_dtype == W.DT_BF16 and w.q_dtype == W.DT_BF16):
        ks.append("tensor_cores")
    only = os.environ.get("PKV_TEST_KERNELS")
    return [k for k in ks if not only or k in only.split(",")]


def _np_cache(t: torch.Tensor) -> np.ndarray:
    t = t.cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


# --------------------------------------------------------------- tiny, fp32

def test_tiny_step_write_decode_copy():
    """The tiny configuration end to end: write one token per sequence
    (lengths 1, 15, 16, 37 -> 2, 16, 17, 38), decode, copy-on-write."""
    w = W.make("tiny")
    c = build_case(w)
    # reading (i): decode over the lengths before the write
    before = w.context_lens - 1
    ref_i = oracle_decode(c, context_lens=before)
    out_i = gpu_decode(c, context_lens=torch.from_numpy(before).cuda(), max_context_len=int(before.max()))
    assert_close(out_i, ref_i, w.cache_dtype, "decode before write")
    # the write is bit-exact
    gpu_write(c)
    oracle_write(c)
    np.testing.assert_array_equal(_np_cache(c.k_cache), c.o_k)
    np.testing.assert_array_equal(_np_cache(c.v_cache), c.o_v)
    # reading (ii): decode over the lengths after the write, every kernel and split
    ref = oracle_decode(c)
    for P in (0, -1, 16, 32):
        out = gpu_decode(c, partition_size=P)
        assert_close(out, ref, w.cache_dtype, f"decode P={P}")
    # copy-on-write: bit-exact, then repointing a holder leaves outputs unchanged
    pkv.copy_blocks([c.k_cache], [c.v_cache], c.cow)
    O.copy_blocks([c.o_k], [c.o_v], w.cow_pairs)
    np.testing.assert_array_equal(_np_cache(c.k_cache), c.o_k)
    np.testing.assert_array_equal(_np_cache(c.v_cache), c.o_v)


def test_tiny_single_token_is_v_exactly():
    w = W.make("tiny")
    c = build_case(w)
    ones = torch.ones(w.S, dtype=torch.int32, device="cuda")
    out = gpu_decode(c, context_lens=ones, max_context_len=1)
    bt = w.block_tables
    for s in range(w.S):
        v0 = c.hv.v_pool[bt[s, 0], 0]                    # [Hkv, d]
        np.testing.assert_array_equal(out[s].cpu().numpy(), np.repeat(v0, w.g, axis=0))


# ------------------------------------------------------ dtype / shape sweep

SWEEP = [
    # (cache, q, d, bs, Hq, Hkv)
    ("f32", "f32", 64, 16, 4, 2), ("f32", "f32", 128, 32, 8, 1), ("f32", "bf16", 128, 16, 6, 6),
    ("bf16", "bf16", 128, 16, 12, 2), ("bf16", "bf16", 64, 32, 16, 2), ("bf16", "bf16", 128, 16, 8, 8),
    ("bf16", "bf16", 128, 32, 28, 4), ("bf16", "f32", 128, 16, 8, 1),
    ("e4m3", "bf16", 128, 16, 28, 4), ("e4m3", "bf16", 128, 32, 7, 1), ("e4m3", "f32", 64, 16, 4, 4),
    # more than 8 query heads per K/V head: several head sets, the last one short
    ("bf16", "bf16", 128, 16, 32, 2), ("e4m3", "bf16", 64, 16, 12, 1),
]


def _sweep_workload(cache, q, d, bs, Hq, Hkv, seed):
    """Ragged lengths around block and partition edges, one empty sequence."""
    import dataclasses
    lens = np.array([1, 1, 2, 15, 16, 17, 31, 32, 33, 63, 64, 65, 200, 513, 1000, 1537], np.int64)
    base = W.make("qwen2.5-1.5b" if bs == 16 else "fp8-bs32", S=len(lens), lengths=lens, seed=seed)
    cl = base.context_lens.copy()
    cl[0] = 0
    return dataclasses.replace(base, Hq=Hq, Hkv=Hkv, d=d, q_dtype=q, cache_dtype=cache, context_lens=cl)


@pytest.mark.parametrize("cfg", SWEEP, ids=["-".join(map(str, c)) for c in SWEEP])
def test_decode_sweep(cfg):
    w = _sweep_workload(*cfg, seed=40 + SWEEP.index(cfg))
    c = build_case(w)
    gpu_write(c)
    oracle_write(c)
    np.testing.assert_array_equal(_np_cache(c.k_cache), c.o_k)
    np.testing.assert_array_equal(_np_cache(c.v_cache), c.o_v)
    ref = oracle_decode(c)
    assert (ref[0] == 0).all()
    for kernel in _kernels_for(w):
        # 128 and 256 cut partial partitions into chunks; at 128 the longer
        # sequences (4+ full partitions) also have their last full one cut
        # (E4M3 caches on tensor cores)
        for P in (0, -1, w.bs, 128, 256):
            out = gpu_decode(c, partition_size=P, kernel=kernel)
            assert_close(out, ref, w.cache_dtype, f"{kernel} P={P}")
            assert (out[0] == 0).all()


@pytest.mark.parametrize("cfg", [("bf16", "bf16", 128, 16, 28, 4), ("e4m3", "bf16", 64, 32, 12, 1)],
                         ids=["bf16-g7", "e4m3-g12"])
def test_split_decode_reuses_workspace(cfg):
    """A split decode leaves the workspace's scheduling header zero, so one
    workspace serves call after call, with bit-identical results."""
    w = _sweep_workload(*cfg, seed=77)
    c = build_case(w)
    ref = oracle_decode(c)
    for P in (w.bs, 64, 128, 512, 0):
        ws = pkv.make_workspace(w.S, w.Hq, w.Hkv, w.d, w.bs, w.max_context_len, P)
        zero = 256
        outs = []
        for _ in range(3):
            out = torch.empty_like(c.q)
            pkv.paged_attention_decode(out, c.q, c.k_cache, c.v_cache, c.block_tables, c.context_lens,
                                       w.max_context_len, scale=w.scale, k_scale=c.k_scale, v_scale=c.v_scale,
                                       partition_size=P, workspace=ws, kernel="tensor_cores")
            torch.cuda.synchronize()
            assert int(ws[:zero].count_nonzero()) == 0, f"P={P}: scheduling state left behind"
            outs.append(out)
        assert_close(outs[0], ref, w.cache_dtype, f"P={P}")
        for o in outs[1:]:
            assert torch.equal(o, outs[0])


# ---------------------------------------------------------------- invariance

@pytest.mark.parametrize("kernel", KERNELS)
def test_permutation_invariance_bit_identical(kernel):
    w = W.make("qwen2.5-1.5b", S=8, lengths=np.array([1, 16, 17, 100, 513, 700, 2049, 4000]))
    c = build_case(w)
    if kernel not in _kernels_for(w):
        pytest.skip("kernel does not apply or is not selected")
    out = gpu_decode(c, kernel=kernel)
    perm = torch.from_numpy(np.random.default_rng(9).permutation(w.NB)).cuda()
    k2 = torch.empty_like(c.k_cache); v2 = torch.empty_like(c.v_cache)
    k2[perm] = c.k_cache; v2[perm] = c.v_cache
    c.k_cache, c.v_cache = k2, v2
    out2 = gpu_decode(c, kernel=kernel, block_tables=perm[c.block_tables.long()].to(torch.int32).contiguous())
    assert torch.equal(out, out2)


@pytest.mark.parametrize("kernel", KERNELS)
def test_shared_prefix_equals_private_copies(kernel):
    w = W.make("qwen2.5-7b-prefix", S=12, lengths=np.array([1030, 1100, 2000, 1025, 5000, 1500, 3, 40, 700,
                                                              1200, 90, 4000]), spare_blocks=64,
               shared_seqs=6)
    assert w.shared_seqs == 6 and (w.block_tables[:6, :64] == w.block_tables[0, :64]).all()
    c = build_case(w)
    if kernel not in _kernels_for(w):
        pytest.skip("kernel does not apply or is not selected")
    out = gpu_decode(c, kernel=kernel)
    ref = oracle_decode(c)
    assert_close(out, ref, w.cache_dtype, "shared prefix")
    # private copy of the 64 prefix blocks for sequence 2 via copy_blocks, then repoint
    used = set(w.block_tables[w.block_tables != 0].tolist()) | set(w.cow_pairs[:, 1].tolist())
    spare = [b for b in range(1, w.NB) if b not in used][:64]
    pairs = np.stack([w.block_tables[2, :64], spare], axis=1).astype(np.int64)
    pkv.copy_blocks([c.k_cache], [c.v_cache], torch.from_numpy(pairs).cuda())
    bt = c.block_tables.clone()
    bt[2, :64] = torch.tensor(spare, dtype=torch.int32)
    out2 = gpu_decode(c, kernel=kernel, block_tables=bt)
    assert torch.equal(out, out2)


# ---------------------------------------------------------------- device errors

def test_bad_block_ids_are_skipped_and_reported():
    w = W.make("qwen2.5-1.5b", S=3, lengths=np.array([40, 600, 33]))
    c = build_case(w)
    bt = c.block_tables.clone()
    bt[1, 3] = w.NB + 1000          # out of range: must be skipped, not read
    bt[2, 1] = -7
    for kernel in _kernels_for(w):
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        out = gpu_decode(c, kernel=kernel, block_tables=bt, err_word=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 1
        assert torch.isfinite(out.float()).all()
        ref = oracle_decode(c)
        assert_close(out[0:1], ref[0:1], w.cache_dtype, "unaffected sequence")


def test_bad_context_len_is_clamped_and_reported():
    w = W.make("qwen2.5-1.5b", S=2, lengths=np.array([40, 60]))
    c = build_case(w)
    cl = c.context_lens.clone()
    cl[1] = w.max_context_len + 50           # above the host bound: clamped, reported
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = gpu_decode(c, context_lens=cl, err_word=err, partition_size=16)
    torch.cuda.synchronize()
    assert int(err.item()) == 2
    assert torch.isfinite(out.float()).all()


def test_bad_slot_is_skipped_and_reported():
    w = W.make("tiny")
    c = build_case(w)
    sm = c.slot_mapping.clone()
    sm[0] = w.NB * w.bs + 3
    sm[1] = -1
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.paged_kv_write(c.new_k, c.new_v, c.k_cache, c.v_cache, sm, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 3
    c.slot_mapping = sm
    ow_slots = c.ow.slot_mapping.copy()
    ow_slots[0] = -1
    ow_slots[1] = -1
    c.ow.slot_mapping = ow_slots
    oracle_write(c)
    np.testing.assert_array_equal(_np_cache(c.k_cache), c.o_k)


def _guarded(cache, G=4):
    """The pool as the middle of a larger buffer: G blocks of a byte pattern
    on each side catch any write past either end of the pool."""
    NB = cache.shape[0]
    big = torch.empty((NB + 2 * G,) + tuple(cache.shape[1:]), dtype=cache.dtype, device=cache.device)
    big.view(torch.uint8).fill_(0x5A)
    big[G:G + NB].copy_(cache)
    return big, big[G:G + NB]


def _guards_intact(big, G=4):
    raw = big.view(torch.uint8)
    return bool((raw[:G] == 0x5A).all()) and bool((raw[-G:] == 0x5A).all())


def test_bad_slots_and_pairs_write_nothing_outside_the_pool():
    """Slots and copy pairs past the pool are skipped: the blocks around the
    pool keep their pattern, and the pool is what the oracle says."""
    w = W.make("tiny")
    c = build_case(w)
    big_k, kc = _guarded(c.k_cache)
    big_v, vc = _guarded(c.v_cache)
    sm = c.slot_mapping.clone()
    sm[0] = w.NB * w.bs + 3                 # one block past the end
    sm[1] = w.NB * w.bs                     # the first slot past the end
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.paged_kv_write(c.new_k, c.new_v, kc, vc, sm, err_word=err)
    pairs = torch.tensor([[1, w.NB], [2, w.NB + 3], [w.NB, 5]], dtype=torch.int64, device="cuda")
    before = kc.clone()
    err2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.copy_blocks([kc], [vc], pairs, err_word=err2)
    torch.cuda.synchronize()
    assert int(err.item()) == 3 and int(err2.item()) == 4
    assert _guards_intact(big_k) and _guards_intact(big_v)
    assert torch.equal(before, kc)


def test_bad_copy_pair_is_skipped_and_reported():
    w = W.make("tiny")
    c = build_case(w)
    before = c.k_cache.clone()
    pairs = torch.tensor([[1, w.NB + 2], [-1, 3]], dtype=torch.int64, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.copy_blocks([c.k_cache], [c.v_cache], pairs, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 4
    assert torch.equal(before, c.k_cache)


def _conflict_free_pairs(pairs, NB):
    """The pairs copy_blocks copies when it checks them: in the pool, and
    with a destination no other in-pool pair writes and no in-pool pair
    (itself included) reads."""
    inpool = [(int(s), int(d)) for s, d in pairs if 0 <= s < NB and 0 <= d < NB]
    keep = []
    for i, (s, d) in enumerate(pairs):
        if not (0 <= s < NB and 0 <= d < NB):
            continue
        dsts = [d2 for j, (_, d2) in enumerate(pairs) if j != i and 0 <= pairs[j][0] < NB and 0 <= d2 < NB]
        if d in dsts or d in [s2 for s2, _ in inpool]:
            continue
        keep.append((s, d))
    return np.array(keep, np.int64).reshape(-1, 2)


@pytest.mark.parametrize("layers", [1, 3])
def test_conflicting_copy_pairs_are_skipped_and_reported(layers):
    """With an error word, a pair whose destination is another pair's
    destination or any pair's source is skipped and reported; the other
    pairs are copied bit for bit as the oracle copies them, and the blocks
    around the pool keep their pattern."""
    w = W.make("tiny")
    c = build_case(w)
    pairs = np.array([[1, 5], [2, 5],            # the same destination twice: both skipped
                      [3, 6], [6, 7],            # 6 is written and read: the first skipped, the second copied
                      [4, 8], [9, 9],            # a plain copy; a block copied onto itself: skipped
                      [10, w.NB], [11, 12]],     # out of the pool: skipped; a plain copy
                     np.int64)
    keep = _conflict_free_pairs(pairs, w.NB)
    assert keep.tolist() == [[6, 7], [4, 8], [11, 12]]
    bigs, kcs, vcs, oks, ovs = [], [], [], [], []
    for layer in range(layers):
        k_l, v_l = (c.k_cache, c.v_cache) if layer == 0 else (c.k_cache * (layer + 1), c.v_cache - layer)
        bk, kc = _guarded(k_l.contiguous())
        bv, vc = _guarded(v_l.contiguous())
        bigs += [bk, bv]
        kcs.append(kc)
        vcs.append(vc)
        oks.append(_np_cache(kc).copy())
        ovs.append(_np_cache(vc).copy())
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.copy_blocks(kcs, vcs, torch.from_numpy(pairs).cuda(), err_word=err)
    O.copy_blocks(oks, ovs, keep)
    torch.cuda.synchronize()
    assert int(err.item()) == 4
    for layer in range(layers):
        np.testing.assert_array_equal(_np_cache(kcs[layer]), oks[layer])
        np.testing.assert_array_equal(_np_cache(vcs[layer]), ovs[layer])
    assert all(_guards_intact(b) for b in bigs)
    # the same pairs without the conflicts: nothing to report, same caches
    err.zero_()
    pkv.copy_blocks(kcs, vcs, torch.from_numpy(keep).cuda(), err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for layer in range(layers):
        np.testing.assert_array_equal(_np_cache(kcs[layer]), oks[layer])


def test_decode_growing_logits_rescale():
    """Keys scaled by 1 + t / 40 along each sequence: every stage's largest
    logit exceeds all earlier ones by far more than 2^8, so the running
    output is rescaled at nearly every stage and each partition starts from
    its own maximum; split or not, the result matches the oracle."""
    from tests.gpu_cases import host_raw, to_device
    lens = np.array([1, 40, 700, 1100, 2049])
    w = W.make("qwen2.5-1.5b", S=len(lens), lengths=lens)
    c = build_case(w)
    for s_ in range(w.S):
        for t in range(int(w.context_lens[s_])):
            c.hv.k_pool[int(w.block_tables[s_, t // w.bs]), t % w.bs] *= np.float32(1.0 + t / 40.0)
    c.k_cache = to_device(c.hv.k_pool, w.cache_dtype)
    c.o_k = host_raw(c.hv.k_pool, w.cache_dtype)
    ref = oracle_decode(c)
    for kernel in _kernels_for(w):
        for P in (-1, 0, 128, 16):
            out = gpu_decode(c, partition_size=P, kernel=kernel)
            assert_close(out, ref, w.cache_dtype, f"growing logits {kernel} P={P}")


# ------------------------------------------------------------ maximum sizes

def _bounded(out, c, w):
    """Finite, and within max |V| (every output is a convex combination of V rows)."""
    of = out.float()
    assert torch.isfinite(of).all()
    vmax = 448.0 * c.v_scale if w.cache_dtype == W.DT_E4M3 else float(c.v_cache.float().abs().max())
    assert float(of.abs().max()) <= vmax * 1.01 + 1e-3


@pytest.mark.parametrize("cache", [W.DT_BF16, W.DT_E4M3])
def test_largest_batch(cache):
    """65,535 sequences, the most one decode takes, of 1..64 tokens: first
    the write of each sequence's new token (65,535 tokens in one launch,
    bit-exact on the sampled sequences' blocks), then the decode unsplit and
    in 16-token partitions (a merge grid of 65,535 blocks of 8 rows, a
    CUDA-core grid of 65,535 sequences).  A sample of sequences (shortest,
    longest, random) against the oracle; every output finite and bounded."""
    import dataclasses
    lens = np.random.default_rng(5).integers(1, 65, size=65535)
    w = dataclasses.replace(W.make("qwen2.5-1.5b", S=65535, lengths=lens), Hq=8, Hkv=1, d=64, cache_dtype=cache)
    c = build_case(w, sample=256)
    gpu_write(c)
    oracle_write(c)
    ids = torch.from_numpy(c.ow.renumber.astype(np.int64)).cuda()
    np.testing.assert_array_equal(_np_cache(c.k_cache[ids]), c.o_k)
    np.testing.assert_array_equal(_np_cache(c.v_cache[ids]), c.o_v)
    ref = oracle_decode(c)
    rows = torch.from_numpy(c.seqs).cuda()
    for P in (-1, 16):
        for kernel in _kernels_for(w):
            out = gpu_decode(c, partition_size=P, kernel=kernel)
            assert_close(out[rows], ref, w.cache_dtype, f"S=65535 P={P} {kernel}")
            _bounded(out, c, w)


@pytest.mark.parametrize("cache", [W.DT_BF16, W.DT_E4M3])
def test_longest_context(cache):
    """A 262,143-token sequence beside a 5-token one: the library's partition
    (about a thousand partial results per row, merged 16 at a time) and
    unsplit (one unit streams the whole sequence).  Every output against the
    oracle."""
    import dataclasses
    lens = np.array([262143, 5])
    w = dataclasses.replace(W.make("qwen2.5-1.5b", S=2, lengths=lens), Hq=8, Hkv=1, d=64, cache_dtype=cache)
    c = build_case(w)
    ref = oracle_decode(c)
    assert pkv.decode_partition_size(w.S, w.Hq, w.Hkv, w.d, w.bs, w.max_context_len, 0) > 0
    for P in (0, -1):
        for kernel in _kernels_for(w):
            out = gpu_decode(c, partition_size=P, kernel=kernel)
            assert_close(out, ref, w.cache_dtype, f"262,143 tokens P={P} {kernel}")
            _bounded(out, c, w)


# ------------------------------------------------------------ full-size runs

FULL = [("qwen2.5-1.5b", None), ("qwen2.5-7b-prefix", None), ("qwen2.5-72b-long", 3), ("fp8-bs16", 4),
        ("fp8-bs32", 4)]


@pytest.mark.parametrize("name,sample", FULL, ids=[f[0] for f in FULL])
def test_full_size_step(name, sample):
    """The configuration at full size, in the launch configuration the
    benchmark times: write -> decode -> copy_blocks.  Every sequence is
    checked where the oracle finishes in seconds, else a sample of sequences
    (shortest, longest, a prefix sharer, random), plus properties that hold
    at any size: outputs are finite and bounded by max |V| (a convex
    combination), and the write is bit-exact on the sampled blocks."""
    w = W.make(name)
    c = build_case(w, sample=sample)
    gpu_write(c)
    oracle_write(c)
    if sample is None:
        np.testing.assert_array_equal(_np_cache(c.k_cache), c.o_k)
        np.testing.assert_array_equal(_np_cache(c.v_cache), c.o_v)
    else:
        ids = torch.from_numpy(c.ow.renumber.astype(np.int64)).cuda()
        np.testing.assert_array_equal(_np_cache(c.k_cache[ids]), c.o_k)
        np.testing.assert_array_equal(_np_cache(c.v_cache[ids]), c.o_v)
    ref = oracle_decode(c)
    for kernel in _kernels_for(w):
        out = gpu_decode(c, kernel=kernel)
        err = assert_close(out[torch.from_numpy(c.seqs).cuda()], ref, w.cache_dtype, f"{name} {kernel}")
        print(f"max |gpu - oracle| {name} {kernel}: {err:.3e} (tolerance {tolerance(w.cache_dtype, out.dtype)})")
        of = out.float()
        assert torch.isfinite(of).all()
        if w.cache_dtype == W.DT_E4M3:
            vmax = 448.0 * c.v_scale
        else:
            vmax = float(c.v_cache.float().abs().max())
        assert float(of.abs().max()) <= vmax * 1.01 + 1e-3
    pkv.copy_blocks([c.k_cache], [c.v_cache], c.cow)
    src = c.cow[:, 0]; dst = c.cow[:, 1]
    assert torch.equal(c.k_cache[src], c.k_cache[dst]) and torch.equal(c.v_cache[src], c.v_cache[dst])
