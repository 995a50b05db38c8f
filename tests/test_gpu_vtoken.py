"""Decode through token tables and token repacking (vToken) through the C
ABI, against the oracle."""
import dataclasses

import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import oracle as O
    import paged_kv_cache_44_gb300 as pkv
    from tests.gpu_cases import ODT, assert_close, host_raw, to_device


def _case(name, lens, Hq, Hkv, d, cache, keep, seed=3):
    w = W.make(name, S=len(lens), lengths=np.array(lens), seed=seed)
    w = dataclasses.replace(w, Hq=Hq, Hkv=Hkv, d=d, cache_dtype=cache)
    hv = W.host_values(w)
    slots, nt = W.token_tables(w, keep)
    return w, hv, slots, nt


def _caches(w, hv, dev="cuda"):
    """Device caches and the oracle's raw pools for the same values (fp8
    through each side's own write, as in the decode tests)."""
    if w.cache_dtype == W.DT_E4M3:
        ks, vs = hv.k_scale, hv.v_scale
        kc = torch.zeros((w.NB, w.bs, w.Hkv, w.d), dtype=torch.uint8, device=dev)
        vc = torch.zeros_like(kc)
        slots = torch.arange(w.NB * w.bs, device=dev, dtype=torch.int64)
        kk = torch.from_numpy(hv.k_pool.reshape(-1, w.Hkv, w.d)).to(dev)
        vv = torch.from_numpy(hv.v_pool.reshape(-1, w.Hkv, w.d)).to(dev)
        pkv.paged_kv_write(kk, vv, kc, vc, slots, ks, vs)
        ok = np.zeros((w.NB, w.bs, w.Hkv, w.d), np.uint8)
        ov = np.zeros_like(ok)
        sl = np.arange(w.NB * w.bs, dtype=np.int64)
        O.paged_kv_write(hv.k_pool.reshape(-1, w.Hkv, w.d), hv.v_pool.reshape(-1, w.Hkv, w.d), O.F32, ok, ov,
                         O.E4M3, sl, w.bs, ks, vs)
        return kc, vc, ok, ov, ks, vs
    kc, vc = to_device(hv.k_pool, w.cache_dtype, dev), to_device(hv.v_pool, w.cache_dtype, dev)
    return kc, vc, host_raw(hv.k_pool, w.cache_dtype), host_raw(hv.v_pool, w.cache_dtype), 1.0, 1.0


def _gpu_token_decode(w, q, kc, vc, slots, nt, ks, vs, P, err=None):
    out = torch.empty_like(q)
    mx = int(nt.max())
    ws = pkv.make_workspace(w.S, w.Hq, w.Hkv, w.d, w.bs, mx, P)
    pkv.token_attention_decode(out, q, kc, vc, torch.from_numpy(slots).cuda(), torch.from_numpy(nt).cuda(), mx,
                               scale=w.scale, k_scale=ks, v_scale=vs, partition_size=P, workspace=ws, err_word=err)
    return out


CASES = [
    # (bs workload, lens, Hq, Hkv, d, cache, keep fraction)
    ("qwen2.5-1.5b", [1, 17, 64, 300, 1000, 2049], 12, 2, 128, W.DT_BF16, 0.5),
    ("qwen2.5-1.5b", [40, 129, 700], 8, 8, 64, W.DT_BF16, 0.3),
    ("qwen2.5-1.5b", [5, 600, 1500], 8, 1, 128, W.DT_BF16, 0.9),
    ("fp8-bs32", [33, 700, 1400], 16, 2, 128, W.DT_E4M3, 0.5),
    ("fp8-bs16", [100, 900], 8, 2, 64, W.DT_E4M3, 0.25),
    # a 262,143-token table with half its tokens live (131,284), beside a short one
    ("qwen2.5-1.5b", [262143, 7], 8, 1, 64, W.DT_BF16, 0.5),
]


@pytest.mark.parametrize("case", CASES, ids=[f"{c[0]}-{c[5]}-g{c[2] // c[3]}-d{c[4]}-k{c[6]}" for c in CASES])
# 128: partial partitions cut into 32-token chunks; with an E4M3 cache the
# longer sequences' last full partition too
@pytest.mark.parametrize("P", [-1, 0, 64, 128])
def test_token_decode_matches_oracle(case, P):
    name, lens, Hq, Hkv, d, cache, keep = case
    w, hv, slots, nt = _case(name, lens, Hq, Hkv, d, cache, keep)
    if P > 0 and P % w.bs:
        P = 2 * w.bs
    kc, vc, ok, ov, ks, vs = _caches(w, hv)
    q32 = W.host_normal(w.seed, "tt-query", (w.S, w.Hq, w.d))
    q = to_device(q32, W.DT_BF16)
    out = _gpu_token_decode(w, q, kc, vc, slots, nt, ks, vs, P)
    ref = O.token_attention_decode(W.bf16_bits(q32), O.BF16, ok, ov, ODT[cache], slots, nt, w.scale, ks, vs)
    assert_close(out, ref, cache, f"token decode P={P}")


@pytest.mark.parametrize("cache", [W.DT_BF16, W.DT_E4M3])
def test_token_table_of_every_token_equals_block_table_decode(cache):
    """Listing every token's slot in order reproduces the block-table decode
    bit for bit (same stages, same arithmetic)."""
    name = "qwen2.5-1.5b" if cache == W.DT_BF16 else "fp8-bs16"
    w, hv, _, _ = _case(name, [1, 100, 513, 2000], 12, 2, 128, cache, 1.0)
    slots, nt = W.token_tables(w, 1.0)
    assert (nt == w.context_lens).all()
    kc, vc, _, _, ks, vs = _caches(w, hv)
    q = to_device(W.host_normal(w.seed, "tt-query", (w.S, w.Hq, w.d)), W.DT_BF16)
    for P in (-1, 256):
        a = _gpu_token_decode(w, q, kc, vc, slots, nt, ks, vs, P)
        b = torch.empty_like(q)
        ws = pkv.make_workspace(w.S, w.Hq, w.Hkv, w.d, w.bs, w.max_context_len, P)
        pkv.paged_attention_decode(b, q, kc, vc, torch.from_numpy(w.block_tables).cuda(),
                                   torch.from_numpy(w.context_lens).cuda(), w.max_context_len, scale=w.scale,
                                   k_scale=ks, v_scale=vs, partition_size=P, workspace=ws, kernel="tensor_cores")
        assert torch.equal(a, b), f"P={P}"


@pytest.mark.parametrize("cache", [W.DT_BF16, W.DT_E4M3])
def test_repack_matches_oracle_and_keeps_attention(cache):
    """Plan on the host (the library's planner), move on the GPU: the caches'
    moved rows and the table equal the oracle's; released blocks are then
    overwritten, and attention is bit-identical to before the repack."""
    name = "qwen2.5-1.5b" if cache == W.DT_BF16 else "fp8-bs16"
    w, hv, slots, nt = _case(name, [300, 1000, 77, 2000], 12, 2, 128, cache, 0.3, seed=9)
    kc, vc, ok, ov, ks, vs = _caches(w, hv)
    kc2 = torch.zeros_like(kc)           # a second layer, to check every layer moves
    kc2.copy_(kc)
    vc2 = vc.clone()
    q = to_device(W.host_normal(w.seed, "tt-query", (w.S, w.Hq, w.d)), W.DT_BF16)
    before = _gpu_token_decode(w, q, kc, vc, slots, nt, ks, vs, 0)
    moves, freed = pkv.vtoken_plan(slots, nt, w.bs, w.NB)
    assert len(moves) and len(freed)
    ts = torch.from_numpy(slots).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.repack_tokens([kc, kc2], [vc, vc2], ts, torch.from_numpy(moves).cuda(), err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ok2, ov2, sl2 = ok.copy(), ov.copy(), slots.copy()
    assert O.repack_tokens([ok2], [ov2], sl2, moves) == 0
    np.testing.assert_array_equal(ts.cpu().numpy(), sl2)
    raw = (lambda t: t.cpu().view(torch.int16).numpy().view(np.uint16)) if cache == W.DT_BF16 else \
        (lambda t: t.cpu().numpy())
    np.testing.assert_array_equal(raw(kc), ok2)
    np.testing.assert_array_equal(raw(vc), ov2)
    assert torch.equal(kc, kc2) and torch.equal(vc, vc2)
    fb = torch.from_numpy(freed.astype(np.int64)).cuda()
    for t in (kc, vc):
        t[fb] = 0x7f if cache == W.DT_E4M3 else 1e30     # released blocks are reused
    after = _gpu_token_decode(w, q, kc, vc, ts.cpu().numpy(), nt, ks, vs, 0)
    assert torch.equal(before, after)


def test_bad_slot_and_bad_move_are_reported():
    w, hv, slots, nt = _case("qwen2.5-1.5b", [100, 200], 8, 2, 128, W.DT_BF16, 0.5)
    kc, vc, ok, ov, ks, vs = _caches(w, hv)
    q32 = W.host_normal(w.seed, "tt-query", (w.S, w.Hq, w.d))
    q = to_device(q32, W.DT_BF16)
    bad = slots.copy()
    bad[1, 3] = w.NB * w.bs + 7
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = _gpu_token_decode(w, q, kc, vc, bad, nt, ks, vs, -1, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 3
    ref = O.token_attention_decode(W.bf16_bits(q32[:1]), O.BF16, ok, ov, O.BF16, slots[:1], nt[:1], w.scale)
    assert_close(out[:1], ref, W.DT_BF16, "the sequence with a valid table")
    ts = torch.from_numpy(slots).cuda()
    mv = torch.tensor([[0, 0, int(slots[0, 0]) + 1, 5], [0, 1, int(slots[0, 1]), w.NB * w.bs]], dtype=torch.int64,
                      device="cuda")
    before = kc.clone()
    err.zero_()
    pkv.repack_tokens([kc], [vc], ts, mv, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 7
    assert torch.equal(ts.cpu(), torch.from_numpy(slots)) and torch.equal(kc, before)
