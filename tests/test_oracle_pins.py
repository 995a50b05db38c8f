"""Pins of the CPU oracle to facts that do not come from the oracle itself:
numbers the pages print, library routines (torch's SDPA, its float8/bf16
casts), closed forms, invariants and brute force on tiny inputs."""
import math
import os

import numpy as np
import pytest
import torch

import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        return [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]


# ------------------------------------------------------------ byte accounting

def test_kv_size_formula_matches_pages(oracle):
    for model, L, hkv, d, b, per_tok, tokens, req in _rows("kv_size_formula.txt"):
        got = oracle.kv_bytes_per_token(int(L), int(hkv), int(d), int(b))
        assert got == int(per_tok), model
        assert got * int(tokens) == int(req), model


def test_kv_size_cross_checks(oracle):
    per_tok = oracle.kv_bytes_per_token(28, 2, 128, 2)
    for check, tokens, bpt, gib, digits in _rows("kv_size_checks.txt"):
        assert per_tok == int(bpt)
        assert round(int(tokens) * per_tok / 2 ** 30, int(digits)) == float(gib), check
    # an fp8 cache (one byte per element) halves the bf16 figure
    assert oracle.kv_bytes_per_token(28, 2, 128, 1) * 2 == per_tok


def test_block_accounting_matches_pages(oracle):
    for tokens, bs, blocks, usable, fill in _rows("block_accounting.txt"):
        n, bs, blocks = int(tokens), int(bs), int(blocks)
        assert oracle.blocks_for_tokens(n, bs) == blocks
        if int(usable) >= 0:
            assert blocks - 1 == int(usable)          # block 0 is the null block
        assert n - (blocks - 1) * bs == int(fill)     # tokens in the last block


def test_last_block_waste_bound(oracle):
    for bs in (8, 16, 32):
        for n in range(1, 300):
            waste = oracle.blocks_for_tokens(n, bs) * bs - n
            assert 0 <= waste <= bs - 1


def test_long_context_pool_is_four_gib():
    w = W.make("qwen2.5-72b-long")
    kv = w.S * int(w.context_lens[0]) * w.Hkv * w.d * 2 * 2     # K and V, bf16
    assert kv == 4 * 2 ** 30


# ------------------------------------------------------------------- formats

def test_e4m3_decode_all_codes_match_torch(oracle):
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_to_float64(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert (np.isnan(ours) == nan).all()
    assert nan.sum() == 2                                       # 0x7F and 0xFF
    np.testing.assert_array_equal(ours[~nan], ref[~nan])
    assert ours[0x7E] == 448.0 and ours[0x01] == 2.0 ** -9


def test_e4m3_encode_roundtrip_and_ties(oracle):
    finite = np.array([c for c in range(256) if c & 0x7F != 0x7F], np.uint8)
    vals = oracle.e4m3_to_float64(finite).astype(np.float32)
    np.testing.assert_array_equal(oracle.e4m3_from_float32(vals), finite)
    # midpoints between neighbouring non-negative codes go to the even code
    pos = np.arange(0, 0x7E, dtype=np.uint8)
    lo = oracle.e4m3_to_float64(pos)
    hi = oracle.e4m3_to_float64(pos + 1)
    mid = ((lo + hi) / 2).astype(np.float32)
    assert ((lo + hi) / 2 == mid.astype(np.float64)).all()      # midpoints exact in fp32
    enc = oracle.e4m3_from_float32(mid)
    expect = np.where(pos % 2 == 0, pos, pos + 1).astype(np.uint8)
    np.testing.assert_array_equal(enc, expect)


def test_e4m3_encode_matches_torch_in_range(oracle):
    rng = np.random.default_rng(11)
    x = np.concatenate([rng.standard_normal(4000).astype(np.float32) * s
                        for s in (1e-3, 0.1, 1.0, 30.0, 150.0)])
    x = x[np.abs(x) <= 448.0]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(oracle.e4m3_from_float32(x), ref)


def test_e4m3_saturates(oracle):
    big = np.array([448.0, 449.0, 463.9, 464.0, 480.0, 1e6, 3e38], np.float32)
    assert (oracle.e4m3_from_float32(big) == 0x7E).all()
    assert (oracle.e4m3_from_float32(-big) == 0xFE).all()
    assert oracle.e4m3_from_float32(np.array([np.nan], np.float32))[0] & 0x7F == 0x7F
    assert oracle.e4m3_from_float32(np.array([-0.0], np.float32))[0] == 0x80
    assert oracle.e4m3_from_float32(np.array([2.0 ** -11], np.float32))[0] == 0x00


def test_bf16_rounding_matches_torch(oracle):
    rng = np.random.default_rng(12)
    x = rng.standard_normal(20000).astype(np.float32) * np.float32(3.0)
    # exact ties: an odd and an even bf16 neighbour with the halfway bit set
    sign = rng.integers(0, 2, 2000, dtype=np.uint32) << 31
    expo = rng.integers(100, 150, 2000, dtype=np.uint32) << 23
    mant = rng.integers(0, 128, 2000, dtype=np.uint32) << 16
    ties = (sign | expo | mant | np.uint32(0x8000)).astype(np.uint32).view(np.float32)
    x = np.concatenate([x, ties, np.array([0.0, -0.0, 1e-40, 3.3e38], np.float32)])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(oracle.bf16_from_float64(x.astype(np.float64)), ref)
    back = oracle.bf16_to_float64(ref)
    np.testing.assert_array_equal(back, torch.from_numpy(ref.view(np.int16)).view(torch.bfloat16)
                                  .to(torch.float64).numpy())


# ------------------------------------------------------------------- decode

def _sdpa_reference(q, k_ctx, v_ctx, scale):
    """Brute force through torch's fp64 SDPA on contiguous K/V.
    q [Hq, d]; k_ctx/v_ctx [n, Hkv, d]."""
    Hq = q.shape[0]
    Hkv = k_ctx.shape[1]
    g = Hq // Hkv
    qt = torch.from_numpy(q.astype(np.float64))[:, None, :]                     # [Hq, 1, d]
    kt = torch.from_numpy(k_ctx.astype(np.float64)).permute(1, 0, 2)             # [Hkv, n, d]
    vt = torch.from_numpy(v_ctx.astype(np.float64)).permute(1, 0, 2)
    kt = kt.repeat_interleave(g, dim=0)
    vt = vt.repeat_interleave(g, dim=0)
    out = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale)
    return out[:, 0, :].numpy()


def _scatter_case(rng, lens, Hq, Hkv, d, bs, extra_blocks=3):
    """Contiguous per-sequence K/V, scattered by the test itself into a pool
    through random block tables."""
    nblk = [-(-n // bs) for n in lens]
    NB = 1 + sum(nblk) + extra_blocks
    perm = rng.permutation(np.arange(1, NB))
    MB = max(max(nblk), 1)
    tables = np.zeros((len(lens), MB), np.int32)
    kpool = rng.standard_normal((NB, bs, Hkv, d)).astype(np.float32)   # garbage in unused slots
    vpool = rng.standard_normal((NB, bs, Hkv, d)).astype(np.float32)
    kctx, vctx = [], []
    i = 0
    for s, n in enumerate(lens):
        kc = rng.standard_normal((n, Hkv, d)).astype(np.float32)
        vc = rng.standard_normal((n, Hkv, d)).astype(np.float32)
        for j in range(nblk[s]):
            pb = perm[i]; i += 1
            tables[s, j] = pb
            m = min(bs, n - j * bs)
            kpool[pb, :m] = kc[j * bs: j * bs + m]
            vpool[pb, :m] = vc[j * bs: j * bs + m]
        kctx.append(kc); vctx.append(vc)
    q = rng.standard_normal((len(lens), Hq, d)).astype(np.float32)
    return q, kpool, vpool, tables, np.array(lens, np.int32), kctx, vctx


@pytest.mark.parametrize("Hq,Hkv", [(4, 2), (8, 8), (8, 1), (6, 2)])
@pytest.mark.parametrize("bs", [16, 32])
def test_decode_brute_force_tiny(oracle, Hq, Hkv, bs):
    rng = np.random.default_rng(100 + Hq * 10 + Hkv + bs)
    d = 64
    lens = [1, 15, 16, 17, 37, 38, 70]
    q, kp, vp, tabs, cl, kctx, vctx = _scatter_case(rng, lens, Hq, Hkv, d, bs)
    scale = float(np.float32(1.0) / np.sqrt(np.float32(d)))
    out = oracle.paged_attention_decode(q, oracle.F32, kp, vp, oracle.F32, tabs, cl, scale)
    for s in range(len(lens)):
        ref = _sdpa_reference(q[s], kctx[s], vctx[s], scale)
        np.testing.assert_allclose(out[s], ref, rtol=0, atol=1e-12)


def test_decode_page_example_tables(oracle):
    """The pages' block-table pictures, used as the actual tables: request A
    (38 tokens in physical 7, 1, 3), request B sharing physical 7, and the
    second page's 0..3 -> 7, 2, 19, 4."""
    rows = {r[0]: (int(r[1]), [int(x) for x in r[2].split(",")]) for r in _rows("block_table_example.txt")}
    rng = np.random.default_rng(5)
    Hq, Hkv, d, bs, NB = 4, 2, 64, 16, 20
    kp = rng.standard_normal((NB, bs, Hkv, d)).astype(np.float32)
    vp = rng.standard_normal((NB, bs, Hkv, d)).astype(np.float32)
    names = ["request_A", "request_B", "page2_seq"]
    MB = max(len(rows[n][1]) for n in names)
    tabs = np.zeros((3, MB), np.int32)
    for i, n in enumerate(names):
        tabs[i, : len(rows[n][1])] = rows[n][1]
    cl = np.array([rows[n][0] for n in names], np.int32)
    q = rng.standard_normal((3, Hq, d)).astype(np.float32)
    scale = 0.125
    out = oracle.paged_attention_decode(q, oracle.F32, kp, vp, oracle.F32, tabs, cl, scale)
    for i, n in enumerate(names):
        tokens, blocks = rows[n]
        kc = np.concatenate([kp[b] for b in blocks])[:tokens]
        vc = np.concatenate([vp[b] for b in blocks])[:tokens]
        np.testing.assert_allclose(out[i], _sdpa_reference(q[i], kc, vc, scale), atol=1e-12, rtol=0)
    # request A's waste is the 10 empty slots of physical block 3
    assert len(rows["request_A"][1]) * bs - rows["request_A"][0] == 10


def test_decode_permutation_invariance(oracle):
    w = W.make("qwen2.5-1.5b", S=6, lengths=np.array([1, 16, 17, 100, 513, 700]))
    hv = W.host_values(w)
    q = W.bf16_bits(hv.query)
    k = W.bf16_bits(hv.k_pool)
    v = W.bf16_bits(hv.v_pool)
    out = oracle.paged_attention_decode(q, oracle.BF16, k, v, oracle.BF16, w.block_tables,
                                        w.context_lens, w.scale)
    perm = np.random.default_rng(9).permutation(w.NB)        # new id of old block b is perm[b]
    k2 = np.empty_like(k); v2 = np.empty_like(v)
    k2[perm] = k; v2[perm] = v
    out2 = oracle.paged_attention_decode(q, oracle.BF16, k2, v2, oracle.BF16,
                                         perm[w.block_tables].astype(np.int32), w.context_lens, w.scale)
    np.testing.assert_array_equal(out, out2)


def test_decode_shared_prefix_equals_private_copies(oracle):
    w = W.make("qwen2.5-7b-prefix", S=6, lengths=np.array([1030, 1100, 2000, 1025, 1040, 1500]),
               spare_blocks=64)
    assert w.shared_prefix_blocks == 64 and w.shared_seqs == 6
    hv = W.host_values(w)
    k, v = hv.k_pool.copy(), hv.v_pool.copy()
    q = hv.query
    out = oracle.paged_attention_decode(q, oracle.F32, k, v, oracle.F32, w.block_tables,
                                        w.context_lens, w.scale)
    # give sequence 2 a private copy of the prefix in spare blocks
    used = set(w.block_tables[w.block_tables != 0].tolist()) | set(w.cow_pairs[:, 1].tolist())
    spare = [b for b in range(1, w.NB) if b not in used][:64]
    tabs = w.block_tables.copy()
    for j in range(64):
        k[spare[j]] = k[tabs[2, j]]; v[spare[j]] = v[tabs[2, j]]
        tabs[2, j] = spare[j]
    out2 = oracle.paged_attention_decode(q, oracle.F32, k, v, oracle.F32, tabs, w.context_lens, w.scale)
    np.testing.assert_array_equal(out, out2)


def test_decode_special_cases(oracle):
    rng = np.random.default_rng(3)
    Hq, Hkv, d, bs = 4, 2, 64, 16
    q, kp, vp, tabs, cl, kctx, vctx = _scatter_case(rng, [1, 0, 20], Hq, Hkv, d, bs)
    out = oracle.paged_attention_decode(q, oracle.F32, kp, vp, oracle.F32, tabs, cl, 0.125)
    # one token: the output is that token's V, exactly
    np.testing.assert_array_equal(out[0], vctx[0][0].astype(np.float64).repeat(2, axis=0))
    # no tokens: zeros
    assert (out[1] == 0).all()
    # all keys equal: uniform weights, the output is the mean of V
    for j in range(tabs.shape[1]):
        kp[tabs[2, j]] = kp[tabs[2, 0], 0]
    out = oracle.paged_attention_decode(q, oracle.F32, kp, vp, oracle.F32, tabs, cl, 0.125)
    mean = vctx[2].astype(np.float64).mean(axis=0).repeat(2, axis=0)
    np.testing.assert_allclose(out[2], mean, atol=1e-13, rtol=0)


def test_decode_scale_enters_linearly(oracle):
    """Doubling the scale equals doubling q (the logits are scale * q.k)."""
    rng = np.random.default_rng(4)
    q, kp, vp, tabs, cl, _, _ = _scatter_case(rng, [40], 4, 2, 64, 16)
    a = oracle.paged_attention_decode(q, oracle.F32, kp, vp, oracle.F32, tabs, cl, 0.25)
    b = oracle.paged_attention_decode((q * 2).astype(np.float32), oracle.F32, kp, vp, oracle.F32,
                                      tabs, cl, 0.125)
    np.testing.assert_allclose(a, b, atol=1e-13, rtol=0)


@pytest.mark.parametrize("partition", [16, 32, 48, 512])
def test_split_merge_identity(oracle, partition):
    rng = np.random.default_rng(partition)
    q, kp, vp, tabs, cl, _, _ = _scatter_case(rng, [1, 16, 17, 500, 1300], 8, 2, 64, 16)
    full = oracle.paged_attention_decode(q, oracle.F32, kp, vp, oracle.F32, tabs, cl, 0.125)
    split = oracle.paged_attention_decode(q, oracle.F32, kp, vp, oracle.F32, tabs, cl, 0.125,
                                          partition=partition)
    np.testing.assert_allclose(split, full, atol=1e-12, rtol=0)


def test_fp8_decode_uses_dequantised_values(oracle):
    rng = np.random.default_rng(8)
    q, kp, vp, tabs, cl, _, _ = _scatter_case(rng, [3, 33], 4, 2, 64, 16)
    kc = rng.integers(0, 256, kp.shape).astype(np.uint8)
    vc = rng.integers(0, 256, vp.shape).astype(np.uint8)
    kc[(kc & 0x7F) == 0x7F] = 0x11                                # no NaN codes
    vc[(vc & 0x7F) == 0x7F] = 0x22
    ks, vs = 0.0123, 0.5
    out = oracle.paged_attention_decode(q, oracle.F32, kc, vc, oracle.E4M3, tabs, cl, 0.125,
                                        k_scale=ks, v_scale=vs)
    kd = (torch.from_numpy(kc).view(torch.float8_e4m3fn).to(torch.float64) * float(np.float32(ks))).numpy()
    vd = (torch.from_numpy(vc).view(torch.float8_e4m3fn).to(torch.float64) * float(np.float32(vs))).numpy()
    for s in range(2):
        nb = -(-int(cl[s]) // 16)
        kk = np.concatenate([kd[b] for b in tabs[s, :nb]])[: cl[s]]
        vv = np.concatenate([vd[b] for b in tabs[s, :nb]])[: cl[s]]
        np.testing.assert_allclose(out[s], _sdpa_reference(q[s], kk, vv, 0.125), atol=1e-12, rtol=0)


# -------------------------------------------------------------------- write

@pytest.mark.parametrize("in_dt,cache_dt", [("f32", "f32"), ("bf16", "bf16"), ("f32", "bf16"),
                                            ("bf16", "f32"), ("f32", "e4m3"), ("bf16", "e4m3")])
def test_write_scatters_to_slots(oracle, in_dt, cache_dt):
    code = {"f32": oracle.F32, "bf16": oracle.BF16, "e4m3": oracle.E4M3}
    npdt = {"f32": np.float32, "bf16": np.uint16, "e4m3": np.uint8}
    rng = np.random.default_rng(21)
    T, Hkv, d, bs, NB = 9, 2, 64, 16, 6
    x32 = (rng.standard_normal((2, T, Hkv, d)) * 3).astype(np.float32)
    x32[0, 0, 0, :4] = [1e4, -1e4, 0.0, -0.0]                    # saturation, signed zero
    x = W.bf16_bits(x32) if in_dt == "bf16" else x32
    xf = W.bf16_bits_to_float32(x) if in_dt == "bf16" else x32  # the values as float32
    slots = np.array([0, 17, -1, 95, 31, 48, -5, 2, 64], np.int64)
    kc = np.full((NB, bs, Hkv, d), 0x3F, npdt[cache_dt]) if cache_dt != "f32" else \
        np.full((NB, bs, Hkv, d), 7.0, np.float32)
    vc = kc.copy()
    before = kc.copy()
    ks, vs = 0.05, 0.02
    assert oracle.paged_kv_write(x[0], x[1], code[in_dt], kc, vc, code[cache_dt], slots, bs, ks, vs) == 0
    touched = np.zeros((NB, bs), bool)
    for i, s in enumerate(slots):
        if s < 0:
            continue
        b, o = divmod(int(s), bs)
        touched[b, o] = True
        for arr, src, sc in ((kc, xf[0, i], ks), (vc, xf[1, i], vs)):
            t = torch.from_numpy(src.copy())
            if cache_dt == "f32":
                ref = src
            elif cache_dt == "bf16":
                ref = t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
            else:
                qv = torch.clamp(t / torch.tensor(sc, dtype=torch.float32), -448.0, 448.0)
                ref = qv.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
            np.testing.assert_array_equal(arr[b, o], ref)
    np.testing.assert_array_equal(kc[~touched], before[~touched])


def test_write_rejects_out_of_range_slot(oracle):
    kc = np.zeros((2, 16, 1, 64), np.float32)
    vc = kc.copy()
    x = np.ones((1, 1, 64), np.float32)
    assert oracle.paged_kv_write(x, x, oracle.F32, kc, vc, oracle.F32, np.array([32]), 16) == -1
    assert (kc == 0).all()


# --------------------------------------------------------------- copy_blocks

def test_copy_blocks_duplicates_bytes(oracle):
    rng = np.random.default_rng(31)
    L, NB = 3, 10
    ks = [rng.integers(0, 255, (NB, 16, 2, 64)).astype(np.uint8) for _ in range(L)]
    vs = [rng.integers(0, 255, (NB, 16, 2, 64)).astype(np.uint8) for _ in range(L)]
    k0 = [a.copy() for a in ks]; v0 = [a.copy() for a in vs]
    pairs = np.array([[1, 7], [4, 8], [4, 9]], np.int64)
    assert oracle.copy_blocks(ks, vs, pairs) == 0
    for l in range(L):
        for s, dd in pairs:
            np.testing.assert_array_equal(ks[l][dd], k0[l][s])
            np.testing.assert_array_equal(vs[l][dd], v0[l][s])
        keep = [b for b in range(NB) if b not in pairs[:, 1]]
        np.testing.assert_array_equal(ks[l][keep], k0[l][keep])
        np.testing.assert_array_equal(vs[l][keep], v0[l][keep])


def test_copy_on_write_then_repoint_keeps_outputs(oracle):
    w = W.make("fp8-bs16", S=4, lengths=np.array([300, 17, 1000, 2]), cow_pairs=8)
    hv = W.host_values(w)
    kc = np.zeros((w.NB, w.bs, w.Hkv, w.d), np.uint8); vc = kc.copy()
    allslots = np.arange(w.NB * w.bs, dtype=np.int64)
    kk = hv.k_pool.reshape(-1, w.Hkv, w.d); vv = hv.v_pool.reshape(-1, w.Hkv, w.d)
    oracle.paged_kv_write(kk, vv, oracle.F32, kc, vc, oracle.E4M3, allslots, w.bs, hv.k_scale, hv.v_scale)
    q = W.bf16_bits(hv.query)
    args = (oracle.E4M3, )
    out = oracle.paged_attention_decode(q, oracle.BF16, kc, vc, oracle.E4M3, w.block_tables,
                                        w.context_lens, w.scale, hv.k_scale, hv.v_scale)
    oracle.copy_blocks([kc], [vc], w.cow_pairs)
    tabs = w.block_tables.copy()
    for src, dst in w.cow_pairs:
        hit = np.argwhere(tabs == src)
        s, j = hit[0]
        tabs[s, j] = dst
    out2 = oracle.paged_attention_decode(q, oracle.BF16, kc, vc, oracle.E4M3, tabs, w.context_lens,
                                         w.scale, hv.k_scale, hv.v_scale)
    np.testing.assert_array_equal(out, out2)
    assert args


# ------------------------------------------------------------------ prefill

def _sdpa_causal_chunk(q, k_ctx, v_ctx, scale):
    """Brute force for a chunk of q_len queries at the end of an n-token
    sequence: torch's fp64 SDPA with an explicit mask (query i sees tokens
    0 .. n - q_len + i).  q [q_len, Hq, d]; k_ctx/v_ctx [n, Hkv, d]."""
    ql, Hq, d = q.shape
    n, Hkv, _ = k_ctx.shape
    g = Hq // Hkv
    qt = torch.from_numpy(q.astype(np.float64)).permute(1, 0, 2)                 # [Hq, ql, d]
    kt = torch.from_numpy(k_ctx.astype(np.float64)).permute(1, 0, 2).repeat_interleave(g, dim=0)
    vt = torch.from_numpy(v_ctx.astype(np.float64)).permute(1, 0, 2).repeat_interleave(g, dim=0)
    pos = torch.arange(n - ql, n)[:, None]
    mask = torch.arange(n)[None, :] <= pos                                          # [ql, n]
    out = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=scale)
    return out.permute(1, 0, 2).numpy()


@pytest.mark.parametrize("Hq,Hkv", [(4, 2), (8, 1), (6, 6)])
def test_prefill_brute_force(oracle, Hq, Hkv):
    rng = np.random.default_rng(200 + Hq + Hkv)
    d, bs = 64, 16
    lens = [1, 16, 17, 40, 70, 33]
    qlens = [1, 3, 17, 40, 5, 0]                    # a whole-sequence chunk, ragged chunks, an empty one
    _, kp, vp, tabs, cl, kctx, vctx = _scatter_case(rng, lens, Hq, Hkv, d, bs)
    qs = np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)
    q = rng.standard_normal((int(qs[-1]), Hq, d)).astype(np.float32)
    out = oracle.paged_attention_prefill(q, oracle.F32, kp, vp, oracle.F32, tabs, cl, qs, 0.125)
    for s in range(len(lens)):
        if qlens[s] == 0:
            continue
        ref = _sdpa_causal_chunk(q[qs[s]:qs[s + 1]], kctx[s], vctx[s], 0.125)
        np.testing.assert_allclose(out[qs[s]:qs[s + 1]], ref, atol=1e-12, rtol=0)


def test_prefill_whole_sequence_is_causal_attention(oracle):
    rng = np.random.default_rng(7)
    _, kp, vp, tabs, cl, kctx, vctx = _scatter_case(rng, [50], 4, 2, 64, 16)
    q = rng.standard_normal((50, 4, 64)).astype(np.float32)
    out = oracle.paged_attention_prefill(q, oracle.F32, kp, vp, oracle.F32, tabs, cl, np.array([0, 50]), 0.125)
    qt = torch.from_numpy(q.astype(np.float64)).permute(1, 0, 2)
    kt = torch.from_numpy(kctx[0].astype(np.float64)).permute(1, 0, 2).repeat_interleave(2, dim=0)
    vt = torch.from_numpy(vctx[0].astype(np.float64)).permute(1, 0, 2).repeat_interleave(2, dim=0)
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=True, scale=0.125)
    np.testing.assert_allclose(out, ref.permute(1, 0, 2).numpy(), atol=1e-12, rtol=0)


def test_prefill_one_query_is_decode(oracle):
    rng = np.random.default_rng(8)
    q, kp, vp, tabs, cl, _, _ = _scatter_case(rng, [1, 30, 99], 8, 2, 64, 16)
    dec = oracle.paged_attention_decode(q, oracle.F32, kp, vp, oracle.F32, tabs, cl, 0.125)
    pre = oracle.paged_attention_prefill(q, oracle.F32, kp, vp, oracle.F32, tabs, cl, np.arange(4), 0.125)
    np.testing.assert_array_equal(dec, pre)


# ------------------------------------------------------------ token table

def _token_case(rng, lens, keep_frac, Hq, Hkv, d, bs):
    """A block-table case whose tokens a deletion policy then thins out at
    random: the token table lists the survivors' slots in logical order."""
    q, kp, vp, tabs, cl, kctx, vctx = _scatter_case(rng, lens, Hq, Hkv, d, bs)
    MT = max(max(lens), 1)
    slots = np.zeros((len(lens), MT), np.int32)
    nt = np.zeros(len(lens), np.int32)
    lk, lv = [], []
    for s, n in enumerate(lens):
        keep = rng.random(n) < keep_frac
        if n and not keep.any():
            keep[rng.integers(0, n)] = True
        idx = np.nonzero(keep)[0]
        slots[s, : idx.size] = [tabs[s, t // bs] * bs + t % bs for t in idx]
        nt[s] = idx.size
        lk.append(kctx[s][idx])
        lv.append(vctx[s][idx])
    return q, kp, vp, tabs, cl, slots, nt, lk, lv


@pytest.mark.parametrize("cache", ["f32", "bf16", "e4m3"])
def test_token_table_of_all_tokens_is_the_block_table(oracle, cache):
    """A token table that lists every token's slot in order gathers exactly
    what the block table gathers: identical outputs."""
    rng = np.random.default_rng(301)
    bs = 16
    q, kp, vp, tabs, cl, _, _ = _scatter_case(rng, [1, 16, 17, 45, 64], 8, 2, 64, bs)
    MT = int(cl.max())
    slots = np.zeros((len(cl), MT), np.int32)
    for s, n in enumerate(cl):
        slots[s, :n] = [tabs[s, t // bs] * bs + t % bs for t in range(n)]
    if cache == "f32":
        kc, vc, dt, ks = kp, vp, oracle.F32, 1.0
    elif cache == "bf16":
        kc, vc, dt, ks = W.bf16_bits(kp), W.bf16_bits(vp), oracle.BF16, 1.0
    else:
        ks = W.e4m3_scale(kp)
        kc, vc, dt = oracle.e4m3_from_float32(kp / np.float32(ks)), oracle.e4m3_from_float32(vp / np.float32(ks)), oracle.E4M3
    a = oracle.paged_attention_decode(q, oracle.F32, kc, vc, dt, tabs, cl, 0.125, ks, ks)
    b = oracle.token_attention_decode(q, oracle.F32, kc, vc, dt, slots, cl, 0.125, ks, ks)
    np.testing.assert_array_equal(a, b)


@pytest.mark.parametrize("Hq,Hkv", [(4, 2), (8, 1), (6, 6)])
def test_token_decode_after_deletion_brute_force(oracle, Hq, Hkv):
    """Deleted tokens are absent from the table: the result is attention over
    the survivors (torch fp64 SDPA on their gathered K/V)."""
    rng = np.random.default_rng(302 + Hq)
    d, bs = 64, 16
    q, kp, vp, _, _, slots, nt, lk, lv = _token_case(rng, [1, 16, 40, 70, 33], 0.4, Hq, Hkv, d, bs)
    out = oracle.token_attention_decode(q, oracle.F32, kp, vp, oracle.F32, slots, nt, 0.125)
    g = Hq // Hkv
    for s in range(len(nt)):
        qt = torch.from_numpy(q[s].astype(np.float64))[:, None, :]                 # [Hq, 1, d]
        kt = torch.from_numpy(lk[s].astype(np.float64)).permute(1, 0, 2).repeat_interleave(g, dim=0)
        vt = torch.from_numpy(lv[s].astype(np.float64)).permute(1, 0, 2).repeat_interleave(g, dim=0)
        ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=0.125)[:, 0].numpy()
        np.testing.assert_allclose(out[s], ref, atol=1e-12, rtol=0)


def test_token_decode_logical_order_does_not_change_attention(oracle):
    rng = np.random.default_rng(303)
    q, kp, vp, _, _, slots, nt, _, _ = _token_case(rng, [50, 90], 0.7, 8, 2, 64, 16)
    out = oracle.token_attention_decode(q, oracle.F32, kp, vp, oracle.F32, slots, nt, 0.125)
    sh = slots.copy()
    for s in range(len(nt)):
        sh[s, : nt[s]] = rng.permutation(slots[s, : nt[s]])
    out2 = oracle.token_attention_decode(q, oracle.F32, kp, vp, oracle.F32, sh, nt, 0.125)
    np.testing.assert_allclose(out, out2, atol=1e-12, rtol=0)


def _scrub_blocks(pools, blocks, bs):
    """A released block's slots are reused: overwrite them."""
    for a in pools:
        for b in blocks:
            a[b] = np.float32(1e30)


def test_repack_keeps_attention_and_releases_blocks(oracle):
    """Plan (oracle/vtoken_plan.py), move the rows, rewrite the table, then
    overwrite every released block: attention is bit-identical to before, each
    sequence's live tokens fill ceil(n / bs) blocks, and no live token is in a
    released block."""
    from oracle.vtoken_plan import plan, apply
    rng = np.random.default_rng(304)
    bs = 16
    q, kp, vp, _, _, slots, nt, _, _ = _token_case(rng, [100, 40, 260, 16, 77], 0.3, 8, 2, 64, bs)
    NB = kp.shape[0]
    before = oracle.token_attention_decode(q, oracle.F32, kp, vp, oracle.F32, slots, nt, 0.125)
    moves, freed = plan(slots, nt, bs, NB)
    assert moves and freed
    kc2, vc2, sl2 = kp.copy(), vp.copy(), slots.copy()
    assert oracle.repack_tokens([kc2], [vc2], sl2, np.array(moves)) == 0
    np.testing.assert_array_equal(sl2, apply(slots, moves))
    for s, t, src, dst in moves:
        np.testing.assert_array_equal(kc2[dst // bs, dst % bs], kp[src // bs, src % bs])
        np.testing.assert_array_equal(vc2[dst // bs, dst % bs], vp[src // bs, src % bs])
    _scrub_blocks([kc2, vc2], freed, bs)
    after = oracle.token_attention_decode(q, oracle.F32, kc2, vc2, oracle.F32, sl2, nt, 0.125)
    np.testing.assert_array_equal(before, after)
    for s in range(len(nt)):
        blocks = {int(x) // bs for x in sl2[s, : nt[s]]}
        assert len(blocks) == -(-int(nt[s]) // bs)
        assert not blocks & set(freed)
    live = [int(x) for s in range(len(nt)) for x in sl2[s, : nt[s]]]
    assert len(live) == len(set(live))


def test_repack_pages_example(oracle):
    from oracle.vtoken_plan import plan
    rows = [ln.split() for ln in open(os.path.join(GOLDEN, "vtoken_repack_example.txt"), encoding="utf-8")
            if ln.strip() and not ln.startswith("#")]
    kv = {r[0]: r[1:] for r in rows if r[0] in ("bs", "NB", "slots", "freed")}
    bs, NB = int(kv["bs"][0]), int(kv["NB"][0])
    slots = np.array([[int(x) for x in kv["slots"]]], np.int32)
    want_moves = [tuple(int(x) for x in r[1:]) for r in rows if r[0] == "move"]
    moves, freed = plan(slots, np.array([slots.shape[1]]), bs, NB)
    assert moves == want_moves and freed == [int(x) for x in kv["freed"]]
    # the oracle's repack applies them
    kp = np.random.default_rng(5).standard_normal((NB, bs, 1, 8)).astype(np.float32)
    vp = kp + 1
    k2, v2, s2 = kp.copy(), vp.copy(), slots.copy()
    assert oracle.repack_tokens([k2], [v2], s2, np.array(moves)) == 0
    assert list(s2[0, 12:]) == [28, 29, 30, 31]
    np.testing.assert_array_equal(k2[1, 12:], kp[2, [0, 5, 10, 15]])
    np.testing.assert_array_equal(v2[1, 12:], vp[2, [0, 5, 10, 15]])


def test_repack_rejects_a_stale_move(oracle):
    """A move whose source is no longer in the table is skipped and reported."""
    rng = np.random.default_rng(305)
    kp = rng.standard_normal((4, 16, 1, 8)).astype(np.float32)
    vp = kp.copy()
    slots = np.array([[0, 1, 2]], np.int32)
    k2 = kp.copy()
    assert oracle.repack_tokens([k2], [vp.copy()], slots, np.array([[0, 1, 5, 40]])) == -1
    assert list(slots[0]) == [0, 1, 2]
    np.testing.assert_array_equal(k2, kp)
