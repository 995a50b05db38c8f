"""The host block manager driving the device calls, end to end.

Prompts with shared prefixes are admitted through the manager (cached
prefix blocks are shared, not rewritten), their K/V written to the slots
the manager names, a sequence is forked and both copies keep decoding (the
first write into the shared last block triggers copy-on-write), and every
sequence is decoded through the manager's block tables.  The oracle runs the
same steps on the host with the tables of the independent Python model of
the manager (which must equal the library's)."""
import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import oracle as O
    import paged_kv_cache_44_gb300 as pkv
    from oracle.block_pool import BlockPoolModel
    from tests.gpu_cases import assert_close


def _kv_of(tokens, pos, Hkv, d, which):
    """K or V of the token at `pos`: a function of the tokens up to it (as a
    model's would be), so equal prefixes give equal K/V."""
    seed = [which, pos] + [int(t) for t in tokens[max(0, pos - 3): pos + 1]]
    return np.random.default_rng(seed).standard_normal((Hkv, d), dtype=np.float32)


@pytest.mark.parametrize("cache", ["bf16", "e4m3"])
def test_manager_drives_write_copy_decode(cache):
    rng = np.random.default_rng(21)
    NB, bs, Hq, Hkv, d = 96, 16, 8, 2, 128
    pool = pkv.BlockPool(NB, bs)
    model = BlockPoolModel(NB, bs)
    dev = "cuda"
    cdt = torch.uint8 if cache == "e4m3" else torch.bfloat16
    odt = O.E4M3 if cache == "e4m3" else O.BF16
    kc = torch.zeros((NB, bs, Hkv, d), dtype=cdt, device=dev)
    vc = torch.zeros_like(kc)
    ok_ = np.zeros((NB, bs, Hkv, d), np.uint8 if cache == "e4m3" else np.uint16)
    ov_ = ok_.copy()
    ks = vs = 4.5 / 448.0

    def write(slots, keys, vals):
        """the same K/V into the same slots on both sides (fp32 input)"""
        kk = np.stack(keys).astype(np.float32)
        vv = np.stack(vals).astype(np.float32)
        sl = np.array(slots, np.int64)
        pkv.paged_kv_write(torch.from_numpy(kk).to(dev), torch.from_numpy(vv).to(dev), kc, vc,
                           torch.from_numpy(sl).to(dev), ks, vs)
        O.paged_kv_write(kk, vv, O.F32, ok_, ov_, odt, sl, bs, ks, vs)

    system = list(rng.integers(1, 1000, 40))                  # a shared 40-token system prompt
    prompts = {0: system + list(rng.integers(1, 1000, 30)), 1: system + list(rng.integers(1, 1000, 5)),
               2: list(rng.integers(1, 1000, 17)), 3: system + list(rng.integers(1, 1000, 60))}
    tokens = {}
    for sid, toks in prompts.items():
        cached = pool.add_sequence(sid, np.array(toks, np.int32))
        assert cached == model.add_sequence(sid, toks)
        if sid in (1, 3):
            assert cached == 32                                # two full blocks of the system prompt
        table = model.block_table(sid)
        assert list(pool.block_table(sid)[0]) == table
        slots = [table[t // bs] * bs + t % bs for t in range(cached, len(toks))]
        write(slots, [_kv_of(toks, t, Hkv, d, 0) for t in range(cached, len(toks))],
              [_kv_of(toks, t, Hkv, d, 1) for t in range(cached, len(toks))])
        tokens[sid] = list(toks)
    pool.fork(0, 4)
    model.fork(0, 4)
    tokens[4] = list(tokens[0])
    copies = 0
    for step in range(20):
        for sid in (0, 4, 1, 2, 3):
            tok = int(rng.integers(1, 1000))
            got = pool.append_token(sid, tok)
            assert got == model.append_token(sid, tok)
            slot, src, dst = got
            tokens[sid].append(tok)
            if src >= 0:
                copies += 1
                pair = np.array([[src, dst]], np.int64)
                pkv.copy_blocks([kc], [vc], torch.from_numpy(pair).to(dev))
                O.copy_blocks([ok_], [ov_], pair)
            t = len(tokens[sid]) - 1
            write([slot], [_kv_of(tokens[sid], t, Hkv, d, 0)], [_kv_of(tokens[sid], t, Hkv, d, 1)])
    assert copies == 1                                         # the fork's shared last block, once
    torch.cuda.synchronize()
    for dev_cache, host_cache in ((kc, ok_), (vc, ov_)):
        got = dev_cache.cpu().view(torch.int16).numpy().view(np.uint16) if cache == "bf16" else dev_cache.cpu().numpy()
        np.testing.assert_array_equal(got, host_cache)
    # decode every sequence through the manager's tables
    sids = sorted(tokens)
    MB = max(len(model.block_table(s)) for s in sids)
    tab = np.zeros((len(sids), MB), np.int32)
    for i, s in enumerate(sids):
        t = model.block_table(s)
        tab[i, : len(t)] = t
    cl = np.array([len(tokens[s]) for s in sids], np.int32)
    q32 = rng.standard_normal((len(sids), Hq, d), dtype=np.float32)
    q = W.bf16_bits(q32)
    out = torch.empty((len(sids), Hq, d), dtype=torch.bfloat16, device=dev)
    ws = pkv.make_workspace(len(sids), Hq, Hkv, d, bs, int(cl.max()), 32)
    scale = float(np.float32(1) / np.sqrt(np.float32(d)))
    pkv.paged_attention_decode(out, torch.from_numpy(q.view(np.int16)).to(dev).view(torch.bfloat16), kc, vc,
                               torch.from_numpy(tab).to(dev), torch.from_numpy(cl).to(dev), int(cl.max()),
                               scale=scale, k_scale=ks, v_scale=vs, partition_size=32, workspace=ws)
    ref = O.paged_attention_decode(q, O.BF16, ok_, ov_, odt, tab, cl, scale, ks, vs)
    assert_close(out, ref, "e4m3" if cache == "e4m3" else "bf16", "manager-driven decode")
