"""Builds matching GPU and oracle inputs for the parity tests.

Both sides get the same host-drawn values (workloads.host_values).  fp8
pools are produced by each side's own write call from the same float32
draws, so the two fp8 pools agree only if the writes agree bit for bit
(which the tests also check).

Full-size workloads are too large to draw on the host in seconds; for them
the device pool is first filled from torch's seeded device generator, then
the blocks of a few sampled sequences are overwritten with host draws, and
the oracle recomputes exactly those sequences from the host draws.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np
import torch

import oracle as O
import paged_kv_cache_44_gb300 as pkv
import workloads as W

ODT = {W.DT_F32: O.F32, W.DT_BF16: O.BF16, W.DT_E4M3: O.E4M3}
TDT = {W.DT_F32: torch.float32, W.DT_BF16: torch.bfloat16, W.DT_E4M3: torch.uint8}


def host_raw(x: np.ndarray, dt: str) -> np.ndarray:
    """float32 draws in the form the oracle takes for dtype dt (not e4m3)."""
    return W.bf16_bits(x) if dt == W.DT_BF16 else np.ascontiguousarray(x, np.float32)


def to_device(x: np.ndarray, dt: str, dev="cuda") -> torch.Tensor:
    if dt == W.DT_BF16:
        return torch.from_numpy(W.bf16_bits(x).view(np.int16)).to(dev).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(dev)


device_normal = W.device_normal


@dataclasses.dataclass
class Case:
    w: W.Workload
    hv: W.HostValues
    in_dt: str                    # dtype of query and new tokens
    # device
    q: torch.Tensor
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    block_tables: torch.Tensor
    context_lens: torch.Tensor
    slot_mapping: torch.Tensor
    new_k: torch.Tensor
    new_v: torch.Tensor
    cow: torch.Tensor
    # oracle (host raw), for the sequences `seqs` of sub-workload `ow`
    seqs: np.ndarray
    ow: W.Workload
    o_q: np.ndarray
    o_k: np.ndarray
    o_v: np.ndarray
    o_new_k: np.ndarray
    o_new_v: np.ndarray

    @property
    def k_scale(self) -> float:
        return self.hv.k_scale

    @property
    def v_scale(self) -> float:
        return self.hv.v_scale


def _write_pool_fp8(cache: torch.Tensor, values: torch.Tensor, blocks: torch.Tensor, bs: int, scale: float):
    """GPU write of float32 `values` [len(blocks), bs, Hkv, d] into `blocks`."""
    n, _, Hkv, d = values.shape
    slots = (blocks.to(torch.int64)[:, None] * bs + torch.arange(bs, device=cache.device)[None, :]).reshape(-1)
    vals = values.reshape(n * bs, Hkv, d).contiguous()
    pkv.paged_kv_write(vals, vals, cache, cache, slots, scale, scale)


def build_case(w: W.Workload, sample: Optional[int] = None, dev="cuda") -> Case:
    """sample=None: every value from the host and every sequence checked.
    sample=k: bulk device fill, host values for k sampled sequences only."""
    in_dt = w.q_dtype
    cdt = w.cache_dtype
    if sample is None:
        seqs = np.arange(w.S)
        ow = w
        hv = W.host_values(w)
    else:
        seqs = W.sample_sequences(w, sample)
        ow = W.sub_workload(w, seqs)
        hv = W.host_values(ow)             # draws for the sampled sequences' blocks (new numbering)
    q_full = W.host_normal(w.seed, "query", (w.S, w.Hq, w.d))
    nk_full = W.host_normal(w.seed, "new-k", (w.S, w.Hkv, w.d))
    nv_full = W.host_normal(w.seed, "new-v", (w.S, w.Hkv, w.d))
    hv.query, hv.new_k, hv.new_v = q_full[seqs], nk_full[seqs], nv_full[seqs]

    shape = (w.NB, w.bs, w.Hkv, w.d)
    numel = int(np.prod(shape))
    if sample is None:
        if cdt == W.DT_E4M3:
            kc = torch.zeros(shape, dtype=torch.uint8, device=dev)
            vc = torch.zeros_like(kc)
            blocks = torch.arange(w.NB, device=dev)
            _write_pool_fp8(kc, torch.from_numpy(hv.k_pool).to(dev), blocks, w.bs, hv.k_scale)
            _write_pool_fp8(vc, torch.from_numpy(hv.v_pool).to(dev), blocks, w.bs, hv.v_scale)
        else:
            kc = to_device(hv.k_pool, cdt, dev)
            vc = to_device(hv.v_pool, cdt, dev)
    else:
        old_ids = torch.from_numpy(ow.renumber.astype(np.int64)).to(dev)   # type: ignore[attr-defined]
        if cdt == W.DT_E4M3:
            kc = torch.zeros(shape, dtype=torch.uint8, device=dev)
            vc = torch.zeros_like(kc)
            all_blocks = torch.arange(w.NB, device=dev)
            chunk = max(1, (1 << 26) // (w.bs * w.Hkv * w.d))
            for which, cache, sc in ((1, kc, hv.k_scale), (2, vc, hv.v_scale)):
                for b0 in range(0, w.NB, chunk):
                    nb = min(chunk, w.NB - b0)
                    vals = device_normal(w.seed, which * 100000 + b0, nb * w.bs * w.Hkv * w.d, dev)
                    _write_pool_fp8(cache, vals.view(nb, w.bs, w.Hkv, w.d), all_blocks[b0:b0 + nb], w.bs, sc)
            _write_pool_fp8(kc, torch.from_numpy(hv.k_pool).to(dev), old_ids, w.bs, hv.k_scale)
            _write_pool_fp8(vc, torch.from_numpy(hv.v_pool).to(dev), old_ids, w.bs, hv.v_scale)
        else:
            caches = []
            for which in (1, 2):
                flat = torch.empty(numel, dtype=TDT[cdt], device=dev)
                for c0, x in W.device_pool_chunks(w.seed, which, numel, dev):
                    flat[c0:c0 + x.numel()] = W.device_bf16_from_draws(x) if cdt == W.DT_BF16 else x
                caches.append(flat.view(shape))
            kc, vc = caches
            kc[old_ids] = to_device(hv.k_pool, cdt, dev)
            vc[old_ids] = to_device(hv.v_pool, cdt, dev)

    q = to_device(q_full, in_dt, dev)
    new_k = to_device(nk_full, in_dt, dev)
    new_v = to_device(nv_full, in_dt, dev)
    bt = torch.from_numpy(w.block_tables).to(dev)
    cl = torch.from_numpy(w.context_lens).to(dev)
    sm = torch.from_numpy(w.slot_mapping).to(dev)
    cow = torch.from_numpy(w.cow_pairs.astype(np.int64)).to(dev)

    # oracle-side pools (host raw) for the checked sequences
    if cdt == W.DT_E4M3:
        o_k = np.zeros((ow.NB, w.bs, w.Hkv, w.d), np.uint8)
        o_v = np.zeros_like(o_k)
        slots = np.arange(ow.NB * w.bs, dtype=np.int64)
        O.paged_kv_write(hv.k_pool.reshape(-1, w.Hkv, w.d), hv.k_pool.reshape(-1, w.Hkv, w.d), O.F32,
                         o_k, np.zeros_like(o_k), O.E4M3, slots, w.bs, hv.k_scale, hv.k_scale)
        O.paged_kv_write(hv.v_pool.reshape(-1, w.Hkv, w.d), hv.v_pool.reshape(-1, w.Hkv, w.d), O.F32,
                         np.zeros_like(o_v), o_v, O.E4M3, slots, w.bs, hv.v_scale, hv.v_scale)
    else:
        o_k = host_raw(hv.k_pool, cdt)
        o_v = host_raw(hv.v_pool, cdt)
    return Case(w=w, hv=hv, in_dt=in_dt, q=q, k_cache=kc, v_cache=vc, block_tables=bt, context_lens=cl,
                slot_mapping=sm, new_k=new_k, new_v=new_v, cow=cow, seqs=seqs, ow=ow,
                o_q=host_raw(hv.query, in_dt), o_k=o_k, o_v=o_v,
                o_new_k=host_raw(hv.new_k, in_dt), o_new_v=host_raw(hv.new_v, in_dt))


def oracle_write(c: Case) -> None:
    """The step's write on the oracle side (sub-workload slots)."""
    O.paged_kv_write(c.o_new_k, c.o_new_v, ODT[c.in_dt], c.o_k, c.o_v, ODT[c.w.cache_dtype],
                     c.ow.slot_mapping, c.w.bs, c.k_scale, c.v_scale)


def oracle_decode(c: Case, context_lens: Optional[np.ndarray] = None, threads=None) -> np.ndarray:
    cl = c.ow.context_lens if context_lens is None else context_lens
    return O.paged_attention_decode(c.o_q, ODT[c.in_dt], c.o_k, c.o_v, ODT[c.w.cache_dtype], c.ow.block_tables,
                                    cl, c.w.scale, c.k_scale, c.v_scale, threads=threads)


def gpu_decode(c: Case, partition_size: Optional[int] = None, kernel="auto", context_lens=None,
               max_context_len=None, block_tables=None, err_word=None) -> torch.Tensor:
    w = c.w
    P = w.partition_size if partition_size is None else partition_size
    cl = c.context_lens if context_lens is None else context_lens
    mc = w.max_context_len if max_context_len is None else max_context_len
    bt = c.block_tables if block_tables is None else block_tables
    out = torch.empty_like(c.q)
    ws = pkv.make_workspace(w.S, w.Hq, w.Hkv, w.d, w.bs, mc, P)
    pkv.paged_attention_decode(out, c.q, c.k_cache, c.v_cache, bt, cl, mc, scale=w.scale, k_scale=c.k_scale,
                               v_scale=c.v_scale, partition_size=P, workspace=ws, kernel=kernel,
                               err_word=err_word)
    return out


def gpu_write(c: Case) -> None:
    pkv.paged_kv_write(c.new_k, c.new_v, c.k_cache, c.v_cache, c.slot_mapping, c.k_scale, c.v_scale)


TOL = {W.DT_F32: (1e-5, 0.0), W.DT_BF16: (2e-2, 1e-2), W.DT_E4M3: (5e-2, 0.0)}


def tolerance(cache_dt: str, out_dtype: torch.dtype):
    """(atol, rtol) for a decode output: the cache dtype's tolerance, 1e-5
    (fp32), 2e-2 + 1e-2 rel (bf16), 5e-2 absolute (E4M3, against the oracle
    fed the same dequantised values).  A bf16 output (bf16 query) of an fp32
    cache is rounded to 8 significant bits, which 1e-5 cannot absorb, so it
    is held to the bf16 tolerance instead.  E4M3 keeps 5e-2 absolute with
    no relative term whatever the output dtype: its outputs are bounded by
    448 * v_scale, where half a bf16 unit in the last place is below 2e-2."""
    atol, rtol = TOL[cache_dt]
    if out_dtype == torch.bfloat16 and cache_dt == W.DT_F32:
        atol, rtol = TOL[W.DT_BF16]
    return atol, rtol


def assert_close(gpu: torch.Tensor, ref: np.ndarray, cache_dt: str, what: str = "") -> float:
    """Elementwise |gpu - ref| <= atol + rtol * |ref| with the tolerance of
    `tolerance(cache_dt, gpu.dtype)`.  Returns the largest |gpu - ref|."""
    atol, rtol = tolerance(cache_dt, gpu.dtype)
    g = gpu.float().cpu().numpy().astype(np.float64)
    err = np.abs(g - ref)
    bad = err > atol + rtol * np.abs(ref)
    if bad.any() or not np.isfinite(g).all():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outside tolerance; max err "
                             f"{float(err.max()):.3e}; first at {idx.tolist()}")
    return float(err.max())
