"""Benchmark of one paged-decode step on GB300.

A step is one pass of the whole hot path over one batch: paged_kv_write of
one new token per sequence, paged_attention_decode of every sequence, and
copy_blocks of the copy-on-write pairs.  The default workload is the
Qwen2.5-72B-shaped long-context decode (32 sequences x 32,768 tokens,
64 query / 8 K/V heads, d = 128, bf16 KV, 512-token partitions): 4 GiB of K/V,
far larger than L2, so every step streams it from HBM.

Prints one JSON line (rank 0).  `value` is algorithmic bytes per step
(query + K/V of the unique blocks read + output + block tables, plus the
write and copy bytes) over the device-timed step, in GB/s, summed over ranks.
A default run (no --workload, --S, --partition or --no-workloads) also
times the same step on the other decode configurations -- the
Qwen2.5-1.5B-shaped, the 7B-shaped shared-prefix and the two fp8 ones --
each with at least 200 steps, its own roofline, clocks and a short oracle
baseline, under the line's `workloads` key; the headline numbers stay
those of the 72B-shaped workload.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--kernel auto|cuda_cores|tensor_cores] [--impl ours|reference]

Under torchrun each rank runs its own replica of the workload (decode
shards by sequence with no exchange, so N GPUs are N independent units).
`--impl reference` times the CPU oracle instead, on a bounded sample of the
same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "paged decode attention KV GB/s and % of HBM peak; seq-steps/s"
NOMINAL_HBM_GBS = 8000.0
L2_BYTES = 129 * 10**6          # GB300; replaced by the device's own figure when torch reports it


def l2_note(pool_bytes: int, n_pools: int) -> str:
    """How a timed step is kept from reading its K/V out of L2."""
    if n_pools == 1:
        return "inputs larger than L2 (pool %.0f MB)" % (pool_bytes / 1e6)
    if (n_pools - 1) * pool_bytes >= 2 * L2_BYTES:
        return "rotating %d copies of the %.0f MB pool: two L2s of other copies read between two uses of one" % (
            n_pools, pool_bytes / 1e6)
    return "not flushed: %d copies of a %.0f MB pool" % (n_pools, pool_bytes / 1e6)
FALLBACK_HBM_GBS = 6800.0
ELEM = {W.DT_F32: 4, W.DT_BF16: 2, W.DT_E4M3: 1}
TORCH_DT = {W.DT_F32: "float32", W.DT_BF16: "bfloat16", W.DT_E4M3: "float8_e4m3fn"}   # torch dtype names


# ------------------------------------------------------------- byte counts

def decode_bytes(w: W.Workload, unique: bool = True) -> int:
    """Algorithmic bytes of one decode: query read + output write + K/V of
    every block read (shared blocks once when unique) + table entries read
    + context lengths."""
    bq = ELEM[w.q_dtype]
    bkv = ELEM[w.cache_dtype]
    qo = 2 * w.S * w.Hq * w.d * bq
    nblk = -(-w.context_lens.astype(np.int64) // w.bs)
    if unique and w.shared_seqs:
        # K/V bytes of distinct physical blocks, counting only the tokens read
        seen = {}
        for s in range(w.S):
            n = int(w.context_lens[s])
            for j in range(int(nblk[s])):
                b = int(w.block_tables[s, j])
                seen[b] = max(seen.get(b, 0), min(w.bs, n - j * w.bs))
        kv_tokens = sum(seen.values())
    else:
        kv_tokens = int(w.context_lens.astype(np.int64).sum())
    kv = kv_tokens * w.Hkv * w.d * 2 * bkv
    return qo + kv + int(nblk.sum()) * 4 + w.S * 4


def write_bytes(w: W.Workload) -> int:
    return w.S * w.Hkv * w.d * 2 * (ELEM[w.q_dtype] + ELEM[w.cache_dtype]) + w.S * 8


def copy_bytes(w: W.Workload) -> int:
    blk = w.bs * w.Hkv * w.d * ELEM[w.cache_dtype]
    return len(w.cow_pairs) * (2 * 2 * blk + 16)


def prefill_flops(w: W.Workload, qlens: np.ndarray) -> int:
    """Algorithmic FLOPs of paged attention over query chunks: every (query,
    head) with the keys its causal range allows (the chunk's query i of a
    sequence of n tokens sees n - q_len + i + 1 keys), 2 d for the logit and
    2 d for the weighted sum per key."""
    n = w.context_lens.astype(np.int64)
    ql = qlens.astype(np.int64)
    keys = ql * (n - ql) + ql * (ql + 1) // 2          # sum over the chunk of (pos + 1)
    return int(keys.sum()) * w.Hq * 4 * w.d


def prefill_bytes(w: W.Workload, qlens: np.ndarray) -> int:
    """Algorithmic bytes: every query read and output written once, the K/V
    of each sequence's tokens once, table entries and lengths."""
    T = int(qlens.sum())
    bq = ELEM[w.q_dtype]
    kv = int(w.context_lens.astype(np.int64).sum()) * w.Hkv * w.d * 2 * ELEM[w.cache_dtype]
    nblk = -(-w.context_lens.astype(np.int64) // w.bs)
    return 2 * T * w.Hq * w.d * bq + kv + int(nblk.sum()) * 4 + w.S * 8


# ------------------------------------------------------------------ clocks

# A clock sampler through NVML, the library nvidia-smi reads from (read-only calls:
# the SM clock, its maximum, the clock-event reasons), polling every PERIOD seconds
# and printing nvidia-smi's CSV fields; it runs as a process of its own so that it
# takes no time from the thread that queues the timed work.
NVML_SAMPLER = r"""
import ctypes, sys, time
uuid, period = sys.argv[1], float(sys.argv[2])
lib = ctypes.CDLL("libnvidia-ml.so.1")
if lib.nvmlInit_v2() != 0:
    sys.exit(3)
h = ctypes.c_void_p()
if lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(h)) != 0:
    sys.exit(4)
get_reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or lib.nvmlDeviceGetCurrentClocksThrottleReasons
sm, mx, r = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
flag = lambda v, b: "Active" if v & b else "Not Active"
while True:
    if (lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(sm)) == 0 and
            lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0 and get_reasons(h, ctypes.byref(r)) == 0):
        v = r.value
        # hw slowdown (with the hardware power brake), hw thermal, sw thermal, sw power cap
        print(sm.value, mx.value, "-", hex(v), flag(v, 0x88), flag(v, 0x40), flag(v, 0x20), flag(v, 0x4), sep=", ", flush=True)
    time.sleep(period)
"""
NVML_PERIOD_S = 0.002


class ClockSampler:
    """Samples the SM clock and the clock-event (throttle) reasons while the
    timed region runs: through NVML every 2 ms where the driver's library
    loads, else with nvidia-smi every 20 ms."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, dev_uuid: str):
        self.uuid = dev_uuid
        self.proc = None
        self.lines = []
        self._t = None
        self.source = None

    def _start(self, cmd) -> bool:
        """Starts a sampler process; true once it has printed its first reading."""
        self.lines = []
        self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        self._t = threading.Thread(target=self._read, daemon=True)
        self._t.start()
        t0 = time.perf_counter()
        while not self.lines and time.perf_counter() - t0 < 5.0 and self.proc.poll() is None:
            time.sleep(0.005)
        if self.lines:
            return True
        self._stop()
        return False

    def __enter__(self):
        # the sampler is live before the timed region starts: its first reading is in
        try:
            if self._start([sys.executable, "-c", NVML_SAMPLER, self.uuid, str(NVML_PERIOD_S)]):
                self.source = "nvml, %g ms" % (NVML_PERIOD_S * 1e3)
            elif self._start(["nvidia-smi", "-i", self.uuid, "--query-gpu=" + self.FIELDS,
                              "--format=csv,noheader,nounits", "-lms", "20"]):
                self.source = "nvidia-smi, 20 ms"
        except (OSError, ValueError):
            self.proc = None
        self._skip = len(self.lines)
        return self

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append(ln.strip())

    def _stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            if self._t is not None:
                self._t.join(timeout=2)
        self.proc = None

    def __exit__(self, *a):
        self._stop()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        # readings taken during the timed region; a region shorter than the sampling
        # interval may have none, and then the reading taken just before it stands in
        lines = self.lines[getattr(self, "_skip", 0):]
        before = not lines
        if before:
            lines = self.lines[-1:]
        for ln in lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        out = {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm),
               "sampler": self.source}
        if before:
            out["sampled_before_region"] = True
        return out


# ----------------------------------------------------------- CPU baseline

class OracleSampler:
    """The CPU oracle on a bounded sample of the workload.

    A sample item is one (sequence, K/V head) slice of at most MAX_TOKENS
    tokens -- the size of one of the GPU's larger work units -- with the
    workload's shapes: one K/V head and its query heads, drawn once on the
    host (drawing is not timed) and then decoded by the oracle as often as
    the time budget allows.  The items follow the lengths of sampled
    sequences of the workload, and are cycled."""

    MAX_TOKENS = 2048

    def __init__(self, w: W.Workload, threads: int, max_items: int = 2):
        import dataclasses
        import oracle as O
        O.build()
        self.O, self.w, self.threads = O, w, threads
        self.odt = {W.DT_F32: O.F32, W.DT_BF16: O.BF16, W.DT_E4M3: O.E4M3}
        self.items = []
        # an item is a batch of one slice per thread (the oracle runs one
        # thread per sequence), following the lengths of sampled sequences
        order = W.sample_sequences(w, w.S, seed_tag="cpu-sample")
        for it in range(max_items):
            pick = [order[(it * threads + k) % len(order)] for k in range(threads)]
            lens = np.array([max(1, min(int(w.context_lens[s]), self.MAX_TOKENS)) for s in pick])
            sw = W.make(w.name, S=threads, lengths=lens, cow_pairs=0, shared_seqs=0, seed=w.seed + 17 * it)
            sw = dataclasses.replace(sw, Hq=w.g, Hkv=1)
            hv = W.host_values(sw)
            q = W.bf16_bits(hv.query) if w.q_dtype == W.DT_BF16 else hv.query
            if w.cache_dtype == W.DT_E4M3:
                kc = np.zeros(hv.k_pool.shape, np.uint8)
                vc = np.zeros_like(kc)
                sl = np.arange(kc.shape[0] * w.bs, dtype=np.int64)
                flat = lambda a: a.reshape(-1, 1, w.d)  # noqa: E731
                O.paged_kv_write(flat(hv.k_pool), flat(hv.v_pool), O.F32, kc, vc, O.E4M3, sl, w.bs,
                                 hv.k_scale, hv.v_scale)
            elif w.cache_dtype == W.DT_BF16:
                kc, vc = W.bf16_bits(hv.k_pool), W.bf16_bits(hv.v_pool)
            else:
                kc, vc = hv.k_pool, hv.v_pool
            self.items.append((sw, hv, q, kc, vc, decode_bytes(sw, unique=False)))
        self.next = 0

    def run(self, budget_s: float):
        """Decode items until `budget_s` of oracle time is spent (at least one).
        Returns (bytes, seconds, items)."""
        done_bytes, spent, n = 0, 0.0, 0
        while n == 0 or spent < budget_s:
            sw, hv, q, kc, vc, nbytes = self.items[self.next % len(self.items)]
            self.next += 1
            t0 = time.perf_counter()
            self.O.paged_attention_decode(q, self.odt[self.w.q_dtype], kc, vc, self.odt[self.w.cache_dtype],
                                          sw.block_tables, sw.context_lens, self.w.scale, hv.k_scale,
                                          hv.v_scale, threads=self.threads)
            spent += time.perf_counter() - t0
            done_bytes += nbytes
            n += 1
        return done_bytes, spent, n

    def describe(self, n: int, spent: float) -> str:
        return (f"{n} batches of {self.threads} (sequence, K/V head) slices of the workload "
                f"(at most {self.MAX_TOKENS} tokens, {self.w.g} query heads each), decode only, "
                f"{spent:.1f} s of oracle time, one thread per slice")

    def seq_steps_per_s(self, gbs: float) -> float:
        """Whole sequences of the workload per second at this byte rate."""
        return gbs * 1e9 / (decode_bytes(self.w, unique=False) / max(1, self.w.S))


def cpu_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ---------------------------------------------------------------- helpers

def peak_hbm():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


KERNEL_SOURCES = {
    "pkv_decode": ["pkv_decode_tc.cu", "pkv_decode_simt.cu", "pkv_common.cuh", "pkv_tc_common.cuh", "pkv_merge.cuh"],
    "pkv_prefill": ["pkv_prefill_umma.cu", "pkv_prefill_umma2.cu", "pkv_prefill_tc.cu", "pkv_qtile.cuh", "pkv_umma.cuh", "pkv_common.cuh",
                    "pkv_tc_common.cuh", "pkv_merge.cuh"],
    "pkv_vtoken": ["pkv_decode_tc.cu", "pkv_decode_simt.cu", "pkv_repack.cu", "pkv_common.cuh", "pkv_tc_common.cuh",
                   "pkv_merge.cuh"],
}


def code_only(text: str) -> str:
    """C/C++/CUDA source with its comments removed and every run of white
    space made one space: what the compiler sees, so that editing a comment
    does not disown a measurement.  String and character literals are kept
    as they are."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            out.append(" ")
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_source_hash(prefix: str = "pkv_decode") -> str:
    """Hash of the code a traffic record was taken on (comments aside): the
    kernels' files, the headers they include, and the parameter struct they
    read."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_cache_44_gb300", "csrc")
    for f in KERNEL_SOURCES[prefix]:
        with open(os.path.join(csrc, f), encoding="utf-8") as fh:
            h.update((f + "\n" + code_only(fh.read())).encode())
    with open(os.path.join(csrc, "pkv_internal.h"), encoding="utf-8") as fh:
        txt = code_only(fh.read())
    i0 = txt.index("struct DecodeParams {")
    h.update(txt[i0: txt.index("};", i0)].encode())
    return h.hexdigest()[:16]


def measured_traffic(workload: str, kernel: str, table: str = "decode_traffic.json", prefix: str = "pkv_decode"):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel sources; else None."""
    p = os.path.join(ROOT, "profiles", table)
    try:
        with open(p) as f:
            rec = json.load(f).get(f"{workload}/{kernel}")
    except (OSError, ValueError):
        return None
    if not rec or rec.get("source_hash") != kernel_source_hash(prefix):
        return None
    return rec.get("dram_bytes_per_launch")


def default_shape(args) -> bool:
    """The stored traffic records were taken on each workload's own size and
    partition; a run with fewer sequences or another partition reports none."""
    return args.S is None and args.partition is None


def max_over_ranks(values, device=None):
    """Element-wise maximum of `values` over all ranks (the job's time is the
    slowest rank's); a no-op without a process group."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor(values, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def whole_job_gbs(world_size: int, bytes_per_rank_step: int, ms_per_step: float) -> float:
    """Throughput of the whole job: every rank's bytes over the slowest rank's time."""
    return world_size * bytes_per_rank_step / (ms_per_step * 1e-3) / 1e9


def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# ------------------------------------------------------------------- arms

def run_reference(args, w: W.Workload):
    ws, rank, _ = dist_setup()
    if rank != 0:
        return
    threads = cpu_threads()
    sampler = OracleSampler(w, threads)
    # the whole run stays within about two minutes of oracle time
    budget = max(0.01, min(10.0, 120.0 / max(1, args.steps + args.warmup)))
    tot_bytes, tot_s, tot_items = 0, 0.0, 0
    per_step_ms = []
    for i in range(args.warmup + args.steps):
        b, sp, n = sampler.run(budget)
        if i >= args.warmup:
            tot_bytes += b
            tot_s += sp
            tot_items += n
            per_step_ms.append(sp * 1e3)
    gbs = tot_bytes / tot_s / 1e9
    sps = sampler.seq_steps_per_s(gbs)
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(statistics.mean(per_step_ms), 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "S": w.S, "Hq": w.Hq, "Hkv": w.Hkv, "d": w.d, "bs": w.bs,
                   "cache_dtype": w.cache_dtype, "max_context_len": w.max_context_len},
        "seq_steps_per_s": round(sps, 4),
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": sampler.describe(tot_items, tot_s)},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def device_caches(w: W.Workload, seed: int, dev, stream):
    """K and V pools of workload `w` filled on the device from seeded draws
    (bf16: the draws' upper halves; fp8: the library's own write with a
    per-tensor scale amax / 448).  Returns (key_cache, value_cache,
    k_scale, v_scale)."""
    import torch
    import paged_kv_cache_44_gb300 as pkv
    tdt = {W.DT_F32: torch.float32, W.DT_BF16: torch.bfloat16, W.DT_E4M3: torch.uint8}
    shape = (w.NB, w.bs, w.Hkv, w.d)
    numel = int(np.prod(shape))
    k_scale = v_scale = 1.0
    caches = []
    with torch.cuda.stream(stream):
        for which in (1, 2):
            if w.cache_dtype == W.DT_E4M3:
                cache = torch.empty(shape, dtype=torch.uint8, device=dev)
                sc = 0.0
                for _, x in W.device_pool_chunks(seed, which, numel, dev):
                    sc = max(sc, float(x.abs().max()))
                scale = float(np.float32(sc) / np.float32(W.E4M3_MAX))
                if which == 1:
                    k_scale = scale
                else:
                    v_scale = scale
                rows = w.Hkv * w.d
                for c0, x in W.device_pool_chunks(seed, which, numel, dev):
                    n = x.numel() // rows
                    slots = torch.arange(c0 // rows, c0 // rows + n, device=dev, dtype=torch.int64)
                    vals = x.view(n, w.Hkv, w.d)
                    pkv.paged_kv_write(vals, vals, cache, cache, slots, scale, scale, stream=stream)
            else:
                cache = torch.empty(numel, dtype=tdt[w.cache_dtype], device=dev)
                for c0, x in W.device_pool_chunks(seed, which, numel, dev):
                    cache[c0:c0 + x.numel()] = W.device_bf16_from_draws(x) if w.cache_dtype == W.DT_BF16 else x
                cache = cache.view(shape)
            caches.append(cache)
    return caches[0], caches[1], k_scale, v_scale


E2E_LOOP = "every step copies its inputs in and its result out (copy streams beside the compute stream); " \
           "two steps in flight"


def overlapped_e2e(dev, stream, h_in: dict, out_like, enqueue, steps: int, barrier=lambda: None):
    """Seconds per step of an end-to-end loop through the public API, run as
    a serving loop would: every step copies its inputs in from pinned host
    memory and its result out, each copy on a stream of its own beside the
    compute stream (step i + 1's inputs go into a second set of device
    buffers while step i computes; step i's result comes out while step
    i + 1 computes), and the host takes step i's result before it queues
    step i + 2.  enqueue(d_in, d_out) queues one step on `stream`.
    Returns (seconds per step, bytes in per step, bytes out per step)."""
    import torch
    d_ins = [{k: torch.empty_like(v, device=dev) for k, v in h_in.items()} for _ in range(2)]
    d_outs = [torch.empty_like(out_like) for _ in range(2)]
    h_outs = [torch.empty(out_like.shape, dtype=out_like.dtype, pin_memory=True) for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def one(i):
        b = i % 2
        if i >= 2:
            ev_out[b].synchronize()        # step i - 2's result is on the host; its buffers are free
        with torch.cuda.stream(s_in):
            for k in h_in:
                d_ins[b][k].copy_(h_in[k], non_blocking=True)
            ev_in[b].record(s_in)
        stream.wait_event(ev_in[b])
        enqueue(d_ins[b], d_outs[b])
        ev_done[b].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_done[b])
            h_outs[b].copy_(d_outs[b], non_blocking=True)
            ev_out[b].record(s_out)

    for i in range(2):
        one(i)
    torch.cuda.synchronize(dev)
    barrier()
    w0 = time.perf_counter()
    for i in range(steps):
        one(i)
    torch.cuda.synchronize(dev)
    secs = (time.perf_counter() - w0) / steps
    h2d = sum(v.numel() * v.element_size() for v in h_in.values())
    return secs, h2d, h_outs[0].numel() * h_outs[0].element_size()


def measure_step(args, w: W.Workload, dev, stream, steps: int, warmup: int, ws: int, rank: int, barrier,
                 e2e: bool = True, partition=None, min_seconds: float = 0.0) -> dict:
    """Time `steps` decode steps of workload `w` (after `warmup` untimed
    ones; more steps if they would take under `min_seconds`) with the K/V
    pools resident in HBM; returns the line's numbers."""
    import torch
    import paged_kv_cache_44_gb300 as pkv

    # ---- inputs, resident in HBM before timing
    seed = w.seed + 7919 * rank
    kc, vc, k_scale, v_scale = device_caches(w, seed, dev, stream)
    with torch.cuda.stream(stream):

        def dev_vals(tag, shp):
            x = W.device_normal(seed, tag, int(np.prod(shp)), dev).view(shp)
            return W.device_bf16_from_draws(x) if w.q_dtype == W.DT_BF16 else x

        q = dev_vals(11, (w.S, w.Hq, w.d))
        new_k = dev_vals(12, (w.S, w.Hkv, w.d))
        new_v = dev_vals(13, (w.S, w.Hkv, w.d))
    bt = torch.from_numpy(w.block_tables).to(dev)
    cl = torch.from_numpy(w.context_lens).to(dev)
    sm = torch.from_numpy(w.slot_mapping).to(dev)
    cow = torch.from_numpy(w.cow_pairs.astype(np.int64)).to(dev)
    out = torch.empty_like(q)
    P = partition if partition is not None else w.partition_size
    # the partition the decode launches with (for an E4M3 cache on the tensor cores it may be
    # twice the one the workspace is planned for)
    Pres = pkv.decode_launch_partition_size(w.S, w.Hq, w.Hkv, w.d, w.bs, w.NB, w.max_context_len, P,
                                            getattr(torch, TORCH_DT[w.q_dtype]),
                                            getattr(torch, TORCH_DT[w.cache_dtype]), args.kernel)
    wsp = pkv.make_workspace(w.S, w.Hq, w.Hkv, w.d, w.bs, w.max_context_len, P, device=dev)
    mc = w.max_context_len
    split = Pres > 0 and -(-mc // Pres) > 1
    launches_per_step = 1 + (2 if split else 1) + (1 if len(w.cow_pairs) else 0)
    torch.cuda.synchronize(dev)

    fused = args.fused and decode_kernel_name(args.kernel, w) == "tensor_cores"
    if fused:
        launches_per_step -= 1

    # A pool that L2 could hold most of is rotated: consecutive steps read different copies, and
    # at least two L2s' worth of other pools' bytes are read between two uses of one copy.
    pool_bytes = (kc.numel() * kc.element_size() + vc.numel() * vc.element_size())
    n_pools = 1 if pool_bytes >= 2 * L2_BYTES else min(64, 1 + -(-2 * L2_BYTES // pool_bytes))
    pools = [(kc, vc)] + [(kc.clone(), vc.clone()) for _ in range(n_pools - 1)]
    turn = [0]
    torch.cuda.synchronize(dev)

    def step(ev0=None, ev1=None, qq=q, nk=new_k, nv=new_v, btab=bt, clen=cl, slots=sm, pairs=cow, o=out,
             evw=None, evc=None):
        kc, vc = pools[turn[0] % n_pools]
        turn[0] += 1
        if fused:
            # one launch writes the new tokens and decodes (the timed "decode" includes the write)
            if ev0 is not None:
                ev0.record(stream)
            pkv.paged_kv_write_decode(o, qq, nk, nv, kc, vc, slots, btab, clen, mc, scale=w.scale,
                                      k_scale=k_scale, v_scale=v_scale, partition_size=P, workspace=wsp,
                                      stream=stream)
        else:
            if evw is not None:
                evw[0].record(stream)
            pkv.paged_kv_write(nk, nv, kc, vc, slots, k_scale, v_scale, stream=stream)
            if evw is not None:
                evw[1].record(stream)
            if ev0 is not None:
                ev0.record(stream)
            pkv.paged_attention_decode(o, qq, kc, vc, btab, clen, mc, scale=w.scale, k_scale=k_scale,
                                       v_scale=v_scale, partition_size=P, workspace=wsp, stream=stream,
                                       kernel=args.kernel)
        if ev1 is not None:
            ev1.record(stream)
        if len(w.cow_pairs):
            if evc is not None:
                evc[0].record(stream)
            pkv.copy_blocks([kc], [vc], pairs, stream=stream)
            if evc is not None:
                evc[1].record(stream)

    # ---- warm-up (timed, to size a timed region that must last a minimum time)
    w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    w0.record(stream)
    for _ in range(warmup):
        step()
    w1.record(stream)
    torch.cuda.synchronize(dev)
    if min_seconds > 0:
        est = w0.elapsed_time(w1) / max(1, warmup) * 1e-3
        steps = max(steps, int(math.ceil(min_seconds / max(est, 1e-6))))
        (steps,) = (int(v) for v in max_over_ranks([steps], dev))   # every rank times the same count

    # ---- timed region: K steps back to back, events on the launching stream around them only
    # (an event between two kernels keeps the second from starting early: every call after
    # the first is launched as a programmatic dependent of the one before)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(uuid) as clk:
        t0.record(stream)
        for i in range(steps):
            step()
        t1.record(stream)
        torch.cuda.synchronize(dev)
    barrier()
    ms_total = t0.elapsed_time(t1)
    (ms_total,) = max_over_ranks([ms_total], dev)
    ms_step = ms_total / steps

    # ---- each call of the step timed on its own, events around it (outside the timed region).
    # A sleep kernel holds the stream while the host queues the calls, so that no interval
    # includes the GPU waiting for the host (a 40 us call is about as long as queueing it).
    n_parts = max(3, min(steps, 200))
    with torch.cuda.stream(stream):
        torch.cuda._sleep(int(0.02 * 2.0e9))
    ev = lambda: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))  # noqa: E731
    evd = [ev() for _ in range(n_parts)]
    evw = [ev() for _ in range(n_parts)]
    evc = [ev() for _ in range(n_parts)]
    for i in range(n_parts):
        step(evd[i][0], evd[i][1], evw=None if fused else evw[i], evc=evc[i] if len(w.cow_pairs) else None)
    torch.cuda.synchronize(dev)
    dec_ms = statistics.mean(a.elapsed_time(b) for a, b in evd)
    (dec_ms,) = max_over_ranks([dec_ms], dev)
    write_ms = None if fused else statistics.mean(a.elapsed_time(b) for a, b in evw)
    copy_ms = statistics.mean(a.elapsed_time(b) for a, b in evc) if len(w.cow_pairs) else None

    # ---- end to end: host buffers in, host result out, through the public API
    e2e_s = h2d = d2h = None
    if e2e:
        pin = lambda t: t.cpu().pin_memory()  # noqa: E731
        h_in = {k: pin(v) for k, v in dict(q=q, nk=new_k, nv=new_v, bt=bt, cl=cl, sm=sm, cow=cow).items()}
        e2e_s, h2d, d2h = overlapped_e2e(
            dev, stream, h_in, out,
            lambda d, o: step(qq=d["q"], nk=d["nk"], nv=d["nv"], btab=d["bt"], clen=d["cl"], slots=d["sm"],
                              pairs=d["cow"], o=o),
            max(3, min(steps, 200)), barrier)
        (e2e_s,) = max_over_ranks([e2e_s], dev)

    # ---- numbers
    dbytes = decode_bytes(w) + (write_bytes(w) if fused else 0)
    sbytes = decode_bytes(w) + write_bytes(w) + copy_bytes(w)
    achieved = dbytes / (dec_ms * 1e-3) / 1e9
    peak, peak_kind = peak_hbm()
    traffic = measured_traffic(w.name, args.kernel) if default_shape(args) and partition is None else None
    kname = decode_kernel_name(args.kernel, w)
    res = {
        "value": whole_job_gbs(ws, sbytes, ms_step), "ms_per_step": ms_step, "steps": steps, "warmup": warmup,
        "config": {"workload": w.name, "S": w.S, "Hq": w.Hq, "Hkv": w.Hkv, "d": w.d, "bs": w.bs,
                   "cache_dtype": w.cache_dtype, "q_dtype": w.q_dtype, "max_context_len": mc,
                   "partition_size": Pres, "decode_kernel": kname, "fused_write_decode": bool(fused),
                   "kv_bytes": int(w.context_lens.astype(np.int64).sum()) * w.Hkv * w.d * 2 * ELEM[w.cache_dtype],
                   "l2": l2_note(pool_bytes, n_pools),
                   "step": ("paged_kv_write_decode(1 token/seq, one launch)" if fused else
                            "paged_kv_write(1 token/seq) + paged_attention_decode") +
                           " + copy_blocks(%d pairs)" % len(w.cow_pairs)},
        "seq_steps_per_s": round(ws * w.S / (ms_step * 1e-3), 1),
        "decode_gbs": round(achieved, 2),
        "decode_ms": round(dec_ms, 5),
        "decode_seq_steps_per_s": round(ws * w.S / (dec_ms * 1e-3), 1),
        "write_ms": None if write_ms is None else round(write_ms, 5),
        "copy_blocks_ms": None if copy_ms is None else round(copy_ms, 5),
        "hbm_frac_of_measured": round(achieved / peak, 4),
        "hbm_frac_of_nominal_8tbs": round(achieved / NOMINAL_HBM_GBS, 4),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_kind": peak_kind,
                     "traffic": None if fused else traffic,
                     "kernel": ("paged_kv_write_decode (" if fused else "paged_attention_decode (") + kname + ")",
                     "algorithmic_bytes_per_launch": dbytes, "launch_ms": round(dec_ms, 5)},
        "gpu_launches": launches_per_step * steps,
        "clocks": clk.summary(),
    }
    if w.shared_seqs:
        res["roofline"]["logical_bytes_per_launch"] = decode_bytes(w, unique=False)
    if e2e:
        res["e2e"] = {"value": round(whole_job_gbs(ws, sbytes, e2e_s * 1e3), 2), "unit": "GB/s",
                      "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_s * 1e3, 4),
                      "loop": E2E_LOOP}
    del pools, kc, vc, wsp
    torch.cuda.synchronize(dev)
    torch.cuda.empty_cache()
    return res


def cpu_baseline(w: W.Workload, seconds: float, one_thread: bool = True) -> dict:
    """The oracle on a bounded sample of workload `w` (see OracleSampler)."""
    threads = cpu_threads()
    sampler = OracleSampler(w, threads)
    b, spent, n = sampler.run(seconds)
    rec = {"value": round(b / spent / 1e9, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
           "sample": sampler.describe(n, spent),
           "seq_steps_per_s": round(sampler.seq_steps_per_s(b / spent / 1e9), 4)}
    if one_thread and threads > 1:
        one = OracleSampler(w, 1)
        b1, spent1, n1 = one.run(max(1.0, seconds / 4))
        rec["one_thread"] = {"value": round(b1 / spent1 / 1e9, 4), "unit": "GB/s", "sample": one.describe(n1, spent1)}
    return rec


# The configurations reported beside the headline one in a default run.
OTHER_WORKLOADS = ("qwen2.5-1.5b", "qwen2.5-7b-prefix", "fp8-bs16", "fp8-bs32")
OTHER_MIN_STEPS = 200     # short steps (the 1.5B-shaped one is ~40 us): more of them for a stable mean
OTHER_MIN_SECONDS = 0.3   # and a timed region long enough for the clock sampler to read the clocks in it


def run_ours(args, w: W.Workload):
    import torch

    ws, rank, local = dist_setup()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if ws > 1 else 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(device=dev)
    global L2_BYTES
    L2_BYTES = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or L2_BYTES)

    def barrier():
        if ws > 1:
            import torch.distributed as dist
            dist.barrier(device_ids=[dev.index])

    m = measure_step(args, w, dev, stream, args.steps, args.warmup, ws, rank, barrier, e2e=True,
                     partition=args.partition)
    line = {
        "metric": METRIC, "value": round(m["value"], 2), "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(m["ms_per_step"], 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if w.cache_dtype == W.DT_BF16 else w.cache_dtype, "data": "synthetic",
    }
    for k, v in m.items():
        if k not in ("value", "ms_per_step", "steps", "warmup"):
            line[k] = v
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds)
    if args.all_workloads:
        # the other configurations, each as its own decode step (same contract, more steps when short)
        line["workloads"] = {w.name: {k: line[k] for k in ("decode_ms", "decode_gbs", "hbm_frac_of_measured",
                                                           "hbm_frac_of_nominal_8tbs", "seq_steps_per_s",
                                                           "decode_seq_steps_per_s", "roofline", "clocks")}}
        line["workloads"][w.name].update(steps=args.steps, partition_size=line["config"]["partition_size"],
                                         headline=True)
        for name in OTHER_WORKLOADS:
            w2 = W.make(name)
            steps2 = max(args.steps, OTHER_MIN_STEPS)
            m2 = measure_step(args, w2, dev, stream, steps2, args.warmup, ws, rank, barrier, e2e=False,
                              min_seconds=OTHER_MIN_SECONDS)
            ent = {k: m2[k] for k in ("decode_ms", "decode_gbs", "hbm_frac_of_measured", "hbm_frac_of_nominal_8tbs",
                                      "seq_steps_per_s", "decode_seq_steps_per_s", "roofline", "clocks",
                                      "write_ms", "copy_blocks_ms", "gpu_launches")}
            ent["step_gbs"] = round(m2["value"], 2)
            ent["ms_per_step"] = round(m2["ms_per_step"], 5)
            ent["steps"] = m2["steps"]
            ent["config"] = m2["config"]
            if rank == 0 and not args.no_cpu_baseline:
                ent["cpu_baseline"] = cpu_baseline(w2, args.other_cpu_seconds, one_thread=False)
            line["workloads"][name] = ent
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def decode_kernel_name(kernel: str, w: W.Workload) -> str:
    if kernel != "auto":
        return kernel
    return "tensor_cores" if (w.cache_dtype == W.DT_E4M3 or
                              (w.cache_dtype == W.DT_BF16 and w.q_dtype == W.DT_BF16)) else "cuda_cores"


def peak_bf16(sustained: bool):
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            rec = json.load(f)
        return float(rec["bf16_tflops_sustained" if sustained else "bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return (1700.0 if sustained else 1900.0), "fallback"


def prefill_kernel_name(kernel: str, w: W.Workload, T: int) -> str:
    """The kernel a prefill call runs: the library's automatic choice takes
    two 128-row query tiles per unit when the (sequence, K/V head) pairs
    average 256 or more (query, head) rows."""
    if kernel != "auto":
        return kernel
    return "tcgen05_2tile" if T * (w.Hq // w.Hkv) >= 2 * 128 * w.S else "tcgen05"


def run_prefill(args, w: W.Workload):
    """Paged attention over query chunks: a step is one call over the
    workload's packed queries (chunked prefill next to decodes, or
    speculative verification), the K/V pools resident in HBM.  Reports both
    TFLOP/s and GB/s; the roofline takes the bound the arithmetic intensity
    selects (FLOPs per byte above the ratio of the measured peaks: tensor)."""
    import torch
    import paged_kv_cache_44_gb300 as pkv

    ws, rank, local = dist_setup()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if ws > 1 else 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(device=dev)
    if w.cache_dtype != W.DT_BF16 or w.q_dtype != W.DT_BF16:
        raise SystemExit("query chunks: bf16 query and cache only")
    seed = w.seed + 7919 * rank
    qlens = W.query_lens(w)
    qs_host = W.query_start(qlens)
    T, mq, mc = int(qs_host[-1]), int(qlens.max()), w.max_context_len
    kc, vc, _, _ = device_caches(w, seed, dev, stream)
    with torch.cuda.stream(stream):
        q = W.device_bf16_from_draws(W.device_normal(seed, 21, T * w.Hq * w.d, dev)).view(T, w.Hq, w.d)
    bt = torch.from_numpy(w.block_tables).to(dev)
    cl = torch.from_numpy(w.context_lens).to(dev)
    qs = torch.from_numpy(qs_host).to(dev)
    out = torch.empty_like(q)
    P = args.partition if args.partition is not None else 0
    wsb = pkv.prefill_workspace_size(w.S, T, mq, w.Hq, w.Hkv, w.d, w.bs, mc, P)
    wsp = torch.zeros(wsb, dtype=torch.uint8, device=dev)
    split = wsb > 256
    torch.cuda.synchronize(dev)

    def step(qq=q, btab=bt, clen=cl, qst=qs, o=out):
        pkv.paged_attention_prefill(o, qq, kc, vc, btab, clen, qst, mq, mc, scale=w.scale, partition_size=P,
                                    workspace=wsp, stream=stream, kernel=args.prefill_kernel)

    def barrier():
        if ws > 1:
            import torch.distributed as dist
            dist.barrier(device_ids=[dev.index])

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(uuid) as clk:
        t0.record(stream)
        for _ in range(args.steps):
            step()
        t1.record(stream)
        torch.cuda.synchronize(dev)
    barrier()
    (ms_total,) = max_over_ranks([t0.elapsed_time(t1)], dev)
    ms_step = ms_total / args.steps

    pin = lambda t: t.cpu().pin_memory()  # noqa: E731
    h_in = {k: pin(v) for k, v in dict(q=q, bt=bt, cl=cl, qs=qs).items()}
    e2e_s, h2d, d2h = overlapped_e2e(
        dev, stream, h_in, out, lambda d, o: step(qq=d["q"], btab=d["bt"], clen=d["cl"], qst=d["qs"], o=o),
        max(3, min(args.steps, 100)), barrier)
    (e2e_s,) = max_over_ranks([e2e_s], dev)

    flops, nbytes = prefill_flops(w, qlens), prefill_bytes(w, qlens)
    tflops = ws * flops / (ms_step * 1e-3) / 1e12
    gbs = whole_job_gbs(ws, nbytes, ms_step)
    hbm, hbm_kind = peak_hbm()
    tc, tc_kind = peak_bf16(sustained=ms_total > 2000.0)
    tensor_bound = flops / nbytes > tc * 1e12 / (hbm * 1e9)
    per_launch_tf, per_launch_gbs = flops / (ms_step * 1e-3) / 1e12, nbytes / (ms_step * 1e-3) / 1e9
    if tensor_bound:
        metric, value, unit = "paged attention over query chunks, TFLOP/s", tflops, "TFLOP/s"
        roof = {"bound": "tensor", "achieved": round(per_launch_tf, 2), "peak": tc, "unit": "TFLOP/s",
                "frac": round(per_launch_tf / tc, 4),
                "peak_kind": tc_kind + (" bf16 sustained" if ms_total > 2000.0 else " bf16 burst")}
        e2e_v = ws * flops / e2e_s / 1e12
    else:
        metric, value, unit = "paged attention over query chunks, KV GB/s", gbs, "GB/s"
        roof = {"bound": "hbm", "achieved": round(per_launch_gbs, 2), "peak": hbm, "unit": "GB/s",
                "frac": round(per_launch_gbs / hbm, 4), "peak_kind": hbm_kind}
        e2e_v = whole_job_gbs(ws, nbytes, e2e_s * 1e3)
    kname = prefill_kernel_name(args.prefill_kernel, w, T)
    roof.update({"traffic": measured_traffic(w.name, kname, "prefill_traffic.json", "pkv_prefill")
                 if default_shape(args) else None,
                 "kernel": "paged_attention_prefill (%s)" % kname,
                 "algorithmic_flops_per_launch": flops,
                 "algorithmic_bytes_per_launch": nbytes, "launch_ms": round(ms_step, 5)})
    line = {
        "component": "prefill", "metric": metric, "value": round(value, 2), "unit": unit, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "S": w.S, "Hq": w.Hq, "Hkv": w.Hkv, "d": w.d, "bs": w.bs,
                   "query_tokens": T, "max_query_len": mq, "max_context_len": mc,
                   "kv_tokens": int(w.context_lens.astype(np.int64).sum()),
                   "partition_size": P, "split": bool(split), "prefill_kernel": kname,
                   "l2": "inputs larger than L2" if nbytes > 2 * L2_BYTES else "not flushed: inputs near L2 size",
                   "step": "paged_attention_prefill over every sequence's query chunk"},
        "tflops": round(tflops, 2), "kv_gbs": round(gbs, 2),
        "query_tokens_per_s": round(ws * T / (ms_step * 1e-3), 1),
        "roofline": roof,
        "e2e": {"value": round(e2e_v, 2), "unit": unit, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_s * 1e3, 4), "loop": E2E_LOOP},
        "gpu_launches": (2 if split else 1) * args.steps,
        "clocks": clk.summary(),
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = prefill_cpu_baseline(w, qlens, args.cpu_seconds, tensor_bound)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def prefill_cpu_baseline(w: W.Workload, qlens: np.ndarray, budget: float, tensor_bound: bool):
    """The oracle on a bounded sample of the workload: batches of one
    sequence per host thread (the oracle's unit of parallel work), each
    keeping the last min(q_len, 16) queries of its chunk (the same keys per
    query as in the full chunk), until about `budget` seconds."""
    import oracle as O
    threads = cpu_threads()
    rng = np.random.default_rng(w.seed)
    order = list(rng.permutation(w.S))
    flops = nbytes = 0
    spent, seqs, queries, keys, calls = 0.0, 0, 0, 0, 0
    used = 1
    while order and spent < budget:
        take, tok = 0, 0                         # at most 2^17 K/V tokens of host draws per call
        while take < min(threads, len(order)) and (take == 0 or tok + int(w.context_lens[order[take]]) <= 1 << 17):
            tok += int(w.context_lens[order[take]])
            take += 1
        batch = np.array(sorted(order[:take]), np.int64)
        order = order[take:]
        used = max(used, take)
        sw = W.sub_workload(w, batch)
        hv = W.host_values(sw)
        ql = np.minimum(qlens[batch], 16).astype(np.int32)
        qst = W.query_start(ql)
        q = W.bf16_bits(W.host_normal(w.seed, "chunk-query:%d" % calls, (int(qst[-1]), w.Hq, w.d)))
        t0 = time.perf_counter()
        O.paged_attention_prefill(q, O.BF16, W.bf16_bits(hv.k_pool), W.bf16_bits(hv.v_pool), O.BF16,
                                  sw.block_tables, sw.context_lens, qst, w.scale, threads=threads)
        spent += time.perf_counter() - t0
        flops += prefill_flops(sw, ql)
        nbytes += prefill_bytes(sw, ql)
        seqs, queries, keys, calls = seqs + len(batch), queries + int(ql.sum()), keys + int(sw.context_lens.sum()), \
            calls + 1
    value = flops / spent / 1e12 if tensor_bound else nbytes / spent / 1e9
    return {"value": round(value, 6), "unit": "TFLOP/s" if tensor_bound else "GB/s", "cores": used,
            "kind": "oracle",
            "sample": "%d sequences in %d calls, the last <=16 queries of each chunk (%d query tokens, %d K/V "
                      "tokens), %.1f s" % (seqs, calls, queries, keys, spent)}


def token_decode_bytes(w: W.Workload, nt: np.ndarray) -> int:
    """Algorithmic bytes of a decode through token tables: query and output,
    the K/V rows of every live token once, and the table entries read."""
    bq, bkv = ELEM[w.q_dtype], ELEM[w.cache_dtype]
    live = int(nt.astype(np.int64).sum())
    return 2 * w.S * w.Hq * w.d * bq + live * w.Hkv * w.d * 2 * bkv + live * 4 + w.S * 4


def run_vtoken(args, w: W.Workload):
    """Token tables after a deletion policy kept half of each sequence's
    tokens at random: decode through the sparse tables, plan and run the
    repacking (every layer's K and V row of each moved token, one layer
    here), then decode through the compacted tables."""
    import torch
    import paged_kv_cache_44_gb300 as pkv

    ws, rank, local = dist_setup()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if ws > 1 else 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(device=dev)
    seed = w.seed + 7919 * rank
    keep = 0.5
    slots_h, nt_h = W.token_tables(w, keep)
    kc, vc, k_scale, v_scale = device_caches(w, seed, dev, stream)
    with torch.cuda.stream(stream):
        q = W.device_bf16_from_draws(W.device_normal(seed, 31, w.S * w.Hq * w.d, dev)).view(w.S, w.Hq, w.d)
    ts0 = torch.from_numpy(slots_h).to(dev)
    nt = torch.from_numpy(nt_h).to(dev)
    mx = int(nt_h.max())
    P = args.partition if args.partition is not None else w.partition_size
    wsp = pkv.make_workspace(w.S, w.Hq, w.Hkv, w.d, w.bs, mx, P, device=dev)
    out = torch.empty_like(q)
    torch.cuda.synchronize(dev)
    nbytes = token_decode_bytes(w, nt_h)

    def decode(ts, qq=q, ntt=nt, o=out):
        pkv.token_attention_decode(o, qq, kc, vc, ts, ntt, mx, scale=w.scale, k_scale=k_scale, v_scale=v_scale,
                                   partition_size=P, workspace=wsp, stream=stream)

    def timed_decode(ts):
        for _ in range(args.warmup):
            decode(ts)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        e0.record(stream)
        for _ in range(args.steps):
            decode(ts)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) / args.steps

    uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    with ClockSampler(uuid) as clk:
        ms_sparse = timed_decode(ts0)
    clocks = clk.summary()

    # repacking: plan on the host, move on the device
    t0 = time.perf_counter()
    moves_h, freed_h = pkv.vtoken_plan(slots_h, nt_h, w.bs, w.NB)
    plan_s = time.perf_counter() - t0
    moves = torch.from_numpy(moves_h).to(dev)
    moved_bytes = 2 * 2 * len(moves_h) * w.Hkv * w.d * ELEM[w.cache_dtype]      # K and V, read and write
    ts = ts0.clone()
    rep_ms = []
    for i in range(args.warmup + 5):
        ts.copy_(ts0)
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        pkv.repack_tokens([kc], [vc], ts, moves, stream=stream)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        if i >= args.warmup:
            rep_ms.append(e0.elapsed_time(e1))
    ms_repack = statistics.median(rep_ms)
    ms_dense = timed_decode(ts)
    (ms_sparse, ms_dense, ms_repack) = max_over_ranks([ms_sparse, ms_dense, ms_repack], dev)

    # end to end: host query and tables in, output out, through the public API
    h_in = {k: v.cpu().pin_memory() for k, v in dict(q=q, ts=ts, nt=nt).items()}
    e2e_s, h2d, d2h = overlapped_e2e(dev, stream, h_in, out,
                                     lambda d, o: decode(d["ts"], qq=d["q"], ntt=d["nt"], o=o),
                                     max(3, min(args.steps, 100)))
    (e2e_s,) = max_over_ranks([e2e_s], dev)

    gbs_sparse = whole_job_gbs(ws, nbytes, ms_sparse)
    gbs_dense = whole_job_gbs(ws, nbytes, ms_dense)
    peak, peak_kind = peak_hbm()
    line = {
        "component": "vtoken", "metric": "token-table decode KV GB/s (live tokens), after repacking",
        "value": round(gbs_dense, 2), "unit": "GB/s", "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_dense, 5), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if w.cache_dtype == W.DT_BF16 else w.cache_dtype, "data": "synthetic",
        "config": {"workload": w.name + "-vtoken", "S": w.S, "Hq": w.Hq, "Hkv": w.Hkv, "d": w.d, "bs": w.bs,
                   "tokens_before_deletion": int(w.context_lens.astype(np.int64).sum()),
                   "live_tokens": int(nt_h.sum()), "deletion": "each token kept with probability %.2f" % keep,
                   "partition_size": P, "l2": "inputs larger than L2",
                   "step": "token_attention_decode over every sequence's live tokens"},
        "decode_before_repack_gbs": round(gbs_sparse, 2), "decode_before_repack_ms": round(ms_sparse, 5),
        "repack": {"moves": int(len(moves_h)), "blocks_released": int(len(freed_h)),
                   "blocks_in_use_before": int(len({int(x) // w.bs for s in range(w.S) for x in slots_h[s, : nt_h[s]]})),
                   "ms": round(ms_repack, 5), "gbs": round(moved_bytes / (ms_repack * 1e-3) / 1e9, 2),
                   "plan_ms_host": round(plan_s * 1e3, 2), "layers": 1},
        "roofline": {"bound": "hbm", "achieved": round(gbs_dense / ws, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(gbs_dense / ws / peak, 4), "peak_kind": peak_kind,
                     "traffic": measured_traffic(w.name, "vtoken", "vtoken_traffic.json", "pkv_vtoken")
                     if default_shape(args) else None,
                     "kernel": "token_attention_decode (tensor cores, cp.async row gather)",
                     "algorithmic_bytes_per_launch": nbytes, "launch_ms": round(ms_dense, 5)},
        "e2e": {"value": round(whole_job_gbs(ws, nbytes, e2e_s * 1e3), 2), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_s * 1e3, 4),
                "loop": E2E_LOOP},
        "gpu_launches": (2 if wsp.numel() > 256 else 1) * args.steps,
        "clocks": clocks,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_block_manager(args):
    """Host block manager throughput, serving-like: S sequences whose
    prompts share a system prefix are admitted (prefix-cache lookups and
    hashing of every full block), each then grows by `steps` tokens (one
    slot per token, a new block every block_size tokens), then all are freed.
    Times the C-ABI calls through the binding (ctypes overhead included)."""
    import paged_kv_cache_44_gb300 as pkv
    rng = np.random.default_rng(0)
    S, bs, prompt, steps = 256, 16, 1024, max(1, min(args.steps, 256))
    system = rng.integers(1, 150_000, 512, dtype=np.int32)
    prompts = [np.concatenate([system, rng.integers(1, 150_000, prompt - 512, dtype=np.int32)]) for _ in range(S)]
    nb = S * (prompt + steps) // bs + S + 8
    pool = pkv.BlockPool(nb, bs)
    t0 = time.perf_counter()
    hits = sum(pool.add_sequence(i, prompts[i]) for i in range(S))
    t1 = time.perf_counter()
    ids = np.arange(S, dtype=np.int64)
    toks = np.full(S, 7, np.int32)
    for _ in range(steps):
        pool.append_tokens(ids, toks)          # one call per decode step: slots + copy pairs
    t2 = time.perf_counter()
    _, cl = pool.block_tables(ids, (prompt + steps + bs - 1) // bs)
    t2b = time.perf_counter()
    step_us, tables_us = (t2 - t1) / steps * 1e6, (t2b - t2) * 1e6
    assert int(cl.min()) == prompt + steps
    t2 = t2b
    for i in range(S):
        pool.free_sequence(i)
    t3 = time.perf_counter()
    line = {"component": "block-manager", "metric": "host block manager operations/s",
            "admit_tokens_per_s": round(S * prompt / (t1 - t0), 1),
            "prefix_hit_tokens": int(hits),
            "append_tokens_per_s": round(S * steps / (t2 - t1), 1),
            "decode_step_us": round(step_us, 2),
            "block_tables_us": round(tables_us, 1),
            "free_sequences_per_s": round(S / (t3 - t2), 1),
            "config": {"sequences": S, "prompt_tokens": prompt, "shared_prefix_tokens": 512, "block_size": bs,
                       "appended_tokens_per_sequence": steps, "blocks": nb},
            "host": {"cpu_threads": cpu_threads()}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default=None, choices=sorted(W.SHAPES),
                    help="default: qwen2.5-72b-long (decode-step), qwen2.5-7b-chunked (prefill)")
    ap.add_argument("--kernel", default="auto", choices=["auto", "cuda_cores", "tensor_cores"])
    ap.add_argument("--partition", type=int, default=None)
    ap.add_argument("--prefill-kernel", default="auto", choices=["auto", "tcgen05", "tcgen05_2tile", "mma_sync"])
    ap.add_argument("--fused", action="store_true",
                    help="decode-step: write the new tokens and decode in one launch")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--S", type=int, default=None, help="fewer sequences (small profiling cases)")
    ap.add_argument("--no-workloads", action="store_true",
                    help="decode-step: time only the headline workload (a default run also reports the "
                         "1.5B-, 7B- and fp8-shaped ones under 'workloads')")
    ap.add_argument("--other-cpu-seconds", type=float, default=3.0,
                    help="oracle seconds for each of the other workloads' cpu_baseline")
    ap.add_argument("--component", default="decode-step", choices=["decode-step", "prefill", "vtoken",
                                                                   "block-manager"],
                    help="prefill: paged attention over query chunks; block-manager: the host block "
                         "manager (each prints its own line)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.component == "block-manager":
        run_block_manager(args)
        return
    args.all_workloads = (args.component == "decode-step" and args.workload is None and args.S is None and
                          args.partition is None and not args.no_workloads and args.impl == "ours")
    if args.workload is None:
        args.workload = "qwen2.5-7b-chunked" if args.component == "prefill" else "qwen2.5-72b-long"
    w = W.make(args.workload, S=args.S) if args.S else W.make(args.workload)
    if args.component == "vtoken":
        if args.impl == "reference":
            ap.error("--impl reference times the decode step")
        run_vtoken(args, w)
        return
    if args.component == "prefill":
        if args.impl == "reference":
            ap.error("--impl reference times the decode step")
        run_prefill(args, w)
        return
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
