// paged_attention_decode on tensor cores (sm_103a).
//
// "LLM推論の基礎とvLLMの内部", section 4: each sequence's K/V is reached
// through its block table; section 2: the query heads of a GQA group share
// one K/V head, so one read of a K/V block serves the whole group; section 1:
// decode is bound by memory bandwidth, so the design goal is to keep HBM
// streaming.
//
// Work unit: (sequence, K/V head, set of <= 8 query heads, partition of P
// tokens).  Each warp is an independent worker: it takes its first unit by
// its index and claims the rest from a counter in the workspace header (or
// takes them round-robin without one),
// and streams the unit's K/V through its own ring of shared-memory stages.
// A stage is 32 tokens of K and V for one K/V head.  The cache is seen by
// the TMA engine as a 2-D tensor [NB * bs rows, Hkv * d elements]; one
// tiled copy (cp.async.bulk.tensor) moves the 128-byte half-rows of one
// K/V head for all bs tokens of the physical block the table names, with
// the 128-byte swizzle (64-byte for 64-byte rows) so that tensor-core
// operand loads are free of bank conflicts.  Copies complete on the stage's
// mbarrier.  The warp keeps up to kStages-1 stages in flight while it works
// on one, and it prefetches across unit boundaries: the next unit's first
// stage, and (bf16 query) its query fragments, loaded into registers when
// the unit is claimed.
//
// Math per stage (mma.sync m16n8k16, fp32 accumulate):
//   S^T[16 tokens x 8 heads] = K[16 x d] . Q^T[d x 8]          (d/16 MMAs per 16 tokens)
//   online softmax over the stage (running max m, sum l, base 2)
//   O^T[d x 8 heads] += V^T[d x 16 tokens] . P^T[16 tokens x 8]  (d/16 MMAs per 16 tokens)
// P^T is the S^T accumulator converted to 16-bit and transposed in registers
// (movmatrix).  bf16 caches use bf16 operands loaded with ldmatrix; E4M3
// caches are widened to fp16 in registers (cvt.rn.f16x2.e4m3x2, exact) and
// use fp16 operands with the query rounded to fp16.  For E4M3 the head
// dimension and the tokens are visited in a fixed permutation (the same on
// both operands of each product) so that every thread reads contiguous bytes.
//
// A unit that covers its whole sequence writes `out`; otherwise it writes
// (m, l, unnormalised O) to the workspace for the merge kernel.
//
// Through a token table (TT): "LLM推論の「見えないメモリ問題」を解く … vToken",
// token-level virtualisation: each live token of a sequence, in logical
// order, names its own slot (block * bs + offset), so a stage's 32 tokens
// may come from anywhere in the pool.  The issue side then copies each
// token's row with 16-byte cp.async requests (eight lanes per 128-byte line)
// straight into the same swizzled stage layout, and the stage's mbarrier
// counts one arrival per lane when its copies land; the math is unchanged.
// (A tensor copy that gathers rows could write only whole 1024-byte swizzle
// atoms, which four 128-byte rows do not fill.)

#include <cuda.h>
#include <cudaTypedefs.h>
#include <math_constants.h>

#include <mutex>

#include "pkv_common.cuh"
#include "pkv_internal.h"
#include "pkv_tc_common.cuh"

namespace pkv {
namespace {

using namespace tc;

// Tuning knobs: workers per CTA, stages per worker, tokens per stage, for
// bf16 and for E4M3 caches (E4M3 does more arithmetic per byte and wants
// more workers).  With two stages a bf16 worker takes 32 KB of shared
// memory, so 7 are as many as fit.  An E4M3 worker takes 16 KB; 11 measured
// fastest (12: 1.2% slower; 13 no longer fit their registers).
#ifndef PKV_TC_WARPS_BF16
#define PKV_TC_WARPS_BF16 7
#endif
#ifndef PKV_TC_STAGES_BF16
#define PKV_TC_STAGES_BF16 2
#endif
#ifndef PKV_TC_TOK_BF16
#define PKV_TC_TOK_BF16 32
#endif
#ifndef PKV_TC_WARPS_FP8
#define PKV_TC_WARPS_FP8 11
#endif
#ifndef PKV_TC_STAGES_FP8
#define PKV_TC_STAGES_FP8 2
#endif
#ifndef PKV_TC_TOK_FP8
#define PKV_TC_TOK_FP8 32
#endif

constexpr int kHeadsPerUnit = 8;
constexpr long long kWaitLimitCycles = 4000000000LL;   // ~2 s: a stage that never lands

template <int D, bool FP8, int QB>
struct Cfg {
    static constexpr int kWarpsWanted = FP8 ? PKV_TC_WARPS_FP8 : PKV_TC_WARPS_BF16;
    static constexpr int kStages = FP8 ? PKV_TC_STAGES_FP8 : PKV_TC_STAGES_BF16;  // ring depth per worker
    static constexpr int kTok = FP8 ? PKV_TC_TOK_FP8 : PKV_TC_TOK_BF16;          // tokens per stage
    static constexpr int kMT = kTok / 16;                        // 16-token m-tiles per stage
    static constexpr int kRowBytes = FP8 ? D : 2 * D;            // one token of one K/V head
    static constexpr int kBoxRow = kRowBytes >= 128 ? 128 : kRowBytes;   // bytes per row of one TMA box
    static constexpr int kHalves = kRowBytes / kBoxRow;         // boxes per (block, K or V)
    static constexpr int kPartBytes = kTok * kRowBytes;         // K (or V) part of a stage
    static constexpr int kStageBytes = 2 * kPartBytes;
    // queued units (claimed, first stage issued, not yet started): at most
    // one per stage in flight
    static constexpr int kQueue = kStages;
    // shared memory: every worker's stages (1024-byte aligned), then one
    // trailer with each worker's barriers, stage masks and unit queue.  The
    // query goes to registers (see qn in the kernel), not to shared memory.
    static constexpr int kWarpBytes = (kStages * kStageBytes + 1023) / 1024 * 1024;
    // trailer per worker: barriers (8 B each), stage masks (4 B each), then
    // the unit queue (32-byte entries, 16-byte aligned)
    static constexpr int kQueueCtlOff = (8 * kStages + 4 * kStages + 15) / 16 * 16;
    static constexpr int kCtlBytes = kQueueCtlOff + 32 * kQueue;
    // workers per CTA: as many as wanted, up to what fits in shared memory
    static constexpr int kWarpsFit = (232448 - 1024) / (kWarpBytes + kCtlBytes);
    static constexpr int kWarps = kWarpsWanted < kWarpsFit ? kWarpsWanted : kWarpsFit;
    static constexpr int kCtlOff = kWarps * kWarpBytes;
    static constexpr int kSmemBytes = kCtlOff + kWarps * kCtlBytes + 1024;   // + room to align the base
    static constexpr int KS = D / 16;     // k-steps of the QK product, m-tiles of the PV product
    static_assert(kTok == 16 || kTok == 32, "stages hold 16 or 32 tokens");
    static_assert(kStageBytes % 1024 == 0 || kRowBytes < 128, "stages must keep the swizzle atoms aligned");
    static_assert(kSmemBytes <= 232448, "shared memory per CTA");
    static_assert(kCtlOff % 1024 == 0 && kCtlBytes % 16 == 0, "trailer alignment");
};

// ------------------------------------------------------------------- units

// Region B ids per (sequence, head set): the full-size chunks of the longest
// remainder (hold * P + P - 1 tokens), then one for the partial chunk.
__host__ __device__ __forceinline__ int chunk_slots(int P, int Q, int hold) {
    const int held = Q < P ? hold : 0;
    return (held * P + P - 1) / Q + 1;
}

struct __align__(16) Unit {
    int s, kvh, h0, nh, part, t0, t1, np;
};

// Unit id -> coordinates.  The ids run over two regions:
//   A: every full partition (P tokens) not held back, partition-major -- the same
//      partition of every sequence is claimed close together in time, so
//      shared prefix blocks are read while still in L2;
//   B: the chunks of each sequence's last, partial partition (and, with
//      p.hold, of the full partitions held back before it): first every
//      full-size chunk (Q tokens), chunk-major, then each sequence's
//      shorter last chunk (and the empty unit of a sequence with no tokens).
// Claimed in id order, the long units go first and the short ones last, so
// the tail of the launch is short.  Returns false for ids that name no
// work (a partition past the sequence's full ones, a chunk past its
// remainder, or a last chunk that does not exist).
__device__ __forceinline__ bool unit_of(const DecodeParams& p, unsigned long long u, int nsets,
                                        unsigned long long region_a, Unit& x) {
    const unsigned long long per_part = (unsigned long long)p.S * p.Hkv * nsets;
    const bool in_a = u < region_a;
    const unsigned long long v = in_a ? u : u - region_a;
    const int idx = (int)(v / per_part);                  // partition (A) or chunk (B) index
    const unsigned long long rem = v - (unsigned long long)idx * per_part;
    x.s = (int)(rem / (unsigned)(p.Hkv * nsets));
    const int r2 = (int)(rem - (unsigned long long)x.s * (p.Hkv * nsets));
    x.kvh = r2 / nsets;
    const int set = r2 - x.kvh * nsets;
    x.h0 = x.kvh * p.g + set * kHeadsPerUnit;
    x.nh = min(kHeadsPerUnit, p.g - set * kHeadsPerUnit);
    int n = __ldg(p.context_lens + x.s);
    if (n < 0 || n > p.max_ctx) {
        if (!in_a && idx == 0 && r2 == 0) report(p.err, PKV_DEVERR_CONTEXT_LEN);
        n = n < 0 ? 0 : p.max_ctx;
    }
    x.np = num_partitions(n, p.P, p.Q, p.hold);
    const int full = whole_partitions(n, p.P, p.Q, p.hold);
    const int tail = n - full * p.P;
    const int cfull = chunk_slots(p.P, p.Q, p.hold) - 1;   // full-size chunks of the longest remainder
    if (in_a) {
        if (idx >= full) return false;
        x.part = idx;
    } else if (idx < cfull) {
        if ((idx + 1) * p.Q > tail) return false;          // full-size chunks first
        x.part = full + idx;
    } else {
        if (idx > cfull) return false;
        if (n > 0 && tail % p.Q == 0) return false;        // then the remainder's partial chunk
        x.part = full + tail / p.Q;
    }
    partition_range(n, p.P, p.Q, p.hold, x.part, x.t0, x.t1);
    return true;
}

template <typename QF>
__device__ __forceinline__ void store_out(const DecodeParams& p, size_t idx, float v) {
    store_elem<QF>(p.out, idx, v);
}

// ------------------------------------------------------------------ kernel

template <int D, bool FP8, typename QF, bool TT>
__global__ void __launch_bounds__(Cfg<D, FP8, QF::bytes>::kWarps * 32, 1)
    decode_tc_kernel(const __grid_constant__ DecodeParams p, const __grid_constant__ CUtensorMap kmap,
                     const __grid_constant__ CUtensorMap vmap, unsigned long long total_units,
                     unsigned long long region_a, int nsets) {
    using C = Cfg<D, FP8, QF::bytes>;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int r = lane >> 2, c = lane & 3;     // fragment row / column-pair of this lane
    // swizzle atoms need 1024-byte alignment: align the base ourselves
    const uint32_t raw_addr = smem_addr(smem_raw);
    const uint32_t base_addr = (raw_addr + 1023u) & ~1023u;
    unsigned char* smem = smem_raw + (base_addr - raw_addr);
    constexpr int kWarps = C::kWarps, kTok = C::kTok;
    unsigned char* ws = smem + warp * C::kWarpBytes;
    const uint32_t ws_addr = base_addr + warp * C::kWarpBytes;
    unsigned char* ctl = smem + C::kCtlOff + warp * C::kCtlBytes;
    const uint32_t ctl_addr = base_addr + C::kCtlOff + warp * C::kCtlBytes;
    uint32_t* masks = reinterpret_cast<uint32_t*>(ctl + 8 * C::kStages);
    Unit* queue = reinterpret_cast<Unit*>(ctl + C::kQueueCtlOff);
    auto bar = [&](int i) { return ctl_addr + 8 * i; };
    auto stage_k = [&](int i) { return ws_addr + i * C::kStageBytes; };
    auto stage_v = [&](int i) { return ws_addr + i * C::kStageBytes + C::kPartBytes; };
    auto lds128 = [&](uint32_t a) { return *reinterpret_cast<const uint4*>(ws + (a - ws_addr)); };
    auto lds64 = [&](uint32_t a) { return *reinterpret_cast<const uint2*>(ws + (a - ws_addr)); };
    // query column of fragment k-step ks: this lane's pairs (d0, d0 + 1) and (d1, d1 + 1)
    auto q_cols = [&](int ks, int& d0, int& d1) {
        if constexpr (FP8) {
            d0 = 64 * (ks / 4) + 16 * c + 4 * (ks % 4);      // 4 consecutive d: j = 0..3
            d1 = d0 + 2;
        } else {
            d0 = 16 * ks + 2 * c;
            d1 = d0 + 8;
        }
    };
    // A bf16 query's fragments for the oldest claimed unit that has not started, as the
    // 32-bit words (bf16 pairs) of head r of the lane, zero past the unit's heads: loaded
    // when that unit is claimed, or when the unit before it starts, so they are in
    // registers by the unit's start.
    uint32_t qn[C::KS][2];
    int qn_for = -1;                      // queue index of the unit they belong to; -1: free
    auto load_qn = [&](int s, int h0, int nh) {
        if constexpr (QF::bytes == 2) {
            const bool hv = r < nh;
            const uint32_t* qw = reinterpret_cast<const uint32_t*>(
                static_cast<const unsigned char*>(p.q) + ((size_t)s * p.Hq + h0 + (hv ? r : 0)) * D * 2);
#pragma unroll
            for (int ks = 0; ks < C::KS; ++ks) {
                int d0, d1;
                q_cols(ks, d0, d1);
                qn[ks][0] = hv ? __ldg(qw + d0 / 2) : 0u;
                qn[ks][1] = hv ? __ldg(qw + d1 / 2) : 0u;
            }
        }
    };

    // the partition merge that may follow can be scheduled now; it waits for this grid's results
    pdl_trigger();
    if (lane == 0) {
        // through a token table every lane's copies arrive on the stage barrier, and lane 0 once more
        for (int i = 0; i < C::kStages; ++i) mbar_init(bar(i), TT ? 33 : 1);
        fence_barrier_init();
    }
    __syncwarp();
    // the previous kernel of the stream (a write of the step's tokens, say) is complete from here on
    pdl_wait();

    // K/V is streamed: its lines go first when L2 needs room, so the partial
    // results (kept with "evict last") and the lines of blocks shared by
    // several sequences, read again soon, stay longer
    const uint64_t kv_pol = l2_policy_evict_first();
    const unsigned long long total_warps = (unsigned long long)gridDim.x * kWarps;
    const unsigned long long my_warp = (unsigned long long)blockIdx.x * kWarps + warp;
    unsigned long long static_next = my_warp;
    const int box_rows = min(p.bs, kTok);                  // tokens one box covers
    const int boxes_per_stage = kTok / box_rows;           // 2 (bs 16, 32-token stages) or 1
    const uint32_t box_bytes = (uint32_t)box_rows * C::kBoxRow;

    // ---- issue side: claims units, fills stages
    bool claiming = true;
    bool i_have = false;
    Unit iu{};
    int i_stage = 0, i_nst = 0;
    unsigned g_issue = 0, q_tail = 0;

    // A worker's first unit is taken without the counter: unit (warp * CTAs +
    // CTA), a one-to-one map of the first round of units onto the workers
    // that spreads consecutive units (neighbouring sequences) over the SMs as
    // the counter's arrival order does, and saves the contended atomic of the
    // launch's ramp.  Later claims come from the counter, offset by the
    // number of workers.
    bool first_claim = true;
    auto claim = [&](unsigned long long& u) -> bool {
        for (;;) {
            unsigned long long v = 0;
            if (first_claim) {
                v = (unsigned long long)warp * gridDim.x + blockIdx.x;   // consecutive units on different SMs
                first_claim = false;
            } else if (lane == 0) {
                if (p.sched != nullptr) {
                    v = atomicAdd(reinterpret_cast<unsigned long long*>(p.sched), 1ull) + total_warps;
                } else {
                    v = static_next;
                }
            }
            v = __shfl_sync(0xffffffffu, v, 0);
            static_next += total_warps;
            if (v >= total_units) return false;
            Unit x;
            if (!unit_of(p, v, nsets, region_a, x)) continue;
            if (x.t1 <= x.t0) {
                // a sequence with no tokens: its output is zero
                for (int i = lane; i < x.nh * D; i += 32)
                    store_out<QF>(p, ((size_t)x.s * p.Hq + x.h0 + i / D) * D + (i % D), 0.f);
                continue;
            }
            u = v;
            return true;
        }
    };

    // block-table entries of the issuing unit, 32 per chunk, one per lane;
    // the next chunk is loaded while the current one is in use
    int tab = 0, tab_next = 0, tab_chunk = 0, tab_blocks = 0;
    auto load_chunk = [&](int chunk) -> int {
        const int rb = 32 * chunk + lane;
        return rb < tab_blocks ? __ldg(p.block_tables + (size_t)iu.s * p.MB + iu.t0 / p.bs + rb) : 0;
    };

    auto issue_one = [&]() -> bool {
        while (!i_have || i_stage == i_nst) {
            if (!claiming) return false;
            unsigned long long u;
            if (!claim(u)) {
                claiming = false;
                return false;
            }
            unit_of(p, u, nsets, region_a, iu);
            if (lane == 0) {
                int4* e = reinterpret_cast<int4*>(queue + q_tail % C::kQueue);
                e[0] = make_int4(iu.s, iu.kvh, iu.h0, iu.nh);
                e[1] = make_int4(iu.part, iu.t0, iu.t1, iu.np);
            }
            if (qn_for < 0) {
                load_qn(iu.s, iu.h0, iu.nh);
                qn_for = (int)q_tail;
            }
            ++q_tail;
            i_have = true;
            i_stage = 0;
            i_nst = (iu.t1 - iu.t0 + kTok - 1) / kTok;
            if constexpr (!TT) {
                tab_blocks = (iu.t1 - iu.t0 + p.bs - 1) / p.bs;
                tab_chunk = 0;
                tab = load_chunk(0);
                tab_next = load_chunk(1);
            }
        }
        const int slot = g_issue % C::kStages;
        const int ts = iu.t0 + i_stage * kTok;
        const int tn = min(kTok, iu.t1 - ts);
        const int rs = i_stage * kTok;                         // token offset of the stage in the unit
        if constexpr (TT) {
            // lane i: the slot of token ts + i; -1 when past the unit or out of the pool
            int tslot = -1;
            if (lane < tn) {
                tslot = __ldg(p.token_slots + (size_t)iu.s * p.MT + ts + lane);
                if (tslot < 0 || (long long)tslot >= (long long)p.NB * p.bs) {
                    report(p.err, PKV_DEVERR_SLOT);
                    tslot = -1;
                }
            }
            const uint32_t m = __ballot_sync(0xffffffffu, tslot >= 0);
            // lanes cover token rows 16 bytes each: CPR lanes per row, 32 / CPR rows per request
            constexpr int CPR = C::kRowBytes / 16;
            constexpr int TPI = 32 / CPR;
            const int j = lane % CPR;
            const unsigned char* kcb = static_cast<const unsigned char*>(p.kc);
            const unsigned char* vcb = static_cast<const unsigned char*>(p.vc);
#pragma unroll 4
            for (int t0 = 0; t0 < kTok; t0 += TPI) {
                const int t = t0 + lane / CPR;
                const int sl = __shfl_sync(0xffffffffu, tslot, t);
                if (sl >= 0) {
                    const size_t row = ((size_t)sl * p.Hkv + iu.kvh) * C::kRowBytes + 16 * j;
                    cp_async16_hint(swz<C::kRowBytes, kTok>(stage_k(slot), t, 16 * j), kcb + row, kv_pol);
                    cp_async16_hint(swz<C::kRowBytes, kTok>(stage_v(slot), t, 16 * j), vcb + row, kv_pol);
                }
            }
            cp_async_mbar_arrive_noinc(bar(slot));
            if (lane == 0) {
                masks[slot] = m;
                mbar_arrive_expect_tx(bar(slot), 0u);
            }
            ++g_issue;
            ++i_stage;
            return true;
        }
        if (rs / p.bs / 32 != tab_chunk) {                     // the stage's blocks start a new chunk
            ++tab_chunk;
            tab = tab_next;
            tab_next = load_chunk(tab_chunk + 1);
        }
        // per token: inside the unit and in a block with a valid id
        const int pb_tok = __shfl_sync(0xffffffffu, tab, ((rs + lane) / p.bs) & 31);
        bool ok = lane < tn;
        if (ok && (pb_tok < 0 || pb_tok >= p.NB)) {
            report(p.err, PKV_DEVERR_BLOCK_ID);
            ok = false;
        }
        const uint32_t m = __ballot_sync(0xffffffffu, ok);
        // one box per (box_rows tokens of the stage, K or V, 128-byte half): lane i issues box i
        const int nbox = boxes_per_stage * 2 * C::kHalves;
        const int b = lane / (2 * C::kHalves), kv = (lane / C::kHalves) & 1, h = lane % C::kHalves;
        const uint32_t rows_mask = box_rows == 32 ? 0xffffffffu : 0xffffu;
        const bool box_live = lane < nbox && ((m >> (b * box_rows)) & rows_mask) != 0;
        const uint32_t nissue = __popc(__ballot_sync(0xffffffffu, box_live));
        const int pb_box = __shfl_sync(0xffffffffu, tab, ((rs + b * box_rows) / p.bs) & 31);
        if (lane == 0) {
            masks[slot] = m;
            mbar_arrive_expect_tx(bar(slot), nissue * box_bytes);
        }
        __syncwarp();
        if (box_live) {
            const int t0b = ts + b * box_rows;                 // first token of the box
            const uint32_t dst = (kv ? stage_v(slot) : stage_k(slot)) + h * (kTok * C::kBoxRow) +
                                 b * box_rows * C::kBoxRow;
            tensor_load_2d_hint(dst, kv ? &vmap : &kmap, iu.kvh * D + h * (C::kBoxRow / (FP8 ? 1 : 2)),
                                pb_box * p.bs + t0b % p.bs, bar(slot), kv_pol);
        }
        ++g_issue;
        ++i_stage;
        return true;
    };

    // ---- consume side
    unsigned g_cons = 0, q_head = 0;
    bool have_unit = false, need_q = false;
    Unit cu{};
    int c_stage = 0, c_nst = 0;
    uint32_t qf[C::KS][2];                // Q^T fragments (n = head r)
    float o[C::KS][4];                    // O^T accumulators, m-tile t of d
    float m_run[2], l_run[2];             // heads 2c, 2c+1
    const float scl = p.logit_scale_log2;
    bool bail = false;

    // Fused write + decode: when this stage holds the sequence's last token,
    // its rows in the stage are replaced by the step's new K and V (converted
    // exactly as paged_kv_write converts them), and the unit of the first
    // head set stores them to the cache slot.  Lanes 0..CPR-1 take 16-byte
    // chunks of the K row, CPR..2 CPR-1 those of the V row.
    auto patch_new_token = [&](uint32_t kb, uint32_t vb) {
        const int n = min(max(__ldg(p.context_lens + cu.s), 0), p.max_ctx);
        const int ts = cu.t0 + c_stage * kTok;
        const int tl = n - 1 - ts;
        if (n < 1 || n > cu.t1 || tl < 0 || tl >= kTok) return;
        const long long sn = __ldg(p.slot_mapping + cu.s);
        if (sn < 0 || sn >= (long long)p.NB * p.bs) return;
        constexpr int CPR = C::kRowBytes / 16;
        static_assert(2 * CPR <= 32, "one chunk per lane");
        if (lane < 2 * CPR) {
            const bool isv = lane >= CPR;
            const int j = lane % CPR;
            const void* src = isv ? p.new_v : p.new_k;
            uint4 chunk;
            float v[8];
            if constexpr (FP8) {
                const size_t e = ((size_t)cu.s * p.Hkv + cu.kvh) * D + 16 * (size_t)j;
                const float sc = isv ? p.v_scale : p.k_scale;
                if (p.new_dt == PKV_F32) load8<F32>(src, e, v); else load8<BF16>(src, e, v);
                const uint2 lo = pack8_e4m3(v, sc);
                if (p.new_dt == PKV_F32) load8<F32>(src, e + 8, v); else load8<BF16>(src, e + 8, v);
                const uint2 hi = pack8_e4m3(v, sc);
                chunk = make_uint4(lo.x, lo.y, hi.x, hi.y);
            } else {
                const size_t e = ((size_t)cu.s * p.Hkv + cu.kvh) * D + 8 * (size_t)j;
                if (p.new_dt == PKV_F32) load8<F32>(src, e, v); else load8<BF16>(src, e, v);
                chunk = pack8_bf16(v);
            }
            *reinterpret_cast<uint4*>(ws + (swz<C::kRowBytes, C::kTok>(isv ? vb : kb, tl, 16 * j) - ws_addr)) = chunk;
            if (cu.h0 == cu.kvh * p.g) {
                unsigned char* cache = static_cast<unsigned char*>(const_cast<void*>(isv ? p.vc : p.kc));
                *reinterpret_cast<uint4*>(cache + ((size_t)sn * p.Hkv + cu.kvh) * C::kRowBytes + 16 * j) = chunk;
            }
        }
        __syncwarp();
    };

    for (int i = 0; i < C::kStages; ++i)
        if (!issue_one()) break;

    for (;;) {
        if (!have_unit) {
            if (q_head == q_tail) break;
            __syncwarp();
            {
                const int4* e = reinterpret_cast<const int4*>(queue + q_head % C::kQueue);
                const int4 a = e[0], b2 = e[1];
                cu.s = a.x; cu.kvh = a.y; cu.h0 = a.z; cu.nh = a.w;
                cu.part = b2.x; cu.t0 = b2.y; cu.t1 = b2.z; cu.np = b2.w;
            }
            ++q_head;
            c_stage = 0;
            c_nst = (cu.t1 - cu.t0 + kTok - 1) / kTok;
            have_unit = true;
            need_q = true;
#pragma unroll
            for (int t = 0; t < C::KS; ++t) o[t][0] = o[t][1] = o[t][2] = o[t][3] = 0.f;
            m_run[0] = m_run[1] = -CUDART_INF_F;
            l_run[0] = l_run[1] = 0.f;
        }

        const int slot = g_cons % C::kStages;
        const uint32_t parity = (g_cons / C::kStages) & 1u;
        if (!mbar_try_wait(bar(slot), parity)) {
            const long long t_start = clock64();
            while (!mbar_try_wait(bar(slot), parity)) {
                if (clock64() - t_start > kWaitLimitCycles) {
                    report(p.err, PKV_DEVERR_TIMEOUT);
                    bail = true;
                    break;
                }
            }
        }
        if (__any_sync(0xffffffffu, bail)) break;
        if (need_q) {
            need_q = false;
            if constexpr (QF::bytes == 2) {
                // this unit's query is in qn (it is the oldest started unit); bf16 pairs as
                // they are, or widened and rounded to fp16 pairs for an E4M3 cache
#pragma unroll
                for (int ks = 0; ks < C::KS; ++ks)
#pragma unroll
                    for (int k = 0; k < 2; ++k) {
                        const uint32_t w = qn[ks][k];
                        qf[ks][k] = FP8 ? pack2<true>(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u)) : w;
                    }
                qn_for = -1;
                if (q_tail > q_head) {
                    // the next queued unit's query, loaded now to be ready at its start
                    const int4 a = reinterpret_cast<const int4*>(queue + q_head % C::kQueue)[0];
                    load_qn(a.x, a.z, a.w);
                    qn_for = (int)q_head;
                }
            } else {
                // an fp32 query: head r of the unit read at its start (zero past its heads)
                const bool hv = r < cu.nh;
                const unsigned char* qs = static_cast<const unsigned char*>(p.q) +
                                          ((size_t)cu.s * p.Hq + cu.h0 + (hv ? r : 0)) * D * QF::bytes;
#pragma unroll
                for (int ks = 0; ks < C::KS; ++ks) {
                    int d0, d1;
                    q_cols(ks, d0, d1);
                    float x0 = 0.f, x1 = 0.f, x2 = 0.f, x3 = 0.f;
                    if (hv) {
                        x0 = load_elem<QF>(qs, d0);
                        x1 = load_elem<QF>(qs, d0 + 1);
                        x2 = load_elem<QF>(qs, d1);
                        x3 = load_elem<QF>(qs, d1 + 1);
                    }
                    qf[ks][0] = pack2<FP8>(x0, x1);
                    qf[ks][1] = pack2<FP8>(x2, x3);
                }
            }
        }
        const uint32_t vmask = masks[slot];
        const uint32_t kb = stage_k(slot), vb = stage_v(slot);
        if constexpr (!TT) {
            if (p.new_k != nullptr) patch_new_token(kb, vb);
        }

        // ---- S^T = K . Q^T for the 16-token m-tiles of the stage
        float sacc[C::kMT][4];
#pragma unroll
        for (int mt = 0; mt < C::kMT; ++mt) {
            sacc[mt][0] = sacc[mt][1] = sacc[mt][2] = sacc[mt][3] = 0.f;
            if constexpr (FP8) {
                // rows of this lane: tokens pi(r) and pi(r+8) of the m-tile,
                // pi(2i+b) = 4i+b, pi(2i+8+b) = 4i+2+b
                const int ta = 16 * mt + 4 * (r >> 1) + (r & 1);
                const int tb = ta + 2;
                uint4 ka[D / 64], kbv[D / 64];
#pragma unroll
                for (int hh = 0; hh < D / 64; ++hh) {
                    ka[hh] = lds128(swz<C::kRowBytes, C::kTok>(kb, ta, 16 * c + 64 * hh));
                    kbv[hh] = lds128(swz<C::kRowBytes, C::kTok>(kb, tb, 16 * c + 64 * hh));
                }
#pragma unroll
                for (int hh = 0; hh < D / 64; ++hh) {
                    const uint32_t wa[4] = {ka[hh].x, ka[hh].y, ka[hh].z, ka[hh].w};
                    const uint32_t wb[4] = {kbv[hh].x, kbv[hh].y, kbv[hh].z, kbv[hh].w};
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int ks = 4 * hh + j;
                        uint32_t a01, a45, a23, a67;
                        e4m3x4_to_f16x2x2(wa[j], a01, a45);     // row r: d j=0,1 | j=2,3
                        e4m3x4_to_f16x2x2(wb[j], a23, a67);     // row r+8
                        mma16816<true>(sacc[mt], a01, a23, a45, a67, qf[ks][0], qf[ks][1]);
                    }
                }
            } else {
                const int mi = lane >> 3;
                const int tok = 16 * mt + 8 * (mi & 1) + (lane & 7);
#pragma unroll
                for (int ks = 0; ks < C::KS; ++ks) {
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4(swz<C::kRowBytes, C::kTok>(kb, tok, 32 * ks + 16 * (mi >> 1)), a0, a1, a2, a3);
                    mma16816<false>(sacc[mt], a0, a1, a2, a3, qf[ks][0], qf[ks][1]);
                }
            }
        }

        // ---- online softmax over the stage's tokens (log2 units)
        float x[C::kMT][4];
        float cmax0 = -CUDART_INF_F, cmax1 = -CUDART_INF_F;
#pragma unroll
        for (int mt = 0; mt < C::kMT; ++mt) {
            int ta, tb;
            if constexpr (FP8) {
                ta = 16 * mt + 4 * (r >> 1) + (r & 1);
                tb = ta + 2;
            } else {
                ta = 16 * mt + r;
                tb = ta + 8;
            }
            const bool va = (vmask >> ta) & 1u, vb2 = (vmask >> tb) & 1u;
            x[mt][0] = va ? sacc[mt][0] * scl : -CUDART_INF_F;
            x[mt][1] = va ? sacc[mt][1] * scl : -CUDART_INF_F;
            x[mt][2] = vb2 ? sacc[mt][2] * scl : -CUDART_INF_F;
            x[mt][3] = vb2 ? sacc[mt][3] * scl : -CUDART_INF_F;
            cmax0 = fmaxf(cmax0, fmaxf(x[mt][0], x[mt][2]));
            cmax1 = fmaxf(cmax1, fmaxf(x[mt][1], x[mt][3]));
        }
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            cmax0 = fmaxf(cmax0, __shfl_xor_sync(0xffffffffu, cmax0, off));
            cmax1 = fmaxf(cmax1, __shfl_xor_sync(0xffffffffu, cmax1, off));
        }
        const float mn0 = fmaxf(m_run[0], cmax0), mn1 = fmaxf(m_run[1], cmax1);
        const float mu0 = mn0 == -CUDART_INF_F ? 0.f : mn0;
        const float mu1 = mn1 == -CUDART_INF_F ? 0.f : mn1;
        const float al0 = fast_exp2(m_run[0] - mu0), al1 = fast_exp2(m_run[1] - mu1);
        m_run[0] = mn0;
        m_run[1] = mn1;
        float ls0 = 0.f, ls1 = 0.f;
        uint32_t pb[C::kMT][2];            // P^T B-fragments, one pair per 16-token k-tile
#pragma unroll
        for (int mt = 0; mt < C::kMT; ++mt) {
            const float p0 = fast_exp2(x[mt][0] - mu0), p1 = fast_exp2(x[mt][1] - mu1);
            const float p2 = fast_exp2(x[mt][2] - mu0), p3 = fast_exp2(x[mt][3] - mu1);
            ls0 += p0 + p2;
            ls1 += p1 + p3;
            pb[mt][0] = movmatrix_t(pack2<FP8>(p0, p1));
            pb[mt][1] = movmatrix_t(pack2<FP8>(p2, p3));
        }
        l_run[0] = l_run[0] * al0 + ls0;
        l_run[1] = l_run[1] * al1 + ls1;
#pragma unroll
        for (int t = 0; t < C::KS; ++t) {
            o[t][0] *= al0;
            o[t][1] *= al1;
            o[t][2] *= al0;
            o[t][3] *= al1;
        }

        // ---- O^T += V^T . P^T
        const bool full = vmask == (kTok == 32 ? 0xffffffffu : 0xffffu);
#pragma unroll
        for (int kt = 0; kt < C::kMT; ++kt) {
            if constexpr (FP8) {
                // this lane's tokens: 16kt + 4c + j, bytes [D/8 * r, D/8 * (r+1)) of each row
                uint32_t w[4][D / 32];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int tok = 16 * kt + 4 * c + j;
                    if constexpr (D == 128) {
                        const uint4 v4 = lds128(swz<C::kRowBytes, C::kTok>(vb, tok, 16 * r));
                        w[j][0] = v4.x; w[j][1] = v4.y; w[j][2] = v4.z; w[j][3] = v4.w;
                    } else {
                        const uint2 v2 = lds64(swz<C::kRowBytes, C::kTok>(vb, tok, 8 * r));
                        w[j][0] = v2.x; w[j][1] = v2.y;
                    }
                    if (!full && !((vmask >> tok) & 1u)) {
#pragma unroll
                        for (int q = 0; q < D / 32; ++q) w[j][q] = 0u;
                    }
                }
#pragma unroll
                for (int t = 0; t < C::KS; ++t) {
                    // d = (D/8) r + 2t (rows r) and +1 (rows r+8): byte 2t and 2t+1 of the lane's bytes
                    const int wi = t >> 1;
                    const uint32_t sel = (t & 1) ? 0x7362u : 0x5140u;
                    const uint32_t p01 = __byte_perm(w[0][wi], w[1][wi], sel);   // tokens 4c, 4c+1
                    const uint32_t p23 = __byte_perm(w[2][wi], w[3][wi], sel);   // tokens 4c+2, 4c+3
                    uint32_t a0, a1, a2, a3;
                    e4m3x4_to_f16x2x2(p01, a0, a1);          // d rows r | r+8, tokens 4c, 4c+1
                    e4m3x4_to_f16x2x2(p23, a2, a3);          // tokens 4c+2, 4c+3
                    mma16816<true>(o[t], a0, a1, a2, a3, pb[kt][0], pb[kt][1]);
                }
            } else {
                const int mi = lane >> 3;
                const int tok = 16 * kt + 8 * (mi >> 1) + (lane & 7);
                const int tk0 = 16 * kt + 2 * c;     // tokens of a0a1/a2a3: tk0, tk0+1; of a4a5/a6a7: +8
                const uint32_t keep01 = (vmask >> tk0) & 3u, keep89 = (vmask >> (tk0 + 8)) & 3u;
                const uint32_t mlo = (keep01 & 1u ? 0x0000ffffu : 0u) | (keep01 & 2u ? 0xffff0000u : 0u);
                const uint32_t mhi = (keep89 & 1u ? 0x0000ffffu : 0u) | (keep89 & 2u ? 0xffff0000u : 0u);
#pragma unroll
                for (int t = 0; t < C::KS; ++t) {
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4_t(swz<C::kRowBytes, C::kTok>(vb, tok, 32 * t + 16 * (mi & 1)), a0, a1, a2, a3);
                    if (!full) {
                        a0 &= mlo; a1 &= mlo; a2 &= mhi; a3 &= mhi;
                    }
                    mma16816<false>(o[t], a0, a1, a2, a3, pb[kt][0], pb[kt][1]);
                }
            }
        }

        // the slot is free again: let the issue side refill it
        __syncwarp();
        fence_proxy_async();
        ++g_cons;
        ++c_stage;
        issue_one();

        if (c_stage == c_nst) {
            // ---- finish the unit: full sums over the 8 lanes that share c
            float l0 = l_run[0], l1 = l_run[1];
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                l0 += __shfl_xor_sync(0xffffffffu, l0, off);
                l1 += __shfl_xor_sync(0xffffffffu, l1, off);
            }
            const int hA = 2 * c, hB = 2 * c + 1;
            const bool wA = hA < cu.nh, wB = hB < cu.nh;
            if (cu.np == 1) {
                const float fA = l0 > 0.f ? p.out_scale / l0 : 0.f;
                const float fB = l1 > 0.f ? p.out_scale / l1 : 0.f;
                const size_t oA = ((size_t)cu.s * p.Hq + cu.h0 + hA) * D, oB = oA + D;
#pragma unroll
                for (int t = 0; t < C::KS; ++t) {
                    int d0, d1;
                    if constexpr (FP8) { d0 = (D / 8) * r + 2 * t; d1 = d0 + 1; }
                    else { d0 = 16 * t + r; d1 = d0 + 8; }
                    if (wA) { store_out<QF>(p, oA + d0, o[t][0] * fA); store_out<QF>(p, oA + d1, o[t][2] * fA); }
                    if (wB) { store_out<QF>(p, oB + d0, o[t][1] * fB); store_out<QF>(p, oB + d1, o[t][3] * fB); }
                }
            } else {
                const uint64_t keep = l2_policy_evict_last();   // held in L2 until the merge reads it
                const size_t uA = ((size_t)cu.s * p.Hq + cu.h0 + hA) * p.Pmax + cu.part;
                const size_t uB = uA + p.Pmax;
#pragma unroll
                for (int t = 0; t < C::KS; ++t) {
                    int d0, d1;
                    if constexpr (FP8) { d0 = (D / 8) * r + 2 * t; d1 = d0 + 1; }
                    else { d0 = 16 * t + r; d1 = d0 + 8; }
                    if (wA) { st_l2_hint(p.part_acc + uA * D + d0, o[t][0], keep); st_l2_hint(p.part_acc + uA * D + d1, o[t][2], keep); }
                    if (wB) { st_l2_hint(p.part_acc + uB * D + d0, o[t][1], keep); st_l2_hint(p.part_acc + uB * D + d1, o[t][3], keep); }
                }
                if (r == 0) {
                    if (wA) { st_l2_hint(p.part_ml + 2 * uA, m_run[0], keep); st_l2_hint(p.part_ml + 2 * uA + 1, l0, keep); }
                    if (wB) { st_l2_hint(p.part_ml + 2 * uB, m_run[1], keep); st_l2_hint(p.part_ml + 2 * uB + 1, l1, keep); }
                }
            }
            have_unit = false;
        }
    }

    // copies of this lane still in flight land before the warp leaves
    if constexpr (TT) asm volatile("cp.async.wait_all;" ::: "memory");

    // ---- leave the scheduling counters at zero for the next launch
    if (p.sched != nullptr && lane == 0) {
        unsigned long long* ctr = reinterpret_cast<unsigned long long*>(p.sched);
        __threadfence();
        const unsigned long long done = atomicAdd(ctr + 1, 1ull);
        if (done == total_warps - 1) {
            atomicExch(ctr, 0ull);
            atomicExch(ctr + 1, 0ull);
        }
    }
}

// ------------------------------------------------------------- host side

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

// The cache [NB, bs, Hkv, d] as a 2-D tensor: rows = NB * bs tokens, row
// length = Hkv * d elements; a box is (one 128-byte half-row of one K/V
// head) x (min(bs, tokens per stage) consecutive tokens of one block).
template <int D, bool FP8>
bool encode_cache_map(CUtensorMap* map, const void* base, const DecodeParams& p) {
    using C = Cfg<D, FP8, 2>;
    auto fn = encode_fn();
    if (fn == nullptr) return false;
    const int esize = FP8 ? 1 : 2;
    const cuuint64_t dims[2] = {(cuuint64_t)p.Hkv * D, (cuuint64_t)p.NB * p.bs};
    const cuuint64_t strides[1] = {(cuuint64_t)p.Hkv * D * esize};
    const cuuint32_t box[2] = {(cuuint32_t)(C::kBoxRow / esize), (cuuint32_t)(p.bs < C::kTok ? p.bs : C::kTok)};
    const cuuint32_t estr[2] = {1, 1};
    const CUtensorMapSwizzle sw = C::kBoxRow == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    const CUresult rc = fn(map, FP8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                           const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return rc == CUDA_SUCCESS;
}

template <int D, bool FP8, typename QF, bool TT>
cudaError_t launch_one(const DecodeParams& p, int num_sms, cudaStream_t st) {
    using C = Cfg<D, FP8, QF::bytes>;
    auto kern = decode_tc_kernel<D, FP8, QF, TT>;
    static SmemOptIn optin;
    cudaError_t e = optin.ensure(reinterpret_cast<const void*>(kern), C::kSmemBytes);
    if (e != cudaSuccess) return e;
    CUtensorMap kmap, vmap;
    if (!encode_cache_map<D, FP8>(&kmap, p.kc, p) || !encode_cache_map<D, FP8>(&vmap, p.vc, p))
        return cudaErrorInvalidValue;
    const int nsets = (p.g + kHeadsPerUnit - 1) / kHeadsPerUnit;
    const unsigned long long per_part = (unsigned long long)p.S * p.Hkv * nsets;
    const unsigned long long region_a = (unsigned long long)(p.max_ctx / p.P) * per_part;   // full partitions
    const unsigned long long units = region_a + (unsigned long long)chunk_slots(p.P, p.Q, p.hold) * per_part;
    unsigned long long want = (units + C::kWarps - 1) / C::kWarps;
    int grid = (int)(want < (unsigned long long)num_sms ? want : (unsigned long long)num_sms);
    if (grid < 1) grid = 1;
    return launch_pdl(kern, dim3(grid), dim3(C::kWarps * 32), C::kSmemBytes, st, p, kmap, vmap, units, region_a,
                      nsets);
}

}  // namespace

bool decode_tc_supports(pkv_dtype q_dt, pkv_dtype c_dt, int d, int bs, int NB) {
    if (!(d == 64 || d == 128) || !(bs == 16 || bs == 32)) return false;
    if ((long long)NB * bs >= (1LL << 31)) return false;      // TMA row coordinates are 32-bit
    if (c_dt == PKV_BF16) return q_dt == PKV_BF16;
    return c_dt == PKV_FP8_E4M3 && (q_dt == PKV_BF16 || q_dt == PKV_F32);
}

template <bool TT>
cudaError_t launch_tc(const DecodeParams& p, pkv_dtype q_dt, pkv_dtype c_dt, int num_sms, cudaStream_t st) {
    if (c_dt == PKV_BF16)
        return p.d == 64 ? launch_one<64, false, BF16, TT>(p, num_sms, st)
                         : launch_one<128, false, BF16, TT>(p, num_sms, st);
    if (q_dt == PKV_BF16)
        return p.d == 64 ? launch_one<64, true, BF16, TT>(p, num_sms, st) : launch_one<128, true, BF16, TT>(p, num_sms, st);
    return p.d == 64 ? launch_one<64, true, F32, TT>(p, num_sms, st) : launch_one<128, true, F32, TT>(p, num_sms, st);
}

cudaError_t launch_decode_tc(const DecodeParams& p, pkv_dtype q_dt, pkv_dtype c_dt, int num_sms, cudaStream_t st,
                             bool token_table) {
    if (p.S == 0) return cudaSuccess;
    return token_table ? launch_tc<true>(p, q_dt, c_dt, num_sms, st) : launch_tc<false>(p, q_dt, c_dt, num_sms, st);
}

}  // namespace pkv
