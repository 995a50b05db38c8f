// Paged attention over query chunks (chunked prefill, speculative
// verification) on the fifth-generation tensor cores, two query tiles per
// unit: tcgen05.mma with the accumulators and the probabilities in tensor
// memory (TMEM).
//
// "LLM推論の基礎とvLLMの内部", section 6: chunked prefill computes a long
// prompt in per-step pieces next to other requests' decodes; section 3: the
// scheduler counts a request's tokens to compute, speculative ones included.
// Query i of a sequence's chunk of q_len (at position n - q_len + i) attends
// to tokens 0 .. n - q_len + i, read through the block table.
//
// Work unit: (sequence, K/V head, pair of tiles of 128 (query, head) rows,
// partition of P key tokens); one persistent CTA per SM claims units in
// order.  Both tiles of a unit read the same K/V stages.  Roles:
//   warp 8      K producer: claims units and streams 128-token K tiles into
//               a ring of shared-memory slots by TMA tensor copies (one box
//               per block and 64-value half row, 128-byte swizzle), with the
//               stage's token masks.  K_j's slot is released once both
//               tiles' S_j are done.
//   warp 11     V producer: the V tiles of the same units into their own
//               ring; V_j's slot is released once both P_j . V_j are done.
//   warp 10     Q loader: each tile's 128 rows of Q into that tile's buffer.
//   warp 9      one thread issues the MMAs, alternating between the tiles:
//                 S_t = Q_t . K_j^T      M 128, N 128, K d   (TMEM, one buffer per tile)
//                 O_t (+)= P_t . V_j     M 128, N d,   K 128 (A = P_t in TMEM)
//               in the order P_A.V_j, S_A(j+1), P_B.V_j, S_B(j+1): while one
//               tile's softmax runs, the tensor core works for the other.
//               P_t is written over S_t's columns, so S_t(j+1) is issued
//               only once P_t . V_j has completed.
//   warps 0-3   softmax of tile A, warps 4-7 of tile B, one thread per row
//               (TMEM lane): read S, causal mask, running maximum in base 2,
//               P = 2^(x - m) packed as bf16 over the first half of S's
//               columns, running sum; at the end O / l, or the partition's
//               (m, l, O).  Two groups keep two softmax warps on every SM
//               sub-partition, so one fills the other's waits.
// The reference maximum m of a row changes only when a stage's maximum
// exceeds it by more than 2^8; O and l are then rescaled (O in TMEM: the
// previous product has completed, since S of this stage was issued after
// it).  Every exponent stays <= 2^8, and the final O / l is the same softmax
// whatever reference was used.
#include <cuda.h>
#include <cuda_bf16.h>
#include <math_constants.h>

#include <mutex>

#include "pkv_common.cuh"
#include "pkv_internal.h"
#include "pkv_qtile.cuh"
#include "pkv_tc_common.cuh"
#include "pkv_umma.cuh"

namespace pkv {
namespace {

using namespace tc;

constexpr int kTok = 128;             // key tokens per stage
constexpr int kTileRows = 128;        // (query, head) rows per tile: M of both products
constexpr int kURows = 2 * kTileRows; // rows per unit
constexpr int kThreads = 384;
constexpr int kProducerWarp = 8, kMmaWarp = 9, kQWarp = 10, kVWarp = 11;
constexpr float kRescaleLog2 = 8.f;
constexpr long long kUWaitLimit = 4000000000LL;   // ~2 s: a barrier that never completes
constexpr uint32_t kTmemCols = 512;               // O_A 0, O_B 128, S_A 256, S_B 384
__host__ __device__ constexpr uint32_t tmem_o(int t) { return 128u * t; }
__host__ __device__ constexpr uint32_t tmem_s(int t) { return 256u + 128u * t; }
// Registers: the kernel is launched with kThreads x kLaunchRegs; each
// softmax warpgroup raises its warps to kSoftmaxRegs, the other warpgroup
// lowers its to kOtherRegs.  The shares add up to the launch's total.
constexpr int kLaunchRegs = 168, kSoftmaxRegs = 200, kOtherRegs = 96;
static_assert(256 * kSoftmaxRegs + 128 * kOtherRegs <= kThreads * kLaunchRegs, "register split");

template <int D>
struct UCfg {
    static constexpr int kHalves = D / 64;                 // 128-byte halves of a Q/K/V row
    static constexpr int kItemBytes = kTok * 2 * D;        // one K or V tile of a stage
    static constexpr int kKItems = D == 128 ? 3 : 4;       // ring of K tiles
    static constexpr int kVItems = D == 128 ? 2 : 4;       // ring of V tiles
    static constexpr int kQBytes = kTileRows * 2 * D;      // one tile of Q
    static constexpr int kVOff = kKItems * kItemBytes;
    static constexpr int kQOff = (kKItems + kVItems) * kItemBytes;
    static constexpr int kCtlOff = kQOff + 2 * kQBytes;
    static constexpr int kCtlBytes = 1024;
    static constexpr int kSmemBytes = kCtlOff + kCtlBytes + 1024;
    static constexpr int KS = D / 16;
    static_assert(kSmemBytes <= 232448, "shared memory per CTA");
};

// control block (byte offsets): mbarriers, then the TMEM slot, the abort
// flag, the token masks of four stages and the ring of two unit records
constexpr uint32_t kBarKFull = 0;         // [4]
constexpr uint32_t kBarKEmpty = 32;       // [4]
constexpr uint32_t kBarVFull = 64;        // [4]
constexpr uint32_t kBarVEmpty = 96;       // [4]
constexpr uint32_t kBarSFull = 128;       // [2 tiles]: S_t of the tile's stage done
constexpr uint32_t kBarPFull = 144;       // [2 tiles]: P_t written (4 warps)
constexpr uint32_t kBarPVDone = 160;      // [2 tiles]: P_t . V done (O_t holds every product so far)
constexpr uint32_t kBarFin = 176;
constexpr uint32_t kBarQFull = 184;       // [2 tiles]
constexpr uint32_t kBarQEmpty = 200;      // [2 tiles]
constexpr uint32_t kBarUFull = 216;       // [2]
constexpr uint32_t kBarUEmpty = 232;      // [2]
constexpr uint32_t kBarMaskFull = 248;    // [4]: masks of stage g published (slot g % 4)
constexpr uint32_t kBarMaskEmpty = 280;   // [4]: masks of stage g read by the eight softmax warps
constexpr uint32_t kTmemSlot = 312, kAbort = 316, kMasks = 320 /* [4][4] words */, kRing = 384 /* [2][4] int4 */;
static_assert(kRing + 128 <= 1024, "control block");

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint4 v) {
    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}
// D[tmem] (+)= A[tmem] . B[smem]: the A operand read from tensor memory
__device__ __forceinline__ void mma_bf16_ts(uint32_t tmem_d, uint32_t tmem_a, uint64_t b, uint32_t idesc,
                                            bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(tmem_d),
        "r"(tmem_a), "l"(b), "r"(idesc), "r"(accumulate ? 1u : 0u));
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_umma2_kernel(const __grid_constant__ DecodeParams p, const int32_t* __restrict__ query_start, int T,
                         int max_q, const __grid_constant__ CUtensorMap kmap,
                         const __grid_constant__ CUtensorMap vmap, unsigned long long total_units, int rt_max) {
    using C = UCfg<D>;
    constexpr int NK = C::kKItems, NV = C::kVItems;
    static_assert(NK <= 4 && NV <= 4, "barrier slots");
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const uint32_t raw_addr = smem_addr(smem_raw);
    const uint32_t base = (raw_addr + 1023u) & ~1023u;
    unsigned char* smem = smem_raw + (base - raw_addr);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t ctl = base + C::kCtlOff;
    unsigned char* ctlp = smem + C::kCtlOff;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(ctlp + kAbort);
    uint32_t* masks = reinterpret_cast<uint32_t*>(ctlp + kMasks);      // [4 stages][4 words]: tokens present
    int4* ring = reinterpret_cast<int4*>(ctlp + kRing);                // [2 units][4 int4]
    auto ktile = [&](uint32_t j) { return base + (j % NK) * C::kItemBytes; };
    auto vtile = [&](uint32_t j) { return base + C::kVOff + (j % NV) * C::kItemBytes; };
    auto qbuf = [&](int t) { return base + C::kQOff + t * C::kQBytes; };
    auto bar = [&](uint32_t off, int i) { return ctl + off + 8 * i; };
    // the partition merge that may follow can be scheduled now; it waits for this grid's results
    asm volatile("griddepcontrol.launch_dependents;");

    if (tid == 0) {
        for (int i = 0; i < NK; ++i) {
            mbar_init(bar(kBarKFull, i), 1);
            mbar_init(bar(kBarKEmpty, i), 1);
        }
        for (int i = 0; i < NV; ++i) {
            mbar_init(bar(kBarVFull, i), 1);
            mbar_init(bar(kBarVEmpty, i), 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(bar(kBarSFull, t), 1);
            mbar_init(bar(kBarPFull, t), 4);
            mbar_init(bar(kBarPVDone, t), 1);
            mbar_init(bar(kBarQFull, t), 1);
            mbar_init(bar(kBarQEmpty, t), 1);
            mbar_init(bar(kBarUFull, t), 1);
            mbar_init(bar(kBarUEmpty, t), 11);   // V producer, Q loader, MMA, eight softmax warps
        }
        for (int i = 0; i < 4; ++i) {
            mbar_init(bar(kBarMaskFull, i), 1);
            mbar_init(bar(kBarMaskEmpty, i), 8);
        }
        mbar_init(bar(kBarFin, 0), 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == kMmaWarp) umma::tmem_alloc(ctl + kTmemSlot, kTmemCols);
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(ctlp + kTmemSlot);

    // bounded wait; false once the limit passes or another role gave up
    auto wait = [&](uint32_t b, uint32_t parity, bool abortable) -> bool {
        if (mbar_try_wait(b, parity)) return true;
        const long long t0 = clock64();
        while (!mbar_try_wait(b, parity)) {
            if (abortable && *abort_flag) return false;
            if (clock64() - t0 > kUWaitLimit) {
                report(p.err, PKV_DEVERR_TIMEOUT);
                *abort_flag = 1;
                return false;
            }
        }
        return true;
    };
    // A parity wait is exact only while the barrier is within one phase of
    // the awaited one, neither behind nor ahead; every wait below has that
    // bound by construction.  K_j sits in slot j % NK of the K ring (phase
    // j / NK), V_j in slot j % NV of the V ring (j counted over the CTA's
    // stages); the per-tile barriers count the stages that tile took part in.

    if (warp == kProducerWarp) {
        // ------------------------------------------------------------ producer
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kOtherRegs));
        unsigned long long static_next = blockIdx.x;
        uint32_t g = 0, un = 0;
        const uint32_t box_bytes = (uint32_t)(p.bs < 32 ? p.bs : 32) * 128u;
        bool ok = true, bad = false;          // bad: warp-uniform
        for (;;) {
            QTile x;
            bool have = false;
            for (;;) {
                unsigned long long v = 0;
                if (lane == 0)
                    v = p.sched != nullptr ? atomicAdd(reinterpret_cast<unsigned long long*>(p.sched), 1ull)
                                           : static_next;
                v = __shfl_sync(0xffffffffu, v, 0);
                static_next += gridDim.x;
                if (v >= total_units) break;
                if (qtile_of<kURows>(p, query_start, T, max_q, v, rt_max, x)) {
                    have = true;
                    break;
                }
            }
            const int slot = un & 1;
            if (un >= 2) ok = wait(bar(kBarUEmpty, slot), ((un >> 1) - 1) & 1, true);
            if (__any_sync(0xffffffffu, !ok)) break;
            if (lane == 0) {
                int4* e = ring + 4 * slot;
                if (have) {
                    e[0] = make_int4(x.s, x.kvh, x.rt, x.part);
                    e[1] = make_int4(x.k0, x.k1, x.n, x.ql);
                    e[2] = make_int4(x.q0, x.np, x.rows, 1);
                } else {
                    e[2] = make_int4(0, 0, 0, 0);
                }
                umma::mbar_arrive(bar(kBarUFull, slot));
            }
            if (!have) break;

            // K tiles; block-table entries come 32 at a time, one chunk ahead
            const int nst = (x.k1 - x.k0 + kTok - 1) / kTok;
            const int bps = kTok / p.bs;                      // blocks per stage: 8 or 4
            const int unit_blocks = (x.k1 - x.k0 + p.bs - 1) / p.bs;
            const int32_t* trow = p.block_tables + (size_t)x.s * p.MB + x.k0 / p.bs;
            auto load_chunk = [&](int c) -> int {
                const int rb = 32 * c + lane;
                return rb < unit_blocks ? __ldg(trow + rb) : 0;
            };
            int tab = load_chunk(0), tab_next = load_chunk(1), tab_chunk = 0;
            for (int j = 0; j < nst; ++j) {
                const uint32_t gs = g + j;
                const int ts = x.k0 + j * kTok;
                const int tn = min(kTok, x.k1 - ts);
                const int nb = (tn + p.bs - 1) / p.bs;
                const int idx0 = j * bps;
                if ((idx0 >> 5) != tab_chunk) {
                    tab_chunk = idx0 >> 5;
                    tab = tab_next;
                    tab_next = load_chunk(tab_chunk + 1);
                }
                const int pb = __shfl_sync(0xffffffffu, tab, (idx0 + (lane & (bps - 1))) & 31);
                const bool bok = lane < nb && pb >= 0 && pb < p.NB;
                if (lane < nb && !bok) report(p.err, PKV_DEVERR_BLOCK_ID);
                const uint32_t bm = __ballot_sync(0xffffffffu, bok);
                const uint32_t kslot = gs % NK, kph = gs / NK;
                if (kph >= 1) ok = wait(bar(kBarKEmpty, kslot), (kph - 1) & 1, true);
                if (gs >= 4) ok = ok && wait(bar(kBarMaskEmpty, gs & 3), ((gs >> 2) - 1) & 1, true);
                if (__any_sync(0xffffffffu, !ok)) {
                    bad = true;
                    break;
                }
                if (lane < 4) {
                    // tokens 32 lane .. 32 lane + 31: present where their block is valid and t < tn
                    uint32_t w;
                    if (p.bs == 16) {
                        const uint32_t b2 = (bm >> (2 * lane)) & 3u;
                        w = ((b2 & 1u) ? 0x0000ffffu : 0u) | ((b2 & 2u) ? 0xffff0000u : 0u);
                    } else {
                        w = ((bm >> lane) & 1u) ? 0xffffffffu : 0u;
                    }
                    const int lo = 32 * lane;
                    const uint32_t tm = tn >= lo + 32 ? 0xffffffffu : (tn <= lo ? 0u : ((1u << (tn - lo)) - 1u));
                    masks[4 * (gs & 3) + lane] = w & tm;
                }
                __syncwarp();
                if (lane == 0) umma::mbar_arrive(bar(kBarMaskFull, gs & 3));
                const int bi = lane / C::kHalves, h = lane % C::kHalves;
                const int pbb = __shfl_sync(0xffffffffu, pb, bi & 31);
                const bool live = bi < nb && ((bm >> bi) & 1u);
                const uint32_t nlive = __popc(__ballot_sync(0xffffffffu, live));
                const uint32_t full = bar(kBarKFull, kslot);
                if (lane == 0) mbar_arrive_expect_tx(full, nlive * box_bytes);
                __syncwarp();
                if (live)
                    tensor_load_2d(ktile(gs) + h * (kTok * 128) + bi * p.bs * 128, &kmap, x.kvh * D + h * 64,
                                   pbb * p.bs, full);
            }
            g += nst;
            if (bad) break;
            ++un;
        }
        // copies still in flight land before the CTA leaves
        for (uint32_t k = 1; k <= (uint32_t)NK && k <= g; ++k)
            wait(bar(kBarKFull, (g - k) % NK), ((g - k) / NK) & 1, false);
        if (p.sched != nullptr && lane == 0) {
            unsigned long long* ctr = reinterpret_cast<unsigned long long*>(p.sched);
            __threadfence();
            const unsigned long long done = atomicAdd(ctr + 1, 1ull);
            if (done == gridDim.x - 1) {
                atomicExch(ctr, 0ull);
                atomicExch(ctr + 1, 0ull);
            }
        }
    } else if (warp == kVWarp) {
        // ---------------------------------------------------------- V producer
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kOtherRegs));
        // follows the units the K producer publishes; V_j waits only for the
        // products of stage j - NV to free its slot
        uint32_t g = 0, un = 0;
        const uint32_t box_bytes = (uint32_t)(p.bs < 32 ? p.bs : 32) * 128u;
        bool ok = true, bad = false;          // bad: warp-uniform
        for (;;) {
            const int slot = un & 1;
            ok = wait(bar(kBarUFull, slot), (un >> 1) & 1, true);
            if (__any_sync(0xffffffffu, !ok)) break;
            const int4 e0 = ring[4 * slot], e1 = ring[4 * slot + 1], e2 = ring[4 * slot + 2];
            __syncwarp();
            if (lane == 0) umma::mbar_arrive(bar(kBarUEmpty, slot));
            if (e2.w == 0) break;
            const int us = e0.x, kvh = e0.y, k0 = e1.x, k1 = e1.y;
            const int nst = (k1 - k0 + kTok - 1) / kTok;
            const int bps = kTok / p.bs;
            const int unit_blocks = (k1 - k0 + p.bs - 1) / p.bs;
            const int32_t* trow = p.block_tables + (size_t)us * p.MB + k0 / p.bs;
            auto load_chunk = [&](int c) -> int {
                const int rb = 32 * c + lane;
                return rb < unit_blocks ? __ldg(trow + rb) : 0;
            };
            int tab = load_chunk(0), tab_next = load_chunk(1), tab_chunk = 0;
            for (int j = 0; j < nst; ++j, ++g) {
                const int tn = min(kTok, k1 - (k0 + j * kTok));
                const int nb = (tn + p.bs - 1) / p.bs;
                const int idx0 = j * bps;
                if ((idx0 >> 5) != tab_chunk) {
                    tab_chunk = idx0 >> 5;
                    tab = tab_next;
                    tab_next = load_chunk(tab_chunk + 1);
                }
                const int pb = __shfl_sync(0xffffffffu, tab, (idx0 + (lane & (bps - 1))) & 31);
                const bool bok = lane < nb && pb >= 0 && pb < p.NB;     // reported by the K producer
                const uint32_t bm = __ballot_sync(0xffffffffu, bok);
                if (g >= (uint32_t)NV) ok = wait(bar(kBarVEmpty, g % NV), ((g / NV) - 1) & 1, true);
                if (__any_sync(0xffffffffu, !ok)) {
                    bad = true;
                    break;
                }
                const int bi = lane / C::kHalves, h = lane % C::kHalves;
                const int pbb = __shfl_sync(0xffffffffu, pb, bi & 31);
                const bool live = bi < nb && ((bm >> bi) & 1u);
                const uint32_t nlive = __popc(__ballot_sync(0xffffffffu, live));
                const uint32_t full = bar(kBarVFull, g % NV);
                if (lane == 0) mbar_arrive_expect_tx(full, nlive * box_bytes);
                __syncwarp();
                if (live)
                    tensor_load_2d(vtile(g) + h * (kTok * 128) + bi * p.bs * 128, &vmap, kvh * D + h * 64, pbb * p.bs,
                                   full);
            }
            if (bad) break;
            ++un;
        }
        for (uint32_t k = 1; k <= (uint32_t)NV && k <= g; ++k)
            wait(bar(kBarVFull, (g - k) % NV), ((g - k) / NV) & 1, false);
    } else if (warp == kQWarp) {
        // ------------------------------------------------------------ Q loader
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kOtherRegs));
        // tile t's buffer is refilled once the unit that used it has issued its last S_t
        uint32_t un = 0, qu[2] = {0u, 0u};
        bool ok = true, bad = false;
        const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(p.q);
        for (;;) {
            const int slot = un & 1;
            ok = wait(bar(kBarUFull, slot), (un >> 1) & 1, true);
            if (__any_sync(0xffffffffu, !ok)) break;
            const int4 e0 = ring[4 * slot], e2 = ring[4 * slot + 2];
            __syncwarp();
            if (lane == 0) umma::mbar_arrive(bar(kBarUEmpty, slot));
            if (e2.w == 0) break;
            const int kvh = e0.y, rt = e0.z, q0 = e2.x, rows = e2.z;
            for (int t = 0; t < 2; ++t) {
                const int r0 = rt * kURows + t * kTileRows;
                if (r0 >= rows) break;                   // the unit's second tile is empty
                if (qu[t] >= 1) ok = wait(bar(kBarQEmpty, t), (qu[t] - 1) & 1, true);
                if (__any_sync(0xffffffffu, !ok)) {
                    bad = true;
                    break;
                }
                constexpr int CH = 2 * D / 16;           // 16-byte chunks per row
                constexpr int kBatch = 16;               // loads in flight per lane
                static_assert((kTileRows * CH / 32) % kBatch == 0, "Q load batches");
                const int rows_here = min(kTileRows, rows - r0);
                const uint32_t qdst = qbuf(t);
                for (int it0 = 0; it0 < kTileRows * CH / 32; it0 += kBatch) {
                    uint4 v[kBatch];
#pragma unroll
                    for (int k = 0; k < kBatch; ++k) {
                        const int idx = (it0 + k) * 32 + lane;
                        const int r = idx / CH, c = idx % CH;
                        v[k] = make_uint4(0u, 0u, 0u, 0u);
                        if (r < rows_here) {
                            const int row = r0 + r;
                            const int qi = row / p.g, hh = row - qi * p.g;
                            const size_t off = ((size_t)(q0 + qi) * p.Hq + kvh * p.g + hh) * D + c * 8;
                            v[k] = __ldg(reinterpret_cast<const uint4*>(q + off));
                        }
                    }
#pragma unroll
                    for (int k = 0; k < kBatch; ++k) {
                        const int idx = (it0 + k) * 32 + lane;
                        const int r = idx / CH, c = idx % CH;
                        st_shared_v4(qdst + (c >> 3) * (kTileRows * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4), v[k]);
                    }
                }
                fence_proxy_async();
                __syncwarp();
                if (lane == 0) umma::mbar_arrive(bar(kBarQFull, t));
                ++qu[t];
            }
            if (bad) break;
            ++un;
        }
    } else if (warp == kMmaWarp) {
        // ---------------------------------------------------------- MMA issue
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kOtherRegs));
        if (lane == 0) {
            constexpr uint32_t idS = umma::idesc_bf16_f32(kTileRows, kTok, false);
            constexpr uint32_t idPV = umma::idesc_bf16_f32(kTileRows, D, true);
            uint32_t g = 0, un = 0, gt[2] = {0u, 0u}, qu[2] = {0u, 0u};
            bool ok = true;
            // S_t = Q_t . K_gs^T into tile t's S buffer
            auto issue_s = [&](int t, uint32_t gs) {
                const uint32_t kb = ktile(gs);
#pragma unroll
                for (int kk = 0; kk < C::KS; ++kk) {
                    const uint64_t a = umma::desc_sw128(qbuf(t) + (kk >> 2) * (kTileRows * 128) + (kk & 3) * 32, 16, 1024);
                    const uint64_t bd = umma::desc_sw128(kb + (kk >> 2) * (kTok * 128) + (kk & 3) * 32, 16, 1024);
                    umma::mma_bf16(tmem + tmem_s(t), a, bd, idS, kk > 0);
                }
                umma::commit(bar(kBarSFull, t));
            };
            // O_t (+)= P_t . V_gs, P_t read from the first half of the S buffer's columns
            auto issue_pv = [&](int t, uint32_t gs, bool first) {
                const uint32_t vb = vtile(gs);
#pragma unroll
                for (int kk = 0; kk < kTok / 16; ++kk) {
                    const uint64_t bd = umma::desc_sw128(vb + kk * 2048, kTok * 128, 1024);
                    mma_bf16_ts(tmem + tmem_o(t), tmem + tmem_s(t) + kk * 8, bd, idPV, !(first && kk == 0));
                }
                umma::commit(bar(kBarPVDone, t));
            };
            for (;;) {
                const int slot = un & 1;
                if (!wait(bar(kBarUFull, slot), (un >> 1) & 1, true)) break;
                const int4 e0 = ring[4 * slot], e1 = ring[4 * slot + 1], e2 = ring[4 * slot + 2];
                umma::mbar_arrive(bar(kBarUEmpty, slot));
                if (e2.w == 0) break;
                const int nst = (e1.y - e1.x + kTok - 1) / kTok;
                const int nt = e0.z * kURows + kTileRows < e2.z ? 2 : 1;      // tiles with rows
                for (int t = 0; t < nt && ok; ++t) ok = wait(bar(kBarQFull, t), qu[t] & 1, true);
                // stage 0: each tile's S, once the tile's previous P . V has read its buffer
                ok = ok && wait(bar(kBarKFull, g % NK), (g / NK) & 1, true);
                for (int t = 0; t < nt && ok; ++t) {
                    if (gt[t] > 0) ok = wait(bar(kBarPVDone, t), (gt[t] - 1) & 1, true);
                    if (!ok) break;
                    umma::fence_after_sync();
                    issue_s(t, g);
                    if (nst == 1) umma::commit(bar(kBarQEmpty, t));
                }
                if (!ok) break;
                umma::commit(bar(kBarKEmpty, g % NK));
                for (int j = 0; j < nst && ok; ++j) {
                    const uint32_t gs = g + j;
                    ok = wait(bar(kBarVFull, gs % NV), (gs / NV) & 1, true);
                    for (int t = 0; t < nt && ok; ++t) {
                        ok = wait(bar(kBarPFull, t), gt[t] & 1, true);
                        if (!ok) break;
                        umma::fence_after_sync();
                        issue_pv(t, gs, j == 0);
                        if (j + 1 < nst) {
                            // the next stage's S_t overwrites P_t: only after P_t . V_gs is done
                            if (t == 0) ok = wait(bar(kBarKFull, (gs + 1) % NK), ((gs + 1) / NK) & 1, true);
                            ok = ok && wait(bar(kBarPVDone, t), gt[t] & 1, true);
                            if (!ok) break;
                            umma::fence_after_sync();
                            issue_s(t, gs + 1);
                            if (j + 2 == nst) umma::commit(bar(kBarQEmpty, t));
                        }
                        ++gt[t];
                    }
                    if (!ok) break;
                    umma::commit(bar(kBarVEmpty, gs % NV));
                    if (j + 1 < nst) umma::commit(bar(kBarKEmpty, (gs + 1) % NK));
                }
                if (!ok) break;
                g += nst;
                for (int t = 0; t < nt; ++t) ++qu[t];
                ++un;
            }
            // every product issued here completes before the CTA releases TMEM
            umma::commit(bar(kBarFin, 0));
            wait(bar(kBarFin, 0), 0, false);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------- softmax
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kSoftmaxRegs));
        const int t = warp >> 2;                              // tile of this warp group
        const int i = tid & (kTileRows - 1);                  // row of the tile, TMEM lane
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t s_col = tmem_s(t), o_col = tmem_o(t);
        const float scl = p.logit_scale_log2;
        uint32_t g = 0, gt = 0, un = 0;
        bool ok = true, bad = false;          // bad: warp-uniform
        for (;;) {
            const int slot = un & 1;
            ok = wait(bar(kBarUFull, slot), (un >> 1) & 1, true);
            if (__any_sync(0xffffffffu, !ok)) break;
            const int4 e0 = ring[4 * slot], e1 = ring[4 * slot + 1], e2 = ring[4 * slot + 2];
            __syncwarp();
            if (lane == 0) umma::mbar_arrive(bar(kBarUEmpty, slot));
            if (e2.w == 0) break;
            const int kvh = e0.y, rt = e0.z, part = e0.w, k0 = e1.x, k1 = e1.y, n = e1.z, ql = e1.w;
            const int q0 = e2.x, np = e2.y, rows = e2.z;
            const int nst = (k1 - k0 + kTok - 1) / kTok;
            const int r0 = rt * kURows + t * kTileRows;
            if (r0 >= rows) {
                // this tile has no rows in the unit: only hand the stages' masks back
                for (int j = 0; j < nst; ++j, ++g) {
                    ok = wait(bar(kBarMaskFull, g & 3), (g >> 2) & 1, true);
                    if (__any_sync(0xffffffffu, !ok)) {
                        bad = true;
                        break;
                    }
                    __syncwarp();
                    if (lane == 0) umma::mbar_arrive(bar(kBarMaskEmpty, g & 3));
                }
                if (bad) break;
                ++un;
                continue;
            }
            const int row = r0 + i;
            const bool rv = row < rows;
            const int qi = rv ? row / p.g : 0;
            const int hh = rv ? row - qi * p.g : 0;
            const int pos = rv ? n - ql + qi : -1;
            float m_ref = -CUDART_INF_F, l = 0.f;
            for (int j = 0; j < nst; ++j, ++g, ++gt) {
                // S of this stage done (so the previous P . V is done too), and the token masks published
                ok = wait(bar(kBarSFull, t), gt & 1, true) && wait(bar(kBarMaskFull, g & 3), (g >> 2) & 1, true);
                if (__any_sync(0xffffffffu, !ok)) {
                    bad = true;
                    break;
                }
                umma::fence_after_sync();
                const int lim = pos - (k0 + j * kTok);           // tokens t <= lim are visible to this row
                uint32_t mw[4];
#pragma unroll
                for (int qq = 0; qq < 4; ++qq) mw[qq] = masks[4 * (g & 3) + qq];
                __syncwarp();
                if (lane == 0) umma::mbar_arrive(bar(kBarMaskEmpty, g & 3));
                const bool all_present = (mw[0] & mw[1] & mw[2] & mw[3]) == 0xffffffffu;
                // rows past the tile's last take the same path: their output is never stored
                const bool whole = ((lim >= kTok - 1 && all_present) || !rv) && scl > 0.f;
                uint32_t sr[4][32];
#pragma unroll
                for (int qq = 0; qq < 4; ++qq) umma::tmem_ld32(tmem + lane_base + s_col + 32 * qq, sr[qq]);
                umma::tmem_wait_ld();
                float mx8[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) mx8[k] = -CUDART_INF_F;
                if (whole) {                 // every token present and visible: max of the raw logits
#pragma unroll
                    for (int qq = 0; qq < 4; ++qq)
#pragma unroll
                        for (int bb = 0; bb < 32; ++bb) mx8[bb & 7] = fmaxf(mx8[bb & 7], __uint_as_float(sr[qq][bb]));
#pragma unroll
                    for (int k = 0; k < 8; ++k) mx8[k] *= scl;
                } else {
#pragma unroll
                    for (int qq = 0; qq < 4; ++qq)
#pragma unroll
                        for (int bb = 0; bb < 32; ++bb) {
                            const bool live = ((mw[qq] >> bb) & 1u) && (32 * qq + bb) <= lim;
                            const float xv = live ? __uint_as_float(sr[qq][bb]) * scl : -CUDART_INF_F;
                            sr[qq][bb] = __float_as_uint(xv);
                            mx8[bb & 7] = fmaxf(mx8[bb & 7], xv);
                        }
                }
                const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                                       fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
                float alpha = 1.f;
                bool resc = false;
                if (j == 0) {
                    m_ref = mx;
                } else if (mx > m_ref + kRescaleLog2) {
                    if (m_ref != -CUDART_INF_F) {
                        alpha = fast_exp2(m_ref - mx);
                        resc = true;
                    }
                    m_ref = mx;
                }
                l *= alpha;
                // V rows of tokens that were not loaded are zeroed (0 * stale data could be NaN);
                // the first tile's group does it for both, before either product reads V
                if (t == 0 && !__all_sync(0xffffffffu, all_present)) {
                    ok = wait(bar(kBarVFull, g % NV), (g / NV) & 1, true);
                    if (__any_sync(0xffffffffu, !ok)) {
                        bad = true;
                        break;
                    }
                    if (!((mw[i >> 5] >> (i & 31)) & 1u)) {
                        const uint32_t vb = vtile(g);
#pragma unroll
                        for (int h = 0; h < C::kHalves; ++h)
#pragma unroll
                            for (int c = 0; c < 8; ++c)
                                st_shared_v4(vb + h * (kTok * 128) + i * 128 + c * 16, make_uint4(0u, 0u, 0u, 0u));
                    }
                    fence_proxy_async();
                }
                // P row: 2^(x - m) as bf16 pairs over columns 0..63 of the S buffer; on the
                // fast path x = scl * s enters through one fused multiply-add
                const float mb = m_ref == -CUDART_INF_F ? 0.f : m_ref;
                const float xs = whole ? scl : 1.f;
                // pairs of columns through paired fp32 instructions: the same roundings
                // and the same eight partial sums as one scalar lane at a time
                const uint64_t xs2 = umma::f2_pack(xs, xs), nmb2 = umma::f2_pack(-mb, -mb);
                uint64_t ls2[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
                for (int hq = 0; hq < 2; ++hq) {
                    uint32_t pw[32];
#pragma unroll
                    for (int k = 0; k < 32; ++k) {
                        const int tt = 64 * hq + 2 * k;
                        const uint64_t s01 = umma::f2_pack(__uint_as_float(sr[tt >> 5][tt & 31]),
                                                           __uint_as_float(sr[(tt + 1) >> 5][(tt + 1) & 31]));
                        float x0, x1;
                        umma::f2_unpack(umma::f2_fma(s01, xs2, nmb2), x0, x1);
                        const float a0 = fast_exp2(x0), a1 = fast_exp2(x1);
                        ls2[k & 3] = umma::f2_add(ls2[k & 3], umma::f2_pack(a0, a1));
                        pw[k] = pack2<false>(a0, a1);
                    }
                    umma::tmem_st32(tmem + lane_base + s_col + 32 * hq, pw);
                }
                float ls[8];
#pragma unroll
                for (int k = 0; k < 4; ++k) umma::f2_unpack(ls2[k], ls[2 * k], ls[2 * k + 1]);
                l += ((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7]));
                if (__any_sync(0xffffffffu, resc)) {
                    // O_t holds the products up to the previous stage: scale it in place (after P,
                    // when the logits are no longer needed, and before P_t . V reads it)
#pragma unroll
                    for (int c0 = 0; c0 < D / 32; ++c0) {
                        uint32_t ov[32];
                        umma::tmem_ld32(tmem + lane_base + o_col + 32 * c0, ov);
                        umma::tmem_wait_ld();
#pragma unroll
                        for (int k = 0; k < 32; ++k) ov[k] = __float_as_uint(__uint_as_float(ov[k]) * alpha);
                        umma::tmem_st32(tmem + lane_base + o_col + 32 * c0, ov);
                    }
                }
                umma::tmem_wait_st();
                umma::fence_before_sync();
                __syncwarp();
                if (lane == 0) umma::mbar_arrive(bar(kBarPFull, t));
            }
            if (bad) break;

            // epilogue: O / l, or the partition's (m, l, O), once the tile's last product is done
            ok = wait(bar(kBarPVDone, t), (gt - 1) & 1, true);
            if (__any_sync(0xffffffffu, !ok)) break;
            umma::fence_after_sync();
            const size_t hrow = (size_t)(q0 + qi) * p.Hq + kvh * p.g + hh;
            const float f = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
            for (int c0 = 0; c0 < D / 32; ++c0) {
                uint32_t ov[32];
                umma::tmem_ld32(tmem + lane_base + o_col + 32 * c0, ov);
                umma::tmem_wait_ld();
                if (!rv) continue;
                if (np == 1) {
                    uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + hrow * D + 32 * c0);
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        dst[k] = make_uint4(pack2<false>(__uint_as_float(ov[8 * k]) * f, __uint_as_float(ov[8 * k + 1]) * f),
                                            pack2<false>(__uint_as_float(ov[8 * k + 2]) * f, __uint_as_float(ov[8 * k + 3]) * f),
                                            pack2<false>(__uint_as_float(ov[8 * k + 4]) * f, __uint_as_float(ov[8 * k + 5]) * f),
                                            pack2<false>(__uint_as_float(ov[8 * k + 6]) * f, __uint_as_float(ov[8 * k + 7]) * f));
                } else {
                    uint4* dst = reinterpret_cast<uint4*>(p.part_acc + (hrow * p.Pmax + part) * D + 32 * c0);
#pragma unroll
                    for (int k = 0; k < 8; ++k) dst[k] = make_uint4(ov[4 * k], ov[4 * k + 1], ov[4 * k + 2], ov[4 * k + 3]);
                }
            }
            if (rv && np > 1) {
                const size_t u = hrow * p.Pmax + part;
                p.part_ml[2 * u] = m_ref;
                p.part_ml[2 * u + 1] = l;
            }
            umma::fence_before_sync();
            ++un;
        }
    }

    umma::fence_before_sync();
    __syncthreads();
    if (warp == kMmaWarp) {
        umma::fence_after_sync();
        umma::tmem_dealloc(tmem, kTmemCols);
    }
}

template <int D>
cudaError_t launch_umma2_d(const DecodeParams& p, const int32_t* query_start, int T, int max_q_len, int num_sms,
                           bool merge, cudaStream_t st) {
    using C = UCfg<D>;
    auto kern = prefill_umma2_kernel<D>;
    // the warpgroups' register shares must fit in what the block is launched
    // with (setmaxnreg waits forever otherwise): checked once, on the binary
    static std::once_flag checked;
    static cudaError_t check = cudaSuccess;
    std::call_once(checked, [&] {
        cudaFuncAttributes fa;
        check = cudaFuncGetAttributes(&fa, kern);
        if (check == cudaSuccess &&
            (fa.numRegs * kThreads < 256 * kSoftmaxRegs + 128 * kOtherRegs || fa.maxThreadsPerBlock < kThreads))
            check = cudaErrorInvalidConfiguration;
    });
    if (check != cudaSuccess) return check;
    static SmemOptIn optin;
    cudaError_t e = optin.ensure(reinterpret_cast<const void*>(kern), C::kSmemBytes);
    if (e != cudaSuccess) return e;
    CUtensorMap kmap, vmap;
    if (!prefill_encode_kv_map(&kmap, p.kc, p) || !prefill_encode_kv_map(&vmap, p.vc, p)) return cudaErrorInvalidValue;
    int rt_max = (max_q_len * p.g + kURows - 1) / kURows;
    if (rt_max < 1) rt_max = 1;
    const unsigned long long units = (unsigned long long)p.Pmax * p.S * p.Hkv * rt_max;
    int grid = (int)(units < (unsigned long long)num_sms ? units : (unsigned long long)num_sms);
    if (grid < 1) grid = 1;
    kern<<<grid, kThreads, C::kSmemBytes, st>>>(p, query_start, T, max_q_len, kmap, vmap, units, rt_max);
    e = cudaGetLastError();
    if (e != cudaSuccess || !merge) return e;
    return launch_prefill_merge(p, query_start, T, kURows, max_q_len, st);
}

}  // namespace

cudaError_t launch_prefill_umma2(const DecodeParams& p, const int32_t* query_start, int T, int max_q_len,
                                 int num_sms, bool merge, cudaStream_t st) {
    if (p.S == 0 || T == 0) return cudaSuccess;
    return p.d == 64 ? launch_umma2_d<64>(p, query_start, T, max_q_len, num_sms, merge, st)
                     : launch_umma2_d<128>(p, query_start, T, max_q_len, num_sms, merge, st);
}

}  // namespace pkv
