// Paged attention for several query tokens per sequence on tensor cores:
// a chunk of prefill, or the tokens a speculative decoder proposes.
//
// "LLM推論の基礎とvLLMの内部", section 6: chunked prefill splits a long prompt
// into per-step pieces that run next to other requests' decodes; section 3:
// the V1 scheduler treats prefill and decode alike (tokens to compute per
// request, speculative tokens included).  The chunk's queries are the
// sequence's last q_len tokens; query i, at position p = n - q_len + i,
// attends to tokens 0..p through the block table.
//
// Work unit: (sequence, K/V head, tile of 16 (query, head) rows, partition of
// P key tokens).  Row r of a sequence's rows for one K/V head is query r / g,
// head r % g (g = Hq / Hkv).  A tile scans keys only up to its last query's
// position.  Each warp is an independent worker with its own ring of
// shared-memory stages of 32 tokens, filled by TMA tensor copies (one box per
// block half-row of the K/V head, 128-byte swizzle), as in the decode kernel.
// Math per stage (mma.sync m16n8k16, bf16 in, fp32 accumulate):
//   S[16 rows x 32 tokens] = Q[16 x d] . K^T            (4 x d/16 MMAs)
//   online softmax per row (running max m, sum l, base 2), causal mask
//   O[16 rows x d] += P[16 x 32 tokens] . V[32 x d]      (2 x d/8 MMAs)
// The S accumulator of two 8-token tiles is exactly the A operand of the
// P.V product; K and V come through ldmatrix (V transposed).  A tile whose
// keys fit one partition writes `out`; otherwise the partition's (m, l, O)
// goes to the workspace and the merge kernel below combines them.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math_constants.h>

#include <mutex>

#include "pkv_common.cuh"
#include "pkv_internal.h"
#include "pkv_merge.cuh"
#include "pkv_qtile.cuh"
#include "pkv_tc_common.cuh"

namespace pkv {
namespace {

using namespace tc;

constexpr int kPWarps = 6;      // workers per CTA
constexpr int kPStages = 2;     // ring depth per worker
constexpr int kPTok = 32;       // key tokens per stage
constexpr int kRows = 16;       // (query, head) rows per tile
constexpr long long kPWaitLimitCycles = 4000000000LL;   // ~2 s: a stage that never lands

template <int D>
struct PCfg {
    static constexpr int kRowBytes = 2 * D;                     // one token of one K/V head (bf16)
    static constexpr int kBoxRow = kRowBytes >= 128 ? 128 : kRowBytes;
    static constexpr int kHalves = kRowBytes / kBoxRow;
    static constexpr int kPartBytes = kPTok * kRowBytes;
    static constexpr int kStageBytes = 2 * kPartBytes;
    static constexpr int kWarpBytes = kPStages * kStageBytes;
    static constexpr int kQueue = kPStages;
    static constexpr int kQueueCtlOff = (12 * kPStages + 15) / 16 * 16;
    static constexpr int kCtlBytes = kQueueCtlOff + 48 * kQueue;
    static constexpr int kCtlOff = kPWarps * kWarpBytes;
    static constexpr int kSmemBytes = kCtlOff + kPWarps * kCtlBytes + 1024;
    static constexpr int KS = D / 16;      // k-steps of Q.K^T
    static constexpr int DT = D / 8;       // 8-wide tiles of d in P.V
    static_assert(kStageBytes % 1024 == 0, "stages keep the swizzle atoms aligned");
    static_assert(kSmemBytes <= 232448, "shared memory per CTA");
};

template <int D>
__global__ void __launch_bounds__(kPWarps * 32, 1)
    prefill_tc_kernel(const __grid_constant__ DecodeParams p, const int32_t* __restrict__ query_start, int T,
                      int max_q, const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                      unsigned long long total_units, int rt_max) {
    using C = PCfg<D>;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int r = lane >> 2, c = lane & 3;
    const uint32_t raw_addr = smem_addr(smem_raw);
    const uint32_t base_addr = (raw_addr + 1023u) & ~1023u;
    unsigned char* smem = smem_raw + (base_addr - raw_addr);
    const uint32_t ws_addr = base_addr + warp * C::kWarpBytes;
    unsigned char* ctl = smem + C::kCtlOff + warp * C::kCtlBytes;
    const uint32_t ctl_addr = base_addr + C::kCtlOff + warp * C::kCtlBytes;
    uint32_t* masks = reinterpret_cast<uint32_t*>(ctl + 8 * kPStages);
    int4* queue = reinterpret_cast<int4*>(ctl + C::kQueueCtlOff);        // 3 int4 per unit
    auto bar = [&](int i) { return ctl_addr + 8 * i; };
    auto stage_k = [&](int i) { return ws_addr + i * C::kStageBytes; };
    auto stage_v = [&](int i) { return ws_addr + i * C::kStageBytes + C::kPartBytes; };
    // the partition merge that may follow can be scheduled now; it waits for this grid's results
    asm volatile("griddepcontrol.launch_dependents;");

    if (lane == 0) {
        for (int i = 0; i < kPStages; ++i) mbar_init(bar(i), 1);
        fence_barrier_init();
    }
    __syncwarp();

    const unsigned long long total_warps = (unsigned long long)gridDim.x * kPWarps;
    unsigned long long static_next = (unsigned long long)blockIdx.x * kPWarps + warp;
    const int box_rows = min(p.bs, kPTok);
    const int boxes_per_stage = kPTok / box_rows;
    const uint32_t box_bytes = (uint32_t)box_rows * C::kBoxRow;

    // ---- issue side
    bool claiming = true, i_have = false;
    QTile iu{};
    int i_stage = 0, i_nst = 0;
    unsigned g_issue = 0, q_tail = 0;
    int tab = 0, tab_next = 0, tab_chunk = 0, tab_blocks = 0;
    auto load_chunk = [&](int chunk) -> int {
        const int rb = 32 * chunk + lane;
        return rb < tab_blocks ? __ldg(p.block_tables + (size_t)iu.s * p.MB + iu.k0 / p.bs + rb) : 0;
    };
    auto claim = [&](unsigned long long& u) -> bool {
        for (;;) {
            unsigned long long v = 0;
            if (lane == 0) v = p.sched != nullptr ? atomicAdd(reinterpret_cast<unsigned long long*>(p.sched), 1ull)
                                                  : static_next;
            v = __shfl_sync(0xffffffffu, v, 0);
            static_next += total_warps;
            if (v >= total_units) return false;
            QTile x;
            if (!qtile_of<kRows>(p, query_start, T, max_q, v, rt_max, x)) continue;
            u = v;
            return true;
        }
    };
    auto issue_one = [&]() -> bool {
        while (!i_have || i_stage == i_nst) {
            if (!claiming) return false;
            unsigned long long u;
            if (!claim(u)) {
                claiming = false;
                return false;
            }
            qtile_of<kRows>(p, query_start, T, max_q, u, rt_max, iu);
            if (lane == 0) {
                int4* e = queue + 3 * (q_tail % C::kQueue);
                e[0] = make_int4(iu.s, iu.kvh, iu.rt, iu.part);
                e[1] = make_int4(iu.k0, iu.k1, iu.n, iu.ql);
                e[2] = make_int4(iu.q0, iu.np, iu.rows, 0);
            }
            ++q_tail;
            i_have = true;
            i_stage = 0;
            i_nst = (iu.k1 - iu.k0 + kPTok - 1) / kPTok;
            tab_blocks = (iu.k1 - iu.k0 + p.bs - 1) / p.bs;
            tab_chunk = 0;
            tab = load_chunk(0);
            tab_next = load_chunk(1);
        }
        const int slot = g_issue % kPStages;
        const int rs = i_stage * kPTok;
        const int ts = iu.k0 + rs;
        const int tn = min(kPTok, iu.k1 - ts);
        if (rs / p.bs / 32 != tab_chunk) {
            ++tab_chunk;
            tab = tab_next;
            tab_next = load_chunk(tab_chunk + 1);
        }
        const int pb_tok = __shfl_sync(0xffffffffu, tab, ((rs + lane) / p.bs) & 31);
        bool ok = lane < tn;
        if (ok && (pb_tok < 0 || pb_tok >= p.NB)) {
            report(p.err, PKV_DEVERR_BLOCK_ID);
            ok = false;
        }
        const uint32_t m = __ballot_sync(0xffffffffu, ok);
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
            const int t0b = ts + b * box_rows;
            const uint32_t dst = (kv ? stage_v(slot) : stage_k(slot)) + h * (kPTok * C::kBoxRow) +
                                 b * box_rows * C::kBoxRow;
            tensor_load_2d(dst, kv ? &vmap : &kmap, iu.kvh * D + h * (C::kBoxRow / 2), pb_box * p.bs + t0b % p.bs,
                           bar(slot));
        }
        ++g_issue;
        ++i_stage;
        return true;
    };

    // ---- consume side
    unsigned g_cons = 0, q_head = 0;
    bool have_unit = false;
    QTile cu{};
    int c_stage = 0, c_nst = 0;
    uint32_t qa[C::KS][4];           // Q A-fragments: rows r, r+8 of the tile
    float o[C::DT][4];               // O accumulators, 8-wide tiles of d
    float m_run[2], l_run[2];        // rows r, r+8
    int pos[2];                      // query positions of rows r, r+8 (-1: padding row)
    const float scl = p.logit_scale_log2;
    bool bail = false;

    for (int i = 0; i < kPStages; ++i)
        if (!issue_one()) break;

    for (;;) {
        if (!have_unit) {
            if (q_head == q_tail) break;
            __syncwarp();
            {
                const int4* e = queue + 3 * (q_head % C::kQueue);
                const int4 a = e[0], b2 = e[1], c3 = e[2];
                cu.s = a.x; cu.kvh = a.y; cu.rt = a.z; cu.part = a.w;
                cu.k0 = b2.x; cu.k1 = b2.y; cu.n = b2.z; cu.ql = b2.w;
                cu.q0 = c3.x; cu.np = c3.y; cu.rows = c3.z;
            }
            ++q_head;
            c_stage = 0;
            c_nst = (cu.k1 - cu.k0 + kPTok - 1) / kPTok;
            have_unit = true;
            size_t qrow[2];
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const int row = cu.rt * kRows + r + 8 * k;
                if (row < cu.rows) {
                    const int qi = row / p.g, hh = row - qi * p.g;
                    pos[k] = cu.n - cu.ql + qi;
                    qrow[k] = ((size_t)(cu.q0 + qi) * p.Hq + cu.kvh * p.g + hh) * D;
                } else {
                    pos[k] = -1;
                    qrow[k] = 0;
                }
            }
            const uint32_t* q32 = static_cast<const uint32_t*>(p.q);
#pragma unroll
            for (int ks = 0; ks < C::KS; ++ks) {
                const int d0 = 16 * ks + 2 * c;
                qa[ks][0] = pos[0] >= 0 ? __ldg(q32 + (qrow[0] + d0) / 2) : 0u;
                qa[ks][1] = pos[1] >= 0 ? __ldg(q32 + (qrow[1] + d0) / 2) : 0u;
                qa[ks][2] = pos[0] >= 0 ? __ldg(q32 + (qrow[0] + d0 + 8) / 2) : 0u;
                qa[ks][3] = pos[1] >= 0 ? __ldg(q32 + (qrow[1] + d0 + 8) / 2) : 0u;
            }
#pragma unroll
            for (int t = 0; t < C::DT; ++t) o[t][0] = o[t][1] = o[t][2] = o[t][3] = 0.f;
            m_run[0] = m_run[1] = -CUDART_INF_F;
            l_run[0] = l_run[1] = 0.f;
        }

        const int slot = g_cons % kPStages;
        const uint32_t parity = (g_cons / kPStages) & 1u;
        if (!mbar_try_wait(bar(slot), parity)) {
            const long long t_start = clock64();
            while (!mbar_try_wait(bar(slot), parity)) {
                if (clock64() - t_start > kPWaitLimitCycles) {
                    report(p.err, PKV_DEVERR_TIMEOUT);
                    bail = true;
                    break;
                }
            }
        }
        if (__any_sync(0xffffffffu, bail)) break;
        const uint32_t vmask = masks[slot];
        const uint32_t kb = stage_k(slot), vb = stage_v(slot);
        const int ts = cu.k0 + c_stage * kPTok;       // first key token of the stage

        // ---- S = Q . K^T: 4 tiles of 8 tokens
        float sacc[4][4];
        const int mi = lane >> 3;
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
            sacc[nt][0] = sacc[nt][1] = sacc[nt][2] = sacc[nt][3] = 0.f;
            const int tok = 8 * nt + (lane & 7);
#pragma unroll
            for (int k2 = 0; k2 < C::KS / 2; ++k2) {
                uint32_t b0, b1, b2, b3;
                ldsm_x4(swz<C::kRowBytes, kPTok>(kb, tok, 32 * (2 * k2 + (mi >> 1)) + 16 * (mi & 1)), b0, b1, b2, b3);
                mma16816<false>(sacc[nt], qa[2 * k2][0], qa[2 * k2][1], qa[2 * k2][2], qa[2 * k2][3], b0, b1);
                mma16816<false>(sacc[nt], qa[2 * k2 + 1][0], qa[2 * k2 + 1][1], qa[2 * k2 + 1][2],
                                qa[2 * k2 + 1][3], b2, b3);
            }
        }

        // ---- online softmax per row, causal mask
        float x[4][4];
        float mx0 = -CUDART_INF_F, mx1 = -CUDART_INF_F;
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int tl = 8 * nt + 2 * c + j;          // token within the stage
                const bool live = (vmask >> tl) & 1u;
                const int t = ts + tl;
                x[nt][j] = live && t <= pos[0] ? sacc[nt][j] * scl : -CUDART_INF_F;
                x[nt][2 + j] = live && t <= pos[1] ? sacc[nt][2 + j] * scl : -CUDART_INF_F;
                mx0 = fmaxf(mx0, x[nt][j]);
                mx1 = fmaxf(mx1, x[nt][2 + j]);
            }
        }
#pragma unroll
        for (int off = 1; off < 4; off <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
        }
        const float mn0 = fmaxf(m_run[0], mx0), mn1 = fmaxf(m_run[1], mx1);
        const float mu0 = mn0 == -CUDART_INF_F ? 0.f : mn0;
        const float mu1 = mn1 == -CUDART_INF_F ? 0.f : mn1;
        const float al0 = fast_exp2(m_run[0] - mu0), al1 = fast_exp2(m_run[1] - mu1);
        m_run[0] = mn0;
        m_run[1] = mn1;
        float ls0 = 0.f, ls1 = 0.f;
        uint32_t pa[2][4];                      // P A-fragments for the two 16-token k-tiles
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
            const float p0 = fast_exp2(x[nt][0] - mu0), p1 = fast_exp2(x[nt][1] - mu0);
            const float p2 = fast_exp2(x[nt][2] - mu1), p3 = fast_exp2(x[nt][3] - mu1);
            ls0 += p0 + p1;
            ls1 += p2 + p3;
            const int kt = nt >> 1, hi = nt & 1;
            pa[kt][0 + 2 * hi] = pack2<false>(p0, p1);      // row r,   tokens 2c, 2c+1 (+8 for hi)
            pa[kt][1 + 2 * hi] = pack2<false>(p2, p3);      // row r+8
        }
        l_run[0] = l_run[0] * al0 + ls0;
        l_run[1] = l_run[1] * al1 + ls1;
#pragma unroll
        for (int t = 0; t < C::DT; ++t) {
            o[t][0] *= al0;
            o[t][1] *= al0;
            o[t][2] *= al1;
            o[t][3] *= al1;
        }

        // ---- O += P . V
        const bool full = vmask == 0xffffffffu;
#pragma unroll
        for (int kt = 0; kt < 2; ++kt) {
            const int tok = 16 * kt + 8 * (mi & 1) + (lane & 7);
            const int tk0 = 16 * kt + 2 * c;      // tokens of b0b1: tk0, tk0+1; of b2b3: +8
            const uint32_t keep01 = (vmask >> tk0) & 3u, keep89 = (vmask >> (tk0 + 8)) & 3u;
            const uint32_t mlo = (keep01 & 1u ? 0x0000ffffu : 0u) | (keep01 & 2u ? 0xffff0000u : 0u);
            const uint32_t mhi = (keep89 & 1u ? 0x0000ffffu : 0u) | (keep89 & 2u ? 0xffff0000u : 0u);
#pragma unroll
            for (int t2 = 0; t2 < C::DT / 2; ++t2) {
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(swz<C::kRowBytes, kPTok>(vb, tok, 32 * t2 + 16 * (mi >> 1)), b0, b1, b2, b3);
                if (!full) {
                    b0 &= mlo; b1 &= mhi; b2 &= mlo; b3 &= mhi;
                }
                mma16816<false>(o[2 * t2], pa[kt][0], pa[kt][1], pa[kt][2], pa[kt][3], b0, b1);
                mma16816<false>(o[2 * t2 + 1], pa[kt][0], pa[kt][1], pa[kt][2], pa[kt][3], b2, b3);
            }
        }

        __syncwarp();
        fence_proxy_async();
        ++g_cons;
        ++c_stage;
        issue_one();

        if (c_stage == c_nst) {
            float l0 = l_run[0], l1 = l_run[1];
#pragma unroll
            for (int off = 1; off < 4; off <<= 1) {
                l0 += __shfl_xor_sync(0xffffffffu, l0, off);
                l1 += __shfl_xor_sync(0xffffffffu, l1, off);
            }
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                if (pos[k] < 0) continue;
                const int row = cu.rt * kRows + r + 8 * k;
                const int qi = row / p.g, hh = row - qi * p.g;
                const size_t hrow = (size_t)(cu.q0 + qi) * p.Hq + cu.kvh * p.g + hh;
                const float l = k ? l1 : l0;
                if (cu.np == 1) {
                    const float f = l > 0.f ? 1.f / l : 0.f;
                    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out) + hrow * D;
#pragma unroll
                    for (int t = 0; t < C::DT; ++t) {
                        const int dd = 8 * t + 2 * c;
                        *reinterpret_cast<__nv_bfloat162*>(out + dd) =
                            __floats2bfloat162_rn(o[t][2 * k] * f, o[t][2 * k + 1] * f);
                    }
                } else {
                    const size_t u = hrow * p.Pmax + cu.part;
#pragma unroll
                    for (int t = 0; t < C::DT; ++t) {
                        const int dd = 8 * t + 2 * c;
                        *reinterpret_cast<float2*>(p.part_acc + u * D + dd) = make_float2(o[t][2 * k], o[t][2 * k + 1]);
                    }
                    if (c == 0) {
                        p.part_ml[2 * u] = m_run[k];
                        p.part_ml[2 * u + 1] = l;
                    }
                }
            }
            have_unit = false;
        }
    }

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

// Merge of a query's partitions, one warp per (query token, head)
// (merge_partitions): the token's sequence by binary search over
// query_start, its tile's partition count from the same formula the decode
// units use.  Launched as a programmatic dependent of the prefill kernel;
// every thread waits for that kernel before it reads anything, so that this
// grid never completes before it (pdl_wait).
template <int D>
__global__ void __launch_bounds__(256) prefill_merge_kernel(DecodeParams p, const int32_t* __restrict__ query_start,
                                                            int T, int tile_rows, int max_q) {
    constexpr int E = D / 32;
    const int lane = threadIdx.x & 31;
    const long long gw = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
    pdl_trigger();
    pdl_wait();
    if (gw >= (long long)T * p.Hq) return;
    const int tq = (int)(gw / p.Hq), h = (int)(gw % p.Hq);
    int lo = 0, hi = p.S;                      // largest s with query_start[s] <= tq
    while (hi - lo > 1) {
        const int mid = (lo + hi) / 2;
        if (query_start[mid] <= tq) lo = mid; else hi = mid;
    }
    const int s = lo;
    const int n = p.context_lens[s], q0 = query_start[s], ql = query_start[s + 1] - q0;
    if (n < 0 || n > p.max_ctx || ql < 0 || ql > n || ql > max_q || q0 < 0 || q0 + ql > T || tq >= q0 + ql)
        return;                                // the sequence the main kernel skipped
    const int kvh = h / p.g, row = (tq - q0) * p.g + (h - kvh * p.g);
    const int rows = ql * p.g, rt = row / tile_rows;
    const int last_row = min(rt * tile_rows + tile_rows - 1, rows - 1);
    const int key_end = n - ql + last_row / p.g + 1;
    const int np = (key_end + p.P - 1) / p.P;
    if (np <= 1) return;
    const size_t u0 = ((size_t)tq * p.Hq + h) * p.Pmax;
    float acc[E];
    const float L = merge_partitions<D>(p.part_ml + 2 * u0, p.part_acc + u0 * D, np, lane, acc);
    const float f = L > 0.f ? 1.f / L : 0.f;
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out) + ((size_t)tq * p.Hq + h) * D + lane * E;
#pragma unroll
    for (int k = 0; k < E; ++k) out[k] = __float2bfloat16_rn(acc[k] * f);
}

template <int D>
cudaError_t launch_prefill_d(const DecodeParams& p, const int32_t* query_start, int T, int max_q_len,
                             int num_sms, bool merge, cudaStream_t st) {
    using C = PCfg<D>;
    auto kern = prefill_tc_kernel<D>;
    static SmemOptIn optin;
    cudaError_t e = optin.ensure(reinterpret_cast<const void*>(kern), C::kSmemBytes);
    if (e != cudaSuccess) return e;
    CUtensorMap kmap, vmap;
    if (!prefill_encode_kv_map(&kmap, p.kc, p) || !prefill_encode_kv_map(&vmap, p.vc, p)) return cudaErrorInvalidValue;
    const int rt_max = (max_q_len * p.g + kRows - 1) / kRows;
    const unsigned long long units = (unsigned long long)p.Pmax * p.S * p.Hkv * (rt_max > 0 ? rt_max : 1);
    const unsigned long long want = (units + kPWarps - 1) / kPWarps;
    int grid = (int)(want < (unsigned long long)num_sms ? want : (unsigned long long)num_sms);
    if (grid < 1) grid = 1;
    kern<<<grid, kPWarps * 32, C::kSmemBytes, st>>>(p, query_start, T, max_q_len, kmap, vmap, units,
                                                    rt_max > 0 ? rt_max : 1);
    e = cudaGetLastError();
    if (e != cudaSuccess || !merge) return e;
    return launch_prefill_merge(p, query_start, T, kRows, max_q_len, st);
}

}  // namespace

bool prefill_encode_kv_map(CUtensorMap* map, const void* base, const DecodeParams& p) {
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
    if (fn == nullptr) return false;
    // rows of one K/V head (d bf16 values), boxes of 64 values x one block
    // of at most 32 tokens, 128-byte swizzle
    const cuuint64_t dims[2] = {(cuuint64_t)p.Hkv * p.d, (cuuint64_t)p.NB * p.bs};
    const cuuint64_t strides[1] = {(cuuint64_t)p.Hkv * p.d * 2};
    const cuuint32_t box[2] = {64u, (cuuint32_t)(p.bs < 32 ? p.bs : 32)};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_prefill_merge(const DecodeParams& p, const int32_t* query_start, int T, int tile_rows,
                                 int max_q, cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    const long long warps = (long long)T * p.Hq;
    cfg.gridDim = dim3((unsigned)((warps + 7) / 8));
    cfg.blockDim = dim3(256);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return p.d == 64 ? cudaLaunchKernelEx(&cfg, prefill_merge_kernel<64>, p, query_start, T, tile_rows, max_q)
                     : cudaLaunchKernelEx(&cfg, prefill_merge_kernel<128>, p, query_start, T, tile_rows, max_q);
}

cudaError_t launch_prefill_tc(const DecodeParams& p, const int32_t* query_start, int T, int max_q_len, int num_sms,
                              bool merge, cudaStream_t st) {
    if (p.S == 0 || T == 0) return cudaSuccess;
    return p.d == 64 ? launch_prefill_d<64>(p, query_start, T, max_q_len, num_sms, merge, st)
                     : launch_prefill_d<128>(p, query_start, T, max_q_len, num_sms, merge, st);
}

}  // namespace pkv
