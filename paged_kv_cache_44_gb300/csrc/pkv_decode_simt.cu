// paged_attention_decode on CUDA cores, and the partition merge.
//
// "LLM推論の基礎とvLLMの内部", section 4: the attention kernel reaches every
// cached token through the sequence's block table; section 2: the query
// heads of one GQA group share a K/V head.  This kernel is the general path
// (every storage format, fp32 included) and the CUDA-core baseline the
// tensor-core kernel is measured against.
//
// Grid (partition, K/V head x head-set, sequence); 128 threads.  A CTA owns
// up to 8 query heads of one K/V head over one partition of tokens.  Tokens
// are taken in chunks of 64: (1) each warp computes logits of its tokens for
// all heads (lanes split d, warp-shuffle sums); (2) per head, the chunk max
// updates the running max m and sum l (online softmax, base-2 exponent);
// (3) thread e accumulates sum_t p_t * V[t][e] for every head.  A sequence
// that fits one partition writes `out` directly; otherwise the partition's
// (m, l, acc) goes to the workspace and the merge kernel combines them.
#include <math_constants.h>

#include "pkv_common.cuh"
#include "pkv_internal.h"
#include "pkv_merge.cuh"

namespace pkv {
namespace {

constexpr int kThreads = 128;
constexpr int kChunk = 64;
constexpr int kHeads = 8;       // query heads per CTA

template <int D, typename QF, typename CF>
__global__ void __launch_bounds__(kThreads) decode_simt_kernel(DecodeParams p) {
    const int s = blockIdx.z;
    const int nsets = (p.g + kHeads - 1) / kHeads;
    const int kvh = blockIdx.y / nsets, set = blockIdx.y % nsets;
    const int part = blockIdx.x;
    const int h0 = kvh * p.g + set * kHeads;
    const int nh = min(kHeads, p.g - set * kHeads);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    // the partition merge that may follow can be scheduled now; it waits for this grid's results
    pdl_trigger();
    pdl_wait();

    int n = p.context_lens[s];
    if (n < 0 || n > p.max_ctx) {   // max_ctx <= MB * bs was checked on the host
        if (part == 0 && blockIdx.y == 0 && threadIdx.x == 0) report(p.err, PKV_DEVERR_CONTEXT_LEN);
        n = n < 0 ? 0 : p.max_ctx;
    }
    const int np = num_partitions(n, p.P, p.Q, p.hold);
    if (part >= np) return;
    int t0, t1;
    partition_range(n, p.P, p.Q, p.hold, part, t0, t1);

    __shared__ float q_s[kHeads][D];
    __shared__ float x_s[kHeads][kChunk];
    __shared__ float m_s[kHeads], l_s[kHeads], alpha_s[kHeads];
    __shared__ int pb_s[kChunk];

    for (int i = threadIdx.x; i < kHeads * D; i += kThreads) {
        const int h = i / D, e = i % D;
        q_s[h][e] = h < nh ? load_elem<QF>(p.q, ((size_t)s * p.Hq + h0 + h) * D + e) : 0.f;
    }
    if (threadIdx.x < kHeads) {
        m_s[threadIdx.x] = -CUDART_INF_F;
        l_s[threadIdx.x] = 0.f;
    }
    float acc[kHeads];
#pragma unroll
    for (int h = 0; h < kHeads; ++h) acc[h] = 0.f;
    __syncthreads();

    const size_t row_stride = (size_t)p.Hkv * D;   // elements between tokens of one block
    for (int c0 = t0; c0 < t1; c0 += kChunk) {
        const int cn = min(kChunk, t1 - c0);
        // physical row of each token of the chunk (-1 when its block id is bad)
        for (int tt = threadIdx.x; tt < cn; tt += kThreads) {
            const int t = c0 + tt;
            const int pb = p.block_tables[(size_t)s * p.MB + t / p.bs];
            if (pb < 0 || pb >= p.NB) {
                report(p.err, PKV_DEVERR_BLOCK_ID);
                pb_s[tt] = -1;
            } else {
                pb_s[tt] = pb * p.bs + t % p.bs;
            }
        }
        __syncthreads();
        // (1) logits, in log2 units
        for (int tt = warp; tt < cn; tt += kThreads / 32) {
            const int row = pb_s[tt];
            float kv[D / 32];
#pragma unroll
            for (int i = 0; i < D / 32; ++i)
                kv[i] = row >= 0 ? load_elem<CF>(p.kc, (size_t)row * row_stride + (size_t)kvh * D + lane + 32 * i) : 0.f;
#pragma unroll
            for (int h = 0; h < kHeads; ++h) {
                if (h >= nh) break;
                float part_dot = 0.f;
#pragma unroll
                for (int i = 0; i < D / 32; ++i) part_dot = fmaf(q_s[h][lane + 32 * i], kv[i], part_dot);
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) part_dot += __shfl_xor_sync(0xffffffffu, part_dot, o);
                if (lane == 0) x_s[h][tt] = row >= 0 ? part_dot * p.logit_scale_log2 : -CUDART_INF_F;
            }
        }
        __syncthreads();
        // (2) online softmax update, one warp per head
        for (int h = warp; h < nh; h += kThreads / 32) {
            float mx = -CUDART_INF_F;
            for (int tt = lane; tt < cn; tt += 32) mx = fmaxf(mx, x_s[h][tt]);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            const float m_old = m_s[h];
            const float m_new = fmaxf(m_old, mx);
            float sum = 0.f;
            for (int tt = lane; tt < cn; tt += 32) {
                const float w = m_new == -CUDART_INF_F ? 0.f : exp2f(x_s[h][tt] - m_new);
                x_s[h][tt] = w;
                sum += w;
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
            __syncwarp();
            if (lane == 0) {
                const float alpha = m_old == -CUDART_INF_F ? 0.f : exp2f(m_old - m_new);
                alpha_s[h] = alpha;
                l_s[h] = l_s[h] * alpha + sum;
                m_s[h] = m_new;
            }
        }
        __syncthreads();
        // (3) acc[h] = acc[h] * alpha[h] + sum_t p[h][t] * V[t][e]
        if (threadIdx.x < D) {
            const int e = threadIdx.x;
#pragma unroll
            for (int h = 0; h < kHeads; ++h) acc[h] *= (h < nh ? alpha_s[h] : 0.f);
            for (int tt = 0; tt < cn; ++tt) {
                const int row = pb_s[tt];
                if (row < 0) continue;
                const float v = load_elem<CF>(p.vc, (size_t)row * row_stride + (size_t)kvh * D + e);
#pragma unroll
                for (int h = 0; h < kHeads; ++h) acc[h] = fmaf(x_s[h][tt], v, acc[h]);
            }
        }
        __syncthreads();
    }

    if (threadIdx.x < D) {
        const int e = threadIdx.x;
        if (np == 1) {
            for (int h = 0; h < nh; ++h) {
                const float l = l_s[h];
                const float o = l > 0.f ? acc[h] / l * p.out_scale : 0.f;
                store_elem<QF>(p.out, ((size_t)s * p.Hq + h0 + h) * D + e, o);
            }
        } else {
            for (int h = 0; h < nh; ++h) {
                const size_t u = ((size_t)s * p.Hq + h0 + h) * p.Pmax + part;
                p.part_acc[u * D + e] = acc[h];
                if (e == 0) {
                    p.part_ml[2 * u] = m_s[h];
                    p.part_ml[2 * u + 1] = l_s[h];
                }
            }
        }
    }
}

// Merge of a sequence's partitions: M = max m_p, L = sum 2^(m_p - M) l_p,
// O = sum 2^(m_p - M) acc_p / L, one warp per (sequence, query head), eight
// warps per CTA (merge_partitions).  Sequences that fit one partition were
// finished by the decode kernel.  Launched as a programmatic dependent of
// the decode kernel, so it is resident when the decode ends; every thread
// waits for the decode before it reads anything, so that this grid never
// completes before the decode (pdl_wait).
constexpr int kMergeWarps = 8;

template <int D, typename QF>
__global__ void __launch_bounds__(kMergeWarps * 32) decode_reduce_kernel(DecodeParams p) {
    constexpr int E = D / 32;
    const int lane = threadIdx.x & 31;
    const long long gw = (long long)blockIdx.x * kMergeWarps + (threadIdx.x >> 5);
    pdl_trigger();
    pdl_wait();         // the decode's partial results
    if (gw >= (long long)p.S * p.Hq) return;
    const int s = (int)(gw / p.Hq), h = (int)(gw % p.Hq);
    int n = p.context_lens[s];
    n = n < 0 ? 0 : min(n, p.max_ctx);     // same clamp as the decode kernel: np <= Pmax
    const int np = num_partitions(n, p.P, p.Q, p.hold);
    if (np <= 1) return;
    const size_t u0 = ((size_t)s * p.Hq + h) * p.Pmax;
    float o[E];
    const float L = merge_partitions<D>(p.part_ml + 2 * u0, p.part_acc + u0 * D, np, lane, o);
    const float f = L > 0.f ? p.out_scale / L : 0.f;
    const size_t ob = ((size_t)s * p.Hq + h) * D + lane * E;
#pragma unroll
    for (int k = 0; k < E; ++k) store_elem<QF>(p.out, ob + k, o[k] * f);
}

template <int D, typename QF>
cudaError_t launch_reduce(const DecodeParams& p, cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const long long warps = (long long)p.S * p.Hq;
    cfg.gridDim = dim3((unsigned)((warps + kMergeWarps - 1) / kMergeWarps));
    cfg.blockDim = dim3(kMergeWarps * 32);
    return cudaLaunchKernelEx(&cfg, decode_reduce_kernel<D, QF>, p);
}

template <int D, typename QF>
cudaError_t launch_simt_q(const DecodeParams& p, pkv_dtype c_dt, dim3 grid, cudaStream_t st) {
    if (c_dt == PKV_F32) return launch_pdl(decode_simt_kernel<D, QF, F32>, grid, dim3(kThreads), 0, st, p);
    if (c_dt == PKV_BF16) return launch_pdl(decode_simt_kernel<D, QF, BF16>, grid, dim3(kThreads), 0, st, p);
    return launch_pdl(decode_simt_kernel<D, QF, E4M3>, grid, dim3(kThreads), 0, st, p);
}

}  // namespace

cudaError_t launch_decode_simt(const DecodeParams& p, pkv_dtype q_dt, pkv_dtype c_dt, cudaStream_t st) {
    if (p.S == 0) return cudaSuccess;
    const int nsets = (p.g + kHeads - 1) / kHeads;
    dim3 grid(p.Pmax, p.Hkv * nsets, p.S);
    if (p.d == 64)
        return q_dt == PKV_F32 ? launch_simt_q<64, F32>(p, c_dt, grid, st) : launch_simt_q<64, BF16>(p, c_dt, grid, st);
    return q_dt == PKV_F32 ? launch_simt_q<128, F32>(p, c_dt, grid, st) : launch_simt_q<128, BF16>(p, c_dt, grid, st);
}

cudaError_t launch_decode_reduce(const DecodeParams& p, pkv_dtype q_dt, cudaStream_t st) {
    if (p.S == 0) return cudaSuccess;
    if (p.d == 64) return q_dt == PKV_F32 ? launch_reduce<64, F32>(p, st) : launch_reduce<64, BF16>(p, st);
    return q_dt == PKV_F32 ? launch_reduce<128, F32>(p, st) : launch_reduce<128, BF16>(p, st);
}

}  // namespace pkv
