// Merge of split-K partitions, shared by the decode and the query-chunk
// merges.  Each partition p of one (query row, head) left m_p (its running
// max, log2 units), l_p (its sum of 2^(s - m_p)) and acc_p (its weighted
// sum of V rows, unnormalised); the full result is
//   M = max m_p,  L = sum 2^(m_p - M) l_p,  O = sum 2^(m_p - M) acc_p / L.
// One warp merges one (row, head).  The partitions are visited in chunks of
// 16 with the maximum carried along (the same rescaling as the online
// softmax inside a partition), so that a chunk's (m, l) pairs and its 16
// acc rows are all requested at once: one memory round trip per chunk
// instead of one per partition.
#pragma once

#include <math_constants.h>

#include <cstddef>
#include <cstdint>

#include "pkv_common.cuh"

namespace pkv {

constexpr int kMergeChunk = 16;

// One row's E elements of this lane, read through L2 (ld.global.cg) with an
// "evict first" hint: each partial result is read exactly once.
template <int E>
__device__ __forceinline__ void merge_load_row(const float* src, float (&a)[E], uint64_t pol) {
    if constexpr (E == 4) {
        asm volatile("ld.global.cg.L2::cache_hint.v4.f32 {%0, %1, %2, %3}, [%4], %5;"
                     : "=f"(a[0]), "=f"(a[1]), "=f"(a[2]), "=f"(a[3])
                     : "l"(src), "l"(pol));
    } else {
        static_assert(E == 2, "rows of 64 or 128 elements");
        asm volatile("ld.global.cg.L2::cache_hint.v2.f32 {%0, %1}, [%2], %3;"
                     : "=f"(a[0]), "=f"(a[1])
                     : "l"(src), "l"(pol));
    }
}

// ml: the (m, l) pairs of the row's partitions [np][2]; acc: their rows
// [np][D].  Lane i ends with o = elements [i*E, i*E+E) of sum 2^(m_p - M)
// acc_p; returns L (the same on every lane).  The data were written by
// another kernel: loads go through L2 (ld.global.cg).
template <int D>
__device__ __forceinline__ float merge_partitions(const float* __restrict__ ml, const float* __restrict__ acc,
                                                  int np, int lane, float (&o)[D / 32]) {
    constexpr int E = D / 32, B = kMergeChunk;
    const uint64_t once = l2_policy_evict_first();
    float M = -CUDART_INF_F, lpart = 0.f;
#pragma unroll
    for (int k = 0; k < E; ++k) o[k] = 0.f;
    for (int c0 = 0; c0 < np; c0 += B) {
        const int cn = min(B, np - c0);
        float m = -CUDART_INF_F, l = 0.f;
        if (lane < cn) {
            asm volatile("ld.global.cg.L2::cache_hint.v2.f32 {%0, %1}, [%2], %3;"
                         : "=f"(m), "=f"(l)
                         : "l"(reinterpret_cast<const float2*>(ml) + c0 + lane), "l"(once));
        }
        float a[B][E];
#pragma unroll
        for (int j = 0; j < B; ++j) {
            if (j < cn) {
                merge_load_row<E>(acc + (size_t)(c0 + j) * D + lane * E, a[j], once);
            } else {
#pragma unroll
                for (int k = 0; k < E; ++k) a[j][k] = 0.f;
            }
        }
        float cm = m;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, off));
        const float Mn = fmaxf(M, cm);
        // a partition with no valid token has m = -inf and weighs nothing
        const float f = M == -CUDART_INF_F ? 0.f : exp2f(M - Mn);
        const float w = m == -CUDART_INF_F ? 0.f : exp2f(m - Mn);
        lpart = fmaf(w, l, lpart * f);
#pragma unroll
        for (int k = 0; k < E; ++k) o[k] *= f;
#pragma unroll
        for (int j = 0; j < B; ++j) {
            const float wj = __shfl_sync(0xffffffffu, w, j);     // 0 past the chunk's end
#pragma unroll
            for (int k = 0; k < E; ++k) o[k] = fmaf(wj, a[j][k], o[k]);
        }
        M = Mn;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) lpart += __shfl_xor_sync(0xffffffffu, lpart, off);
    return lpart;
}

}  // namespace pkv
