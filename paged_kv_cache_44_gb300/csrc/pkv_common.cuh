// Device helpers shared by the pkv kernels: element loads/stores for the
// three storage formats, and the device-side error report.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/pkv.h"

namespace pkv {

// Storage formats as template tags.
struct F32 { using T = float; static constexpr int bytes = 4; };
struct BF16 { using T = __nv_bfloat16; static constexpr int bytes = 2; };
struct E4M3 { using T = uint8_t; static constexpr int bytes = 1; };

// Programmatic dependent launch.  The library's kernels are launched so
// that each may be scheduled while the previous kernel of the stream is
// still running (once that kernel has called pdl_trigger()).  Every such
// kernel calls pdl_wait() in every thread before its first access to global
// memory: it returns once the previous kernel has completed and its writes
// are visible.  Since no grid can then complete before its predecessor, the
// stream keeps its order through any chain of such launches.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;"); }

// Record the first device-side problem; never traps.
__device__ __forceinline__ void report(int32_t* err, int code) {
    if (err != nullptr) atomicCAS(err, 0, code);
}

// L2 eviction priorities for the split-K partial results: the decode writes
// them with "evict last", so that the K/V streaming through L2 does not push
// them out before the merge, which reads each of them once with "evict
// first".  (PTX createpolicy / .L2::cache_hint, sm_80 and later.)
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ void st_l2_hint(float* p, float v, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(p), "f"(v), "l"(pol) : "memory");
}

// Split-K layout of a sequence of n tokens: full partitions of P tokens,
// then the rest cut into chunks of Q tokens (Q = P: one partial partition);
// a sequence with no tokens has one, empty, partition.  With hold > 0 (and
// Q < P), a sequence of at least kTailHoldMin full partitions has its last
// `hold` full partitions cut into chunks as well: more of the work is in
// the small units handed out last.
constexpr int kTailHoldMin = 4;

__host__ __device__ __forceinline__ int whole_partitions(int n, int P, int Q, int hold) {
    const int full = n / P;
    return Q < P && hold > 0 && full >= kTailHoldMin ? full - hold : full;
}

__host__ __device__ __forceinline__ int num_partitions(int n, int P, int Q, int hold) {
    if (n <= 0) return 1;
    const int fa = whole_partitions(n, P, Q, hold);
    return fa + (n - fa * P + Q - 1) / Q;
}

// Tokens [t0, t1) of partition `part` of a sequence of n tokens.
__host__ __device__ __forceinline__ void partition_range(int n, int P, int Q, int hold, int part, int& t0,
                                                        int& t1) {
    const int fa = whole_partitions(n, P, Q, hold);
    if (part < fa) {
        t0 = part * P;
        t1 = t0 + P;
    } else {
        t0 = fa * P + (part - fa) * Q;
        t1 = min(t0 + Q, n);
    }
}

// ---- scalar element -> float (fp8: the code's value, scale applied by caller)

__device__ __forceinline__ float to_float(float x) { return x; }
__device__ __forceinline__ float to_float(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ float e4m3_to_float(uint8_t c) {
    uint16_t c16 = c;
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(c16));
    return __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFF)));
}

template <typename Fmt>
__device__ __forceinline__ float load_elem(const void* base, size_t i);
template <>
__device__ __forceinline__ float load_elem<F32>(const void* base, size_t i) {
    return static_cast<const float*>(base)[i];
}
template <>
__device__ __forceinline__ float load_elem<BF16>(const void* base, size_t i) {
    return __bfloat162float(static_cast<const __nv_bfloat16*>(base)[i]);
}
template <>
__device__ __forceinline__ float load_elem<E4M3>(const void* base, size_t i) {
    return e4m3_to_float(static_cast<const uint8_t*>(base)[i]);
}

template <typename Fmt>
__device__ __forceinline__ void store_elem(void* base, size_t i, float v);
template <>
__device__ __forceinline__ void store_elem<F32>(void* base, size_t i, float v) {
    static_cast<float*>(base)[i] = v;
}
template <>
__device__ __forceinline__ void store_elem<BF16>(void* base, size_t i, float v) {
    static_cast<__nv_bfloat16*>(base)[i] = __float2bfloat16_rn(v);
}

// Two floats -> two E4M3 codes (low byte = a), round to nearest even,
// saturating to +-448.
__device__ __forceinline__ uint16_t f32x2_to_e4m3x2(float a, float b) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(b), "f"(a));
    return r;
}

// ---- the conversions of a new token's K/V into the cache format, shared by
// paged_kv_write and the fused write + decode

// 8 consecutive input elements as fp32
template <typename In>
__device__ __forceinline__ void load8(const void* base, size_t i, float v[8]);
template <>
__device__ __forceinline__ void load8<F32>(const void* base, size_t i, float v[8]) {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(base) + i);
    float4 a = __ldg(p), b = __ldg(p + 1);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
template <>
__device__ __forceinline__ void load8<BF16>(const void* base, size_t i, float v[8]) {
    uint4 r = __ldg(reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(base) + i));
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        v[2 * k] = __uint_as_float(w[k] << 16);
        v[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
    }
}
// 8 elements in bf16: round to nearest even
__device__ __forceinline__ uint4 pack8_bf16(const float v[8]) {
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * k], v[2 * k + 1]);
        w[k] = *reinterpret_cast<uint32_t*>(&h);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}
// 8 elements in E4M3: one IEEE fp32 divide by the scale per element, then
// round to nearest even with saturation
__device__ __forceinline__ uint2 pack8_e4m3(const float v[8], float scale) {
    uint32_t w[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        uint32_t lo = f32x2_to_e4m3x2(__fdiv_rn(v[4 * k + 0], scale), __fdiv_rn(v[4 * k + 1], scale));
        uint32_t hi = f32x2_to_e4m3x2(__fdiv_rn(v[4 * k + 2], scale), __fdiv_rn(v[4 * k + 3], scale));
        w[k] = lo | (hi << 16);
    }
    return make_uint2(w[0], w[1]);
}

template <typename Out>
__device__ __forceinline__ void store8(void* base, size_t i, const float v[8], float scale);
template <>
__device__ __forceinline__ void store8<F32>(void* base, size_t i, const float v[8], float) {
    float4* p = reinterpret_cast<float4*>(static_cast<float*>(base) + i);
    p[0] = make_float4(v[0], v[1], v[2], v[3]);
    p[1] = make_float4(v[4], v[5], v[6], v[7]);
}
template <>
__device__ __forceinline__ void store8<BF16>(void* base, size_t i, const float v[8], float) {
    *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(base) + i) = pack8_bf16(v);
}
template <>
__device__ __forceinline__ void store8<E4M3>(void* base, size_t i, const float v[8], float scale) {
    *reinterpret_cast<uint2*>(static_cast<uint8_t*>(base) + i) = pack8_e4m3(v, scale);
}

}  // namespace pkv
