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

// Record the first device-side problem; never traps.
__device__ __forceinline__ void report(int32_t* err, int code) {
    if (err != nullptr) atomicCAS(err, 0, code);
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

}  // namespace pkv
