// paged_kv_write: scatter each new token's K and V into its slot.
//
// "LLM推論の基礎とvLLMの内部", section 4: blocks are handed to a request one
// at a time, so a new token occupies one slot (block, offset) of the pool;
// section 2: with --kv-cache-dtype fp8 each element is one byte.
//
// One thread moves 8 consecutive elements of one (token, K-or-V, head) row:
// a 16-byte (bf16) or two 16-byte (fp32) loads, and 32/16/8-byte stores.
#include "pkv_common.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

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
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * k], v[2 * k + 1]);
        w[k] = *reinterpret_cast<uint32_t*>(&h);
    }
    *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(base) + i) = make_uint4(w[0], w[1], w[2], w[3]);
}
template <>
__device__ __forceinline__ void store8<E4M3>(void* base, size_t i, const float v[8], float scale) {
    uint32_t w[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        // one IEEE fp32 divide per element, then RNE + saturation to e4m3
        uint32_t lo = f32x2_to_e4m3x2(__fdiv_rn(v[4 * k + 0], scale), __fdiv_rn(v[4 * k + 1], scale));
        uint32_t hi = f32x2_to_e4m3x2(__fdiv_rn(v[4 * k + 2], scale), __fdiv_rn(v[4 * k + 3], scale));
        w[k] = lo | (hi << 16);
    }
    *reinterpret_cast<uint2*>(static_cast<uint8_t*>(base) + i) = make_uint2(w[0], w[1]);
}

template <typename In, typename Out>
__global__ void __launch_bounds__(256) write_kernel(WriteParams p) {
    const int chunks = p.d / 8;
    const long long total = (long long)p.T * 2 * p.Hkv * chunks;
    const long long slots = (long long)p.NB * p.bs;
    for (long long it = (long long)blockIdx.x * blockDim.x + threadIdx.x; it < total;
         it += (long long)gridDim.x * blockDim.x) {
        const int c = (int)(it % chunks);
        long long r = it / chunks;
        const int h = (int)(r % p.Hkv);
        r /= p.Hkv;
        const int which = (int)(r & 1);       // 0 = K, 1 = V
        const long long i = r >> 1;           // token
        const long long s = p.slot_mapping[i];
        if (s < 0) continue;
        if (s >= slots) {
            if (which == 0 && h == 0 && c == 0) report(p.err, PKV_DEVERR_SLOT);
            continue;
        }
        const long long blk = s / p.bs, off = s % p.bs;
        const size_t src = ((size_t)i * p.Hkv + h) * p.d + (size_t)c * 8;
        const size_t dst = (((size_t)blk * p.bs + off) * p.Hkv + h) * p.d + (size_t)c * 8;
        float v[8];
        load8<In>(which ? p.value : p.key, src, v);
        store8<Out>(which ? p.value_cache : p.key_cache, dst, v, which ? p.v_scale : p.k_scale);
    }
}

// bf16 -> bf16 is a pure copy of the bits.
__global__ void __launch_bounds__(256) write_copy16_kernel(WriteParams p, int elem_bytes) {
    const int chunks = p.d * elem_bytes / 16;
    const long long total = (long long)p.T * 2 * p.Hkv * chunks;
    const long long slots = (long long)p.NB * p.bs;
    for (long long it = (long long)blockIdx.x * blockDim.x + threadIdx.x; it < total;
         it += (long long)gridDim.x * blockDim.x) {
        const int c = (int)(it % chunks);
        long long r = it / chunks;
        const int h = (int)(r % p.Hkv);
        r /= p.Hkv;
        const int which = (int)(r & 1);
        const long long i = r >> 1;
        const long long s = p.slot_mapping[i];
        if (s < 0) continue;
        if (s >= slots) {
            if (which == 0 && h == 0 && c == 0) report(p.err, PKV_DEVERR_SLOT);
            continue;
        }
        const long long blk = s / p.bs, off = s % p.bs;
        const size_t row = (size_t)p.d * elem_bytes;
        const char* src = static_cast<const char*>(which ? p.value : p.key) + ((size_t)i * p.Hkv + h) * row;
        char* dst = static_cast<char*>(which ? p.value_cache : p.key_cache) +
                    (((size_t)blk * p.bs + off) * p.Hkv + h) * row;
        reinterpret_cast<uint4*>(dst)[c] = __ldg(reinterpret_cast<const uint4*>(src) + c);
    }
}

}  // namespace

cudaError_t launch_write(const WriteParams& p, pkv_dtype in_dt, pkv_dtype cache_dt, cudaStream_t st) {
    if (p.T == 0) return cudaSuccess;
    const int threads = 256;
    const bool same = (in_dt == cache_dt);
    const long long items = (long long)p.T * 2 * p.Hkv * (same ? p.d * (in_dt == PKV_F32 ? 4 : 2) / 16 : p.d / 8);
    const long long want = (items + threads - 1) / threads;
    const int blocks = (int)(want < 65536 ? want : 65536);
    if (same) {
        write_copy16_kernel<<<blocks, threads, 0, st>>>(p, in_dt == PKV_F32 ? 4 : 2);
    } else if (in_dt == PKV_F32 && cache_dt == PKV_BF16) {
        write_kernel<F32, BF16><<<blocks, threads, 0, st>>>(p);
    } else if (in_dt == PKV_BF16 && cache_dt == PKV_F32) {
        write_kernel<BF16, F32><<<blocks, threads, 0, st>>>(p);
    } else if (in_dt == PKV_F32 && cache_dt == PKV_FP8_E4M3) {
        write_kernel<F32, E4M3><<<blocks, threads, 0, st>>>(p);
    } else if (in_dt == PKV_BF16 && cache_dt == PKV_FP8_E4M3) {
        write_kernel<BF16, E4M3><<<blocks, threads, 0, st>>>(p);
    } else {
        return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace pkv
