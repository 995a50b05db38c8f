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

template <typename In, typename Out>
__global__ void __launch_bounds__(256) write_kernel(WriteParams p) {
    pdl_trigger();
    pdl_wait();
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
    pdl_trigger();
    pdl_wait();
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
    const dim3 g(blocks), b(threads);
    if (same) return launch_pdl(write_copy16_kernel, g, b, 0, st, p, in_dt == PKV_F32 ? 4 : 2);
    if (in_dt == PKV_F32 && cache_dt == PKV_BF16) return launch_pdl(write_kernel<F32, BF16>, g, b, 0, st, p);
    if (in_dt == PKV_BF16 && cache_dt == PKV_F32) return launch_pdl(write_kernel<BF16, F32>, g, b, 0, st, p);
    if (in_dt == PKV_F32 && cache_dt == PKV_FP8_E4M3) return launch_pdl(write_kernel<F32, E4M3>, g, b, 0, st, p);
    if (in_dt == PKV_BF16 && cache_dt == PKV_FP8_E4M3) return launch_pdl(write_kernel<BF16, E4M3>, g, b, 0, st, p);
    return cudaErrorInvalidValue;
}

}  // namespace pkv
