// copy_blocks: copy-on-write duplication of physical blocks.
//
// "LLM推論の基礎とvLLMの内部", section 4: blocks of a shared prefix carry a
// reference count; a write into a shared block first copies it.  The host
// decides the (src, dst) pairs; this kernel moves the bytes, for every layer.
//
// Grid: (pair, layer, K-or-V x chunk of 16 KB).  Each CTA moves one chunk of
// one block with 16-byte vectors, all of a thread's loads in flight before
// its stores (a chunk is four vectors per thread): a copy of a few MB is a
// single memory round trip after the launch.  The layer pointers travel in
// the kernel parameters.
#include "pkv_common.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kCopyThreads = 256;
constexpr long long kChunkVecs = 1024;              // 16-byte vectors per CTA
constexpr int kPerThread = (int)(kChunkVecs / kCopyThreads);

// kCheck (the caller passed an error word): besides ids outside the pool,
// a pair is skipped when its destination is also written by another pair or
// read by any pair, since the copies run in no fixed order and the result
// would depend on it.  Every CTA of the pair decides the same way from the
// read-only mapping: its threads scan all P pairs (16 bytes each, from L2).
template <bool kCheck>
__global__ void __launch_bounds__(kCopyThreads) copy_blocks_kernel(const __grid_constant__ CopyParams p) {
    pdl_trigger();
    pdl_wait();
    const int pair = blockIdx.x, layer = blockIdx.y, which = blockIdx.z & 1, chunk = blockIdx.z >> 1;
    const long long src = p.mapping[2 * pair], dst = p.mapping[2 * pair + 1];
    const bool first = layer == 0 && blockIdx.z == 0 && threadIdx.x == 0;
    if (src < 0 || src >= p.NB || dst < 0 || dst >= p.NB) {
        if (first) report(p.err, PKV_DEVERR_COPY_PAIR);
        return;
    }
    if constexpr (kCheck) {
        bool clash = false;
        for (int q = threadIdx.x; q < p.P; q += kCopyThreads) {
            const long long s2 = p.mapping[2 * q], d2 = p.mapping[2 * q + 1];
            const bool in_pool = s2 >= 0 && s2 < p.NB && d2 >= 0 && d2 < p.NB;
            clash |= in_pool && (s2 == dst || (q != pair && d2 == dst));
        }
        if (__syncthreads_or(clash)) {
            if (first) report(p.err, PKV_DEVERR_COPY_PAIR);
            return;
        }
    }
    char* base = static_cast<char*>(which ? p.v[layer] : p.k[layer]);
    const uint4* s = reinterpret_cast<const uint4*>(base + (size_t)src * p.block_bytes);
    uint4* d = reinterpret_cast<uint4*>(base + (size_t)dst * p.block_bytes);
    const long long n = (long long)(p.block_bytes / 16);
    const long long i0 = chunk * kChunkVecs + threadIdx.x;
    uint4 v[kPerThread];
#pragma unroll
    for (int k = 0; k < kPerThread; ++k) {
        const long long i = i0 + (long long)k * kCopyThreads;
        if (i < n) v[k] = __ldg(s + i);
    }
#pragma unroll
    for (int k = 0; k < kPerThread; ++k) {
        const long long i = i0 + (long long)k * kCopyThreads;
        if (i < n) d[i] = v[k];
    }
}

}  // namespace

cudaError_t launch_copy(const CopyParams& p, cudaStream_t st) {
    if (p.P == 0 || p.L == 0) return cudaSuccess;
    const long long n = (long long)(p.block_bytes / 16);
    const long long chunks = (n + kChunkVecs - 1) / kChunkVecs;
    if (chunks < 1 || 2 * chunks > 65535) return cudaErrorInvalidValue;
    dim3 grid(p.P, p.L, (unsigned)(2 * chunks));
    if (p.err != nullptr) return launch_pdl(copy_blocks_kernel<true>, grid, dim3(kCopyThreads), 0, st, p);
    return launch_pdl(copy_blocks_kernel<false>, grid, dim3(kCopyThreads), 0, st, p);
}

}  // namespace pkv
