// copy_blocks: copy-on-write duplication of physical blocks.
//
// "LLM推論の基礎とvLLMの内部", section 4: blocks of a shared prefix carry a
// reference count; a write into a shared block first copies it.  The host
// decides the (src, dst) pairs; this kernel moves the bytes, for every layer.
//
// Grid: (pair, layer, K-or-V).  Each CTA streams one block with 16-byte
// vectors; the layer pointers travel in the kernel parameters.
#include "pkv_common.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

__global__ void __launch_bounds__(256) copy_blocks_kernel(const __grid_constant__ CopyParams p) {
    const int pair = blockIdx.x, layer = blockIdx.y, which = blockIdx.z;
    const long long src = p.mapping[2 * pair], dst = p.mapping[2 * pair + 1];
    if (src < 0 || src >= p.NB || dst < 0 || dst >= p.NB) {
        if (layer == 0 && which == 0 && threadIdx.x == 0) report(p.err, PKV_DEVERR_COPY_PAIR);
        return;
    }
    char* base = static_cast<char*>(which ? p.v[layer] : p.k[layer]);
    const uint4* s = reinterpret_cast<const uint4*>(base + (size_t)src * p.block_bytes);
    uint4* d = reinterpret_cast<uint4*>(base + (size_t)dst * p.block_bytes);
    const long long n = (long long)(p.block_bytes / 16);
    long long i = threadIdx.x;
    // four independent 16-byte loads in flight per thread
    for (; i + 3 * blockDim.x < n; i += 4 * blockDim.x) {
        uint4 a = __ldg(s + i), b = __ldg(s + i + blockDim.x);
        uint4 c = __ldg(s + i + 2 * blockDim.x), e = __ldg(s + i + 3 * blockDim.x);
        d[i] = a; d[i + blockDim.x] = b; d[i + 2 * blockDim.x] = c; d[i + 3 * blockDim.x] = e;
    }
    for (; i < n; i += blockDim.x) d[i] = __ldg(s + i);
}

}  // namespace

cudaError_t launch_copy(const CopyParams& p, cudaStream_t st) {
    if (p.P == 0 || p.L == 0) return cudaSuccess;
    dim3 grid(p.P, p.L, 2);
    copy_blocks_kernel<<<grid, 256, 0, st>>>(p);
    return cudaGetLastError();
}

}  // namespace pkv
