// Repacking of live tokens ("LLM推論の「見えないメモリ問題」を解く … vToken",
// asynchronous repacking): each move names a sequence, the logical index of
// one of its live tokens, the token's current slot and a free destination
// slot.  The first kernel copies the token's K and V rows of every layer
// from the source slot to the destination; the second, ordered after it on
// the stream, rewrites the token-table entry.  Keeping them apart means no
// copy ever reads an entry that another block has already rewritten.  A move
// whose indices are out of range, or whose source is not what the table
// holds, is skipped by both and reported (PKV_DEVERR_MOVE).
#include "pkv_common.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

__device__ __forceinline__ bool move_ok(const RepackParams& p, int m, int64_t& seq, int64_t& idx, int64_t& src,
                                        int64_t& dst) {
    const int64_t* mv = p.moves + 4 * (size_t)m;
    seq = mv[0];
    idx = mv[1];
    src = mv[2];
    dst = mv[3];
    const int64_t slots = (int64_t)p.NB * p.bs;
    return seq >= 0 && seq < p.S && idx >= 0 && idx < p.MT && src >= 0 && src < slots && dst >= 0 && dst < slots &&
           p.token_slots[seq * p.MT + idx] == src;
}

// grid (moves / 8, layers), a warp per move: the token's K and V rows of one
// layer, each lane's 16-byte loads issued before its stores
constexpr int kMovesPerBlock = 8;
__global__ void __launch_bounds__(32 * kMovesPerBlock) repack_copy_kernel(const __grid_constant__ RepackParams p) {
    const int lane = threadIdx.x & 31;
    const long long m = (long long)blockIdx.x * kMovesPerBlock + (threadIdx.x >> 5);
    int64_t seq, idx, src, dst;
    if (m >= p.M || !move_ok(p, (int)m, seq, idx, src, dst)) return;
    const int l = blockIdx.y;
    const size_t n16 = p.token_bytes / 16;
    const uint4* ks = reinterpret_cast<const uint4*>(static_cast<const char*>(p.k[l]) + src * p.token_bytes);
    const uint4* vs = reinterpret_cast<const uint4*>(static_cast<const char*>(p.v[l]) + src * p.token_bytes);
    uint4* kd = reinterpret_cast<uint4*>(static_cast<char*>(p.k[l]) + dst * p.token_bytes);
    uint4* vd = reinterpret_cast<uint4*>(static_cast<char*>(p.v[l]) + dst * p.token_bytes);
    constexpr int kBatch = 4;            // chunks of K (and of V) per lane in flight
    for (size_t i0 = 0; i0 < n16; i0 += 32 * kBatch) {
        uint4 a[kBatch], b[kBatch];
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
            const size_t i = i0 + 32 * j + lane;
            if (i < n16) {
                a[j] = ks[i];
                b[j] = vs[i];
            }
        }
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
            const size_t i = i0 + 32 * j + lane;
            if (i < n16) {
                kd[i] = a[j];
                vd[i] = b[j];
            }
        }
    }
}

// one thread per move: the table entry now names the destination slot
__global__ void __launch_bounds__(256) repack_table_kernel(const __grid_constant__ RepackParams p) {
    const long long m = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (m >= p.M) return;
    int64_t seq, idx, src, dst;
    if (!move_ok(p, (int)m, seq, idx, src, dst)) {
        report(p.err, PKV_DEVERR_MOVE);
        return;
    }
    p.token_slots[seq * p.MT + idx] = (int32_t)dst;
}

}  // namespace

cudaError_t launch_repack(const RepackParams& p, cudaStream_t st) {
    if (p.M == 0 || p.L == 0) return cudaSuccess;
    repack_copy_kernel<<<dim3((unsigned)((p.M + kMovesPerBlock - 1) / kMovesPerBlock), (unsigned)p.L),
                         32 * kMovesPerBlock, 0, st>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    repack_table_kernel<<<(unsigned)((p.M + 255) / 256), 256, 0, st>>>(p);
    return cudaGetLastError();
}

}  // namespace pkv
