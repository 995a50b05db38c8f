// Work units of paged attention over query chunks, shared by the kernels
// that compute it and by the merge of their partitions.
//
// A sequence s with n tokens computes its last q_len tokens as queries
// (a chunk of prefill, or the tokens a speculative decoder proposes).  For
// K/V head kvh its rows are the pairs (query i, head kvh * g + j), row
// r = i * g + j, cut into tiles of ROWS rows; a tile needs the keys up to
// its last query's position n - q_len + i_last, cut into partitions of P
// tokens.  Unit ids run partition-major, then sequence, K/V head, row tile,
// so the tiles of one key range are claimed together and share the K/V
// reads in L2.
#pragma once

#include "pkv_common.cuh"
#include "pkv_internal.h"

namespace pkv {

struct __align__(16) QTile {
    int s, kvh, rt, part;      // sequence, K/V head, row tile, key partition
    int k0, k1;                // key tokens [k0, k1)
    int n, ql;                 // sequence length, queries in the chunk
    int q0, np, rows, pad;     // first query token, partitions of the tile, rows of the sequence
};

// Unit id -> coordinates; false for ids that name no work.  A sequence whose
// length exceeds the host bound, whose query count is outside [0, n] or
// above the host's max_q, or whose queries leave [0, T) is skipped and
// reported once.  rt_max = ceil(max_q * g / ROWS) tiles per (sequence, K/V
// head).
template <int ROWS>
__device__ __forceinline__ bool qtile_of(const DecodeParams& p, const int32_t* query_start, int T, int max_q,
                                         unsigned long long u, int rt_max, QTile& x) {
    const unsigned long long per_part = (unsigned long long)p.S * p.Hkv * rt_max;
    x.part = (int)(u / per_part);
    const unsigned long long rem = u - (unsigned long long)x.part * per_part;
    x.s = (int)(rem / ((unsigned long long)p.Hkv * rt_max));
    const int r2 = (int)(rem - (unsigned long long)x.s * p.Hkv * rt_max);
    x.kvh = r2 / rt_max;
    x.rt = r2 - x.kvh * rt_max;
    const int n = __ldg(p.context_lens + x.s);
    x.q0 = __ldg(query_start + x.s);
    x.ql = __ldg(query_start + x.s + 1) - x.q0;
    if (n < 0 || n > p.max_ctx || x.ql < 0 || x.ql > n || x.ql > max_q || x.q0 < 0 || x.q0 + x.ql > T) {
        if (x.part == 0 && r2 == 0) report(p.err, PKV_DEVERR_QUERY_LEN);
        return false;
    }
    x.n = n;
    x.rows = x.ql * p.g;
    if (x.rt * ROWS >= x.rows) return false;
    const int last_row = min(x.rt * ROWS + ROWS - 1, x.rows - 1);
    const int key_end = n - x.ql + last_row / p.g + 1;
    x.np = (key_end + p.P - 1) / p.P;
    if (x.part >= x.np) return false;
    x.k0 = x.part * p.P;
    x.k1 = min(key_end, x.k0 + p.P);
    return true;
}

}  // namespace pkv
