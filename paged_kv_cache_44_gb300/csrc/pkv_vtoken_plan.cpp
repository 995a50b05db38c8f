// Host planner for token repacking ("LLM推論の「見えないメモリ問題」を解く …
// vToken", asynchronous repacking): decides which live tokens move where so
// that each sequence's tokens fill as few blocks as possible and the blocks
// they leave can be released.  Policy, per sequence, over the blocks only
// that sequence references: it needs k = ceil(live tokens there / bs)
// blocks; the k with the most live tokens stay (lower block id first on
// ties); its tokens in the other blocks move, in logical order, to the free
// slots of the kept blocks, lowest slot first; the other blocks are then
// empty and released.  A block several sequences reference (a shared
// prefix) stays where it is and lends no free slots.
#include <algorithm>
#include <vector>

#include "../../include/pkv.h"

// Flat arrays instead of hash sets: one bit per slot of the pool marks the
// slots the current sequence lists (set while a sequence is examined, then
// cleared through its own row), and per-block counters are reset through
// the list of blocks the sequence touched.  Host memory: one bit per slot
// and about ten bytes per block.

extern "C" {

pkv_status pkv_vtoken_plan(const int32_t* token_slots, int MT, const int32_t* num_tokens, int S, int bs, int NB,
                           int64_t* moves, int64_t max_moves, int64_t* num_moves, int32_t* freed,
                           int64_t max_freed, int64_t* num_freed) {
    if (S < 0 || MT < 1 || bs < 1 || NB < 1 || max_moves < 0 || max_freed < 0 || !num_moves || !num_freed)
        return PKV_ERR_INVALID_ARG;
    if (S > 0 && (!token_slots || !num_tokens)) return PKV_ERR_INVALID_ARG;
    const long long slots = (long long)NB * bs;
    std::vector<uint64_t> listed((size_t)((slots + 63) / 64), 0);
    auto test_set = [&](int32_t sl) {                     // true if the bit was already set
        uint64_t& w = listed[(size_t)sl >> 6];
        const uint64_t bit = 1ull << (sl & 63);
        const bool was = (w & bit) != 0;
        w |= bit;
        return was;
    };
    auto clear_row = [&](const int32_t* row, int n) {
        for (int t = 0; t < n; ++t) listed[(size_t)row[t] >> 6] = 0;
    };
    // which sequences reference each block (1 = private; 2 = two or more)
    std::vector<uint8_t> users(NB, 0);
    std::vector<int32_t> last_user(NB, -1);
    for (int s = 0; s < S; ++s) {
        const int n = num_tokens[s];
        if (n < 0 || n > MT) return PKV_ERR_INVALID_ARG;
        const int32_t* row = token_slots + (size_t)s * MT;
        for (int t = 0; t < n; ++t) {
            const int32_t sl = row[t];
            if (sl < 0 || sl >= slots) return PKV_ERR_INVALID_ARG;
            if (test_set(sl)) return PKV_ERR_INVALID_ARG;     // listed twice by one sequence
            const int b = sl / bs;
            if (last_user[b] != s) {
                last_user[b] = s;
                if (users[b] < 2) ++users[b];
            }
        }
        clear_row(row, n);
    }
    long long total = 0;
    for (int s = 0; s < S; ++s) total += num_tokens[s];
    std::vector<int64_t> mv;
    std::vector<int32_t> fr;
    mv.reserve((size_t)std::min<long long>(4 * total, 4 * (long long)max_moves + 4));
    std::vector<int32_t> count(NB, 0);       // live tokens of the current sequence per private block
    std::vector<uint8_t> dropped(NB, 0);
    std::vector<int32_t> touched, keep, drop, holes;
    for (int s = 0; s < S; ++s) {
        const int n = num_tokens[s];
        const int32_t* row = token_slots + (size_t)s * MT;
        touched.clear();
        long long live = 0;
        for (int t = 0; t < n; ++t) {
            test_set(row[t]);
            const int b = row[t] / bs;
            if (users[b] != 1) continue;
            if (count[b]++ == 0) touched.push_back(b);
            ++live;
        }
        const size_t k = (size_t)((live + bs - 1) / bs);
        if (touched.size() > k) {
            // the k blocks with the most live tokens stay (lower id first on ties)
            std::sort(touched.begin(), touched.end(), [&](int a, int b) {
                return count[a] != count[b] ? count[a] > count[b] : a < b;
            });
            keep.assign(touched.begin(), touched.begin() + k);
            drop.assign(touched.begin() + k, touched.end());
            std::sort(keep.begin(), keep.end());
            std::sort(drop.begin(), drop.end());
            // free slots of the kept blocks, lowest first
            holes.clear();
            for (int b : keep)
                for (int o = 0; o < bs; ++o) {
                    const long long sl = (long long)b * bs + o;
                    if (!((listed[(size_t)sl >> 6] >> (sl & 63)) & 1ull)) holes.push_back((int32_t)sl);
                }
            for (int b : drop) dropped[b] = 1;
            size_t hi = 0;
            for (int t = 0; t < n; ++t) {
                if (!dropped[row[t] / bs]) continue;
                mv.push_back(s);
                mv.push_back(t);
                mv.push_back(row[t]);
                mv.push_back(holes[hi++]);
            }
            for (int b : drop) dropped[b] = 0;
            fr.insert(fr.end(), drop.begin(), drop.end());
        }
        for (int b : touched) count[b] = 0;
        clear_row(row, n);
    }
    *num_moves = (int64_t)(mv.size() / 4);
    *num_freed = (int64_t)fr.size();
    if (*num_moves > max_moves || *num_freed > max_freed) return PKV_ERR_WORKSPACE;
    if (!mv.empty()) {
        if (!moves) return PKV_ERR_INVALID_ARG;
        std::copy(mv.begin(), mv.end(), moves);
    }
    if (!fr.empty()) {
        if (!freed) return PKV_ERR_INVALID_ARG;
        std::copy(fr.begin(), fr.end(), freed);
    }
    return PKV_OK;
}

}  // extern "C"
