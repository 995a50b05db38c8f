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
#include <unordered_map>
#include <unordered_set>
#include <vector>

#include "../../include/pkv.h"

extern "C" {

pkv_status pkv_vtoken_plan(const int32_t* token_slots, int MT, const int32_t* num_tokens, int S, int bs, int NB,
                           int64_t* moves, int64_t max_moves, int64_t* num_moves, int32_t* freed,
                           int64_t max_freed, int64_t* num_freed) {
    if (S < 0 || MT < 1 || bs < 1 || NB < 1 || max_moves < 0 || max_freed < 0 || !num_moves || !num_freed)
        return PKV_ERR_INVALID_ARG;
    if (S > 0 && (!token_slots || !num_tokens)) return PKV_ERR_INVALID_ARG;
    const long long slots = (long long)NB * bs;
    // which sequences reference each block (1 = private; 2 = two or more)
    std::vector<uint8_t> users(NB, 0);
    std::vector<int32_t> last_user(NB, -1);
    for (int s = 0; s < S; ++s) {
        const int n = num_tokens[s];
        if (n < 0 || n > MT) return PKV_ERR_INVALID_ARG;
        std::unordered_set<int32_t> seen;
        seen.reserve(n * 2 + 1);
        for (int t = 0; t < n; ++t) {
            const int32_t sl = token_slots[(size_t)s * MT + t];
            if (sl < 0 || sl >= slots) return PKV_ERR_INVALID_ARG;
            if (!seen.insert(sl).second) return PKV_ERR_INVALID_ARG;
            const int b = sl / bs;
            if (last_user[b] != s) {
                last_user[b] = s;
                if (users[b] < 2) ++users[b];
            }
        }
    }
    std::vector<int64_t> mv;
    std::vector<int32_t> fr;
    for (int s = 0; s < S; ++s) {
        const int n = num_tokens[s];
        const int32_t* row = token_slots + (size_t)s * MT;
        std::unordered_map<int, int> count;
        for (int t = 0; t < n; ++t) {
            const int b = row[t] / bs;
            if (users[b] == 1) ++count[b];
        }
        if (count.empty()) continue;
        long long live = 0;
        for (auto& kv : count) live += kv.second;
        const size_t k = (size_t)((live + bs - 1) / bs);
        if (count.size() <= k) continue;
        std::vector<std::pair<int, int>> order(count.begin(), count.end());   // (block, live)
        std::sort(order.begin(), order.end(), [](const std::pair<int, int>& a, const std::pair<int, int>& b) {
            return a.second != b.second ? a.second > b.second : a.first < b.first;
        });
        std::vector<int> keep, drop;
        for (size_t i = 0; i < order.size(); ++i) (i < k ? keep : drop).push_back(order[i].first);
        std::sort(keep.begin(), keep.end());
        std::sort(drop.begin(), drop.end());
        std::unordered_set<int32_t> used(row, row + n);
        std::vector<int32_t> holes;
        for (int b : keep)
            for (int o = 0; o < bs; ++o)
                if (!used.count(b * bs + o)) holes.push_back(b * bs + o);
        std::unordered_set<int> dropset(drop.begin(), drop.end());
        size_t hi = 0;
        for (int t = 0; t < n; ++t) {
            if (!dropset.count(row[t] / bs)) continue;
            mv.push_back(s);
            mv.push_back(t);
            mv.push_back(row[t]);
            mv.push_back(holes[hi++]);
        }
        fr.insert(fr.end(), drop.begin(), drop.end());
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
