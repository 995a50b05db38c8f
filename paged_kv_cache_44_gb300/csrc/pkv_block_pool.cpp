// Host block manager for the paged KV cache: the bookkeeping that produces
// the block tables, slot mappings and copy-on-write pairs the device calls
// consume.
//
// "LLM推論の基礎とvLLMの内部", section 4: physical blocks of block_size
// tokens are handed to a request one at a time as it grows; a per-request
// block table maps logical to physical blocks; block 0 is reserved as the
// null block; free blocks sit in a doubly linked queue; shared blocks carry
// a reference count and are copied before a write (copy-on-write).
// Section 5: a full block's hash chains its parent's hash, its tokens and
// extra keys; only full blocks are cached, so hits come in whole blocks, and
// the last prompt token is always recomputed; a finished request returns its
// blocks with their hashes kept, tail first, and free blocks are reused from
// the front of the queue (least recently freed first).
// Reading where the pages are silent: a free block with no hash holds
// nothing worth keeping and is handed out before any cached block.
#include <cstdint>
#include <cstring>
#include <new>
#include <unordered_map>
#include <vector>

#include "../../include/pkv.h"

namespace {

constexpr int kNone = -1;

struct Block {
    int ref = 0;
    int prev = kNone, next = kNone;   // free-queue links
    bool queued = false;
    bool hashed = false;
    uint64_t hash = 0;
};

struct Seq {
    std::vector<int32_t> table;       // physical block per logical block
    std::vector<int32_t> tokens;      // every token (prompt + appended)
    std::vector<uint64_t> hashes;     // chain hash of each full block
    uint64_t mark = 0;                // last batch call that named this sequence
};

// 64-bit mixing (splitmix64 finaliser) for the prefix-hash chain.
uint64_t mix(uint64_t x) {
    x += 0x9e3779b97f4a7c15ull;
    x = (x ^ (x >> 30)) * 0xbf58476d1ce4e5b9ull;
    x = (x ^ (x >> 27)) * 0x94d049bb133111ebull;
    return x ^ (x >> 31);
}

}  // namespace

struct pkv_block_pool {
    int num_blocks = 0, bs = 0;
    bool caching = false;
    uint64_t extra_key = 0;
    std::vector<Block> blocks;
    int head = kNone, tail = kNone;   // free queue: head is reused first
    int nfree = 0;
    std::unordered_map<uint64_t, int> cached;   // hash -> block
    std::unordered_map<int64_t, Seq> seqs;
    uint64_t batch = 0;                         // batch calls so far
    std::vector<Seq*> batch_seqs;

    // ---- free queue
    void q_remove(int b) {
        Block& x = blocks[b];
        if (x.prev != kNone) blocks[x.prev].next = x.next; else head = x.next;
        if (x.next != kNone) blocks[x.next].prev = x.prev; else tail = x.prev;
        x.prev = x.next = kNone;
        x.queued = false;
        --nfree;
    }
    void q_push_back(int b) {
        Block& x = blocks[b];
        x.prev = tail;
        x.next = kNone;
        if (tail != kNone) blocks[tail].next = b; else head = b;
        tail = b;
        x.queued = true;
        ++nfree;
    }
    void q_push_front(int b) {
        Block& x = blocks[b];
        x.next = head;
        x.prev = kNone;
        if (head != kNone) blocks[head].prev = b; else tail = b;
        head = b;
        x.queued = true;
        ++nfree;
    }

    // A block for new contents: the front of the queue, its old hash dropped.
    int take_block() {
        if (head == kNone) return kNone;
        const int b = head;
        q_remove(b);
        Block& x = blocks[b];
        if (x.hashed) {
            auto it = cached.find(x.hash);
            if (it != cached.end() && it->second == b) cached.erase(it);
            x.hashed = false;
        }
        x.ref = 1;
        return b;
    }

    // One reference fewer; a block nobody holds goes back to the queue:
    // cached blocks at the back (kept as long as possible), others at the front.
    void release(int b) {
        Block& x = blocks[b];
        if (--x.ref > 0) return;
        if (x.hashed) q_push_back(b); else q_push_front(b);
    }

    uint64_t chain(uint64_t parent, const int32_t* toks) const {
        uint64_t h = mix(parent ^ mix(extra_key + 0x51ed27ull));
        for (int i = 0; i < bs; ++i) h = mix(h ^ (uint64_t)(uint32_t)toks[i]);
        return h;
    }

    // One token more for `s`: its slot, and the copy-on-write pair if its
    // last block was shared.
    pkv_status append(Seq& s, int32_t token, int64_t* slot, int64_t* cow_src, int64_t* cow_dst) {
        const int pos = (int)s.tokens.size();
        int64_t src = -1, dst = -1;
        if (pos % bs == 0) {
            // the last block is full: a new block
            const int b = take_block();
            if (b == kNone) return PKV_ERR_WORKSPACE;
            s.table.push_back(b);
        } else {
            // the last block has room; a block that is not full carries no hash
            const int last = s.table.back();
            if (blocks[last].ref > 1) {
                // shared with another sequence (a fork): copy before writing
                const int b = take_block();
                if (b == kNone) return PKV_ERR_WORKSPACE;
                src = last;
                dst = b;
                release(last);
                s.table.back() = b;
            }
        }
        s.tokens.push_back(token);
        if ((int)s.tokens.size() % bs == 0) seal(s, (int)s.tokens.size() / bs - 1);
        if (slot) *slot = (int64_t)s.table.back() * bs + pos % bs;
        if (cow_src) *cow_src = src;
        if (cow_dst) *cow_dst = dst;
        return PKV_OK;
    }

    // Give full block j of `s` its chain hash and make it findable.
    void seal(Seq& s, int j) {
        const uint64_t parent = j > 0 ? s.hashes[j - 1] : 0x6b767065ull;
        const uint64_t h = chain(parent, s.tokens.data() + (size_t)j * bs);
        s.hashes.push_back(h);
        if (!caching) return;
        Block& x = blocks[s.table[j]];
        if (x.hashed) return;
        if (cached.find(h) != cached.end()) return;   // an equal block is already cached
        x.hashed = true;
        x.hash = h;
        cached.emplace(h, s.table[j]);
    }
};

extern "C" {

pkv_status pkv_pool_create(int num_blocks, int block_size, int enable_prefix_caching, pkv_block_pool** out) {
    if (!out || num_blocks < 2 || block_size < 1) return PKV_ERR_INVALID_ARG;
    pkv_block_pool* p = new (std::nothrow) pkv_block_pool();
    if (!p) return PKV_ERR_INVALID_ARG;
    p->num_blocks = num_blocks;
    p->bs = block_size;
    p->caching = enable_prefix_caching != 0;
    p->blocks.resize(num_blocks);
    for (int b = 1; b < num_blocks; ++b) p->q_push_back(b);   // block 0 is the null block
    *out = p;
    return PKV_OK;
}

void pkv_pool_destroy(pkv_block_pool* p) { delete p; }

pkv_status pkv_pool_set_extra_key(pkv_block_pool* p, uint64_t extra_key) {
    if (!p) return PKV_ERR_INVALID_ARG;
    p->extra_key = extra_key;
    return PKV_OK;
}

int pkv_pool_num_free_blocks(const pkv_block_pool* p) { return p ? p->nfree : -1; }

int pkv_pool_num_cached_blocks(const pkv_block_pool* p) { return p ? (int)p->cached.size() : -1; }

pkv_status pkv_pool_add_sequence(pkv_block_pool* p, int64_t seq_id, const int32_t* tokens, int n_tokens,
                                 int* num_cached_tokens) {
    if (!p || n_tokens < 1 || !tokens) return PKV_ERR_INVALID_ARG;
    if (p->seqs.count(seq_id)) return PKV_ERR_INVALID_ARG;
    const int bs = p->bs;
    const int nblk = (n_tokens + bs - 1) / bs, nfull = n_tokens / bs;
    // longest cached prefix of whole blocks, leaving at least the last token to compute
    std::vector<int> hits;
    if (p->caching) {
        uint64_t parent = 0x6b767065ull;
        for (int j = 0; j < nfull && (j + 1) * bs <= n_tokens - 1; ++j) {
            const uint64_t h = p->chain(parent, tokens + (size_t)j * bs);
            auto it = p->cached.find(h);
            if (it == p->cached.end()) break;
            hits.push_back(it->second);
            parent = h;
        }
    }
    int held = 0;
    for (int b : hits) held += p->blocks[b].ref == 0;
    if (nblk - (int)hits.size() > p->nfree - held) return PKV_ERR_WORKSPACE;   // not enough free blocks
    Seq s;
    s.tokens.assign(tokens, tokens + n_tokens);
    for (int b : hits) {
        Block& x = p->blocks[b];
        if (x.queued) p->q_remove(b);
        ++x.ref;
        s.table.push_back(b);
    }
    while ((int)s.table.size() < nblk) s.table.push_back(p->take_block());
    for (int j = 0; j < nfull; ++j) p->seal(s, j);
    if (num_cached_tokens) *num_cached_tokens = (int)hits.size() * bs;
    p->seqs.emplace(seq_id, std::move(s));
    return PKV_OK;
}

pkv_status pkv_pool_append_token(pkv_block_pool* p, int64_t seq_id, int32_t token, int64_t* slot,
                                 int64_t* cow_src, int64_t* cow_dst) {
    if (!p) return PKV_ERR_INVALID_ARG;
    auto it = p->seqs.find(seq_id);
    if (it == p->seqs.end()) return PKV_ERR_INVALID_ARG;
    return p->append(it->second, token, slot, cow_src, cow_dst);
}

pkv_status pkv_pool_fork(pkv_block_pool* p, int64_t parent_id, int64_t child_id) {
    if (!p) return PKV_ERR_INVALID_ARG;
    auto it = p->seqs.find(parent_id);
    if (it == p->seqs.end() || p->seqs.count(child_id)) return PKV_ERR_INVALID_ARG;
    Seq child = it->second;
    for (int b : child.table) ++p->blocks[b].ref;
    p->seqs.emplace(child_id, std::move(child));
    return PKV_OK;
}

pkv_status pkv_pool_free_sequence(pkv_block_pool* p, int64_t seq_id) {
    if (!p) return PKV_ERR_INVALID_ARG;
    auto it = p->seqs.find(seq_id);
    if (it == p->seqs.end()) return PKV_ERR_INVALID_ARG;
    const std::vector<int32_t>& t = it->second.table;
    for (int j = (int)t.size() - 1; j >= 0; --j) p->release(t[j]);   // tail first
    p->seqs.erase(it);
    return PKV_OK;
}

pkv_status pkv_pool_block_table(const pkv_block_pool* p, int64_t seq_id, int32_t* table, int max_blocks,
                                int* num_blocks, int* num_tokens) {
    if (!p) return PKV_ERR_INVALID_ARG;
    auto it = p->seqs.find(seq_id);
    if (it == p->seqs.end()) return PKV_ERR_INVALID_ARG;
    const Seq& s = it->second;
    const int n = (int)s.table.size();
    if (num_blocks) *num_blocks = n;
    if (num_tokens) *num_tokens = (int)s.tokens.size();
    if (table) {
        if (max_blocks < n) return PKV_ERR_INVALID_ARG;
        std::memcpy(table, s.table.data(), sizeof(int32_t) * n);
        for (int j = n; j < max_blocks; ++j) table[j] = 0;    // padding: the null block
    }
    return PKV_OK;
}

pkv_status pkv_pool_append_tokens(pkv_block_pool* p, const int64_t* seq_ids, const int32_t* tokens, int n,
                                  int64_t* slot_mapping, int64_t* block_mapping, int* num_copies) {
    if (!p || n < 0 || (n > 0 && (!seq_ids || !tokens || !slot_mapping || !block_mapping || !num_copies)))
        return PKV_ERR_INVALID_ARG;
    // every id must exist and appear once; enough free blocks for the worst case
    int worst = 0;
    const uint64_t mark = ++p->batch;
    p->batch_seqs.resize((size_t)n);
    for (int i = 0; i < n; ++i) {
        auto it = p->seqs.find(seq_ids[i]);
        if (it == p->seqs.end() || it->second.mark == mark) return PKV_ERR_INVALID_ARG;
        Seq& s = it->second;
        s.mark = mark;
        p->batch_seqs[i] = &s;
        worst += (s.tokens.size() % p->bs == 0) || p->blocks[s.table.back()].ref > 1;
    }
    if (worst > p->nfree) return PKV_ERR_WORKSPACE;
    int nc = 0;
    for (int i = 0; i < n; ++i) {
        int64_t src = -1, dst = -1;
        const pkv_status st = p->append(*p->batch_seqs[i], tokens[i], slot_mapping + i, &src, &dst);
        if (st != PKV_OK) return st;   // cannot happen after the checks above
        if (src >= 0) {
            block_mapping[2 * nc] = src;
            block_mapping[2 * nc + 1] = dst;
            ++nc;
        }
    }
    *num_copies = nc;
    return PKV_OK;
}

pkv_status pkv_pool_block_tables(const pkv_block_pool* p, const int64_t* seq_ids, int n, int32_t* tables,
                                 int max_blocks, int32_t* context_lens) {
    if (!p || n < 0 || max_blocks < 1 || (n > 0 && (!seq_ids || !tables || !context_lens)))
        return PKV_ERR_INVALID_ARG;
    for (int i = 0; i < n; ++i) {
        int nb = 0, nt = 0;
        const pkv_status st =
            pkv_pool_block_table(p, seq_ids[i], tables + (size_t)i * max_blocks, max_blocks, &nb, &nt);
        if (st != PKV_OK) return st;
        context_lens[i] = nt;
    }
    return PKV_OK;
}

int pkv_pool_block_ref_count(const pkv_block_pool* p, int block) {
    if (!p || block < 0 || block >= p->num_blocks) return -1;
    return p->blocks[block].ref;
}

}  // extern "C"
