/*
 * pkv -- paged KV-cache decode attention for GB300 (sm_103a).
 *
 * C ABI of libpkv.so.  Every pointer argument is a DEVICE pointer unless its
 * comment says "host".  Every call is asynchronous on `stream`: it validates
 * its arguments on the host, enqueues kernels, and returns without waiting
 * for the GPU.  No call allocates memory or synchronises the host, so the
 * write, decode and copy calls can be recorded into a CUDA graph (tested);
 * pkv_paged_attention_decode_static is described on its own below.  The
 * caller owns every buffer, including the decode workspace.
 *
 * Layouts (all row-major, contiguous, 16-byte aligned base pointers):
 *   new tokens  key / value        [T,  Hkv, d]
 *   query / out                    [S,  Hq,  d]
 *   caches      key / value_cache  [NB, bs,  Hkv, d]   (one layer)
 *   block_tables                   int32 [S, MB]
 *   context_lens                   int32 [S]
 *   slot_mapping                   int64 [T]
 *   block_mapping                  int64 [P, 2]  (src, dst)
 * Sizes: Hq = query heads, Hkv = K/V heads (Hq % Hkv == 0; query head h
 * reads K/V head h / (Hq / Hkv)), d = head dimension, bs = tokens per
 * physical block, NB = physical blocks in the pool, MB = table entries per
 * sequence.
 *
 * Error behaviour.  Problems visible on the host (null pointers, bad sizes,
 * unsupported dtypes or shapes, a workspace that is too small) return a
 * status other than PKV_OK before anything is enqueued.  Problems visible
 * only on the device (a block id outside [0, NB), a context length above
 * max_context_len, a slot outside [0, NB * bs), a copy pair out of range) never
 * fault: the offending block, token or pair is skipped and, when `err_word`
 * is not NULL, the first such problem's code (PKV_DEVERR_*) is stored there
 * with an atomic compare-and-swap from 0.  A launch failure returns
 * PKV_ERR_CUDA.
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PKV_API __attribute__((visibility("default")))
#else
#define PKV_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* pkv_stream_t;   /* same handle as cudaStream_t; NULL = legacy stream */

typedef enum {
    PKV_OK = 0,
    PKV_ERR_INVALID_ARG = 1,
    PKV_ERR_UNSUPPORTED = 2,
    PKV_ERR_WORKSPACE = 3,
    PKV_ERR_CUDA = 4
} pkv_status;

typedef enum {
    PKV_F32 = 0,       /* IEEE binary32 */
    PKV_BF16 = 1,      /* bfloat16 */
    PKV_FP8_E4M3 = 2   /* OCP fp8 E4M3 ("fn": max 448, no infinities); value = code * scale */
} pkv_dtype;

/* Device-side error codes stored into *err_word. */
enum {
    PKV_DEVERR_NONE = 0,
    PKV_DEVERR_BLOCK_ID = 1,      /* a block table entry outside [0, NB) */
    PKV_DEVERR_CONTEXT_LEN = 2,   /* context_lens[s] < 0 or > max_context_len (clamped) */
    PKV_DEVERR_SLOT = 3,          /* slot_mapping[i] >= NB * bs, or a token-table slot outside [0, NB * bs) */
    PKV_DEVERR_COPY_PAIR = 4,     /* a copy pair with an id outside [0, NB), or whose destination another
                                     pair also writes or any pair reads (see pkv_copy_blocks) */
    PKV_DEVERR_TIMEOUT = 5,       /* a staged copy did not land within ~2 s; the kernel gave up */
    PKV_DEVERR_QUERY_LEN = 6,     /* prefill: a sequence's queries are < 0, more than its length or
                                     than max_query_len, or outside [0, T) (the sequence is skipped) */
    PKV_DEVERR_MOVE = 7           /* repack: a move out of range, or whose source is not the slot the
                                     token table holds (the move is skipped) */
};

/*
 * paged_kv_write -- store each new token's K and V into its slot
 * (vLLM's reshape_and_cache).
 *
 * Source: "LLM推論の基礎とvLLMの内部", section 4 "PagedAttentionとブロック
 * 管理": the KV cache is cut into fixed-size blocks that are handed to a
 * request one at a time as its tokens arrive, so each new token lands in one
 * slot of one physical block; section 2 of the same page: an fp8 KV cache
 * (--kv-cache-dtype fp8) stores one byte per element.
 *
 * For token i with s = slot_mapping[i]: s < 0 skips the token; otherwise
 * key_cache[s / bs][s % bs][h][:] = convert(key[i][h][:]) for every K/V head
 * h, and the same for value.  Conversions: f32->f32, bf16->bf16, bf16->f32
 * exact; f32->bf16 round to nearest even; (f32|bf16)->E4M3 stores
 * e4m3(float(x) / k_scale) (v_scale for V) with one IEEE fp32 divide,
 * round-to-nearest-even and saturation to +-448.
 * Supported: in_dtype in {F32, BF16}; cache_dtype in {F32, BF16, FP8_E4M3};
 * d a multiple of 8, at most 512.  T == 0 is a no-op.  Duplicate slots in
 * one call race (which token wins is unspecified).
 */
PKV_API pkv_status pkv_paged_kv_write(const void* key, const void* value, pkv_dtype in_dtype,
                              void* key_cache, void* value_cache, pkv_dtype cache_dtype,
                              const int64_t* slot_mapping, int T,
                              int NB, int bs, int Hkv, int d,
                              float k_scale, float v_scale,
                              int32_t* err_word, pkv_stream_t stream);

/*
 * Bytes of workspace pkv_paged_attention_decode needs for these sizes and
 * this partition request (see below); 0 for invalid arguments.  The
 * workspace holds a 256-byte scheduling header and, when a sequence may span
 * several partitions, one (max, sum, weighted sum) triple per (sequence,
 * query head, partition or chunk; see below).  The header must be zero before a workspace is
 * first used (every decode leaves it zero when it completes, so zero-filling
 * once at allocation is enough).  One workspace must not be used by two
 * decodes that may run at the same time.
 */
PKV_API size_t pkv_decode_workspace_size(int S, int Hq, int Hkv, int d, int bs,
                                 int max_context_len, int partition_size);

/*
 * Partition size (tokens) that a decode with these arguments will use:
 * the request itself when it is > 0, no split (returns 0) when it is -1,
 * and the library's choice when it is 0 (an E4M3 cache on the tensor-core
 * kernel may then take twice this size, in the same workspace; see
 * pkv_paged_attention_decode).  Returns -1 for invalid arguments.
 */
PKV_API int pkv_decode_partition_size(int S, int Hq, int Hkv, int d, int bs,
                              int max_context_len, int partition_size);

/*
 * paged_attention_decode -- one query token per sequence attends to every
 * cached token of that sequence, read through its block table.
 *
 * Source: "LLM推論の基礎とvLLMの内部", section 4: each request keeps a table
 * from logical blocks to physical blocks and the attention kernel reads K/V
 * through it; section 12 of the same page: PagedAttention changes where K/V
 * live, not what attention computes; section 2: GQA lets several query
 * heads share one K/V head.  "vLLM 内部構造 (2) — PagedAttention", section
 * "ブロックテーブル": logically contiguous, physically scattered blocks.
 *
 * For sequence s with n = context_lens[s] and query head h (K/V head
 * kvh = h / (Hq / Hkv)):
 *   k_t, v_t = key/value_cache[block_tables[s][t / bs]][t % bs][kvh], t < n
 *   x_t = scale * <query[s][h], k_t>,  p = softmax(x),  out[s][h] = sum p_t v_t
 * (for E4M3 caches k_t and v_t are code * k_scale and code * v_scale).  A
 * sequence with n == 0 gets zeros.  Arithmetic is fp32 with fp32
 * accumulation; out has the dtype of query.
 *
 * Long contexts are split into partitions of `partition_size` tokens
 * (a multiple of bs): each partition keeps its own running max and sum, and
 * a second pass merges them (M = max m_p, L = sum e^(m_p - M) l_p,
 * O = sum e^(m_p - M) acc_p / L).  When a decode is split, each sequence's
 * last, partial partition is processed in chunks of a quarter partition
 * (rounded down to a multiple of 32 tokens; partitions under 128 tokens are
 * not cut), which are merged like partitions: the launch then ends on small
 * pieces of work.  With an E4M3 cache on the tensor-core kernel, a sequence
 * of four or more full partitions has its last full partition cut into
 * chunks too.  partition_size: 0 = library choice,
 * -1 = never split, > 0 = that size.  The library's choice depends on the
 * sizes alone (so does the workspace size); an E4M3 cache on the
 * tensor-core kernel then takes twice that partition where the launch keeps
 * at least half as many units and the same workspace holds its partial
 * results (its units are bound by their own arithmetic, and fewer, longer
 * ones end the launch sooner).  When any sequence may span more than
 * one partition, `workspace` must hold pkv_decode_workspace_size(...) bytes,
 * else PKV_ERR_WORKSPACE is returned.
 *
 * max_context_len (host) must be >= every context_lens[s] and <= MB * bs; it
 * sizes the launch without reading device memory.  Supported: q_dtype in
 * {F32, BF16}; cache_dtype in {F32, BF16, FP8_E4M3}; d in {64, 128};
 * bs in {16, 32}; any group size Hq / Hkv >= 1 (a K/V head's query heads
 * are processed up to 8 at a time, each such set reading the head's K/V).
 * For E4M3 caches the query is rounded to fp16 for the tensor-core
 * products, so |query| must stay below 65504.
 */
PKV_API pkv_status pkv_paged_attention_decode(void* out, const void* query, pkv_dtype q_dtype,
                                      const void* key_cache, const void* value_cache,
                                      pkv_dtype cache_dtype,
                                      const int32_t* block_tables, int MB,
                                      const int32_t* context_lens, int S, int max_context_len,
                                      int Hq, int Hkv, int d, int bs, int NB,
                                      float scale, float k_scale, float v_scale,
                                      int partition_size,
                                      void* workspace, size_t workspace_bytes,
                                      int32_t* err_word, pkv_stream_t stream);

/*
 * paged_kv_write_decode -- pkv_paged_kv_write of one new token per sequence
 * followed by pkv_paged_attention_decode, in one launch (plus the merge
 * when split).  key/value [S, Hkv, d] (in_dtype f32 or bf16) are the new
 * tokens, slot_mapping [S] int64 their slots, which must be the slots of
 * the sequences' last positions (context_lens[s] - 1, through
 * block_tables); a negative slot skips that sequence's write, as in
 * paged_kv_write.  The caches end up as after the two calls and the output
 * equals theirs bit for bit.  The decode unit that holds a sequence's last
 * token puts the converted new K/V into its staged rows and stores them to
 * the slot.  Supported: the tensor-core decode's dtypes (see
 * pkv_paged_attention_decode_ex); anything else returns PKV_ERR_UNSUPPORTED.
 * Source: the two calls' passages; one launch per step instead of two.
 */
PKV_API pkv_status pkv_paged_kv_write_decode(void* out, const void* query, pkv_dtype q_dtype,
                                             const void* key, const void* value, pkv_dtype in_dtype,
                                             void* key_cache, void* value_cache, pkv_dtype cache_dtype,
                                             const int64_t* slot_mapping,
                                             const int32_t* block_tables, int MB,
                                             const int32_t* context_lens, int S, int max_context_len,
                                             int Hq, int Hkv, int d, int bs, int NB,
                                             float scale, float k_scale, float v_scale,
                                             int partition_size,
                                             void* workspace, size_t workspace_bytes,
                                             int32_t* err_word, pkv_stream_t stream);

/* Kernel choice for pkv_paged_attention_decode_ex. */
typedef enum {
    PKV_DECODE_AUTO = 0,          /* tensor cores where supported, else CUDA cores */
    PKV_DECODE_CUDA_CORES = 1,    /* the CUDA-core kernel (every dtype) */
    PKV_DECODE_TENSOR_CORES = 2   /* the tensor-core kernel; PKV_ERR_UNSUPPORTED where it does not apply
                                     (it needs a bf16 query with a bf16 cache, or an E4M3 cache) */
} pkv_decode_kernel;

/*
 * Same as pkv_paged_attention_decode, with an explicit kernel choice
 * (`kernel` is a pkv_decode_kernel).  Both kernels compute the same
 * function; the choice exists so the two can be measured against each
 * other.
 */
PKV_API pkv_status pkv_paged_attention_decode_ex(void* out, const void* query, pkv_dtype q_dtype,
                                         const void* key_cache, const void* value_cache,
                                         pkv_dtype cache_dtype,
                                         const int32_t* block_tables, int MB,
                                         const int32_t* context_lens, int S, int max_context_len,
                                         int Hq, int Hkv, int d, int bs, int NB,
                                         float scale, float k_scale, float v_scale,
                                         int partition_size,
                                         void* workspace, size_t workspace_bytes,
                                         int32_t* err_word, pkv_stream_t stream, int kernel);

/*
 * Partition size (tokens) a decode launch with these arguments uses:
 * pkv_decode_partition_size's answer, except that with the library's choice
 * (partition_size 0) an E4M3 cache on the tensor-core kernel may take twice
 * it (see pkv_paged_attention_decode; the workspace size is the same).
 * `kernel` is a pkv_decode_kernel; NB is the number of cache blocks.  The
 * paged decode, the fused write + decode and the token-table decode follow
 * the same rule.  Returns 0 for no split, -1 for invalid arguments (and
 * for PKV_DECODE_TENSOR_CORES where that kernel does not apply).  Touches
 * no device memory.
 */
PKV_API int pkv_decode_launch_partition_size(int S, int Hq, int Hkv, int d, int bs, int NB,
                                             int max_context_len, int partition_size,
                                             pkv_dtype q_dtype, pkv_dtype cache_dtype, int kernel);

/*
 * copy_blocks -- copy-on-write duplication of physical blocks.
 *
 * Source: "LLM推論の基礎とvLLMの内部", section 4: blocks of a shared prefix
 * carry a reference count and are copied when written (copy-on-write);
 * "vLLM 内部構造 (2) — PagedAttention", section "共有": many requests with
 * the same system prompt point at one set of physical blocks.
 *
 * For every layer l < num_layers and pair p < P with
 * (src, dst) = block_mapping[p]: block dst of key_caches[l] and of
 * value_caches[l] becomes a byte copy of block src (block_bytes bytes each,
 * = bs * Hkv * d * element size).  key_caches / value_caches are HOST arrays
 * of num_layers device pointers (at most 256 layers); the call copies them
 * into the launch, so the arrays may be freed when it returns.  block_bytes
 * must be a multiple of 16.
 *
 * The pairs are copied in no fixed order, so the destinations must be
 * distinct and must not be sources (the host that decides copy-on-write
 * guarantees this).  A pair with an id outside [0, NB) is always skipped.
 * When err_word is not NULL the pairs are also checked against each other:
 * a pair whose destination another in-pool pair also writes, or any
 * in-pool pair (itself included) reads, is skipped, and PKV_DEVERR_COPY_PAIR
 * is reported; the other pairs are copied.  This check scans the whole
 * mapping in every CTA of the copy (16 bytes per pair, from L2), which is
 * negligible for tens of pairs and grows with P * P for thousands.  With
 * err_word NULL nothing is checked and such pairs race.
 */
PKV_API pkv_status pkv_copy_blocks(void* const* key_caches, void* const* value_caches, int num_layers,
                           const int64_t* block_mapping, int P, int NB, size_t block_bytes,
                           int32_t* err_word, pkv_stream_t stream);

/*
 * Bytes of fixed device scratch behind pkv_paged_attention_decode_static
 * (32 MiB).
 */
#define PKV_STATIC_SCRATCH_BYTES (32u << 20)

/*
 * pkv_paged_attention_decode_static -- the same decode, for callers that
 * cannot allocate device memory.
 *
 * This call has no counterpart on the pages: it is a convenience of this
 * library.  pkv_paged_attention_decode needs a workspace that its caller
 * allocates.  Some callers cannot allocate device memory where they decode:
 * an engine that reserves all of its memory at start-up and forbids later
 * allocations, a latency-critical loop that must not wait on the allocator,
 * a foreign-language caller that holds raw pointers but no allocator.  This
 * entry point takes the same arguments minus the workspace and allocates
 * nothing: its scratch is a fixed array of PKV_STATIC_SCRATCH_BYTES in
 * device memory that the library defines at file scope.  Every GPU that
 * loads the library holds that array until the process exits.  The caller
 * still passes and owns every input and output.
 *
 * Limits and behaviour:
 *  - The arguments are checked as pkv_paged_attention_decode checks them,
 *    with the same status codes, before anything is enqueued.
 *  - The scratch the call needs is pkv_decode_workspace_size(...) for the
 *    same sizes and partition request.  If that exceeds
 *    PKV_STATIC_SCRATCH_BYTES the call returns PKV_ERR_WORKSPACE and
 *    enqueues nothing; a larger partition_size needs less scratch.
 *  - `stream` must belong to the current device (the array used is the
 *    current device's); a stream of another device gives
 *    PKV_ERR_INVALID_ARG and nothing is enqueued.
 *  - The first call on a device looks up the array's device address (with
 *    that device current) and caches it with the device's CUDA context.
 *    After a device reset (a new context) the next call looks the address
 *    up again.
 *  - Each call clears the array's 256-byte work-counter header on `stream`
 *    (a memset) before the decode; the rest keeps the previous call's
 *    contents and needs no clearing.
 *  - All calls share the one array per device: two calls whose work may
 *    overlap on the GPU (different streams, or different host threads)
 *    race and give wrong results.  Serialise them.
 *  - The call makes no cudaMalloc or cudaFree and no other allocating call.
 */
PKV_API pkv_status pkv_paged_attention_decode_static(void* out, const void* query, pkv_dtype q_dtype,
                                                     const void* key_cache, const void* value_cache,
                                                     pkv_dtype cache_dtype,
                                                     const int32_t* block_tables, int MB,
                                                     const int32_t* context_lens, int S, int max_context_len,
                                                     int Hq, int Hkv, int d, int bs, int NB,
                                                     float scale, float k_scale, float v_scale,
                                                     int partition_size,
                                                     int32_t* err_word, pkv_stream_t stream);

/*
 * paged_attention_prefill -- several query tokens per sequence, causal: a
 * chunk of a prompt (chunked prefill) or the tokens a speculative decoder
 * proposes, attending through the same block tables.
 *
 * Source: "LLM推論の基礎とvLLMの内部", section 6: chunked prefill runs a
 * long prompt in per-step pieces next to other requests' decodes; section 3:
 * the V1 scheduler gives every request the tokens it still has to compute,
 * speculative ones included, without separate prefill and decode phases.
 *
 * query/out [T, Hq, d] pack every sequence's queries: those of sequence s
 * are rows query_start[s] .. query_start[s+1] (int32 [S+1], device, rising,
 * query_start[S] = T).  They are the sequence's last q_len tokens, whose
 * K/V are already in the cache (pkv_paged_kv_write first): query i sits at
 * position p = context_lens[s] - q_len + i and attends to tokens 0..p.
 * partition_size splits long key ranges like the decode's (0 = library
 * choice, -1 = never, > 0 = that many tokens, a multiple of bs); then
 * `workspace` must hold pkv_prefill_workspace_size(...) bytes, its first
 * 256 bytes zero before first use.  max_query_len >= every q_len and
 * max_context_len >= every length (host values that size the launch).
 * Supported: bf16 query and bf16 cache (tensor cores), d in {64, 128}, bs in
 * {16, 32}; anything else returns PKV_ERR_UNSUPPORTED.  Runs a tcgen05
 * kernel (PKV_PREFILL_AUTO of pkv_paged_attention_prefill_ex).
 */
PKV_API size_t pkv_prefill_workspace_size(int S, int num_query_tokens, int max_query_len, int Hq, int Hkv, int d,
                                          int bs, int max_context_len, int partition_size);
PKV_API pkv_status pkv_paged_attention_prefill(void* out, const void* query, pkv_dtype q_dtype,
                                               const void* key_cache, const void* value_cache,
                                               pkv_dtype cache_dtype,
                                               const int32_t* block_tables, int MB,
                                               const int32_t* context_lens, const int32_t* query_start,
                                               int S, int num_query_tokens, int max_query_len,
                                               int max_context_len, int Hq, int Hkv, int d, int bs, int NB,
                                               float scale, int partition_size,
                                               void* workspace, size_t workspace_bytes,
                                               int32_t* err_word, pkv_stream_t stream);

/* Kernel choice for pkv_paged_attention_prefill_ex. */
typedef enum {
    PKV_PREFILL_AUTO = 0,         /* a tcgen05 kernel: two tiles per unit when the (sequence, K/V head)
                                     pairs average 256 or more (query, head) rows, else one */
    PKV_PREFILL_MMA_SYNC = 1,     /* warp-level mma.sync: tiles of 16 (query, head) rows, one warp each */
    PKV_PREFILL_TCGEN05 = 2,      /* tcgen05.mma with tensor-memory accumulators: tiles of 128 rows,
                                     one CTA each */
    PKV_PREFILL_TCGEN05_2TILE = 3 /* the same with two 128-row tiles per unit reading each K/V stage
                                     once, each tile with its own softmax warpgroup */
} pkv_prefill_kernel;

/*
 * Same as pkv_paged_attention_prefill, with an explicit kernel choice
 * (`kernel` is a pkv_prefill_kernel).  Both kernels compute the same
 * function with the same partitioning and workspace; the choice exists so
 * the two can be measured against each other.
 */
PKV_API pkv_status pkv_paged_attention_prefill_ex(void* out, const void* query, pkv_dtype q_dtype,
                                                  const void* key_cache, const void* value_cache,
                                                  pkv_dtype cache_dtype,
                                                  const int32_t* block_tables, int MB,
                                                  const int32_t* context_lens, const int32_t* query_start,
                                                  int S, int num_query_tokens, int max_query_len,
                                                  int max_context_len, int Hq, int Hkv, int d, int bs, int NB,
                                                  float scale, int partition_size,
                                                  void* workspace, size_t workspace_bytes,
                                                  int32_t* err_word, pkv_stream_t stream, int kernel);

/* ------------------------------------------------------------------------
 * Token tables and repacking.
 *
 * Source: "LLM推論の「見えないメモリ問題」を解く：トークンレベル仮想化でKV
 * キャッシュを再利用可能にする「vToken」", sections on token-level
 * virtualisation and asynchronous repacking: a token table maps each live
 * token of a sequence, in logical order, to its physical slot; a deletion
 * policy removes tokens from the table; repacking moves the survivors of
 * sparse blocks to free slots of other blocks, rewrites their table entries
 * and releases the emptied blocks.  Attention reads through the table, so
 * the cache pools and captured CUDA graphs are untouched by repacking.
 *
 * A slot is block * bs + offset, i.e. the row of the cache seen as
 * [NB * bs, Hkv, d].
 * ------------------------------------------------------------------------ */

/*
 * token_attention_decode -- the decode of pkv_paged_attention_decode, with
 * each sequence's K/V reached through its token table instead of a block
 * table: token_slots [S, MT] int32 (device) lists the slots of the
 * sequence's live tokens in logical order; num_tokens [S] (device) how many;
 * max_tokens >= every num_tokens (host value; <= MT).  Output, scales,
 * partitioning and workspace are those of the decode
 * (pkv_decode_workspace_size(S, Hq, d, max_tokens, partition_size)).
 * Supported: the tensor-core decode's dtypes (bf16 query and cache, or an
 * E4M3 cache with a bf16 or fp32 query), d in {64, 128}, bs in {16, 32};
 * anything else returns PKV_ERR_UNSUPPORTED.  A slot outside the pool is
 * treated as an absent token and reported (PKV_DEVERR_SLOT).
 */
PKV_API pkv_status pkv_token_attention_decode(void* out, const void* query, pkv_dtype q_dtype,
                                              const void* key_cache, const void* value_cache,
                                              pkv_dtype cache_dtype,
                                              const int32_t* token_slots, int MT,
                                              const int32_t* num_tokens, int S, int max_tokens,
                                              int Hq, int Hkv, int d, int bs, int NB,
                                              float scale, float k_scale, float v_scale,
                                              int partition_size,
                                              void* workspace, size_t workspace_bytes,
                                              int32_t* err_word, pkv_stream_t stream);

/*
 * repack_tokens -- apply moves [M, 4] int64 (device) = (sequence, logical
 * index, source slot, destination slot): for every layer, the token's K and
 * V rows (token_bytes = Hkv * d * element size bytes each) are copied from
 * the source slot to the destination, then token_slots[sequence][index]
 * becomes the destination.  key_caches / value_caches are host arrays of
 * num_layers (<= 256) device pointers.  Preconditions: destinations are free
 * slots, distinct, and no move's destination is another move's source; each
 * (sequence, index) appears once.  A move out of range or whose source is
 * not what the table holds is skipped and reported (PKV_DEVERR_MOVE).
 */
PKV_API pkv_status pkv_repack_tokens(void* const* key_caches, void* const* value_caches, int num_layers,
                                     int32_t* token_slots, int MT, int S, const int64_t* moves, int M,
                                     int NB, int bs, size_t token_bytes, int32_t* err_word,
                                     pkv_stream_t stream);

/*
 * vtoken_plan -- host planner for repacking (host arrays).  Per sequence,
 * over the blocks only that sequence uses (a block several sequences
 * reference is left alone): the sequence needs k = ceil(live tokens in
 * those blocks / bs) blocks; the k with the most live tokens stay (lower id
 * first on ties); its tokens in the others move, in logical order, to the
 * free slots of the kept blocks, lowest slot first; the others are then
 * empty and are listed in `freed` (ascending per sequence).  Writes up to
 * max_moves moves [.., 4] and max_freed block ids, and the counts needed in
 * *num_moves / *num_freed.  Returns PKV_ERR_INVALID_ARG for a slot outside
 * the pool or a sequence holding one slot twice, PKV_ERR_WORKSPACE when an
 * output array is too small (counts still set, arrays untouched).  Scratch
 * host memory during the call: one bit per slot of the pool and about ten
 * bytes per block, plus the moves found.
 */
PKV_API pkv_status pkv_vtoken_plan(const int32_t* token_slots, int MT, const int32_t* num_tokens, int S, int bs,
                                   int NB, int64_t* moves, int64_t max_moves, int64_t* num_moves,
                                   int32_t* freed, int64_t max_freed, int64_t* num_freed);

/* ------------------------------------------------------------------------
 * Host block manager: the bookkeeping that produces the block tables, slot
 * mappings and copy-on-write pairs the device calls consume.  Host memory
 * only; nothing here touches the GPU.
 *
 * Source: "LLM推論の基礎とvLLMの内部", section 4 "PagedAttentionとブロック
 * 管理": blocks are handed to a request one at a time as it grows, each
 * request keeps a block table, block 0 is reserved as the null block, free
 * blocks wait in a doubly linked queue, and shared blocks carry a reference
 * count and are copied before a write.  Section 5: a full block's hash
 * chains its parent's hash, its tokens and extra keys; only full blocks are
 * cached; the last prompt token is always recomputed; a finished request
 * returns its blocks tail first with their hashes kept, and the queue is
 * reused from its front (least recently freed first).  Free blocks without
 * a hash are handed out before any cached block.
 *
 * Errors: PKV_ERR_INVALID_ARG for a null pool, an unknown or duplicate
 * sequence id, or bad sizes; PKV_ERR_WORKSPACE when the pool has too few
 * free blocks (nothing is changed then).  A pool is not thread-safe.
 * ---------------------------------------------------------------------- */
typedef struct pkv_block_pool pkv_block_pool;

/* A pool of num_blocks blocks of block_size tokens (block 0 reserved, so
 * num_blocks - 1 usable).  enable_prefix_caching != 0 turns on the hash
 * chain and reuse of cached blocks. */
PKV_API pkv_status pkv_pool_create(int num_blocks, int block_size, int enable_prefix_caching,
                                   pkv_block_pool** out);
PKV_API void pkv_pool_destroy(pkv_block_pool* pool);
/* Extra key mixed into every block hash (a LoRA id, a cache salt, ...):
 * pools with different keys never share cached blocks. */
PKV_API pkv_status pkv_pool_set_extra_key(pkv_block_pool* pool, uint64_t extra_key);
PKV_API int pkv_pool_num_free_blocks(const pkv_block_pool* pool);
PKV_API int pkv_pool_num_cached_blocks(const pkv_block_pool* pool);
/* Reference count of a physical block (-1 for a bad id). */
PKV_API int pkv_pool_block_ref_count(const pkv_block_pool* pool, int block);

/* Start sequence seq_id with its prompt tokens[0..n_tokens): reuse the
 * longest cached prefix of whole blocks (never the block holding the last
 * token's position if that would leave no token to compute), take new blocks
 * for the rest.  *num_cached_tokens (optional) receives the tokens found in
 * the cache.  The prompt's K/V then go to slots block_table[t / bs] * bs +
 * t % bs for t >= *num_cached_tokens. */
PKV_API pkv_status pkv_pool_add_sequence(pkv_block_pool* pool, int64_t seq_id, const int32_t* tokens,
                                         int n_tokens, int* num_cached_tokens);

/* One more token for seq_id.  *slot receives the cache slot of its K/V.  If
 * the last block was full a new block is taken; if it is shared with another
 * sequence (after pkv_pool_fork) it is copied first: *cow_src / *cow_dst
 * receive the (src, dst) pair to pass to pkv_copy_blocks before the write,
 * else -1. */
PKV_API pkv_status pkv_pool_append_token(pkv_block_pool* pool, int64_t seq_id, int32_t token, int64_t* slot,
                                         int64_t* cow_src, int64_t* cow_dst);

/* child_id shares every block of parent_id (reference counts + 1), as for
 * parallel sampling or beam search. */
PKV_API pkv_status pkv_pool_fork(pkv_block_pool* pool, int64_t parent_id, int64_t child_id);

/* End seq_id: its blocks lose one reference each, last block first. */
PKV_API pkv_status pkv_pool_free_sequence(pkv_block_pool* pool, int64_t seq_id);

/* One decode step for n sequences at once: token tokens[i] is appended to
 * seq_ids[i] (each id once).  slot_mapping[i] receives its slot -- the input
 * of pkv_paged_kv_write -- and the copy-on-write pairs go to
 * block_mapping[0 .. 2 * *num_copies) as (src, dst) -- the input of
 * pkv_copy_blocks, to run before the write.  block_mapping must have room
 * for 2 * n entries.  If the pool cannot cover the step, PKV_ERR_WORKSPACE is
 * returned and nothing changes. */
PKV_API pkv_status pkv_pool_append_tokens(pkv_block_pool* pool, const int64_t* seq_ids, const int32_t* tokens,
                                          int n, int64_t* slot_mapping, int64_t* block_mapping, int* num_copies);

/* The decode's inputs for n sequences: tables [n, max_blocks] (padded with
 * the null block) and context_lens [n]. */
PKV_API pkv_status pkv_pool_block_tables(const pkv_block_pool* pool, const int64_t* seq_ids, int n,
                                         int32_t* tables, int max_blocks, int32_t* context_lens);

/* Copy seq_id's block table into table[0..max_blocks), padded with the null
 * block 0; *num_blocks and *num_tokens (optional) receive its length.  A
 * NULL table only queries the lengths. */
PKV_API pkv_status pkv_pool_block_table(const pkv_block_pool* pool, int64_t seq_id, int32_t* table,
                                        int max_blocks, int* num_blocks, int* num_tokens);

/* Static, human-readable text for a status. */
PKV_API const char* pkv_status_string(pkv_status status);

/* Version of this library, e.g. "pkv 0.1.0 sm_103a". */
PKV_API const char* pkv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H */
