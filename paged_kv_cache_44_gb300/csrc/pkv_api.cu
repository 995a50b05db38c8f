// C ABI of libpkv.so: host-side validation, workspace planning, dispatch.
// Nothing here allocates, synchronises or reads device memory.
#include <math.h>
#include <string.h>

#include <cudaTypedefs.h>

#include <mutex>

#include "pkv_common.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
// Units of work (sequence x K/V head x head-set x partition) the default
// partition size aims for, counted as if every sequence had the maximum
// length: about four per worker warp of a full GB300 (152 SMs x 8 warps),
// so that dynamic scheduling evens out ragged lengths and the last units to
// finish are short next to the whole launch.  It depends on no dtype, so the
// workspace size and the launch always agree.
constexpr long long kTargetUnits = 152LL * 8 * 4;
constexpr int kMinDefaultPartition = 512;
// A small launch: fewer than about 1.3 units per worker warp of a full
// GB300 (152 SMs x 7 bf16 workers) even if every sequence had the maximum
// length.
constexpr long long kSmallLaunchUnits = 152LL * 9;
constexpr int kMinSmallPartition = 256;
constexpr long long kPrefillTargetUnits = 152LL * 4;
constexpr int kPrefillTileRows = 128;       // (query, head) rows per tcgen05 tile
constexpr int kHeadSet = 8;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool finite_pos(float x) { return isfinite(x) && x > 0.f; }

bool decode_shape_ok(int S, int Hq, int Hkv, int d, int bs, int max_ctx) {
    return S >= 0 && S <= 65535 && Hkv >= 1 && Hq >= Hkv && Hq % Hkv == 0 && (d == 64 || d == 128) &&
           (bs == 16 || bs == 32) && max_ctx >= 0;
}

// Partition size in tokens (0 = no split) for a request; -1 if invalid.
int resolve_partition(int S, int Hq, int Hkv, int d, int bs, int max_ctx, int req) {
    if (!decode_shape_ok(S, Hq, Hkv, d, bs, max_ctx)) return -1;
    if (req > 0) return req % bs == 0 ? req : -1;
    if (req == -1) return 0;
    if (req != 0) return -1;
    const long long sets = (long long)S * Hkv * ((Hq / Hkv + kHeadSet - 1) / kHeadSet);
    if (sets == 0 || max_ctx <= kMinDefaultPartition) return 0;
    int P = 1 << 20;
    while (P > kMinDefaultPartition && sets * ((max_ctx + P - 1) / P) < kTargetUnits) P >>= 1;
    // A small launch gives each worker warp about one long unit, streamed at
    // a single warp's latency-bound rate, and the longest units set the
    // launch's length: take the largest partition, in steps of 128 tokens
    // down to 256, that gives that many units at the maximum length.
    // 64 sequences of 512..4096 tokens, 2 K/V heads: 384 instead of 512,
    // decode 35.3-35.4 vs 37.5-37.9 us (256: 38.1, 320: 35.6, 448: 36.0).
    while (P > kMinSmallPartition && sets * ((max_ctx + P - 1) / P) < kSmallLaunchUnits) P -= 128;
    if (P >= max_ctx) return 0;
    return P;
}

// The last, partial partition of a sequence is cut into chunks of Q tokens
// (a quarter partition, a multiple of 32 tokens and so of the block size):
// those chunks are the last units a launch hands out, so the launch ends on
// small units instead of on whichever partial partitions happened to be large.
int tail_chunk(int P) { return P >= 128 ? (P / 4) / 32 * 32 : P; }

// Full partitions held back into chunks at a long sequence's end
// (num_partitions), for E4M3 caches on the tensor-core kernel: a worker
// streams E4M3 at the pace of its own arithmetic (about 17 tokens/us, a
// full 1024-token unit lasts ~60 us), so the units claimed last decide when
// the launch ends, and small ones end it sooner.  On bf16 caches the same
// layout was slower (more units and partial results for the same tail).
constexpr int kTailHold = 1;
int tail_hold(pkv_dtype cache_dtype, bool tensor_cores) {
    return cache_dtype == PKV_FP8_E4M3 && tensor_cores ? kTailHold : 0;
}

// Partial results per row for lengths up to max_ctx with `hold` held-back
// partitions: the count (num_partitions) grows with n between multiples of
// P, so its largest value is at max_ctx, just below the last multiple of P,
// or just below the length from which partitions are held back.
int max_partitions(int max_ctx, int P, int Q, int hold) {
    int m = num_partitions(max_ctx, P, Q, hold);
    const int F = max_ctx / P;
    if (F >= 1) m = max(m, num_partitions(F * P - 1, P, Q, hold));
    m = max(m, num_partitions(min(max_ctx, kTailHoldMin * P - 1), P, Q, hold));
    return m > 1 ? m : 1;
}

DecodePlan make_plan(int S, int Hq, int d, int max_ctx, int P) {
    DecodePlan pl{};
    pl.P = P;
    pl.Q = P;
    pl.Pmax = P > 0 ? (max_ctx > 0 ? (max_ctx + P - 1) / P : 1) : 1;
    pl.Pmax_plain = pl.Pmax;
    pl.split = P > 0 && pl.Pmax > 1;
    pl.bytes = kWorkspaceHeaderBytes;
    if (!pl.split) return pl;
    pl.Q = tail_chunk(P);
    // the workspace fits both layouts; each launch uses its own row stride
    pl.Pmax_plain = max_partitions(max_ctx, P, pl.Q, 0);
    pl.Pmax = max(pl.Pmax_plain, max_partitions(max_ctx, P, pl.Q, kTailHold));
    auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
    const size_t units = (size_t)S * Hq * pl.Pmax;
    pl.ml_offset = kWorkspaceHeaderBytes;
    pl.acc_offset = up(pl.ml_offset + units * 2 * sizeof(float));
    pl.bytes = up(pl.acc_offset + units * d * sizeof(float));
    return pl;
}

// Partition a launch uses.  With the library's choice (request 0), an E4M3
// cache on the tensor-core kernel takes twice the planned partition where
// that still leaves half of kTargetUnits units: an E4M3 worker streams at
// the pace of its own arithmetic and every unit has a fixed cost (its
// claim, its first stage in flight, its partial result and merge row), so
// fewer, longer units end the launch sooner.  Measured on the fp8 workloads
// (128 sequences of 256..16384 tokens, bs 16 and 32): 2048-token partitions
// 1.1-1.5% faster than 1024, 3072 and 4096 slower.  The workspace is planned
// for the dtype-independent partition; a partition twice as large never
// needs more partial results per row, and the larger one is taken only when
// the plan's row stride holds them.
int launch_partition(const DecodePlan& pl, int S, int Hq, int Hkv, int max_ctx, int req, bool e4m3_tc) {
    if (req != 0 || !pl.split || !e4m3_tc) return pl.P;
    const int P2 = 2 * pl.P;
    const long long sets = (long long)S * Hkv * ((Hq / Hkv + kHeadSet - 1) / kHeadSet);
    if (P2 >= max_ctx || sets * ((max_ctx + P2 - 1) / P2) < kTargetUnits / 2) return pl.P;
    return max_partitions(max_ctx, P2, tail_chunk(P2), kTailHold) <= pl.Pmax ? P2 : pl.P;
}

// Fills the partition fields of a launch: P, its chunk Q, the row stride.
void set_partitions(DecodeParams& p, const DecodePlan& pl, int Pl, int no_split_P, int hold) {
    p.P = Pl > 0 ? Pl : no_split_P;      // no split: one partition covers every token
    p.Q = Pl <= 0 ? p.P : (Pl == pl.P ? pl.Q : tail_chunk(Pl));
    p.hold = hold;
    p.Pmax = hold ? pl.Pmax : pl.Pmax_plain;
}

pkv_status from_cuda(cudaError_t e) { return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA; }

int num_sms_current() {
    static std::mutex mu;
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152;
    std::lock_guard<std::mutex> g(mu);
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 152;
        cache[dev] = n;
    }
    return cache[dev];
}

}  // namespace

CUcontext current_context() {
    static std::once_flag once;
    static PFN_cuCtxGetCurrent_v4000 fn = nullptr;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f);
    });
    CUcontext ctx = nullptr;
    if (fn == nullptr || fn(&ctx) != CUDA_SUCCESS) return nullptr;
    return ctx;
}

}  // namespace pkv

using namespace pkv;

extern "C" {

const char* pkv_status_string(pkv_status st) {
    switch (st) {
        case PKV_OK: return "ok";
        case PKV_ERR_INVALID_ARG: return "invalid argument";
        case PKV_ERR_UNSUPPORTED: return "unsupported dtype or shape";
        case PKV_ERR_WORKSPACE: return "workspace missing or too small";
        case PKV_ERR_CUDA: return "CUDA launch failed";
    }
    return "unknown status";
}

const char* pkv_version(void) { return "pkv 0.1.0 sm_103a"; }

pkv_status pkv_paged_kv_write(const void* key, const void* value, pkv_dtype in_dtype, void* key_cache,
                              void* value_cache, pkv_dtype cache_dtype, const int64_t* slot_mapping, int T,
                              int NB, int bs, int Hkv, int d, float k_scale, float v_scale, int32_t* err_word,
                              pkv_stream_t stream) {
    if (T < 0 || NB < 1 || bs < 1 || Hkv < 1 || d < 8) return PKV_ERR_INVALID_ARG;
    if (in_dtype != PKV_F32 && in_dtype != PKV_BF16) return PKV_ERR_UNSUPPORTED;
    if (cache_dtype != PKV_F32 && cache_dtype != PKV_BF16 && cache_dtype != PKV_FP8_E4M3)
        return PKV_ERR_UNSUPPORTED;
    if (d % 8 != 0 || d > 512) return PKV_ERR_UNSUPPORTED;
    if (cache_dtype == PKV_FP8_E4M3 && (!finite_pos(k_scale) || !finite_pos(v_scale))) return PKV_ERR_INVALID_ARG;
    if ((long long)NB * bs > (1LL << 40)) return PKV_ERR_INVALID_ARG;
    if (T == 0) return PKV_OK;
    if (!key || !value || !key_cache || !value_cache || !slot_mapping) return PKV_ERR_INVALID_ARG;
    if (!aligned16(key) || !aligned16(value) || !aligned16(key_cache) || !aligned16(value_cache) ||
        (reinterpret_cast<uintptr_t>(slot_mapping) & 7u))
        return PKV_ERR_INVALID_ARG;
    WriteParams p{};
    p.key = key; p.value = value; p.key_cache = key_cache; p.value_cache = value_cache;
    p.slot_mapping = slot_mapping; p.err = err_word;
    p.T = T; p.NB = NB; p.bs = bs; p.Hkv = Hkv; p.d = d; p.k_scale = k_scale; p.v_scale = v_scale;
    return from_cuda(launch_write(p, in_dtype, cache_dtype, reinterpret_cast<cudaStream_t>(stream)));
}

int pkv_decode_partition_size(int S, int Hq, int Hkv, int d, int bs, int max_context_len, int partition_size) {
    return resolve_partition(S, Hq, Hkv, d, bs, max_context_len, partition_size);
}

int pkv_decode_launch_partition_size(int S, int Hq, int Hkv, int d, int bs, int NB, int max_context_len,
                                     int partition_size, pkv_dtype q_dtype, pkv_dtype cache_dtype, int kernel) {
    if (kernel < PKV_DECODE_AUTO || kernel > PKV_DECODE_TENSOR_CORES || NB < 1) return -1;
    if (q_dtype != PKV_F32 && q_dtype != PKV_BF16) return -1;
    if (cache_dtype != PKV_F32 && cache_dtype != PKV_BF16 && cache_dtype != PKV_FP8_E4M3) return -1;
    const int P = resolve_partition(S, Hq, Hkv, d, bs, max_context_len, partition_size);
    if (P < 0) return -1;
    const bool tc_ok = decode_tc_supports(q_dtype, cache_dtype, d, bs, NB);
    if (kernel == PKV_DECODE_TENSOR_CORES && !tc_ok) return -1;      // the decode would refuse it
    const bool use_tc = kernel != PKV_DECODE_CUDA_CORES && tc_ok;
    const DecodePlan pl = make_plan(S, Hq, d, max_context_len, P);
    return launch_partition(pl, S, Hq, Hkv, max_context_len, partition_size, use_tc && cache_dtype == PKV_FP8_E4M3);
}

size_t pkv_decode_workspace_size(int S, int Hq, int Hkv, int d, int bs, int max_context_len, int partition_size) {
    const int P = resolve_partition(S, Hq, Hkv, d, bs, max_context_len, partition_size);
    if (P < 0) return 0;
    return make_plan(S, Hq, d, max_context_len, P).bytes;
}

}  // extern "C"

namespace pkv {

pkv_status check_decode_args(const void* out, const void* query, pkv_dtype q_dtype, const void* key_cache,
                             const void* value_cache, pkv_dtype cache_dtype, const int32_t* block_tables, int MB,
                             const int32_t* context_lens, int S, int max_context_len, int Hq, int Hkv, int d,
                             int bs, int NB, float scale, float k_scale, float v_scale, int partition_size,
                             int kernel) {
    if (S < 0 || MB < 1 || NB < 1 || Hkv < 1 || Hq < 1 || max_context_len < 0) return PKV_ERR_INVALID_ARG;
    if (Hq % Hkv != 0) return PKV_ERR_INVALID_ARG;
    if (q_dtype != PKV_F32 && q_dtype != PKV_BF16) return PKV_ERR_UNSUPPORTED;
    if (cache_dtype != PKV_F32 && cache_dtype != PKV_BF16 && cache_dtype != PKV_FP8_E4M3)
        return PKV_ERR_UNSUPPORTED;
    if (!(d == 64 || d == 128) || !(bs == 16 || bs == 32)) return PKV_ERR_UNSUPPORTED;
    if (S > 65535) return PKV_ERR_UNSUPPORTED;
    if ((long long)max_context_len > (long long)MB * bs) return PKV_ERR_INVALID_ARG;
    if (!isfinite(scale)) return PKV_ERR_INVALID_ARG;
    if (cache_dtype == PKV_FP8_E4M3 && (!finite_pos(k_scale) || !finite_pos(v_scale))) return PKV_ERR_INVALID_ARG;
    if (partition_size < -1 || (partition_size > 0 && partition_size % bs != 0)) return PKV_ERR_INVALID_ARG;
    if (kernel < 0 || kernel > 2) return PKV_ERR_INVALID_ARG;
    if (S == 0) return PKV_OK;
    if (!out || !query || !key_cache || !value_cache || !block_tables || !context_lens) return PKV_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(query) || !aligned16(key_cache) || !aligned16(value_cache) ||
        (reinterpret_cast<uintptr_t>(block_tables) & 3u) || (reinterpret_cast<uintptr_t>(context_lens) & 3u))
        return PKV_ERR_INVALID_ARG;
    if (resolve_partition(S, Hq, Hkv, d, bs, max_context_len, partition_size) < 0) return PKV_ERR_INVALID_ARG;
    if (kernel == PKV_DECODE_TENSOR_CORES && !decode_tc_supports(q_dtype, cache_dtype, d, bs, NB))
        return PKV_ERR_UNSUPPORTED;
    return PKV_OK;
}

}  // namespace pkv

extern "C" {

pkv_status pkv_paged_attention_decode_ex(void* out, const void* query, pkv_dtype q_dtype, const void* key_cache,
                                         const void* value_cache, pkv_dtype cache_dtype,
                                         const int32_t* block_tables, int MB, const int32_t* context_lens, int S,
                                         int max_context_len, int Hq, int Hkv, int d, int bs, int NB, float scale,
                                         float k_scale, float v_scale, int partition_size, void* workspace,
                                         size_t workspace_bytes, int32_t* err_word, pkv_stream_t stream,
                                         int kernel) {
    const pkv_status chk = check_decode_args(out, query, q_dtype, key_cache, value_cache, cache_dtype, block_tables,
                                             MB, context_lens, S, max_context_len, Hq, Hkv, d, bs, NB, scale,
                                             k_scale, v_scale, partition_size, kernel);
    if (chk != PKV_OK || S == 0) return chk;

    const int P = resolve_partition(S, Hq, Hkv, d, bs, max_context_len, partition_size);
    const bool use_tc = kernel != PKV_DECODE_CUDA_CORES && decode_tc_supports(q_dtype, cache_dtype, d, bs, NB);
    const DecodePlan pl = make_plan(S, Hq, d, max_context_len, P);
    if (pl.split) {
        if (!workspace || workspace_bytes < pl.bytes) return PKV_ERR_WORKSPACE;
        if (!aligned16(workspace)) return PKV_ERR_INVALID_ARG;
    }

    DecodeParams p{};
    p.out = out; p.q = query; p.kc = key_cache; p.vc = value_cache;
    p.block_tables = block_tables; p.context_lens = context_lens; p.err = err_word;
    p.S = S; p.MB = MB; p.Hq = Hq; p.Hkv = Hkv; p.g = Hq / Hkv; p.d = d; p.bs = bs; p.NB = NB;
    set_partitions(p, pl,
                   launch_partition(pl, S, Hq, Hkv, max_context_len, partition_size,
                                    use_tc && cache_dtype == PKV_FP8_E4M3),
                   MB * bs, tail_hold(cache_dtype, use_tc));
    p.max_ctx = max_context_len;
    const float ks = cache_dtype == PKV_FP8_E4M3 ? k_scale : 1.f;
    p.logit_scale_log2 = scale * ks * kLog2e;
    p.out_scale = cache_dtype == PKV_FP8_E4M3 ? v_scale : 1.f;
    if (pl.split) {
        char* ws = static_cast<char*>(workspace);
        p.sched = reinterpret_cast<unsigned*>(ws);
        p.part_ml = reinterpret_cast<float*>(ws + pl.ml_offset);
        p.part_acc = reinterpret_cast<float*>(ws + pl.acc_offset);
    } else if (workspace && workspace_bytes >= kWorkspaceHeaderBytes && aligned16(workspace)) {
        p.sched = reinterpret_cast<unsigned*>(workspace);
    }
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = use_tc ? launch_decode_tc(p, q_dtype, cache_dtype, num_sms_current(), st)
                           : launch_decode_simt(p, q_dtype, cache_dtype, st);
    if (e != cudaSuccess) return PKV_ERR_CUDA;
    if (pl.split) e = launch_decode_reduce(p, q_dtype, st);
    return from_cuda(e);
}

pkv_status pkv_paged_kv_write_decode(void* out, const void* query, pkv_dtype q_dtype, const void* key,
                                     const void* value, pkv_dtype in_dtype, void* key_cache, void* value_cache,
                                     pkv_dtype cache_dtype, const int64_t* slot_mapping, const int32_t* block_tables,
                                     int MB, const int32_t* context_lens, int S, int max_context_len, int Hq, int Hkv,
                                     int d, int bs, int NB, float scale, float k_scale, float v_scale,
                                     int partition_size, void* workspace, size_t workspace_bytes, int32_t* err_word,
                                     pkv_stream_t stream) {
    if (S < 0 || MB < 1 || NB < 1 || Hkv < 1 || Hq < 1 || max_context_len < 0) return PKV_ERR_INVALID_ARG;
    if (Hq % Hkv != 0) return PKV_ERR_INVALID_ARG;
    if (q_dtype != PKV_F32 && q_dtype != PKV_BF16) return PKV_ERR_UNSUPPORTED;
    if (in_dtype != PKV_F32 && in_dtype != PKV_BF16) return PKV_ERR_UNSUPPORTED;
    if (cache_dtype != PKV_F32 && cache_dtype != PKV_BF16 && cache_dtype != PKV_FP8_E4M3)
        return PKV_ERR_UNSUPPORTED;
    if (!decode_tc_supports(q_dtype, cache_dtype, d, bs, NB)) return PKV_ERR_UNSUPPORTED;
    if (S > 65535) return PKV_ERR_UNSUPPORTED;
    if ((long long)max_context_len > (long long)MB * bs) return PKV_ERR_INVALID_ARG;
    if (!isfinite(scale)) return PKV_ERR_INVALID_ARG;
    if (cache_dtype == PKV_FP8_E4M3 && (!finite_pos(k_scale) || !finite_pos(v_scale))) return PKV_ERR_INVALID_ARG;
    if (partition_size < -1 || (partition_size > 0 && partition_size % bs != 0)) return PKV_ERR_INVALID_ARG;
    if (S == 0) return PKV_OK;
    if (!out || !query || !key || !value || !key_cache || !value_cache || !slot_mapping || !block_tables ||
        !context_lens)
        return PKV_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(query) || !aligned16(key) || !aligned16(value) || !aligned16(key_cache) ||
        !aligned16(value_cache) || (reinterpret_cast<uintptr_t>(slot_mapping) & 7u) ||
        (reinterpret_cast<uintptr_t>(block_tables) & 3u) || (reinterpret_cast<uintptr_t>(context_lens) & 3u))
        return PKV_ERR_INVALID_ARG;
    const int P = resolve_partition(S, Hq, Hkv, d, bs, max_context_len, partition_size);
    if (P < 0) return PKV_ERR_INVALID_ARG;
    const DecodePlan pl = make_plan(S, Hq, d, max_context_len, P);
    if (pl.split) {
        if (!workspace || workspace_bytes < pl.bytes) return PKV_ERR_WORKSPACE;
        if (!aligned16(workspace)) return PKV_ERR_INVALID_ARG;
    }
    DecodeParams p{};
    p.out = out; p.q = query; p.kc = key_cache; p.vc = value_cache;
    p.block_tables = block_tables; p.context_lens = context_lens; p.err = err_word;
    p.S = S; p.MB = MB; p.Hq = Hq; p.Hkv = Hkv; p.g = Hq / Hkv; p.d = d; p.bs = bs; p.NB = NB;
    set_partitions(p, pl,
                   launch_partition(pl, S, Hq, Hkv, max_context_len, partition_size, cache_dtype == PKV_FP8_E4M3),
                   MB * bs, tail_hold(cache_dtype, true));
    p.max_ctx = max_context_len;
    const float ks = cache_dtype == PKV_FP8_E4M3 ? k_scale : 1.f;
    p.logit_scale_log2 = scale * ks * kLog2e;
    p.out_scale = cache_dtype == PKV_FP8_E4M3 ? v_scale : 1.f;
    p.new_k = key; p.new_v = value; p.slot_mapping = slot_mapping; p.new_dt = in_dtype;
    p.k_scale = k_scale; p.v_scale = v_scale;
    if (pl.split) {
        char* ws = static_cast<char*>(workspace);
        p.sched = reinterpret_cast<unsigned*>(ws);
        p.part_ml = reinterpret_cast<float*>(ws + pl.ml_offset);
        p.part_acc = reinterpret_cast<float*>(ws + pl.acc_offset);
    } else if (workspace && workspace_bytes >= kWorkspaceHeaderBytes && aligned16(workspace)) {
        p.sched = reinterpret_cast<unsigned*>(workspace);
    }
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = launch_decode_tc(p, q_dtype, cache_dtype, num_sms_current(), st);
    if (e != cudaSuccess) return PKV_ERR_CUDA;
    if (pl.split) e = launch_decode_reduce(p, q_dtype, st);
    return from_cuda(e);
}

pkv_status pkv_token_attention_decode(void* out, const void* query, pkv_dtype q_dtype, const void* key_cache,
                                      const void* value_cache, pkv_dtype cache_dtype, const int32_t* token_slots,
                                      int MT, const int32_t* num_tokens, int S, int max_tokens, int Hq, int Hkv,
                                      int d, int bs, int NB, float scale, float k_scale, float v_scale,
                                      int partition_size, void* workspace, size_t workspace_bytes,
                                      int32_t* err_word, pkv_stream_t stream) {
    if (S < 0 || MT < 1 || NB < 1 || Hkv < 1 || Hq < 1 || max_tokens < 0 || max_tokens > MT)
        return PKV_ERR_INVALID_ARG;
    if (Hq % Hkv != 0) return PKV_ERR_INVALID_ARG;
    if (q_dtype != PKV_F32 && q_dtype != PKV_BF16) return PKV_ERR_UNSUPPORTED;
    if (cache_dtype != PKV_F32 && cache_dtype != PKV_BF16 && cache_dtype != PKV_FP8_E4M3)
        return PKV_ERR_UNSUPPORTED;
    if (!decode_tc_supports(q_dtype, cache_dtype, d, bs, NB)) return PKV_ERR_UNSUPPORTED;
    if (S > 65535) return PKV_ERR_UNSUPPORTED;
    if (!isfinite(scale)) return PKV_ERR_INVALID_ARG;
    if (cache_dtype == PKV_FP8_E4M3 && (!finite_pos(k_scale) || !finite_pos(v_scale))) return PKV_ERR_INVALID_ARG;
    if (partition_size < -1 || (partition_size > 0 && partition_size % bs != 0)) return PKV_ERR_INVALID_ARG;
    if (S == 0) return PKV_OK;
    if (!out || !query || !key_cache || !value_cache || !token_slots || !num_tokens) return PKV_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(query) || !aligned16(key_cache) || !aligned16(value_cache) ||
        (reinterpret_cast<uintptr_t>(token_slots) & 3u) || (reinterpret_cast<uintptr_t>(num_tokens) & 3u))
        return PKV_ERR_INVALID_ARG;
    const int P = resolve_partition(S, Hq, Hkv, d, bs, max_tokens, partition_size);
    if (P < 0) return PKV_ERR_INVALID_ARG;
    const DecodePlan pl = make_plan(S, Hq, d, max_tokens, P);
    if (pl.split) {
        if (!workspace || workspace_bytes < pl.bytes) return PKV_ERR_WORKSPACE;
        if (!aligned16(workspace)) return PKV_ERR_INVALID_ARG;
    }
    DecodeParams p{};
    p.out = out; p.q = query; p.kc = key_cache; p.vc = value_cache;
    p.token_slots = token_slots; p.MT = MT; p.context_lens = num_tokens; p.err = err_word;
    p.S = S; p.MB = 1; p.Hq = Hq; p.Hkv = Hkv; p.g = Hq / Hkv; p.d = d; p.bs = bs; p.NB = NB;
    set_partitions(p, pl,
                   launch_partition(pl, S, Hq, Hkv, max_tokens, partition_size, cache_dtype == PKV_FP8_E4M3),
                   max_tokens > 0 ? max_tokens : 1, tail_hold(cache_dtype, true));
    p.max_ctx = max_tokens;
    const float ks = cache_dtype == PKV_FP8_E4M3 ? k_scale : 1.f;
    p.logit_scale_log2 = scale * ks * kLog2e;
    p.out_scale = cache_dtype == PKV_FP8_E4M3 ? v_scale : 1.f;
    if (pl.split) {
        char* ws = static_cast<char*>(workspace);
        p.sched = reinterpret_cast<unsigned*>(ws);
        p.part_ml = reinterpret_cast<float*>(ws + pl.ml_offset);
        p.part_acc = reinterpret_cast<float*>(ws + pl.acc_offset);
    } else if (workspace && workspace_bytes >= kWorkspaceHeaderBytes && aligned16(workspace)) {
        p.sched = reinterpret_cast<unsigned*>(workspace);
    }
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = launch_decode_tc(p, q_dtype, cache_dtype, num_sms_current(), st, true);
    if (e != cudaSuccess) return PKV_ERR_CUDA;
    if (pl.split) e = launch_decode_reduce(p, q_dtype, st);
    return from_cuda(e);
}

pkv_status pkv_repack_tokens(void* const* key_caches, void* const* value_caches, int num_layers,
                             int32_t* token_slots, int MT, int S, const int64_t* moves, int M, int NB, int bs,
                             size_t token_bytes, int32_t* err_word, pkv_stream_t stream) {
    if (num_layers < 0 || num_layers > kMaxCopyLayers || M < 0 || MT < 1 || S < 0 || NB < 1 || bs < 1)
        return PKV_ERR_INVALID_ARG;
    if (token_bytes == 0 || token_bytes % 16 != 0) return PKV_ERR_INVALID_ARG;
    if (M == 0 || num_layers == 0) return PKV_OK;
    if (!key_caches || !value_caches || !moves || !token_slots) return PKV_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(moves) & 7u) || (reinterpret_cast<uintptr_t>(token_slots) & 3u))
        return PKV_ERR_INVALID_ARG;
    RepackParams p{};
    for (int l = 0; l < num_layers; ++l) {
        if (!key_caches[l] || !value_caches[l] || !aligned16(key_caches[l]) || !aligned16(value_caches[l]))
            return PKV_ERR_INVALID_ARG;
        p.k[l] = key_caches[l];
        p.v[l] = value_caches[l];
    }
    p.moves = moves; p.token_slots = token_slots; p.err = err_word;
    p.M = M; p.L = num_layers; p.S = S; p.MT = MT; p.NB = NB; p.bs = bs; p.token_bytes = token_bytes;
    return from_cuda(launch_repack(p, reinterpret_cast<cudaStream_t>(stream)));
}

pkv_status pkv_paged_attention_decode(void* out, const void* query, pkv_dtype q_dtype, const void* key_cache,
                                      const void* value_cache, pkv_dtype cache_dtype, const int32_t* block_tables,
                                      int MB, const int32_t* context_lens, int S, int max_context_len, int Hq,
                                      int Hkv, int d, int bs, int NB, float scale, float k_scale, float v_scale,
                                      int partition_size, void* workspace, size_t workspace_bytes,
                                      int32_t* err_word, pkv_stream_t stream) {
    return pkv_paged_attention_decode_ex(out, query, q_dtype, key_cache, value_cache, cache_dtype, block_tables, MB,
                                         context_lens, S, max_context_len, Hq, Hkv, d, bs, NB, scale, k_scale,
                                         v_scale, partition_size, workspace, workspace_bytes, err_word, stream,
                                         PKV_DECODE_AUTO);
}

}  // extern "C"

namespace pkv {
namespace {

// Prefill partition size (0 = no split; -1 = invalid): tiles of 16 (query,
// head) rows already give parallelism, so split only when there are few.
int resolve_prefill_partition(int S, int max_q_len, int Hq, int Hkv, int d, int bs, int max_ctx, int req) {
    if (!decode_shape_ok(S, Hq, Hkv, d, bs, max_ctx) || max_q_len < 0 || max_q_len > max_ctx) return -1;
    if (req > 0) return req % bs == 0 ? req : -1;
    if (req == -1) return 0;
    if (req != 0) return -1;
    // counted in tiles of 128 rows (the tcgen05 kernel's unit); about four
    // units per SM keep the persistent CTAs busy to the end
    const long long tiles = (long long)S * Hkv * ((max_q_len * (long long)(Hq / Hkv) + 127) / 128);
    if (tiles == 0 || tiles >= kPrefillTargetUnits || max_ctx <= kMinDefaultPartition) return 0;
    int P = 1 << 20;
    while (P > kMinDefaultPartition && tiles * ((max_ctx + P - 1) / P) < kPrefillTargetUnits) P >>= 1;
    return P >= max_ctx ? 0 : P;
}

struct PrefillPlan {
    int P, Pmax;
    bool split;
    size_t ml_offset, acc_offset, bytes;
};

PrefillPlan plan_prefill(int T, int Hq, int d, int max_ctx, int P) {
    PrefillPlan pl{};
    pl.P = P;
    pl.Pmax = P > 0 ? (max_ctx > 0 ? (max_ctx + P - 1) / P : 1) : 1;
    pl.split = P > 0 && pl.Pmax > 1;
    pl.bytes = kWorkspaceHeaderBytes;
    if (!pl.split) return pl;
    auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
    const size_t units = (size_t)T * Hq * pl.Pmax;
    pl.ml_offset = kWorkspaceHeaderBytes;
    pl.acc_offset = up(pl.ml_offset + units * 2 * sizeof(float));
    pl.bytes = up(pl.acc_offset + units * d * sizeof(float));
    return pl;
}

}  // namespace
}  // namespace pkv

extern "C" {

size_t pkv_prefill_workspace_size(int S, int num_query_tokens, int max_query_len, int Hq, int Hkv, int d, int bs,
                                  int max_context_len, int partition_size) {
    if (num_query_tokens < 0) return 0;
    const int P = resolve_prefill_partition(S, max_query_len, Hq, Hkv, d, bs, max_context_len, partition_size);
    if (P < 0) return 0;
    return plan_prefill(num_query_tokens, Hq, d, max_context_len, P).bytes;
}

pkv_status pkv_paged_attention_prefill(void* out, const void* query, pkv_dtype q_dtype, const void* key_cache,
                                       const void* value_cache, pkv_dtype cache_dtype, const int32_t* block_tables,
                                       int MB, const int32_t* context_lens, const int32_t* query_start, int S,
                                       int num_query_tokens, int max_query_len, int max_context_len, int Hq,
                                       int Hkv, int d, int bs, int NB, float scale, int partition_size,
                                       void* workspace, size_t workspace_bytes, int32_t* err_word,
                                       pkv_stream_t stream) {
    return pkv_paged_attention_prefill_ex(out, query, q_dtype, key_cache, value_cache, cache_dtype, block_tables, MB,
                                          context_lens, query_start, S, num_query_tokens, max_query_len,
                                          max_context_len, Hq, Hkv, d, bs, NB, scale, partition_size, workspace,
                                          workspace_bytes, err_word, stream, PKV_PREFILL_AUTO);
}

pkv_status pkv_paged_attention_prefill_ex(void* out, const void* query, pkv_dtype q_dtype, const void* key_cache,
                                          const void* value_cache, pkv_dtype cache_dtype,
                                          const int32_t* block_tables, int MB, const int32_t* context_lens,
                                          const int32_t* query_start, int S, int num_query_tokens,
                                          int max_query_len, int max_context_len, int Hq, int Hkv, int d, int bs,
                                          int NB, float scale, int partition_size, void* workspace,
                                          size_t workspace_bytes, int32_t* err_word, pkv_stream_t stream,
                                          int kernel) {
    if (kernel < PKV_PREFILL_AUTO || kernel > PKV_PREFILL_TCGEN05_2TILE) return PKV_ERR_INVALID_ARG;
    if (S < 0 || MB < 1 || NB < 1 || Hkv < 1 || Hq < 1 || max_context_len < 0 || num_query_tokens < 0 ||
        max_query_len < 0 || max_query_len > max_context_len)
        return PKV_ERR_INVALID_ARG;
    if (Hq % Hkv != 0) return PKV_ERR_INVALID_ARG;
    if (q_dtype != PKV_BF16 || cache_dtype != PKV_BF16) return PKV_ERR_UNSUPPORTED;
    if (!(d == 64 || d == 128) || !(bs == 16 || bs == 32)) return PKV_ERR_UNSUPPORTED;
    if (S > 65535 || (long long)NB * bs >= (1LL << 31)) return PKV_ERR_UNSUPPORTED;
    if ((long long)max_context_len > (long long)MB * bs) return PKV_ERR_INVALID_ARG;
    if (!isfinite(scale)) return PKV_ERR_INVALID_ARG;
    if (partition_size < -1 || (partition_size > 0 && partition_size % bs != 0)) return PKV_ERR_INVALID_ARG;
    if (S == 0 || num_query_tokens == 0) return PKV_OK;
    if (!out || !query || !key_cache || !value_cache || !block_tables || !context_lens || !query_start)
        return PKV_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(query) || !aligned16(key_cache) || !aligned16(value_cache) ||
        (reinterpret_cast<uintptr_t>(block_tables) & 3u) || (reinterpret_cast<uintptr_t>(context_lens) & 3u) ||
        (reinterpret_cast<uintptr_t>(query_start) & 3u))
        return PKV_ERR_INVALID_ARG;
    const int P = resolve_prefill_partition(S, max_query_len, Hq, Hkv, d, bs, max_context_len, partition_size);
    if (P < 0) return PKV_ERR_INVALID_ARG;
    const PrefillPlan pl = plan_prefill(num_query_tokens, Hq, d, max_context_len, P);
    if (pl.split && (!workspace || workspace_bytes < pl.bytes)) return PKV_ERR_WORKSPACE;
    if (workspace && !aligned16(workspace)) return PKV_ERR_INVALID_ARG;
    DecodeParams p{};
    p.out = out; p.q = query; p.kc = key_cache; p.vc = value_cache;
    p.block_tables = block_tables; p.context_lens = context_lens; p.err = err_word;
    p.S = S; p.MB = MB; p.Hq = Hq; p.Hkv = Hkv; p.g = Hq / Hkv; p.d = d; p.bs = bs; p.NB = NB;
    p.P = pl.P > 0 ? pl.P : MB * bs;
    p.Q = p.P;                            // query chunks: whole partitions only
    p.Pmax = pl.Pmax;
    p.max_ctx = max_context_len;
    p.logit_scale_log2 = scale * kLog2e;
    p.out_scale = 1.f;
    if (workspace && workspace_bytes >= kWorkspaceHeaderBytes) p.sched = reinterpret_cast<unsigned*>(workspace);
    if (pl.split) {
        char* ws = static_cast<char*>(workspace);
        p.part_ml = reinterpret_cast<float*>(ws + pl.ml_offset);
        p.part_acc = reinterpret_cast<float*>(ws + pl.acc_offset);
    }
    auto st = reinterpret_cast<cudaStream_t>(stream);
    if (kernel == PKV_PREFILL_MMA_SYNC)
        return from_cuda(launch_prefill_tc(p, query_start, num_query_tokens, max_query_len, num_sms_current(),
                                           pl.split, st));
    // two query tiles per unit pay when a (sequence, K/V head) has 256 or
    // more (query, head) rows on average: prompt chunks, not speculative tokens
    const bool two_tiles = kernel == PKV_PREFILL_TCGEN05_2TILE ||
                           (kernel == PKV_PREFILL_AUTO &&
                            (long long)num_query_tokens * (Hq / Hkv) >= 2LL * kPrefillTileRows * S);
    if (two_tiles)
        return from_cuda(launch_prefill_umma2(p, query_start, num_query_tokens, max_query_len, num_sms_current(),
                                              pl.split, st));
    return from_cuda(launch_prefill_umma(p, query_start, num_query_tokens, max_query_len, num_sms_current(),
                                         pl.split, st));
}

pkv_status pkv_copy_blocks(void* const* key_caches, void* const* value_caches, int num_layers,
                           const int64_t* block_mapping, int P, int NB, size_t block_bytes, int32_t* err_word,
                           pkv_stream_t stream) {
    if (num_layers < 0 || num_layers > kMaxCopyLayers || P < 0 || NB < 1) return PKV_ERR_INVALID_ARG;
    if (block_bytes == 0 || block_bytes % 16 != 0) return PKV_ERR_INVALID_ARG;
    if (P == 0 || num_layers == 0) return PKV_OK;
    if (!key_caches || !value_caches || !block_mapping) return PKV_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(block_mapping) & 7u) return PKV_ERR_INVALID_ARG;
    CopyParams p{};
    for (int l = 0; l < num_layers; ++l) {
        if (!key_caches[l] || !value_caches[l] || !aligned16(key_caches[l]) || !aligned16(value_caches[l]))
            return PKV_ERR_INVALID_ARG;
        p.k[l] = key_caches[l];
        p.v[l] = value_caches[l];
    }
    p.mapping = block_mapping; p.err = err_word; p.P = P; p.NB = NB; p.L = num_layers;
    p.block_bytes = block_bytes;
    return from_cuda(launch_copy(p, reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
