// Internal launch interface between the C ABI (pkv_api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>
#include <mutex>
#include <utility>

#include "../../include/pkv.h"

namespace pkv {

// The calling thread's current CUDA context (the driver's cuCtxGetCurrent,
// reached through the runtime's entry-point query), or nullptr when there is
// none or the query is unavailable.  A device reset gives a device ordinal a
// new primary context, in which per-context state (module globals, kernel
// attributes) starts afresh: caches keyed by ordinal alone would outlive it.
CUcontext current_context();

// A kernel's opt-in to more than 48 KB of dynamic shared memory, made once
// per device and context (the attribute belongs to the context).  One
// instance per kernel; safe when several host threads make their first call
// at once.
class SmemOptIn {
  public:
    cudaError_t ensure(const void* kernel, int bytes) {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        const bool cached = dev >= 0 && dev < kDevices;
        CUcontext ctx = current_context();
        if (cached && ctx != nullptr && done_[dev].load(std::memory_order_acquire) == ctx) return cudaSuccess;
        std::lock_guard<std::mutex> lock(mu_);
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        // the call makes the device's primary context current if it was not yet
        if (e == cudaSuccess && cached && (ctx = current_context()) != nullptr)
            done_[dev].store(ctx, std::memory_order_release);
        return e;
    }

  private:
    static constexpr int kDevices = 64;
    std::atomic<CUcontext> done_[kDevices] = {};
    std::mutex mu_;
};

// Launch `kernel` on `st` as a programmatic dependent of the stream's
// previous kernel (pdl_wait / pdl_trigger in pkv_common.cuh).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

constexpr int kMaxCopyLayers = 256;
constexpr size_t kWorkspaceHeaderBytes = 256;   // scheduler counters, zero between calls

struct WriteParams {
    const void* key;
    const void* value;
    void* key_cache;
    void* value_cache;
    const int64_t* slot_mapping;
    int32_t* err;
    int T, NB, bs, Hkv, d;
    float k_scale, v_scale;
};
cudaError_t launch_write(const WriteParams& p, pkv_dtype in_dt, pkv_dtype cache_dt, cudaStream_t st);

struct CopyParams {
    const int64_t* mapping;
    int32_t* err;
    int P, NB, L;
    unsigned long long block_bytes;
    void* k[kMaxCopyLayers];
    void* v[kMaxCopyLayers];
};
cudaError_t launch_copy(const CopyParams& p, cudaStream_t st);

struct RepackParams {
    const int64_t* moves;     // [M][4]: sequence, logical index, source slot, destination slot
    int32_t* token_slots;     // [S][MT]
    int32_t* err;
    int M, L, S, MT, NB, bs;
    unsigned long long token_bytes;
    void* k[kMaxCopyLayers];
    void* v[kMaxCopyLayers];
};
cudaError_t launch_repack(const RepackParams& p, cudaStream_t st);

struct DecodeParams {
    void* out;
    const void* q;
    const void* kc;
    const void* vc;
    const int32_t* block_tables;
    const int32_t* token_slots;   // [S][MT]: decoding through a token table (then block_tables is unused)
    const int32_t* context_lens;  // tokens per sequence (live tokens, with a token table)
    float* part_ml;       // [S][Hq][Pmax][2]: running max (log2 units) and sum
    float* part_acc;      // [S][Hq][Pmax][d]: un-normalised weighted sums of V
    unsigned* sched;      // scheduling counters in the workspace header (or null)
    int32_t* err;
    int S, MB, Hq, Hkv, g, d, bs, NB;
    int MT;               // row length of token_slots
    int P;                // tokens per partition (> 0)
    int Q;                // a sequence's last, partial partition is cut into chunks of Q tokens (Q <= P)
    int hold;             // full partitions at a long sequence's end also cut into chunks (num_partitions)
    int Pmax;             // partitions (and chunks) of the longest sequence: partial results per row
    int max_ctx;
    float logit_scale_log2;   // scale * k_scale * log2(e)
    float out_scale;          // v_scale for E4M3 caches, else 1
    // fused write + decode (new_k != null): each sequence's new token, K and
    // V [S][Hkv][d] of type new_dt, goes to slot_mapping[s], the slot of its
    // last position, before the decode reads it
    const void* new_k;
    const void* new_v;
    const int64_t* slot_mapping;
    pkv_dtype new_dt;
    float k_scale, v_scale;   // E4M3 write scales
};

// Resolved layout of the decode workspace.
struct DecodePlan {
    int P;            // tokens per partition; 0 = one partition per sequence
    int Q;            // chunk of the last, partial partition (= P when not split)
    int Pmax;         // partial results per row the workspace holds (either layout)
    int Pmax_plain;   // ... needed without held-back partitions
    bool split;       // a reduce pass is needed
    size_t ml_offset, acc_offset, bytes;
};

// Host checks of pkv_paged_attention_decode_ex's arguments, with its status
// codes, short of the workspace: PKV_OK when the decode can be enqueued (or,
// with S == 0, has nothing to do).  Touches neither the GPU nor the CUDA
// runtime, so a caller can run it before enqueueing anything of its own.
pkv_status check_decode_args(const void* out, const void* query, pkv_dtype q_dtype, const void* key_cache,
                             const void* value_cache, pkv_dtype cache_dtype, const int32_t* block_tables, int MB,
                             const int32_t* context_lens, int S, int max_context_len, int Hq, int Hkv, int d,
                             int bs, int NB, float scale, float k_scale, float v_scale, int partition_size,
                             int kernel);

cudaError_t launch_decode_simt(const DecodeParams& p, pkv_dtype q_dt, pkv_dtype c_dt, cudaStream_t st);
cudaError_t launch_decode_tc(const DecodeParams& p, pkv_dtype q_dt, pkv_dtype c_dt, int num_sms,
                             cudaStream_t st, bool token_table = false);
cudaError_t launch_decode_reduce(const DecodeParams& p, pkv_dtype q_dt, cudaStream_t st);
bool decode_tc_supports(pkv_dtype q_dt, pkv_dtype c_dt, int d, int bs, int NB);
cudaError_t launch_prefill_tc(const DecodeParams& p, const int32_t* query_start, int T, int max_q_len, int num_sms,
                              bool merge, cudaStream_t st);
cudaError_t launch_prefill_umma(const DecodeParams& p, const int32_t* query_start, int T, int max_q_len, int num_sms,
                                bool merge, cudaStream_t st);
// the same with two 128-row query tiles per unit sharing each K/V stage
cudaError_t launch_prefill_umma2(const DecodeParams& p, const int32_t* query_start, int T, int max_q_len,
                                 int num_sms, bool merge, cudaStream_t st);
cudaError_t launch_prefill_merge(const DecodeParams& p, const int32_t* query_start, int T, int tile_rows,
                                 int max_q, cudaStream_t st);
// 2-D tensor map over a bf16 K or V cache [NB * bs tokens, Hkv * d]: boxes of
// 64 values by min(bs, 32) tokens, 128-byte swizzle
bool prefill_encode_kv_map(CUtensorMap* map, const void* base, const DecodeParams& p);

}  // namespace pkv
