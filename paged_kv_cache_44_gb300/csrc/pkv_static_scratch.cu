// A decode entry point that allocates nothing.
//
// pkv_paged_attention_decode needs scratch memory (the partition triples and
// the work counter) that its caller allocates.  Some callers cannot allocate
// device memory at the point where they decode.  Examples: an engine that
// reserves all of its device memory at start-up and forbids later
// allocations; a real-time loop that must not take the allocator's locks or
// its implicit synchronisation; a foreign-language caller that only holds
// raw pointers and has no device allocator.  This entry point serves them
// with scratch that lives in a fixed array in device memory, owned by the
// library for the life of the process.
#include <mutex>

#include "pkv_internal.h"

// Fixed scratch for pkv_paged_attention_decode_static.  Every GPU that loads
// the library holds this much device memory until the process exits.
static __device__ __align__(256) unsigned char g_decode_scratch[PKV_STATIC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {nullptr};

// Device address of g_decode_scratch on the current device.  In host code
// the array's name is only a host-side stand-in, so the address is looked up
// once per device, with that device current, and cached.
pkv_status scratch_on_current_device(void** addr) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PKV_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_scratch_addr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr) return PKV_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *addr = g_scratch_addr[dev];
    return PKV_OK;
}

}  // namespace

extern "C" pkv_status pkv_paged_attention_decode_static(
    void* out, const void* query, pkv_dtype q_dtype, const void* key_cache, const void* value_cache,
    pkv_dtype cache_dtype, const int32_t* block_tables, int MB, const int32_t* context_lens, int S,
    int max_context_len, int Hq, int Hkv, int d, int bs, int NB, float scale, float k_scale, float v_scale,
    int partition_size, int32_t* err_word, pkv_stream_t stream) {
    if (S < 0) return PKV_ERR_INVALID_ARG;
    if (S == 0) return PKV_OK;
    const size_t need = pkv_decode_workspace_size(S, Hq, Hkv, d, bs, max_context_len, partition_size);
    if (need == 0) return PKV_ERR_INVALID_ARG;                       // sizes the decode would reject
    if (need > (size_t)PKV_STATIC_SCRATCH_BYTES) return PKV_ERR_WORKSPACE;   // beyond the fixed maximum
    void* scratch = nullptr;
    const pkv_status st = scratch_on_current_device(&scratch);
    if (st != PKV_OK) return st;
    // The array keeps whatever the previous call left.  The work counter at
    // its start must be zero; a completed decode leaves it zero, but clear it
    // anyway so that one interrupted call cannot disturb the next.
    if (cudaMemsetAsync(scratch, 0, pkv::kWorkspaceHeaderBytes, reinterpret_cast<cudaStream_t>(stream)) !=
        cudaSuccess)
        return PKV_ERR_CUDA;
    return pkv_paged_attention_decode(out, query, q_dtype, key_cache, value_cache, cache_dtype, block_tables, MB,
                                      context_lens, S, max_context_len, Hq, Hkv, d, bs, NB, scale, k_scale,
                                      v_scale, partition_size, scratch, (size_t)PKV_STATIC_SCRATCH_BYTES,
                                      err_word, stream);
}
