// decode_noalloc.cu -- paged decode attention for callers that cannot allocate.
//
// pkv_paged_decode_attention needs a caller-provided device workspace (the
// work list, arrival counters and split-KV partial states).  Some callers
// cannot call cudaMalloc when they decode: plugins whose host framework owns
// every device allocation (its caching allocator must see all memory),
// servers held to a device-memory budget fixed at start-up, and latency-
// critical loops in which a cudaMalloc, which may synchronise the device, is
// not allowed.  For them this file keeps the workspace in a fixed, file-scope
// device array that the module carries on every device that loads the
// library, and passes its device address to the same kernels.  Nothing here
// allocates.
#include <mutex>

#include "../../include/pagedkv.h"
#include <cuda_runtime.h>

namespace {

constexpr size_t kScratchBytes = PKV_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// The scratch.  In host code this name is only a host-side stand-in for the
// device array, never a usable address: kernels get the address that
// cudaGetSymbolAddress returns for the current device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

// Once per device, with that device current: look up the array's device address.
pkv_status scratch_for_current_device(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return PKV_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (g_scratch_ptr[dev] == nullptr) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr)
            return PKV_ERR_CUDA;
        g_scratch_ptr[dev] = ptr;
    }
    *out = g_scratch_ptr[dev];
    return PKV_OK;
}

}  // namespace

extern "C" PKV_API pkv_status pkv_paged_decode_attention_noalloc(
    const void* query, const void* k_cache, const void* v_cache, const int32_t* block_tables,
    const int32_t* context_lens, int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
    int block_size, int num_blocks, int max_blocks_per_seq, int max_context_len, float scale,
    pkv_dtype q_dtype, pkv_dtype kv_dtype, float kv_scale, void* out, pkv_stream_t stream) {
    const size_t need = pkv_decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                                   block_size, max_context_len, kv_dtype);
    if (need > kScratchBytes) return PKV_ERR_WORKSPACE;   // beyond the static scratch
    void* scratch = nullptr;
    const pkv_status st = scratch_for_current_device(&scratch);
    if (st != PKV_OK) return st;
    // The planning kernel rewrites the counters and the work list on every
    // call, so the previous call's contents need no clearing here.
    return pkv_paged_decode_attention(query, k_cache, v_cache, block_tables, context_lens,
                                      num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                                      num_blocks, max_blocks_per_seq, max_context_len, scale,
                                      q_dtype, kv_dtype, kv_scale, scratch, kScratchBytes, out,
                                      stream);
}
