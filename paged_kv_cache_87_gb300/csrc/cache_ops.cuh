// cache_ops.cuh -- parameters and host launchers of the cache-writing kernels.
#pragma once

#include "common.cuh"

namespace pkv {

struct ReshapeParams {
    const void* key;
    const void* value;
    void* k_cache;
    void* v_cache;
    const int64_t* slot_mapping;
    unsigned* status;
    int num_tokens, num_kv_heads, head_dim, block_size, num_blocks;
    float kv_scale;
};

struct CopyParams {
    const void* src_k;    // source pool (device memory or mapped pinned host memory)
    const void* src_v;
    void* dst_k;          // destination pool (same pool for copy-on-write)
    void* dst_v;
    const int32_t* pairs;
    unsigned* status;
    int64_t block_bytes;   // num_kv_heads * block_size * head_dim * element bytes
    int src_num_blocks, dst_num_blocks;
};

cudaError_t launch_reshape_and_cache(const ReshapeParams& p, pkv_dtype src, bool quant,
                                     int num_sms, cudaStream_t stream);
cudaError_t launch_copy_blocks(const CopyParams& p, int num_pairs, cudaStream_t stream);

// A kernel whose pipeline wait can never complete: it flags PKV_DEV_WAIT_TIMEOUT in
// `status` once the wait's bound has passed, and returns.
cudaError_t launch_wait_bound_probe(unsigned* status, cudaStream_t stream);

}  // namespace pkv
