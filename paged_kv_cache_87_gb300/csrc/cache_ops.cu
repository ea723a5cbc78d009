// cache_ops.cu -- the kernels that write the paged KV cache.
//
//  * reshape_and_cache ("PagedAttention: Mathematical Foundations ..." §7
//    kernel 1, "Fused Reshape and Block Write"): each new token's key and
//    value rows go straight to their physical slot, optionally quantised to
//    FP8 e4m3 with a per-tensor scale.
//  * copy_blocks (§5 Parallel Sampling step 4 and §7 kernel 3, "Batched Block
//    Copy-on-Write"): every copy-on-write block copy of a step in one launch.
//  * swap_blocks (§6 Preemption, swapping): the same batched block copy
//    between two pools, one of which may be pinned host memory that the GPU
//    reaches directly (NVLink-C2C on Grace-based systems).
// All are pure data movement: one thread moves one 16-byte chunk per
// iteration with vector loads/stores, in a grid-stride loop.
#include "cache_ops.cuh"

namespace pkv {

// Two fp32 values -> two e4m3 codes (round to nearest even, saturate to
// +-448, NaN -> NaN), packed little-endian: `lo` lands in the lower byte.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

template <typename ST>
__device__ __forceinline__ void load16_as_float(const uint8_t* src, float* f);

template <>
__device__ __forceinline__ void load16_as_float<F32>(const uint8_t* src, float* f) {
    const uint4* s = reinterpret_cast<const uint4*>(src);
#pragma unroll
    for (int i = 0; i < 4; ++i) Chunk<F32>::to_float(s[i], f + 4 * i);
}
template <>
__device__ __forceinline__ void load16_as_float<F16>(const uint8_t* src, float* f) {
    const uint4* s = reinterpret_cast<const uint4*>(src);
#pragma unroll
    for (int i = 0; i < 2; ++i) Chunk<F16>::to_float(s[i], f + 8 * i);
}
template <>
__device__ __forceinline__ void load16_as_float<BF16>(const uint8_t* src, float* f) {
    const uint4* s = reinterpret_cast<const uint4*>(src);
#pragma unroll
    for (int i = 0; i < 2; ++i) Chunk<BF16>::to_float(s[i], f + 8 * i);
}

// One thread = one 16-byte chunk of one (token, kv head) row of the cache.
template <typename ST, bool QUANT>
__global__ void __launch_bounds__(256) reshape_and_cache_kernel(ReshapeParams p) {
    pdl_launch_dependents();   // the decode launched next may start its launch now
    constexpr int KB = QUANT ? 1 : ST::bytes;          // cache element bytes
    const int row_chunks = p.head_dim * KB / 16;
    const int64_t total = (int64_t)p.num_tokens * p.num_kv_heads * row_chunks;
    const int64_t pool_slots = (int64_t)p.num_blocks * p.block_size;
    for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int c = (int)(idx % row_chunks);
        const int64_t th = idx / row_chunks;
        const int h = (int)(th % p.num_kv_heads);
        const int64_t t = th / p.num_kv_heads;
        const int64_t slot = p.slot_mapping[t];
        if (slot < 0) continue;
        if (slot >= pool_slots) {
            if (c == 0 && h == 0) set_status(p.status, PKV_DEV_BAD_SLOT);
            continue;
        }
        const int64_t blk = slot / p.block_size, off = slot % p.block_size;
        const int64_t drow = ((blk * p.num_kv_heads + h) * p.block_size + off) * p.head_dim;
        const int64_t srow = (t * p.num_kv_heads + h) * p.head_dim;
        if constexpr (!QUANT) {
            const int64_t db = drow * KB + (int64_t)c * 16, sb = srow * KB + (int64_t)c * 16;
            *reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.k_cache) + db) =
                *reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(p.key) + sb);
            *reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.v_cache) + db) =
                *reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(p.value) + sb);
        } else {
            // 16 cache elements from 16 source elements
            const int64_t e0 = (int64_t)c * 16;
            const int64_t sb = (srow + e0) * ST::bytes;
            const void* srcs[2] = {p.key, p.value};
            void* dsts[2] = {p.k_cache, p.v_cache};
#pragma unroll
            for (int kv = 0; kv < 2; ++kv) {
                float f[16];
                load16_as_float<ST>(static_cast<const uint8_t*>(srcs[kv]) + sb, f);
                uint32_t w[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float a = __fdiv_rn(f[4 * i + 0], p.kv_scale);
                    const float b = __fdiv_rn(f[4 * i + 1], p.kv_scale);
                    const float cc = __fdiv_rn(f[4 * i + 2], p.kv_scale);
                    const float d = __fdiv_rn(f[4 * i + 3], p.kv_scale);
                    w[i] = cvt_e4m3x2(a, b) | (cvt_e4m3x2(cc, d) << 16);
                }
                *reinterpret_cast<uint4*>(static_cast<uint8_t*>(dsts[kv]) + drow + e0) =
                    make_uint4(w[0], w[1], w[2], w[3]);
            }
        }
    }
}

// grid = (pairs, slices of a block, 2 caches); one 16-byte chunk per thread-iteration.
// Block pairs[i][0] of the source pool -> block pairs[i][1] of the destination.
__global__ void __launch_bounds__(256) copy_blocks_kernel(CopyParams p) {
    pdl_launch_dependents();
    const int pair = blockIdx.x;
    const int32_t src = p.pairs[2 * pair], dst = p.pairs[2 * pair + 1];
    if (src < 0 || src >= p.src_num_blocks || dst < 0 || dst >= p.dst_num_blocks) {
        if (threadIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0)
            set_status(p.status, PKV_DEV_BAD_PAIR);
        return;
    }
    const uint8_t* sc = static_cast<const uint8_t*>(blockIdx.z == 0 ? p.src_k : p.src_v);
    uint8_t* dc = static_cast<uint8_t*>(blockIdx.z == 0 ? p.dst_k : p.dst_v);
    const uint4* s = reinterpret_cast<const uint4*>(sc + (int64_t)src * p.block_bytes);
    uint4* d = reinterpret_cast<uint4*>(dc + (int64_t)dst * p.block_bytes);
    const int64_t n = p.block_bytes / 16;
    for (int64_t i = (int64_t)blockIdx.y * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.y * blockDim.x)
        d[i] = s[i];
}

cudaError_t launch_reshape_and_cache(const ReshapeParams& p, pkv_dtype src, bool quant,
                                     int num_sms, cudaStream_t stream) {
    const int kb = quant ? 1 : (src == PKV_F32 ? 4 : 2);
    const int64_t total = (int64_t)p.num_tokens * p.num_kv_heads * (p.head_dim * kb / 16);
    int64_t want = (total + 255) / 256;
    const int64_t cap = (int64_t)num_sms * 8;
    const int grid = (int)(want < cap ? (want < 1 ? 1 : want) : cap);
    switch (src) {
    case PKV_F32:
        if (quant) reshape_and_cache_kernel<F32, true><<<grid, 256, 0, stream>>>(p);
        else reshape_and_cache_kernel<F32, false><<<grid, 256, 0, stream>>>(p);
        break;
    case PKV_F16:
        if (quant) reshape_and_cache_kernel<F16, true><<<grid, 256, 0, stream>>>(p);
        else reshape_and_cache_kernel<F16, false><<<grid, 256, 0, stream>>>(p);
        break;
    case PKV_BF16:
        if (quant) reshape_and_cache_kernel<BF16, true><<<grid, 256, 0, stream>>>(p);
        else reshape_and_cache_kernel<BF16, false><<<grid, 256, 0, stream>>>(p);
        break;
    default:
        return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

cudaError_t launch_copy_blocks(const CopyParams& p, int num_pairs, cudaStream_t stream) {
    const int64_t chunks = p.block_bytes / 16;
    int slices = (int)((chunks + 255) / 256);
    if (slices > 64) slices = 64;
    if (slices < 1) slices = 1;
    dim3 grid(num_pairs, slices, 2);
    copy_blocks_kernel<<<grid, 256, 0, stream>>>(p);
    return cudaGetLastError();
}

// One thread waits on an mbarrier that nothing arrives at: the bounded wait every
// pipeline uses gives up after kWaitNs and the kernel flags PKV_DEV_WAIT_TIMEOUT.
__global__ void wait_bound_probe_kernel(unsigned* status) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
        if (!mbar_wait(&bar, 0)) set_status(status, PKV_DEV_WAIT_TIMEOUT);
    }
}

cudaError_t launch_wait_bound_probe(unsigned* status, cudaStream_t stream) {
    wait_bound_probe_kernel<<<1, 32, 0, stream>>>(status);
    return cudaGetLastError();
}

}  // namespace pkv
