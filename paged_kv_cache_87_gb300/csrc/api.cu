// api.cu -- the extern "C" entry points of libpagedkv.so (include/pagedkv.h).
//
// Host-side validation, workspace layout, dtype/shape dispatch and the
// per-device status word.  Every check that can be made from scalars and
// pointers happens here, before any CUDA call.
#include <math.h>

#include "cache_ops.cuh"
#include "decode_launch.cuh"
#include "mq_attention.cuh"

// Per-device status word written by the kernels (bit-or of PKV_DEV_*).
__device__ unsigned int g_pkv_status = 0u;

namespace pkv {
namespace {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
    bool ready = false;
    int num_sms = 0;
    unsigned* status = nullptr;
};
DeviceInfo g_devices[kMaxDevices];

cudaError_t device_info(DeviceInfo** out) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    DeviceInfo& d = g_devices[dev];
    if (!d.ready) {
        err = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev);
        if (err != cudaSuccess) return err;
        void* sym = nullptr;
        err = cudaGetSymbolAddress(&sym, g_pkv_status);
        if (err != cudaSuccess) return err;
        d.status = static_cast<unsigned*>(sym);
        d.ready = true;
    }
    *out = &d;
    return cudaSuccess;
}

int dtype_bytes(pkv_dtype t) {
    switch (t) {
    case PKV_F32: return 4;
    case PKV_F16: return 2;
    case PKV_BF16: return 2;
    case PKV_FP8_E4M3: return 1;
    default: return 0;
    }
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Work decomposition shared by pkv_decode_workspace_bytes and the decode call.
struct Plan {
    int group, hpi, nsub;
    int chunk_tokens, max_chunks, part_stride;
    size_t off_hdr, off_ctx, off_items, off_recp, off_recc, off_workers, off_seq, off_common,
        off_units, off_expect, off_pm, off_pl, off_pacc, total;
};

// Chunk length: at least 512 tokens, a multiple of 64 (every stage size and
// block size divides it), long enough that a sequence has at most
// kMaxMergeChunks chunks, and at most kMaxItemBlocks blocks.
pkv_status make_plan(int S, int Hq, int Hkv, int HD, int B, int max_ctx, Plan* pl) {
    if (S < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || max_ctx < 0) return PKV_ERR_INVALID_ARG;
    if (HD != 64 && HD != 128) return PKV_ERR_UNSUPPORTED;
    if (B != 8 && B != 16 && B != 32) return PKV_ERR_UNSUPPORTED;
    Plan p{};
    p.group = Hq / Hkv;
    p.hpi = p.group <= 1 ? 1 : (p.group <= 2 ? 2 : 4);
    p.nsub = (p.group + p.hpi - 1) / p.hpi;
    const int per_chunk_min = (max_ctx + kMaxMergeChunks - 1) / kMaxMergeChunks;
    int C = (per_chunk_min + 63) / 64 * 64;
    if (C < 512) C = 512;
    if (C > kMaxItemBlocks * B) return PKV_ERR_UNSUPPORTED;   // context too long
    p.chunk_tokens = C;
    p.max_chunks = max_ctx > 0 ? (max_ctx + C - 1) / C : 1;
    // partial states per (sequence, query head): a fixed-chunk split has at most
    // max_chunks; a balanced split (quota >= one chunk) cuts a unit into at most
    // max_chunks + 1 segments, and a sequence in a shared-prefix group merges
    // the segments of its group's shared unit and of its private unit
    p.part_stride = 2 * (p.max_chunks + 1);
    const size_t s = (size_t)S, mc = (size_t)p.max_chunks;
    const size_t units = s * Hkv * p.nsub;      // nsub of the CUDA-core split: an upper bound
    size_t off = 0;
    p.off_hdr = off;     off += 256;
    p.off_ctx = off;     off = round_up(off + s * 4, 256);
    p.off_items = off;   off = round_up(off + s * mc * 8, 256);
    p.off_recp = off;    off = round_up(off + (2 * s + 1) * 4, 256);
    p.off_recc = off;    off = round_up(off + 2 * s * 16, 256);
    p.off_workers = off; off = round_up(off + (size_t)kMaxWorkers * 32, 256);
    p.off_seq = off;     off = round_up(off + s * 16, 256);
    p.off_common = off;  off = round_up(off + s * 4, 256);
    p.off_units = off;   off = round_up(off + units * 4, 256);
    p.off_expect = off;  off = round_up(off + units * 4, 256);
    const size_t partial_states = max_ctx > 0 ? s * Hq * (size_t)p.part_stride : 0;
    p.off_pm = off;      off = round_up(off + partial_states * 4, 256);
    p.off_pl = off;      off = round_up(off + partial_states * 4, 256);
    p.off_pacc = off;    off = round_up(off + partial_states * HD * 4, 256);
    p.total = off;
    *pl = p;
    return PKV_OK;
}

pkv_status cuda_status(cudaError_t e) { return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA; }

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" {

size_t pkv_decode_workspace_bytes(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                  int block_size, int max_context_len, pkv_dtype kv_dtype) {
    if (dtype_bytes(kv_dtype) == 0) return 0;
    Plan p;
    if (make_plan(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, max_context_len,
                  &p) != PKV_OK)
        return 0;
    return p.total;
}

}  // extern "C"

namespace {

pkv_status decode_impl(const void* query, const void* k_cache, const void* v_cache,
                       const int32_t* block_tables, const int32_t* context_lens, int num_seqs,
                       int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                       int num_blocks, int max_blocks_per_seq, int max_context_len, float scale,
                       pkv_dtype q_dtype, pkv_dtype kv_dtype, float kv_scale, void* workspace,
                       size_t workspace_bytes, void* out, pkv_stream_t stream,
                       int allow_groups) {
    if (num_seqs < 0 || num_blocks <= 0 || max_blocks_per_seq <= 0 || max_context_len < 0)
        return PKV_ERR_INVALID_ARG;
    if (q_dtype != PKV_F32 && q_dtype != PKV_F16 && q_dtype != PKV_BF16)
        return dtype_bytes(q_dtype) ? PKV_ERR_UNSUPPORTED : PKV_ERR_INVALID_ARG;
    if (kv_dtype != q_dtype && kv_dtype != PKV_FP8_E4M3)
        return dtype_bytes(kv_dtype) ? PKV_ERR_UNSUPPORTED : PKV_ERR_INVALID_ARG;
    if (!isfinite(scale) || !isfinite(kv_scale) || !(kv_scale > 0.f)) return PKV_ERR_INVALID_ARG;
    Plan plan;
    pkv_status st = make_plan(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                              max_context_len, &plan);
    if (st != PKV_OK) return st;
    if ((int64_t)max_context_len > (int64_t)max_blocks_per_seq * block_size)
        return PKV_ERR_INVALID_ARG;
    if (num_seqs == 0) return PKV_OK;
    if (!query || !k_cache || !v_cache || !block_tables || !context_lens || !out)
        return PKV_ERR_INVALID_ARG;
    if (!aligned(query, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
        !aligned(out, 16) || !aligned(block_tables, 4) || !aligned(context_lens, 4))
        return PKV_ERR_INVALID_ARG;
    if (!workspace || !aligned(workspace, 256) || workspace_bytes < plan.total)
        return PKV_ERR_WORKSPACE;

    DeviceInfo* dev = nullptr;
    cudaError_t err = device_info(&dev);
    if (err != cudaSuccess) return PKV_ERR_CUDA;

    uint8_t* ws = static_cast<uint8_t*>(workspace);
    DecodeParams p{};
    p.q = query;
    p.k_cache = k_cache;
    p.v_cache = v_cache;
    p.block_tables = block_tables;
    p.context_lens = context_lens;
    p.out = out;
    p.ws.counter = reinterpret_cast<unsigned*>(ws + plan.off_hdr);
    p.ws.total = p.ws.counter + 1;
    p.ws.quota = reinterpret_cast<int*>(p.ws.counter + 2);
    p.ws.ctx_eff = reinterpret_cast<int*>(ws + plan.off_ctx);
    p.ws.items = reinterpret_cast<int2*>(ws + plan.off_items);
    p.ws.rec_prefix = reinterpret_cast<int*>(ws + plan.off_recp);
    p.ws.rec = reinterpret_cast<int4*>(ws + plan.off_recc);
    p.ws.worker_first = reinterpret_cast<int4*>(ws + plan.off_workers);
    p.ws.seq_info = reinterpret_cast<int4*>(ws + plan.off_seq);
    p.ws.common = reinterpret_cast<int*>(ws + plan.off_common);
    p.ws.unit_expect = reinterpret_cast<int*>(ws + plan.off_expect);
    p.ws.unit_done = reinterpret_cast<unsigned*>(ws + plan.off_units);
    p.ws.pm = reinterpret_cast<float*>(ws + plan.off_pm);
    p.ws.pl = reinterpret_cast<float*>(ws + plan.off_pl);
    p.ws.pacc = reinterpret_cast<float*>(ws + plan.off_pacc);
    p.status = dev->status;
    p.num_seqs = num_seqs;
    p.num_q_heads = num_q_heads;
    p.num_kv_heads = num_kv_heads;
    p.group = plan.group;
    p.nsub = plan.nsub;
    p.head_dim = head_dim;
    p.block_size = block_size;
    p.num_blocks = num_blocks;
    p.max_blocks = max_blocks_per_seq;
    p.max_context_len = max_context_len;
    p.chunk_tokens = plan.chunk_tokens;
    p.max_chunks = plan.max_chunks;
    p.part_stride = plan.part_stride;
    p.allow_groups = allow_groups;
    const bool fp8 = kv_dtype == PKV_FP8_E4M3;
    p.qk_scale_log2 = scale * 1.4426950408889634f * (fp8 ? kv_scale : 1.f);
    p.out_scale = fp8 ? kv_scale : 1.f;

    // 16-bit q with 16-bit K/V (any head_dim) or FP8 K/V (head_dim 128) run on
    // tensor cores, 8 query heads per item; fp32 and the rest on CUDA cores
    // (plan.hpi heads per item).
    const bool mma = (q_dtype == PKV_F16 || q_dtype == PKV_BF16) &&
                     (kv_dtype == q_dtype || (kv_dtype == PKV_FP8_E4M3 && head_dim == 128)) &&
                     (int64_t)num_blocks * num_kv_heads * block_size <= 0x7fffffffLL;
    const int hpi = mma ? kMmaHeadsPerItem : plan.hpi;
    p.nsub = (plan.group + hpi - 1) / hpi;   // never above plan.nsub: the workspace fits
    // CUDA-core path with every context within one chunk: no split, no merge, so the
    // decode kernel takes its work items straight from the sequence index (one launch)
    p.self_plan = !mma && max_context_len <= plan.chunk_tokens;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    switch (q_dtype) {
    case PKV_F32: err = decode_dispatch_f32(p, kv_dtype, hpi, s); break;
    case PKV_F16: err = decode_dispatch_f16(p, kv_dtype, hpi, s); break;
    default: err = decode_dispatch_bf16(p, kv_dtype, hpi, s); break;
    }
    return cuda_status(err);
}

}  // namespace

extern "C" {

pkv_status pkv_paged_decode_attention(const void* query, const void* k_cache, const void* v_cache,
                                      const int32_t* block_tables, const int32_t* context_lens,
                                      int num_seqs, int num_q_heads, int num_kv_heads,
                                      int head_dim, int block_size, int num_blocks,
                                      int max_blocks_per_seq, int max_context_len, float scale,
                                      pkv_dtype q_dtype, pkv_dtype kv_dtype, float kv_scale,
                                      void* workspace, size_t workspace_bytes, void* out,
                                      pkv_stream_t stream) {
    return decode_impl(query, k_cache, v_cache, block_tables, context_lens, num_seqs,
                       num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                       max_blocks_per_seq, max_context_len, scale, q_dtype, kv_dtype, kv_scale,
                       workspace, workspace_bytes, out, stream, 0);
}

pkv_status pkv_paged_decode_attention_prefix(
    const void* query, const void* k_cache, const void* v_cache, const int32_t* block_tables,
    const int32_t* context_lens, int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
    int block_size, int num_blocks, int max_blocks_per_seq, int max_context_len, float scale,
    pkv_dtype q_dtype, pkv_dtype kv_dtype, float kv_scale, void* workspace,
    size_t workspace_bytes, void* out, pkv_stream_t stream) {
    return decode_impl(query, k_cache, v_cache, block_tables, context_lens, num_seqs,
                       num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                       max_blocks_per_seq, max_context_len, scale, q_dtype, kv_dtype, kv_scale,
                       workspace, workspace_bytes, out, stream, 1);
}

pkv_status pkv_reshape_and_cache(const void* key, const void* value, void* k_cache,
                                 void* v_cache, const int64_t* slot_mapping, int num_tokens,
                                 int num_kv_heads, int head_dim, int block_size, int num_blocks,
                                 pkv_dtype src_dtype, pkv_dtype kv_dtype, float kv_scale,
                                 pkv_stream_t stream) {
    if (num_tokens < 0 || num_kv_heads <= 0 || num_blocks <= 0) return PKV_ERR_INVALID_ARG;
    if (src_dtype != PKV_F32 && src_dtype != PKV_F16 && src_dtype != PKV_BF16)
        return dtype_bytes(src_dtype) ? PKV_ERR_UNSUPPORTED : PKV_ERR_INVALID_ARG;
    if (kv_dtype != src_dtype && kv_dtype != PKV_FP8_E4M3)
        return dtype_bytes(kv_dtype) ? PKV_ERR_UNSUPPORTED : PKV_ERR_INVALID_ARG;
    if (head_dim != 64 && head_dim != 128) return PKV_ERR_UNSUPPORTED;
    if (block_size != 8 && block_size != 16 && block_size != 32) return PKV_ERR_UNSUPPORTED;
    const bool quant = kv_dtype == PKV_FP8_E4M3;
    if (quant && (!isfinite(kv_scale) || !(kv_scale > 0.f))) return PKV_ERR_INVALID_ARG;
    if (num_tokens == 0) return PKV_OK;
    if (!key || !value || !k_cache || !v_cache || !slot_mapping) return PKV_ERR_INVALID_ARG;
    if (!aligned(key, 16) || !aligned(value, 16) || !aligned(k_cache, 16) ||
        !aligned(v_cache, 16) || !aligned(slot_mapping, 8))
        return PKV_ERR_INVALID_ARG;
    DeviceInfo* dev = nullptr;
    if (device_info(&dev) != cudaSuccess) return PKV_ERR_CUDA;
    ReshapeParams p{key, value, k_cache, v_cache, slot_mapping, dev->status, num_tokens,
                    num_kv_heads, head_dim, block_size, num_blocks, kv_scale};
    return cuda_status(launch_reshape_and_cache(p, src_dtype, quant, dev->num_sms,
                                                reinterpret_cast<cudaStream_t>(stream)));
}

pkv_status pkv_copy_blocks(void* k_cache, void* v_cache, const int32_t* src_dst_pairs,
                           int num_pairs, int num_kv_heads, int head_dim, int block_size,
                           int num_blocks, pkv_dtype kv_dtype, pkv_stream_t stream) {
    if (num_pairs < 0 || num_kv_heads <= 0 || num_blocks <= 0) return PKV_ERR_INVALID_ARG;
    if (dtype_bytes(kv_dtype) == 0) return PKV_ERR_INVALID_ARG;
    if (head_dim != 64 && head_dim != 128) return PKV_ERR_UNSUPPORTED;
    if (block_size != 8 && block_size != 16 && block_size != 32) return PKV_ERR_UNSUPPORTED;
    if (num_pairs > 65535) return PKV_ERR_UNSUPPORTED;
    if (num_pairs == 0) return PKV_OK;
    if (!k_cache || !v_cache || !src_dst_pairs) return PKV_ERR_INVALID_ARG;
    if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(src_dst_pairs, 4))
        return PKV_ERR_INVALID_ARG;
    DeviceInfo* dev = nullptr;
    if (device_info(&dev) != cudaSuccess) return PKV_ERR_CUDA;
    CopyParams p{k_cache, v_cache, k_cache, v_cache, src_dst_pairs, dev->status,
                 (int64_t)num_kv_heads * block_size * head_dim * dtype_bytes(kv_dtype),
                 num_blocks, num_blocks};
    return cuda_status(launch_copy_blocks(p, num_pairs, reinterpret_cast<cudaStream_t>(stream)));
}

pkv_status pkv_swap_blocks(const void* src_k, const void* src_v, int src_num_blocks,
                           void* dst_k, void* dst_v, int dst_num_blocks,
                           const int32_t* src_dst_pairs, int num_pairs, int num_kv_heads,
                           int head_dim, int block_size, pkv_dtype kv_dtype,
                           pkv_stream_t stream) {
    if (num_pairs < 0 || num_kv_heads <= 0 || src_num_blocks <= 0 || dst_num_blocks <= 0)
        return PKV_ERR_INVALID_ARG;
    if (dtype_bytes(kv_dtype) == 0) return PKV_ERR_INVALID_ARG;
    if (head_dim != 64 && head_dim != 128) return PKV_ERR_UNSUPPORTED;
    if (block_size != 8 && block_size != 16 && block_size != 32) return PKV_ERR_UNSUPPORTED;
    if (num_pairs > 65535) return PKV_ERR_UNSUPPORTED;
    if (num_pairs == 0) return PKV_OK;
    if (!src_k || !src_v || !dst_k || !dst_v || !src_dst_pairs) return PKV_ERR_INVALID_ARG;
    if (!aligned(src_k, 16) || !aligned(src_v, 16) || !aligned(dst_k, 16) ||
        !aligned(dst_v, 16) || !aligned(src_dst_pairs, 4))
        return PKV_ERR_INVALID_ARG;
    DeviceInfo* dev = nullptr;
    if (device_info(&dev) != cudaSuccess) return PKV_ERR_CUDA;
    // every buffer must be reachable from this device: device memory, or pinned
    // host memory mapped into the device's address space
    const void* in[5] = {src_k, src_v, dst_k, dst_v, src_dst_pairs};
    void* mapped[5];
    for (int i = 0; i < 5; ++i) {
        cudaPointerAttributes a{};
        if (cudaPointerGetAttributes(&a, in[i]) != cudaSuccess) {
            cudaGetLastError();
            return PKV_ERR_INVALID_ARG;
        }
        if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) {
            mapped[i] = const_cast<void*>(in[i]);
        } else if (a.type == cudaMemoryTypeHost && a.devicePointer != nullptr) {
            mapped[i] = a.devicePointer;
        } else {
            return PKV_ERR_INVALID_ARG;   // pageable or unmapped host memory
        }
    }
    CopyParams p{mapped[0], mapped[1], mapped[2], mapped[3],
                 static_cast<const int32_t*>(mapped[4]), dev->status,
                 (int64_t)num_kv_heads * block_size * head_dim * dtype_bytes(kv_dtype),
                 src_num_blocks, dst_num_blocks};
    return cuda_status(launch_copy_blocks(p, num_pairs, reinterpret_cast<cudaStream_t>(stream)));
}

pkv_status pkv_selftest_wait_bound(pkv_stream_t stream) {
    DeviceInfo* dev = nullptr;
    if (device_info(&dev) != cudaSuccess) return PKV_ERR_CUDA;
    return cuda_status(launch_wait_bound_probe(dev->status, static_cast<cudaStream_t>(stream)));
}

pkv_status pkv_get_device_status(unsigned int* host_code) {
    if (!host_code) return PKV_ERR_INVALID_ARG;
    DeviceInfo* dev = nullptr;
    if (device_info(&dev) != cudaSuccess) return PKV_ERR_CUDA;
    if (cudaDeviceSynchronize() != cudaSuccess) return PKV_ERR_CUDA;
    unsigned v = 0u;
    if (cudaMemcpy(&v, dev->status, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess)
        return PKV_ERR_CUDA;
    const unsigned zero = 0u;
    if (cudaMemcpy(dev->status, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
        return PKV_ERR_CUDA;
    *host_code = v;
    return PKV_OK;
}

const char* pkv_status_string(pkv_status status) {
    switch (status) {
    case PKV_OK: return "ok";
    case PKV_ERR_INVALID_ARG: return "invalid argument";
    case PKV_ERR_UNSUPPORTED: return "unsupported head_dim, block_size, dtype or length";
    case PKV_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case PKV_ERR_CUDA: return "CUDA error";
    case PKV_ERR_OUT_OF_BLOCKS: return "no free KV blocks left";
    default: return "unknown status";
    }
}

int pkv_version(void) { return 100; }


size_t pkv_multi_query_workspace_bytes(int num_seqs) {
    if (num_seqs < 0) return 0;
    return round_up(((size_t)num_seqs + 1) * 4, 256) + round_up((size_t)num_seqs * 4, 256) + 256;
}

namespace {

// The multi-query entry points: causal (tree == nullptr) or draft-tree verification.
pkv_status multi_query_attention(
    const void* query, const void* k_cache, const void* v_cache, const int32_t* block_tables,
    const int32_t* context_lens, const int32_t* query_start, const uint64_t* tree, int num_seqs,
    int total_q, int num_q_heads, int num_kv_heads, int head_dim, int block_size, int num_blocks,
    int max_blocks_per_seq, int max_context_len, float scale, pkv_dtype q_dtype,
    pkv_dtype kv_dtype, float kv_scale, void* workspace, size_t workspace_bytes, void* out,
    pkv_stream_t stream) {
    if (num_seqs < 0 || total_q < 0 || num_q_heads <= 0 || num_kv_heads <= 0 ||
        num_q_heads % num_kv_heads != 0 || num_blocks <= 0 || max_blocks_per_seq <= 0 ||
        max_context_len < 0)
        return PKV_ERR_INVALID_ARG;
    if (!dtype_bytes(q_dtype) || !dtype_bytes(kv_dtype)) return PKV_ERR_INVALID_ARG;
    if (!isfinite(scale) || !isfinite(kv_scale) || !(kv_scale > 0.f)) return PKV_ERR_INVALID_ARG;
    const int group = num_q_heads / num_kv_heads;
    if ((q_dtype != PKV_F16 && q_dtype != PKV_BF16) || kv_dtype != q_dtype || head_dim != 128 ||
        (block_size != 8 && block_size != 16 && block_size != 32) || 128 % group != 0)
        return PKV_ERR_UNSUPPORTED;
    if ((int64_t)num_blocks * num_kv_heads * block_size > INT32_MAX) return PKV_ERR_UNSUPPORTED;
    if ((int64_t)max_context_len > (int64_t)max_blocks_per_seq * block_size)
        return PKV_ERR_INVALID_ARG;
    if (num_seqs == 0 || total_q == 0) return PKV_OK;
    if (!query || !k_cache || !v_cache || !block_tables || !context_lens || !query_start || !out)
        return PKV_ERR_INVALID_ARG;
    if (!aligned(query, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
        !aligned(out, 16) || !aligned(block_tables, 4) || !aligned(context_lens, 4) ||
        !aligned(query_start, 4) || !aligned(tree, 8))
        return PKV_ERR_INVALID_ARG;
    if (!workspace || !aligned(workspace, 256) ||
        workspace_bytes < pkv_multi_query_workspace_bytes(num_seqs))
        return PKV_ERR_WORKSPACE;
    DeviceInfo* dev = nullptr;
    if (device_info(&dev) != cudaSuccess) return PKV_ERR_CUDA;
    MqParams p{};
    p.q = query;
    p.k_cache = k_cache;
    p.v_cache = v_cache;
    p.block_tables = block_tables;
    p.context_lens = context_lens;
    p.query_start = query_start;
    p.tree = tree;
    p.out = out;
    p.item_prefix = static_cast<int*>(workspace);
    p.seq_order = reinterpret_cast<int*>(static_cast<char*>(workspace) +
                                         round_up(((size_t)num_seqs + 1) * 4, 256));
    p.work_next = reinterpret_cast<int*>(static_cast<char*>(workspace) +
                                         round_up(((size_t)num_seqs + 1) * 4, 256) +
                                         round_up((size_t)num_seqs * 4, 256));
    p.status = dev->status;
    p.num_seqs = num_seqs;
    p.total_q = total_q;
    p.num_q_heads = num_q_heads;
    p.num_kv_heads = num_kv_heads;
    p.group = group;
    p.head_dim = head_dim;
    p.block_size = block_size;
    p.num_blocks = num_blocks;
    p.max_blocks = max_blocks_per_seq;
    p.max_context_len = max_context_len;
    p.qk_scale_log2 = scale * 1.4426950408889634f;
    const int64_t items = mq_max_items(num_seqs, total_q, group, num_kv_heads);
    return cuda_status(launch_mq_attention(p, q_dtype, items, dev->num_sms,
                                           static_cast<cudaStream_t>(stream)));
}

}  // namespace

pkv_status pkv_paged_multi_query_attention(
    const void* query, const void* k_cache, const void* v_cache, const int32_t* block_tables,
    const int32_t* context_lens, const int32_t* query_start, int num_seqs, int total_q,
    int num_q_heads, int num_kv_heads, int head_dim, int block_size, int num_blocks,
    int max_blocks_per_seq, int max_context_len, float scale, pkv_dtype q_dtype,
    pkv_dtype kv_dtype, float kv_scale, void* workspace, size_t workspace_bytes, void* out,
    pkv_stream_t stream) {
    return multi_query_attention(query, k_cache, v_cache, block_tables, context_lens,
                                 query_start, nullptr, num_seqs, total_q, num_q_heads,
                                 num_kv_heads, head_dim, block_size, num_blocks,
                                 max_blocks_per_seq, max_context_len, scale, q_dtype, kv_dtype,
                                 kv_scale, workspace, workspace_bytes, out, stream);
}

pkv_status pkv_paged_tree_attention(
    const void* query, const void* k_cache, const void* v_cache, const int32_t* block_tables,
    const int32_t* context_lens, const int32_t* query_start, const uint64_t* tree_mask,
    int num_seqs, int total_q, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
    int num_blocks, int max_blocks_per_seq, int max_context_len, float scale, pkv_dtype q_dtype,
    pkv_dtype kv_dtype, float kv_scale, void* workspace, size_t workspace_bytes, void* out,
    pkv_stream_t stream) {
    if (!tree_mask && num_seqs > 0 && total_q > 0) return PKV_ERR_INVALID_ARG;
    return multi_query_attention(query, k_cache, v_cache, block_tables, context_lens,
                                 query_start, tree_mask, num_seqs, total_q, num_q_heads,
                                 num_kv_heads, head_dim, block_size, num_blocks,
                                 max_blocks_per_seq, max_context_len, scale, q_dtype, kv_dtype,
                                 kv_scale, workspace, workspace_bytes, out, stream);
}

}  // extern "C"
