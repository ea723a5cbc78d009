// common.cuh -- device helpers shared by the pagedkv kernels (sm_103a).
//
// Inline PTX for the asynchronous-copy machinery (mbarrier, 1-D bulk copies
// into shared memory), element conversions, and the per-device status word.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/pagedkv.h"

namespace pkv {

// Upper bound on the time one mbarrier wait may take before the kernel gives
// up, flags PKV_DEV_WAIT_TIMEOUT and returns.  A correct pipeline completes a
// wait in microseconds; the bound is two seconds of device time.
constexpr uint64_t kWaitNs = 2000000000ull;

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void set_status(unsigned int* status, unsigned int bit) {
    if (status) atomicOr(status, bit);
}

// Arrival on a gpu-scope counter: a release of every write that happens before
// it (a warp barrier first makes the other lanes' writes count) and, for the
// last arriver, an acquire of the writes the earlier arrivals released.
__device__ __forceinline__ unsigned atom_add_acq_rel_gpu(unsigned* ctr, unsigned v) {
    unsigned old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;"
                 : "=r"(old) : "l"(ctr), "r"(v) : "memory");
    return old;
}

// Bring the 128-byte line holding `ptr` into L2 (no register result).
__device__ __forceinline__ void prefetch_l2(const void* ptr) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(ptr));
}

// ------------------------------------------------------------- mbarrier --

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialisation may start while the previous kernel on its stream still runs;
// pdl_wait blocks until that kernel has completed and its memory is visible.
// pdl_launch_dependents lets the next such kernel start launching.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar))
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;"
                 ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase with the given parity.  Returns false on timeout.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    while (true) {
        for (int i = 0; i < 256; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (global_ns() - t0 > kWaitNs) return false;
    }
}

// -------------------------------------------------------- bulk copies --

// 1-D bulk copy global -> shared (this CTA), completing on `bar` with `bytes`
// of transaction count.  Both addresses 16-byte aligned, bytes % 16 == 0.
__device__ __forceinline__ void bulk_g2s(void* smem_dst, const void* gmem_src, uint32_t bytes,
                                         uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_addr(smem_dst)), "l"(gmem_src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// Same, with an L2 eviction-priority hint (the KV stream is read once).
__device__ __forceinline__ void bulk_g2s_hint(void* smem_dst, const void* gmem_src,
                                              uint32_t bytes, uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;"
        ::"r"(smem_addr(smem_dst)), "l"(gmem_src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

// 2-D TMA tile load global -> shared, completing on `bar`; (x, y) = (column, row).
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;"
        ::"r"(smem_addr(smem_dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y),
        "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Order this thread's generic-proxy shared-memory writes before later
// async-proxy accesses (TMA writes, tensor-core reads) of the same bytes.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t l2_evict_last_policy() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// ------------------------------------------------------ named barriers --

__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// ----------------------------------------------------------- math ------

// 2^x on the SFU (ex2.approx.ftz): 2^-inf = +0, 2^0 = 1.
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// --------------------------------------------------------- dtype traits --

struct F32 {
    using storage = float;
    static constexpr int bytes = 4;
    static constexpr pkv_dtype code = PKV_F32;
};
struct F16 {
    using storage = __half;
    static constexpr int bytes = 2;
    static constexpr pkv_dtype code = PKV_F16;
};
struct BF16 {
    using storage = __nv_bfloat16;
    static constexpr int bytes = 2;
    static constexpr pkv_dtype code = PKV_BF16;
};
struct E4M3 {
    using storage = uint8_t;
    static constexpr int bytes = 1;
    static constexpr pkv_dtype code = PKV_FP8_E4M3;
};

// Convert one 16-byte chunk of T elements into 16 / T::bytes floats.
template <typename T>
struct Chunk;

template <>
struct Chunk<F32> {
    static constexpr int n = 4;
    __device__ __forceinline__ static void to_float(const uint4& r, float* f) {
        f[0] = __uint_as_float(r.x);
        f[1] = __uint_as_float(r.y);
        f[2] = __uint_as_float(r.z);
        f[3] = __uint_as_float(r.w);
    }
};

template <>
struct Chunk<F16> {
    static constexpr int n = 8;
    __device__ __forceinline__ static void to_float(const uint4& r, float* f) {
        const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __half2 h = *reinterpret_cast<const __half2*>(&w[i]);
            float2 v = __half22float2(h);
            f[2 * i] = v.x;
            f[2 * i + 1] = v.y;
        }
    }
};

template <>
struct Chunk<BF16> {
    static constexpr int n = 8;
    __device__ __forceinline__ static void to_float(const uint4& r, float* f) {
        const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {   // bf16 is the top half of an fp32
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
};

template <>
struct Chunk<E4M3> {
    static constexpr int n = 16;
    __device__ __forceinline__ static void to_float(const uint4& r, float* f) {
        const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                __nv_fp8x2_storage_t pair = static_cast<__nv_fp8x2_storage_t>(w[i] >> (16 * k));
                __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(pair, __NV_E4M3);
                float2 v = __half22float2(*reinterpret_cast<__half2*>(&hr));
                f[4 * i + 2 * k] = v.x;
                f[4 * i + 2 * k + 1] = v.y;
            }
        }
    }
};

// Scalar load of element i of a q/out-typed buffer as float.
template <typename T>
__device__ __forceinline__ float load_as_float(const void* p, int64_t i);
template <>
__device__ __forceinline__ float load_as_float<F32>(const void* p, int64_t i) {
    return static_cast<const float*>(p)[i];
}
template <>
__device__ __forceinline__ float load_as_float<F16>(const void* p, int64_t i) {
    return __half2float(static_cast<const __half*>(p)[i]);
}
template <>
__device__ __forceinline__ float load_as_float<BF16>(const void* p, int64_t i) {
    return __bfloat162float(static_cast<const __nv_bfloat16*>(p)[i]);
}

// Round-to-nearest-even store of a float into a q/out-typed buffer.
template <typename T>
__device__ __forceinline__ void store_from_float(void* p, int64_t i, float v);
template <>
__device__ __forceinline__ void store_from_float<F32>(void* p, int64_t i, float v) {
    static_cast<float*>(p)[i] = v;
}
template <>
__device__ __forceinline__ void store_from_float<F16>(void* p, int64_t i, float v) {
    static_cast<__half*>(p)[i] = __float2half_rn(v);
}
template <>
__device__ __forceinline__ void store_from_float<BF16>(void* p, int64_t i, float v) {
    static_cast<__nv_bfloat16*>(p)[i] = __float2bfloat16_rn(v);
}

}  // namespace pkv
