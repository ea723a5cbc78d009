// decode_launch.cuh -- host-side launch of the planning + decode kernels for
// one query type.  Each decode_<qtype>.cu includes this and instantiates the
// (kv type, head_dim, heads-per-item) variants it serves, so the variants
// compile in parallel translation units.
#pragma once

#include <type_traits>

#include "decode.cuh"
#include "decode_mma.cuh"
#include "tmap.cuh"

namespace pkv {

// Per-device cache of a kernel's resident CTAs per SM (0 = not yet queried).
struct OccCache {
    int ctas[64] = {0};
};

template <typename QT, typename KT, int HD, int HPI>
cudaError_t launch_decode_simt(const DecodeParams& p, cudaStream_t stream) {
    using Cfg = SimtCfg<QT, KT, HD, HPI>;
    const size_t smem = SimtSmem<Cfg>::total;
    static OccCache occ;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    auto kernel = decode_simt_kernel<QT, KT, HD, HPI>;
    if (occ.ctas[dev] == 0) {
        err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (err != cudaSuccess) return err;
        int per_sm = 0, sms = 0;
        err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, Cfg::THREADS, smem);
        if (err != cudaSuccess) return err;
        err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (err != cudaSuccess) return err;
        occ.ctas[dev] = (per_sm > 0 ? per_sm : 1) * sms;
    }
    // the decode kernel starts launching while its predecessor runs and waits for it
    // on the device (programmatic dependent launch)
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)occ.ctas[dev], 1, 1);
    cfg.blockDim = dim3(Cfg::THREADS, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    if (p.self_plan) {
        // every context within one chunk: the decode kernel plans for itself
        const long long units = (long long)p.num_seqs * p.num_kv_heads * p.nsub;
        cfg.gridDim.x = (unsigned)(units < occ.ctas[dev] ? units : occ.ctas[dev]);
        return cudaLaunchKernelEx(&cfg, kernel, p);
    }
    plan_kernel<QT><<<1, 1024, 0, stream>>>(p);
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    return cudaLaunchKernelEx(&cfg, kernel, p);
}

// Tensor-core variant: 16-bit q, 16-bit or FP8 K/V, 8 query heads per item.
// The prefix-aware entry point groups sequences that share leading blocks
// (up to 16 query heads per shared unit) when a kv head has at most 8 query
// heads: the NT = 2 kernel.  Otherwise NT = 1.
template <typename QT, typename KT, int HD, int NT>
cudaError_t launch_decode_mma_nt(const DecodeParams& p, cudaStream_t stream) {
    using Cfg = MmaCfg<QT, KT, HD, NT>;
    static OccCache occ;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    auto kernel = decode_mma_kernel<QT, KT, HD, NT>;
    if (occ.ctas[dev] == 0) {
        err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   (int)Cfg::SMEM);
        if (err != cudaSuccess) return err;
        int per_sm = 0, sms = 0;
        err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, Cfg::THREADS,
                                                            Cfg::SMEM);
        if (err != cudaSuccess) return err;
        err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (err != cudaSuccess) return err;
        occ.ctas[dev] = min((per_sm > 0 ? per_sm : 1) * sms, kMaxWorkers);
    }
    CUtensorMap tk, tv;
    const long long rows = (long long)p.num_blocks * p.num_kv_heads * p.block_size;
    if (!encode_pool_map(&tk, p.k_cache, HD, KT::bytes, rows, p.block_size) ||
        !encode_pool_map(&tv, p.v_cache, HD, KT::bytes, rows, p.block_size))
        return cudaErrorInvalidValue;
    DecodeParams ps = p;
    ps.num_workers = occ.ctas[dev];
    // the planner (after the shared-prefix detection of a prefix-aware launch), decode
    // and merge kernels start launching while their predecessor runs and wait for it
    // on the device (programmatic dependent launch)
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    const bool grouping = ps.allow_groups && ps.nsub == 1 && ps.group <= kMmaHeadsPerItem;
    if (grouping) {
        prefix_common_kernel<QT><<<(unsigned)((ps.num_seqs + 7) / 8), 256, 0, stream>>>(ps);
        err = cudaGetLastError();
        if (err != cudaSuccess) return err;
        cudaLaunchConfig_t pc = {};
        pc.gridDim = dim3(1, 1, 1);
        pc.blockDim = dim3(1024, 1, 1);
        pc.stream = stream;
        pc.attrs = pdl;
        pc.numAttrs = 1;
        err = cudaLaunchKernelEx(&pc, plan_split_kernel<QT>, ps);
    } else {
        cudaLaunchConfig_t pc = {};
        pc.gridDim = dim3(1, 1, 1);
        pc.blockDim = dim3(1024, 1, 1);
        pc.stream = stream;
        pc.attrs = pdl;
        pc.numAttrs = 1;
        err = cudaLaunchKernelEx(&pc, plan_split_kernel<QT>, ps);
    }
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ps.num_workers, 1, 1);
    cfg.blockDim = dim3(Cfg::THREADS, 1, 1);
    cfg.dynamicSmemBytes = Cfg::SMEM;
    cfg.stream = stream;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    err = cudaLaunchKernelEx(&cfg, kernel, ps, tk, tv);
    if (err != cudaSuccess || !ps.allow_groups) return err;
    const int units = ps.num_seqs * ps.num_kv_heads * ps.nsub;
    cfg.gridDim = dim3((unsigned)((units + 7) / 8), 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.dynamicSmemBytes = 0;
    return cudaLaunchKernelEx(&cfg, merge_units_kernel<QT, HD>, ps);
}

template <typename QT, typename KT, int HD>
cudaError_t launch_decode_mma(const DecodeParams& p, cudaStream_t stream) {
    return p.allow_groups && p.nsub == 1 ? launch_decode_mma_nt<QT, KT, HD, 2>(p, stream)
                                         : launch_decode_mma_nt<QT, KT, HD, 1>(p, stream);
}

template <typename QT, typename KT>
cudaError_t dispatch_decode_kv(const DecodeParams& p, int hpi, cudaStream_t stream) {
    if constexpr (!std::is_same<QT, F32>::value) {
        if (hpi == kMmaHeadsPerItem) {
            if constexpr (std::is_same<KT, E4M3>::value)
                return launch_decode_mma<QT, KT, 128>(p, stream);
            else
                return p.head_dim == 128 ? launch_decode_mma<QT, KT, 128>(p, stream)
                                         : launch_decode_mma<QT, KT, 64>(p, stream);
        }
    }
    if (p.head_dim == 128) {
        if (hpi == 1) return launch_decode_simt<QT, KT, 128, 1>(p, stream);
        if (hpi == 2) return launch_decode_simt<QT, KT, 128, 2>(p, stream);
        return launch_decode_simt<QT, KT, 128, 4>(p, stream);
    }
    if (hpi == 1) return launch_decode_simt<QT, KT, 64, 1>(p, stream);
    if (hpi == 2) return launch_decode_simt<QT, KT, 64, 2>(p, stream);
    return launch_decode_simt<QT, KT, 64, 4>(p, stream);
}

// Defined in decode_f32.cu / decode_f16.cu / decode_bf16.cu.
cudaError_t decode_dispatch_f32(const DecodeParams& p, pkv_dtype kv, int hpi, cudaStream_t s);
cudaError_t decode_dispatch_f16(const DecodeParams& p, pkv_dtype kv, int hpi, cudaStream_t s);
cudaError_t decode_dispatch_bf16(const DecodeParams& p, pkv_dtype kv, int hpi, cudaStream_t s);

}  // namespace pkv
