// decode_bf16.cu -- decode variants whose query/output type is bf16
// (KV cache in bf16 or FP8 e4m3).
#include "decode_launch.cuh"

namespace pkv {

cudaError_t decode_dispatch_bf16(const DecodeParams& p, pkv_dtype kv, int hpi, cudaStream_t s) {
    if (kv == PKV_FP8_E4M3) return dispatch_decode_kv<BF16, E4M3>(p, hpi, s);
    return dispatch_decode_kv<BF16, BF16>(p, hpi, s);
}

}  // namespace pkv
