// decode_f16.cu -- decode variants whose query/output type is f16
// (KV cache in f16 or FP8 e4m3).
#include "decode_launch.cuh"

namespace pkv {

cudaError_t decode_dispatch_f16(const DecodeParams& p, pkv_dtype kv, int hpi, cudaStream_t s) {
    if (kv == PKV_FP8_E4M3) return dispatch_decode_kv<F16, E4M3>(p, hpi, s);
    return dispatch_decode_kv<F16, F16>(p, hpi, s);
}

}  // namespace pkv
