// decode_f32.cu -- decode variants whose query/output type is f32
// (KV cache in f32 or FP8 e4m3).
#include "decode_launch.cuh"

namespace pkv {

cudaError_t decode_dispatch_f32(const DecodeParams& p, pkv_dtype kv, int hpi, cudaStream_t s) {
    if (kv == PKV_FP8_E4M3) return dispatch_decode_kv<F32, E4M3>(p, hpi, s);
    return dispatch_decode_kv<F32, F32>(p, hpi, s);
}

}  // namespace pkv
