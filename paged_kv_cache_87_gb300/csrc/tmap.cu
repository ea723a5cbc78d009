// tmap.cu -- TMA tensor maps over the K/V pools.
//
// A pool [num_blocks][num_kv_heads][B][d] is viewed as a 2-D tensor of
// num_blocks*num_kv_heads*B rows by d columns.  One box = 128 bytes of a row
// (64 two-byte or 128 one-byte elements) x B rows, with the 128-byte swizzle,
// so one (block, kv head) tile of a 128-byte-row half lands as B swizzled rows.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "tmap.cuh"

namespace pkv {
namespace {

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                 const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                 const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encoder() {
    static EncodeTiled fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiled>(p);
    });
    return fn;
}

}  // namespace

bool encode_pool_map(CUtensorMap* map, const void* pool, int head_dim, int elem_bytes,
                     long long rows, int box_rows) {
    EncodeTiled enc = encoder();
    if (!enc || rows <= 0 || rows > 0x7fffffffLL) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)head_dim, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)head_dim * elem_bytes};
    const cuuint32_t box[2] = {(cuuint32_t)(128 / elem_bytes), (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUtensorMapDataType dt =
        elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
    return enc(map, dt, 2, const_cast<void*>(pool), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

bool encode_pool_map_grouped(CUtensorMap* map, const void* pool, long long rows, int box_rows) {
    EncodeTiled enc = encoder();
    if (!enc || rows <= 0 || rows % 8 != 0 || rows / 8 > 0x7fffffffLL || box_rows % 8 != 0)
        return false;
    // 16-bit rows of 128 elements viewed as (64 elements, 8 rows, 2 halves, rows / 8):
    // a box of box_rows rows lands as [group of 8 rows][half][8 rows][128 bytes]
    const cuuint64_t dims[4] = {64, 8, 2, (cuuint64_t)(rows / 8)};
    const cuuint64_t strides[3] = {256, 128, 2048};
    const cuuint32_t box[4] = {64, 8, 2, (cuuint32_t)(box_rows / 8)};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 4, const_cast<void*>(pool), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

bool encode_q_map(CUtensorMap* map, const void* q, long long total_q, int num_q_heads, int group) {
    EncodeTiled enc = encoder();
    if (!enc || total_q <= 0 || total_q > 0x7fffffffLL || num_q_heads <= 0 || group <= 0 ||
        128 % group != 0 || num_q_heads % group != 0)
        return false;
    // [total_q][num_q_heads][128] 16-bit elements as (element, head, token); a box of
    // 64 elements x group heads x 128 / group tokens lands as 128 rows of 128 bytes,
    // row = token * group + head, 128-byte swizzled; rows past total_q read zeros
    const cuuint64_t dims[3] = {128, (cuuint64_t)num_q_heads, (cuuint64_t)total_q};
    const cuuint64_t strides[2] = {256, (cuuint64_t)num_q_heads * 256};
    const cuuint32_t box[3] = {64, (cuuint32_t)group, (cuuint32_t)(128 / group)};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<void*>(q), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

}  // namespace pkv
