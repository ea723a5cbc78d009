// tmap.cuh -- host encoding of the TMA tensor maps over the K/V pools.
#pragma once

#include <cuda.h>

namespace pkv {

// 2-D map over `rows` rows of `head_dim` elements of `elem_bytes` bytes; box =
// 128 bytes x `box_rows` rows, 128-byte swizzle.  False if it cannot be encoded.
bool encode_pool_map(CUtensorMap* map, const void* pool, int head_dim, int elem_bytes,
                     long long rows, int box_rows);

}  // namespace pkv
