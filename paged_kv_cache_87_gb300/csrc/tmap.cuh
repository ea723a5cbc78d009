// tmap.cuh -- host encoding of the TMA tensor maps over the K/V pools and the queries.
#pragma once

#include <cuda.h>

namespace pkv {

// 2-D map over `rows` rows of `head_dim` elements of `elem_bytes` bytes; box =
// 128 bytes x `box_rows` rows, 128-byte swizzle.  False if it cannot be encoded.
bool encode_pool_map(CUtensorMap* map, const void* pool, int head_dim, int elem_bytes,
                     long long rows, int box_rows);

// The same pool for 16-bit rows of 128 elements as a 4-D tensor (64 elements,
// 8 rows, 2 halves, row groups): one box of box_rows (a multiple of 8) rows carries
// both 128-byte halves and lands as [group of 8 rows][half][8 rows][128 B], 128-byte
// swizzled, so the 8-row groups of a half are 2 KB apart across blocks.
bool encode_pool_map_grouped(CUtensorMap* map, const void* pool, long long rows, int box_rows);

// The queries [total_q][num_q_heads][128] (16-bit) as (element, head, token): one box
// of 64 elements x `group` heads x 128 / group tokens is one 128-byte half of the
// 128 (query token, head of a kv head's group) rows of a multi-query row tile,
// landing as [row][128 B], 128-byte swizzled.  False if it cannot be encoded.
bool encode_q_map(CUtensorMap* map, const void* q, long long total_q, int num_q_heads, int group);

}  // namespace pkv
