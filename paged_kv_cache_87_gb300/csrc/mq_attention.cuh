// mq_attention.cuh -- parameters and launcher of the multi-query (causal) paged
// attention: several query tokens per sequence over the paged KV cache, for
// prefill, chunked prefill and the verification of a chain of draft tokens.
#pragma once

#include "common.cuh"

namespace pkv {

constexpr int kMqRows = 256;     // (query token, head of the group) rows per CTA: two tiles of 128

struct MqParams {
    const void* q;                 // [total_q, Hq, d]
    const void* k_cache;           // [NB, Hkv, B, d]
    const void* v_cache;
    const int32_t* block_tables;   // [S, max_blocks]
    const int32_t* context_lens;   // [S]: tokens in the cache, the queries' own included
    const int32_t* query_start;    // [S + 1]: query rows of sequence s
    const uint64_t* tree;          // [total_q] draft-tree ancestor bits, or null (causal)
    void* out;                     // [total_q, Hq, d]
    int* item_prefix;              // workspace [S + 1]: items before the k-th launched sequence
    int* seq_order;                // workspace [S]: the sequence launched k-th
    int* work_next;                // workspace: the next item a CTA takes
    unsigned* status;
    int num_seqs, total_q, num_q_heads, num_kv_heads, group, head_dim, block_size, num_blocks;
    int max_blocks;
    int max_context_len;
    float qk_scale_log2;           // scale * log2(e)
};

// Upper bound of the work items of a launch (items of every sequence).
int64_t mq_max_items(int num_seqs, int total_q, int group, int num_kv_heads);

// Launches the planner and min(max_items, num_sms) persistent attention CTAs.
cudaError_t launch_mq_attention(const MqParams& p, pkv_dtype q_dtype, int64_t max_items,
                                int num_sms, cudaStream_t stream);

}  // namespace pkv
