// block_manager.cpp -- host-side block manager of the paged KV cache.
//
// "PagedAttention: Mathematical Foundations ..." §4 (Allocation Lifecycle:
// prefill takes ceil(N/B) blocks from a free list, decoding appends to the
// last block, a full last block makes the manager take a new one, completion
// decrements reference counts and returns blocks that reach zero) and §5
// (parallel sampling / beam search: sequences fork by sharing every block with
// reference count + 1; writing into a shared, partially filled block first
// copies it to a private block -- copy-on-write).  "Pytorch implementation of
// paper ..." §3 hands blocks out from the front of a FIFO free list and
// returns freed ones to its back; this manager does the same.
//
// The manager owns no device memory: it produces block tables, slot ids and
// (src, dst) copy pairs for the device kernels (reshape_and_cache,
// copy_blocks, paged_decode_attention).
#include <deque>
#include <new>
#include <unordered_map>
#include <vector>

#include "../../include/pagedkv.h"

namespace {

struct Sequence {
    std::vector<int32_t> blocks;
    int64_t num_tokens = 0;
};

}  // namespace

struct pkv_block_manager {
    int num_blocks = 0;
    int block_size = 0;
    std::deque<int32_t> free_list;
    std::vector<int32_t> refcount;
    std::unordered_map<int64_t, Sequence> seqs;

    bool take(int32_t* out) {
        if (free_list.empty()) return false;
        *out = free_list.front();
        free_list.pop_front();
        refcount[*out] = 1;
        return true;
    }
    void release(int32_t b) {
        if (--refcount[b] == 0) free_list.push_back(b);
    }
};

extern "C" {

PKV_API pkv_block_manager* pkv_bm_create(int num_blocks, int block_size,
                                         const int32_t* free_order, int num_free) {
    if (num_blocks <= 0 || block_size <= 0) return nullptr;
    pkv_block_manager* m = new (std::nothrow) pkv_block_manager();
    if (!m) return nullptr;
    m->num_blocks = num_blocks;
    m->block_size = block_size;
    m->refcount.assign((size_t)num_blocks, 0);
    if (free_order) {
        std::vector<char> seen((size_t)num_blocks, 0);
        for (int i = 0; i < num_free; ++i) {
            const int32_t b = free_order[i];
            if (b < 0 || b >= num_blocks || seen[(size_t)b]) {
                delete m;
                return nullptr;
            }
            seen[(size_t)b] = 1;
            m->free_list.push_back(b);
        }
    } else {
        for (int32_t b = 0; b < num_blocks; ++b) m->free_list.push_back(b);
    }
    return m;
}

PKV_API void pkv_bm_destroy(pkv_block_manager* m) { delete m; }

PKV_API int pkv_bm_num_free(const pkv_block_manager* m) {
    return m ? (int)m->free_list.size() : -1;
}

PKV_API int pkv_bm_refcount(const pkv_block_manager* m, int32_t block) {
    if (!m || block < 0 || block >= m->num_blocks) return -1;
    return m->refcount[(size_t)block];
}

PKV_API pkv_status pkv_bm_add_sequence(pkv_block_manager* m, int64_t seq_id,
                                       int64_t num_tokens) {
    if (!m || num_tokens < 0 || m->seqs.count(seq_id)) return PKV_ERR_INVALID_ARG;
    const int64_t need = (num_tokens + m->block_size - 1) / m->block_size;
    if (need > (int64_t)m->free_list.size()) return PKV_ERR_OUT_OF_BLOCKS;
    Sequence s;
    s.num_tokens = num_tokens;
    s.blocks.resize((size_t)need);
    for (int64_t i = 0; i < need; ++i) m->take(&s.blocks[(size_t)i]);
    m->seqs.emplace(seq_id, std::move(s));
    return PKV_OK;
}

PKV_API pkv_status pkv_bm_fork(pkv_block_manager* m, int64_t parent, int64_t child) {
    if (!m || m->seqs.count(child)) return PKV_ERR_INVALID_ARG;
    auto it = m->seqs.find(parent);
    if (it == m->seqs.end()) return PKV_ERR_INVALID_ARG;
    Sequence s = it->second;
    for (int32_t b : s.blocks) ++m->refcount[(size_t)b];
    m->seqs.emplace(child, std::move(s));
    return PKV_OK;
}

PKV_API pkv_status pkv_bm_append_slot(pkv_block_manager* m, int64_t seq_id, int64_t* slot,
                                      int32_t* cow_src, int32_t* cow_dst) {
    if (!m || !slot || !cow_src || !cow_dst) return PKV_ERR_INVALID_ARG;
    auto it = m->seqs.find(seq_id);
    if (it == m->seqs.end()) return PKV_ERR_INVALID_ARG;
    Sequence& s = it->second;
    const int B = m->block_size;
    const int64_t j = s.num_tokens / B, off = s.num_tokens % B;
    *cow_src = *cow_dst = -1;
    if (j >= (int64_t)s.blocks.size()) {               // block overflow: take a new block
        int32_t b;
        if (!m->take(&b)) return PKV_ERR_OUT_OF_BLOCKS;
        s.blocks.push_back(b);
    } else if (m->refcount[(size_t)s.blocks[(size_t)j]] > 1) {   // shared: copy on write
        int32_t b;
        if (!m->take(&b)) return PKV_ERR_OUT_OF_BLOCKS;
        *cow_src = s.blocks[(size_t)j];
        *cow_dst = b;
        --m->refcount[(size_t)*cow_src];
        s.blocks[(size_t)j] = b;
    }
    *slot = (int64_t)s.blocks[(size_t)j] * B + off;
    ++s.num_tokens;
    return PKV_OK;
}

PKV_API pkv_status pkv_bm_free_sequence(pkv_block_manager* m, int64_t seq_id) {
    if (!m) return PKV_ERR_INVALID_ARG;
    auto it = m->seqs.find(seq_id);
    if (it == m->seqs.end()) return PKV_ERR_INVALID_ARG;
    for (int32_t b : it->second.blocks) m->release(b);
    m->seqs.erase(it);
    return PKV_OK;
}

PKV_API pkv_status pkv_bm_sequence(const pkv_block_manager* m, int64_t seq_id,
                                   int32_t* table, int max_blocks, int* num_blocks,
                                   int64_t* num_tokens) {
    if (!m || !num_blocks || !num_tokens) return PKV_ERR_INVALID_ARG;
    auto it = m->seqs.find(seq_id);
    if (it == m->seqs.end()) return PKV_ERR_INVALID_ARG;
    const Sequence& s = it->second;
    *num_blocks = (int)s.blocks.size();
    *num_tokens = s.num_tokens;
    if (table) {
        if ((int)s.blocks.size() > max_blocks) return PKV_ERR_INVALID_ARG;
        for (size_t i = 0; i < s.blocks.size(); ++i) table[i] = s.blocks[i];
        for (int i = (int)s.blocks.size(); i < max_blocks; ++i) table[i] = -1;
    }
    return PKV_OK;
}

PKV_API pkv_status pkv_bm_prepare_step(pkv_block_manager* m, const int64_t* seq_ids, int n,
                                       int64_t* slot_mapping, int32_t* cow_pairs,
                                       int* num_cow, int32_t* block_tables, int max_blocks,
                                       int32_t* context_lens) {
    if (!m || n < 0 || (n && (!seq_ids || !slot_mapping || !cow_pairs || !num_cow)))
        return PKV_ERR_INVALID_ARG;
    // validate first, so a failure leaves the manager unchanged.  Blocks the step
    // takes: one per sequence whose last block is full, and, for a shared block
    // with reference count r that k of the step's sequences write into, min(k, r-1)
    // copies -- each writer but the last to find it shared copies it and drops the
    // count by one, so once it reaches 1 the remaining writer owns it
    int64_t new_blocks = 0;
    std::unordered_map<int32_t, int64_t> writers;   // shared block -> writers this step
    for (int i = 0; i < n; ++i) {
        auto it = m->seqs.find(seq_ids[i]);
        if (it == m->seqs.end()) return PKV_ERR_INVALID_ARG;
        for (int k = 0; k < i; ++k)
            if (seq_ids[k] == seq_ids[i]) return PKV_ERR_INVALID_ARG;
        const Sequence& s = it->second;
        const int64_t j = s.num_tokens / m->block_size;
        if (j >= (int64_t)s.blocks.size()) {
            ++new_blocks;
        } else {
            const int32_t b = s.blocks[(size_t)j];
            if (m->refcount[(size_t)b] > 1) ++writers[b];
        }
        if (block_tables && (int64_t)s.blocks.size() + 1 > max_blocks) return PKV_ERR_INVALID_ARG;
    }
    for (const auto& kv : writers) {
        const int64_t r = m->refcount[(size_t)kv.first];
        new_blocks += kv.second < r - 1 ? kv.second : r - 1;
    }
    if (new_blocks > (int64_t)m->free_list.size()) return PKV_ERR_OUT_OF_BLOCKS;
    int ncow = 0;
    for (int i = 0; i < n; ++i) {
        int32_t src, dst;
        pkv_bm_append_slot(m, seq_ids[i], &slot_mapping[i], &src, &dst);
        if (src >= 0) {
            cow_pairs[2 * ncow] = src;
            cow_pairs[2 * ncow + 1] = dst;
            ++ncow;
        }
    }
    *num_cow = ncow;
    for (int i = 0; i < n; ++i) {
        const Sequence& s = m->seqs.find(seq_ids[i])->second;
        if (block_tables) {
            int32_t* row = block_tables + (int64_t)i * max_blocks;
            for (size_t k = 0; k < s.blocks.size(); ++k) row[k] = s.blocks[k];
            for (int k = (int)s.blocks.size(); k < max_blocks; ++k) row[k] = -1;
        }
        if (context_lens) context_lens[i] = (int32_t)s.num_tokens;
    }
    return PKV_OK;
}

}  // extern "C"
