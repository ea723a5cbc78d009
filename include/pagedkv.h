/*
 * pagedkv.h -- C ABI of libpagedkv.so: the data-parallel hot path of
 * PagedAttention on one GB300 (sm_103a).
 *
 * Three operations, after "PagedAttention: Mathematical Foundations, Virtual
 * Memory Block Allocation, and Zero-Waste KV Cache Serving" (llms.blog):
 *   - pkv_paged_decode_attention: §3 (block-wise attention over a context
 *     split into B-token blocks) and §7 kernel 2 / the decode pseudocode
 *     (one pass over the block table with a running max, rescale and sum);
 *   - pkv_reshape_and_cache: §7 kernel 1 (write each new token's key and
 *     value straight into its physical block slot);
 *   - pkv_copy_blocks: §5 Parallel Sampling step 4 and §7 kernel 3 (all
 *     copy-on-write block copies of a step in one launch).
 *
 * Conventions shared by every call
 *   Memory:  every pointer argument except `host_code` is a DEVICE pointer
 *            on the current CUDA device.  The caller owns every buffer,
 *            including the decode workspace; the library never allocates.
 *   Streams: `stream` is a cudaStream_t (NULL = the legacy default stream).
 *            All calls are stream-ordered and asynchronous; none synchronises
 *            the device (pkv_get_device_status excepted).
 *   Errors:  scalar/pointer/alignment checks run on the host before any
 *            launch and return a pkv_status without touching the GPU.  A
 *            failed launch returns PKV_ERR_CUDA.  Contract violations that
 *            live in device data (a block id outside the pool, a context
 *            length above the table's capacity, a slot outside the pool) are
 *            caught by the kernels, which skip the offending access (never
 *            trapping) and set a bit in a per-device status word that
 *            pkv_get_device_status reads.
 *
 * KV cache layout (this library's contract; the pages disagree with each
 * other -- "Pytorch implementation of paper ..." (aishastr.live) §2 stores K
 * as [blocks, heads, head_dim, B], the 10100.com page §2 quotes a 5-D K and a
 * head_dim-major V): k_cache and v_cache are both
 *     [num_blocks][num_kv_heads][block_size][head_dim], head_dim contiguous,
 * so every (physical block, kv head) tile is one contiguous run of
 * block_size * head_dim elements.  Token row `off` of physical block `blk`
 * holds logical position j*B + off of every sequence whose table entry j is
 * `blk`.
 */
#ifndef PAGEDKV_H
#define PAGEDKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element types.  PKV_FP8_E4M3 is the OCP 8-bit "e4m3fn" format (bias 7, no
 * infinities, S.1111.111 = NaN, largest finite 448); it is a KV storage type
 * only. */
typedef enum pkv_dtype {
    PKV_F32 = 0,
    PKV_F16 = 1,
    PKV_BF16 = 2,
    PKV_FP8_E4M3 = 3
} pkv_dtype;

typedef enum pkv_status {
    PKV_OK = 0,
    PKV_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, bad size, bad scale */
    PKV_ERR_UNSUPPORTED = 2,   /* head_dim, block_size or dtype combination not built */
    PKV_ERR_WORKSPACE = 3,     /* decode workspace too small or misaligned */
    PKV_ERR_CUDA = 4,          /* a CUDA runtime call or launch failed */
    PKV_ERR_OUT_OF_BLOCKS = 5  /* block manager: the free list cannot satisfy the request */
} pkv_status;

/* Bits of the device status word (see pkv_get_device_status). */
#define PKV_DEV_BAD_BLOCK_ID   0x1u  /* table entry outside [0, num_blocks): block skipped */
#define PKV_DEV_BAD_CONTEXT    0x2u  /* context_len < 0 or above max_context_len or
                                        max_blocks_per_seq * block_size: clamped */
#define PKV_DEV_BAD_SLOT       0x4u  /* slot >= num_blocks * block_size: token skipped */
#define PKV_DEV_BAD_PAIR       0x8u  /* copy pair id outside [0, num_blocks): pair skipped */
#define PKV_DEV_WAIT_TIMEOUT   0x10u /* a pipeline wait exceeded its bound: kernel returned */

/* Symbols of the C ABI are the only ones the library exports. */
#if defined(__GNUC__)
#define PKV_API __attribute__((visibility("default")))
#else
#define PKV_API
#endif

/* Opaque stand-in for cudaStream_t, so this header needs no CUDA include. */
typedef struct CUstream_st* pkv_stream_t;

/*
 * Bytes of device workspace pkv_paged_decode_attention needs for these sizes.
 * The workspace holds the per-call work list, one arrival counter per
 * (sequence, kv head group) and the split-KV partial states (m, l, acc[d]) of
 * every chunk of every (sequence, query head).  It need not be zeroed.
 * Returns 0 for unsupported or invalid sizes.
 */
PKV_API size_t pkv_decode_workspace_bytes(int num_seqs, int num_q_heads, int num_kv_heads,
                                  int head_dim, int block_size, int max_context_len,
                                  pkv_dtype kv_dtype);

/*
 * Single-query decode attention over a paged KV cache.
 *
 * For every sequence s and query head h (kv head g = h / (num_q_heads /
 * num_kv_heads), contiguous GQA groups), over the context_lens[s] tokens
 * whose rows are found through block_tables[s][t / block_size], row
 * t % block_size:
 *     out[s][h] = sum_t softmax_t(scale * q[s][h] . k_t) * v_t
 * ("...Mathematical Foundations" §3: a_ij and o_i; the kernel evaluates it
 * in one pass with the running-max rescale of §7's pseudocode, splitting long
 * contexts into chunks whose partial states are merged by the same rescale).
 * A sequence with context_len 0 gets an all-zero output.
 * With kv_dtype PKV_FP8_E4M3 every K/V element is decode(code) * kv_scale.
 *
 *   query         [num_seqs][num_q_heads][head_dim], q_dtype, 16-byte aligned
 *   k_cache,
 *   v_cache       [num_blocks][num_kv_heads][block_size][head_dim], kv_dtype,
 *                 16-byte aligned (layout above); rows at or beyond a
 *                 sequence's context length are never used (may hold NaN)
 *   block_tables  int32 [num_seqs][max_blocks_per_seq]; only the first
 *                 ceil(context_lens[s] / block_size) entries of a row are read
 *   context_lens  int32 [num_seqs]
 *   max_context_len  host-known upper bound of context_lens (sizes the
 *                 workspace and the split plan); must be <= max_blocks_per_seq
 *                 * block_size.  Longer device values are clamped to it and
 *                 flagged PKV_DEV_BAD_CONTEXT.
 *   scale         logit scale (1/sqrt(head_dim) for standard attention)
 *   q_dtype       PKV_F32 / PKV_F16 / PKV_BF16; out has the same type
 *   kv_dtype      q_dtype or PKV_FP8_E4M3
 *   kv_scale      dequantisation scale for FP8 KV (> 0, finite; pass 1 otherwise)
 *   workspace     device buffer of >= pkv_decode_workspace_bytes(...) bytes,
 *                 256-byte aligned; calls sharing a workspace must be ordered
 *                 on one stream
 *   out           [num_seqs][num_q_heads][head_dim], q_dtype, 16-byte aligned
 * Supported: head_dim in {64, 128}; block_size in {8, 16, 32}; any
 * num_q_heads that is a multiple of num_kv_heads.
 * Two launches on `stream`: a one-CTA planning kernel and the decode kernel.
 */
PKV_API pkv_status pkv_paged_decode_attention(const void* query, const void* k_cache, const void* v_cache,
                                      const int32_t* block_tables, const int32_t* context_lens,
                                      int num_seqs, int num_q_heads, int num_kv_heads,
                                      int head_dim, int block_size, int num_blocks,
                                      int max_blocks_per_seq, int max_context_len, float scale,
                                      pkv_dtype q_dtype, pkv_dtype kv_dtype, float kv_scale,
                                      void* workspace, size_t workspace_bytes, void* out,
                                      pkv_stream_t stream);

/*
 * Prefix-aware decode: the same result as pkv_paged_decode_attention (same
 * arguments, workspace size and errors), for batches in which sequences
 * share the physical blocks of a common prompt ("...Mathematical
 * Foundations" §5 Parallel Sampling and System Prompt Prefix Sharing).
 * Consecutive sequences whose block-table rows start with the same physical
 * block are grouped (at most 16 query heads per kv head in a group); the
 * blocks every member's row shares with the first member's are streamed
 * once for the whole group, and each member's remaining tokens separately;
 * the two parts are merged per (sequence, query head).  Grouping applies when
 * q and K/V are 16-bit or FP8 with 16-bit q (head_dim 128 for FP8) and a kv
 * head has at most 8 query heads; otherwise this is the plain decode.  The
 * rounding differs from the plain call's (the summation is split
 * differently), within the same tolerances.
 */
PKV_API pkv_status pkv_paged_decode_attention_prefix(
    const void* query, const void* k_cache, const void* v_cache, const int32_t* block_tables,
    const int32_t* context_lens, int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
    int block_size, int num_blocks, int max_blocks_per_seq, int max_context_len, float scale,
    pkv_dtype q_dtype, pkv_dtype kv_dtype, float kv_scale, void* workspace,
    size_t workspace_bytes, void* out, pkv_stream_t stream);

/*
 * Multi-query (causal) paged attention: several query tokens per sequence --
 * prefill, chunked prefill, or the verification of a chain of draft tokens
 * ("...Mathematical Foundations" §1 The Prefill (Prompt) Phase: a prompt's
 * tokens are processed in parallel as dense tensor-core products, and a token
 * attends to every earlier token and itself; §3 o = softmax(q K^T / sqrt(d)) V
 * through the block table).
 *
 * Sequence s owns query rows query_start[s] .. query_start[s+1]-1 (n_s rows);
 * its cache holds context_lens[s] >= n_s tokens, the last n_s being the
 * queries' own keys and values (written beforehand, e.g. by
 * pkv_reshape_and_cache).  Query row query_start[s] + i is the token at
 * position p = context_lens[s] - n_s + i; for each query head h
 *   out[row][h][:] = softmax_t(scale * q[row][h] . k_t) v_t over t = 0 .. p,
 * k_t / v_t of kv head h / (num_q_heads / num_kv_heads) found through the
 * table as in pkv_paged_decode_attention.
 *
 *   query        [total_q][num_q_heads][head_dim], q_dtype, 16-byte aligned
 *   query_start  device int32 [num_seqs + 1], query_start[0] = 0,
 *                non-decreasing, query_start[num_seqs] = total_q
 *   context_lens device int32 [num_seqs], n_s <= context_lens[s] <= the table's
 *                capacity; a sequence breaking this is skipped (its rows are
 *                left untouched) and flagged PKV_DEV_BAD_CONTEXT
 *   workspace    >= pkv_multi_query_workspace_bytes(num_seqs), 256-byte aligned
 *   out          [total_q][num_q_heads][head_dim], q_dtype, 16-byte aligned
 *   other arguments as in pkv_paged_decode_attention.
 * Supported: q_dtype PKV_F16 or PKV_BF16 with kv_dtype == q_dtype,
 * head_dim 128, block_size in {8, 16, 32}, num_q_heads / num_kv_heads a
 * divisor of 128; others return PKV_ERR_UNSUPPORTED.  Q K^T and P V run on the
 * tcgen05 tensor cores with fp32 accumulation in tensor memory; P is rounded
 * to q_dtype before P V (the softmax denominator sums the fp32 weights).
 * Two launches on `stream`: a one-CTA planning kernel (it orders the
 * sequences by context length, longest first, when there are at most 1024)
 * and the attention kernel: one persistent CTA per SM, each taking work
 * items (a sequence, a kv head and 256 (query, head) rows) in that order
 * from a counter.  The workspace holds the plan: per-sequence item offsets,
 * the order and the counter.
 */
PKV_API size_t pkv_multi_query_workspace_bytes(int num_seqs);

PKV_API pkv_status pkv_paged_multi_query_attention(
    const void* query, const void* k_cache, const void* v_cache, const int32_t* block_tables,
    const int32_t* context_lens, const int32_t* query_start, int num_seqs, int total_q,
    int num_q_heads, int num_kv_heads, int head_dim, int block_size, int num_blocks,
    int max_blocks_per_seq, int max_context_len, float scale, pkv_dtype q_dtype,
    pkv_dtype kv_dtype, float kv_scale, void* workspace, size_t workspace_bytes, void* out,
    pkv_stream_t stream);

/*
 * Verification of draft-token trees (speculative decoding trees: "...Mathematical
 * Foundations" §9 lists them among the uses of shared paged memory; the
 * attention is that of §3).  As pkv_paged_multi_query_attention, except that
 * the n_s <= 64 query tokens of sequence s are a tree of draft tokens, laid
 * out so that every token comes after its ancestors, and query i of the
 * sequence (row query_start[s] + i, position p = context_lens[s] - n_s + i)
 * attends to
 *   every token at a position < context_lens[s] - n_s (the prior context),
 *   itself (position p), and
 *   each tree token j < i whose bit j is set in tree_mask[query_start[s] + i]
 *   (its ancestors); bits j >= i are ignored.
 * With bits 0 .. i-1 set this is the causal attention of
 * pkv_paged_multi_query_attention.
 *
 *   tree_mask    device uint64 [total_q], 8-byte aligned; not null unless
 *                num_seqs or total_q is 0 (PKV_ERR_INVALID_ARG)
 *   a sequence with more than 64 queries is skipped (its rows are left
 *   untouched) and flagged PKV_DEV_BAD_CONTEXT.
 * Workspace: pkv_multi_query_workspace_bytes(num_seqs).  Supported shapes and
 * types, launches and the other arguments as pkv_paged_multi_query_attention.
 */
PKV_API pkv_status pkv_paged_tree_attention(
    const void* query, const void* k_cache, const void* v_cache, const int32_t* block_tables,
    const int32_t* context_lens, const int32_t* query_start, const uint64_t* tree_mask,
    int num_seqs, int total_q, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
    int num_blocks, int max_blocks_per_seq, int max_context_len, float scale, pkv_dtype q_dtype,
    pkv_dtype kv_dtype, float kv_scale, void* workspace, size_t workspace_bytes, void* out,
    pkv_stream_t stream);

/*
 * Write new tokens' keys and values into their cache slots
 * ("...Mathematical Foundations" §7 kernel 1; §4 Allocation Lifecycle step 2).
 *
 * For every token t with slot_mapping[t] >= 0 and every kv head h:
 *   block = slot / block_size, row = slot % block_size,
 *   k_cache[block][h][row][:] = key[t][h][:]   (same for value / v_cache).
 * Same element type: a bit copy.  kv_dtype PKV_FP8_E4M3: each element becomes
 * e4m3(x / kv_scale), the quotient taken in fp32 with IEEE rounding, then
 * rounded to nearest-even with saturation to +-448 (NaN stays NaN).
 *
 *   key, value    [num_tokens][num_kv_heads][head_dim], src_dtype, contiguous,
 *                 16-byte aligned
 *   slot_mapping  int64 [num_tokens]; negative = padding, skipped; slots at or
 *                 beyond num_blocks * block_size are skipped and flagged
 *                 PKV_DEV_BAD_SLOT.  Two tokens with the same slot race.
 *   src_dtype     PKV_F32 / PKV_F16 / PKV_BF16;  kv_dtype: src_dtype or FP8
 * One launch on `stream` (none when num_tokens == 0).
 */
PKV_API pkv_status pkv_reshape_and_cache(const void* key, const void* value, void* k_cache,
                                 void* v_cache, const int64_t* slot_mapping, int num_tokens,
                                 int num_kv_heads, int head_dim, int block_size, int num_blocks,
                                 pkv_dtype src_dtype, pkv_dtype kv_dtype, float kv_scale,
                                 pkv_stream_t stream);

/*
 * Batched copy-on-write ("...Mathematical Foundations" §5 step 4, §7 kernel 3):
 * for every pair i, physical block pairs[i][1] of both caches becomes a byte
 * copy of block pairs[i][0] (all kv heads), in one launch.
 *
 *   src_dst_pairs int32 [num_pairs][2] (device).  The dst ids must be distinct
 *                 and no dst may also be a src (the result would depend on
 *                 order); the library cannot check this without reading the
 *                 pairs back, so callers validate it.  Ids outside the pool
 *                 are skipped and flagged PKV_DEV_BAD_PAIR.
 * One launch on `stream` (none when num_pairs == 0).
 */
PKV_API pkv_status pkv_copy_blocks(void* k_cache, void* v_cache, const int32_t* src_dst_pairs,
                           int num_pairs, int num_kv_heads, int head_dim, int block_size,
                           int num_blocks, pkv_dtype kv_dtype, pkv_stream_t stream);

/*
 * Swapping ("...Mathematical Foundations" §6 Preemption and Memory Recovery:
 * evict blocks from GPU HBM to host memory and bring them back): for every
 * pair i, block pairs[i][1] of the destination pool becomes a byte copy of
 * block pairs[i][0] of the source pool, K and V, in one launch.  Either pool
 * may be pinned (page-locked) host memory -- on Grace-based systems the GPU
 * reads and writes it directly over NVLink-C2C -- or device memory; so may the
 * pairs array.  Pageable or unmapped host memory is refused
 * (PKV_ERR_INVALID_ARG) before any launch.  Both pools have the layout of the
 * cache ([blocks][kv heads][B][d]) with their own block counts.  Ids outside a
 * pool are skipped and flagged PKV_DEV_BAD_PAIR; the dst ids must be distinct.
 */
PKV_API pkv_status pkv_swap_blocks(const void* src_k, const void* src_v, int src_num_blocks,
                                   void* dst_k, void* dst_v, int dst_num_blocks,
                                   const int32_t* src_dst_pairs, int num_pairs,
                                   int num_kv_heads, int head_dim, int block_size,
                                   pkv_dtype kv_dtype, pkv_stream_t stream);

/*
 * Paged decode attention without a caller-provided workspace.  No
 * counterpart on the pages: this entry point exists for callers that cannot
 * allocate device memory when they decode -- plugins whose host framework
 * owns every device allocation (its caching allocator must account for all
 * memory, so a library may not call cudaMalloc behind its back), servers that
 * run under a fixed device-memory budget set at start-up, and latency-critical
 * loops where a cudaMalloc (which may synchronise the device) is not allowed.
 *
 * Same arguments, semantics and errors as pkv_paged_decode_attention, minus
 * `workspace` / `workspace_bytes`.  The workspace is a static device array of
 * PKV_NOALLOC_SCRATCH_BYTES that the library holds on every device that loads
 * it, until the process exits; nothing is allocated by this call.
 *   - Limit: if pkv_decode_workspace_bytes(...) for these sizes exceeds
 *     PKV_NOALLOC_SCRATCH_BYTES the call returns PKV_ERR_WORKSPACE and
 *     launches nothing.
 *   - Set-up: the first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current), and the first call of
 *     each (q_dtype, kv_dtype, head_dim) combination on a device sets its
 *     kernel's shared-memory limit and queries its occupancy.  Make those
 *     first calls (one warm-up call per combination is enough) before any
 *     stream capture.
 *   - Sharing: every call on a device uses the same array, which keeps the
 *     last call's contents (each call rewrites what must start at zero before
 *     its kernels read it).  Calls whose kernels overlap on the GPU -- on two
 *     streams, or from two host threads without ordering -- race on it and
 *     give wrong results; order them on one stream.
 */
#define PKV_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)

PKV_API pkv_status pkv_paged_decode_attention_noalloc(
    const void* query, const void* k_cache, const void* v_cache, const int32_t* block_tables,
    const int32_t* context_lens, int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
    int block_size, int num_blocks, int max_blocks_per_seq, int max_context_len, float scale,
    pkv_dtype q_dtype, pkv_dtype kv_dtype, float kv_scale, void* out, pkv_stream_t stream);

/*
 * Self-test of the pipeline waits: launches one CTA on `stream` whose mbarrier
 * wait can never complete (nothing arrives at it).  The wait gives up after the
 * bound every kernel's waits use (2 s of device time), the kernel sets
 * PKV_DEV_WAIT_TIMEOUT in the device status word (read it with
 * pkv_get_device_status) and returns: a stalled pipeline reports an error
 * instead of hanging, and the context stays usable.
 */
PKV_API pkv_status pkv_selftest_wait_bound(pkv_stream_t stream);

/*
 * Read and clear the status word of the current device (a bit-or of
 * PKV_DEV_* flags set by kernels since the last read).  Synchronous: waits
 * for the device's work to finish.  `host_code` is a host pointer.
 */
PKV_API pkv_status pkv_get_device_status(unsigned int* host_code);

/* ------------------------------------------------------------------------
 * Host block manager ("...Mathematical Foundations" §4 Virtual Memory
 * Architecture and Block Tables, Allocation Lifecycle; §5 Parallel Sampling
 * and Beam Search).  Plain host code: no GPU, no CUDA calls.  It hands out
 * physical block ids from a FIFO free list, keeps a reference count per block
 * and a block table + token count per sequence, and tells the caller which
 * slot each new token goes to and which copy-on-write copies to run first.
 * Not thread-safe: one manager per scheduler thread.
 * ------------------------------------------------------------------------ */
typedef struct pkv_block_manager pkv_block_manager;

/* A manager over blocks [0, num_blocks).  `free_order` (host, may be NULL)
 * lists the ids of the initial free list in hand-out order (num_free entries,
 * no repeats; blocks not listed are never handed out); NULL means 0, 1, ...
 * Returns NULL on bad arguments or allocation failure. */
PKV_API pkv_block_manager* pkv_bm_create(int num_blocks, int block_size,
                                         const int32_t* free_order, int num_free);
PKV_API void pkv_bm_destroy(pkv_block_manager* m);
/* Free blocks left, or -1 for a NULL manager. */
PKV_API int pkv_bm_num_free(const pkv_block_manager* m);
/* Reference count of a block (0 = free), or -1 for a bad id. */
PKV_API int pkv_bm_refcount(const pkv_block_manager* m, int32_t block);

/* Prefill: a new sequence holding num_tokens tokens in ceil(num_tokens / B)
 * fresh blocks (their slots are table[t / B] * B + t % B).  Fails with
 * PKV_ERR_INVALID_ARG for a known id, PKV_ERR_OUT_OF_BLOCKS without changes. */
PKV_API pkv_status pkv_bm_add_sequence(pkv_block_manager* m, int64_t seq_id,
                                       int64_t num_tokens);
/* Fork (parallel sampling, beam search): `child` shares every block of
 * `parent`; each shared block's reference count goes up by one. */
PKV_API pkv_status pkv_bm_fork(pkv_block_manager* m, int64_t parent, int64_t child);
/* Slot of the sequence's next token, growing the table on overflow.  If the
 * token's block is shared (reference count > 1) it is first replaced by a
 * fresh private block: *cow_src / *cow_dst receive the copy the caller must
 * run (pkv_copy_blocks) before writing; otherwise both are -1. */
PKV_API pkv_status pkv_bm_append_slot(pkv_block_manager* m, int64_t seq_id, int64_t* slot,
                                      int32_t* cow_src, int32_t* cow_dst);
/* Completion / pruning: drop the sequence; blocks reaching count 0 go to the
 * back of the free list. */
PKV_API pkv_status pkv_bm_free_sequence(pkv_block_manager* m, int64_t seq_id);
/* The sequence's block table (up to max_blocks entries, rest -1; table may be
 * NULL), its number of blocks and tokens. */
PKV_API pkv_status pkv_bm_sequence(const pkv_block_manager* m, int64_t seq_id,
                                   int32_t* table, int max_blocks, int* num_blocks,
                                   int64_t* num_tokens);
/* One decode step for n distinct sequences: append one token to each (in the
 * given order), writing slot_mapping[n], the copy-on-write pairs
 * cow_pairs[*num_cow][2] (room for n), and optionally the updated block_tables
 * [n][max_blocks] (-1 padded) and context_lens[n].  Validates first: on error
 * nothing changes.  The free-block check counts exactly the blocks the step
 * takes: one per full last block, and for a shared block of reference count r
 * written by k of the n sequences, min(k, r - 1) copies (the last writer to
 * find it shared becomes its sole owner). */
PKV_API pkv_status pkv_bm_prepare_step(pkv_block_manager* m, const int64_t* seq_ids, int n,
                                       int64_t* slot_mapping, int32_t* cow_pairs,
                                       int* num_cow, int32_t* block_tables, int max_blocks,
                                       int32_t* context_lens);

/* Static description of a pkv_status. */
PKV_API const char* pkv_status_string(pkv_status status);

/* Library version: major * 10000 + minor * 100 + patch. */
PKV_API int pkv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H */
