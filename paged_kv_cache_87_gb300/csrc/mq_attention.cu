// mq_attention.cu -- multi-query causal paged attention on the 5th-generation
// tensor cores (tcgen05: accumulators in TMEM, K/V staged by TMA).
//
// What it computes ("PagedAttention: Mathematical Foundations, Virtual Memory
// Block Allocation, and Zero-Waste KV Cache Serving"): §1 -- in the prefill
// phase a prompt's tokens are processed in parallel as dense tensor-core
// matrix products, and a token's attention covers every earlier token and
// itself; §3 -- o = softmax(scale * q K^T) V with K and V gathered block by
// block through the sequence's table; §7 -- the running max / rescale /
// running sum of the decode pseudocode, applied here per query row.
// Query row i of sequence s (query_start[s] + i) is the token at position
// ctx_s - n_s + i and attends to tokens 0 .. ctx_s - n_s + i.
//
// Organisation: work items of (sequence, kv head, 256 rows), a row being a
// (query token, query head of the kv head's group) pair, so the G heads that
// share a kv head share every K/V tile.  The 256 rows are two tiles A and B of
// 128 (TMEM lanes); every K/V tile staged in shared memory feeds both.  One
// persistent CTA per SM takes items from a launch-wide counter in the planner's
// order (longest sequences first); the K/V ring, the MMAs and the softmax run on
// from one item into the next, so an item's first tiles overlap the previous
// item's last ones and its epilogue.  Twelve warps (the third warpgroup hands
// most of its registers to the first two):
//   warps 0-3  tile A, one thread per row: the softmax of each S tile, the
//              rescale of O, the epilogue;
//   warps 4-7  the same for tile B;
//   warp 8     takes the items and decodes each into the CTA's item ring (a
//              sequence, a kv head, row ranges, tile counts); TMA producer: the
//              item's Q rows, then K_0, V_0, K_1, V_1, ... into a 5-stage ring,
//              one 4-D box per (block, kv head) row of the pool;
//   warp 9     TMEM allocation; one lane issues the MMAs;
//   warp 10    prefetches each published item's Q rows into L2 (the Q buffer
//              frees only with the previous item's last S MMAs); warp 11 idle.
// Per 128-token tile j and row tile X:  S_X = Q_X K_j^T (M 128, N 128, K 128;
// Q from shared memory, S in TMEM), then O_X += P_X V_j (P in TMEM, written
// over the first 64 columns of S_X as 16-bit pairs; V an MN-major operand).
// The MMAs go out as PV_A(j), S_A(j+1), PV_B(j), S_B(j+1): while one tile's
// softmax runs, the tensor pipe works on the other tile.  S_X(j+1) is issued
// after PV_X(j) by the same thread, and its completion (the commit that
// publishes S_X(j+1)) covers PV_X(j): the softmax may then rescale O_X and
// overwrite P_X without a further wait.
// The running max only moves when a tile's max exceeds it by more than 2^8 (in
// the log2 domain), and O is rescaled in TMEM only then.
// Draft-tree verification (§9 speculative decoding trees: each draft token sees
// the prior context, itself and its ancestors) is a second instantiation: every
// row holds its uint64 of ancestor bits and the tiles reaching the tree take the
// masked path.
// Every mbarrier wait is bounded (2 s); on a timeout the CTA flags
// PKV_DEV_WAIT_TIMEOUT, drains its MMAs and releases its TMEM.
#include <type_traits>

#include "mq_attention.cuh"
#include "tcgen05.cuh"
#include "tmap.cuh"

namespace pkv {
namespace {

constexpr int kHD = 128;                              // head dim of this kernel
constexpr int kTile = 128;                            // rows of a row tile; tokens of a K/V tile
constexpr int kTileBytes = kTile * 256;               // 128 rows x 256 B
constexpr int kHalfBytes = kTile * 128;               // one 128-byte half of d of a tile
// K and V tiles arrive as [group of 8 tokens][half of d][8 tokens][128 B]
constexpr int kGroupHalf = 8 * 128;                   // one half of d of an 8-token group
constexpr int kGroupBytes = 2 * kGroupHalf;           // an 8-token group
constexpr int kStages = 5;                            // K/V ring: K_0, V_0, K_1, V_1, ...
constexpr int kOffQ = 0;                              // Q_A, Q_B: [half][128 rows][128 B]
constexpr int kOffRing = kOffQ + 2 * kTileBytes;
constexpr int kOffBars = kOffRing + kStages * kTileBytes;
constexpr int kOffItems = kOffBars + 256;             // the two-slot ring of decoded items
constexpr int kSmem = kOffItems + 2 * 64 + 1024;      // barriers, TMEM slot, flag; item ring; alignment
constexpr int kThreads = 384;                         // 8 row warps; producer, MMA, Q prefetch, idle
// registers per thread after the split: the row warpgroups take what the third
// warpgroup gives back (216 x 256 + 72 x 128 = 168 x 384, the launch's budget)
constexpr int kRowRegs = 216;
constexpr int kAuxRegs = 72;
// TMEM columns (lane = row): S_X (fp32) at 128 X, its first 64 columns reused
// for P_X (16-bit, two per column); O_X (fp32) at 256 + 128 X
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;
constexpr uint32_t kColO = 256;
constexpr float kMaxSlack = 8.0f;                     // log2-domain headroom before the max moves
constexpr int kMaxTree = 64;                          // draft tokens of a tree (one uint64 of bits)

static_assert(kMqRows == 2 * kTile, "a CTA holds two row tiles");
static_assert(kRowRegs * 256 + kAuxRegs * 128 <= (65536 / kThreads) / 8 * 8 * kThreads,
              "the register split fits the launch's registers");
static_assert(kSmem <= 227 * 1024, "shared memory per CTA");
constexpr int kItemReaders = 10;                      // warps reading each item
constexpr int kNumBars = 2 * kStages + 2 + 2 + 1 + 1 + 1 + 2 + 2 + 2 + 1;
static_assert(kNumBars * 8 + 8 <= 256, "barriers, TMEM slot and flag fit their region");

template <typename QT>
__device__ __forceinline__ uint32_t pack2(float a, float b, float& ra, float& rb) {
    if constexpr (std::is_same<QT, BF16>::value) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        ra = __low2float(h);
        rb = __high2float(h);
        return *reinterpret_cast<const uint32_t*>(&h);
    } else {
        const __half2 h = __floats2half2_rn(a, b);
        ra = __low2float(h);
        rb = __high2float(h);
        return *reinterpret_cast<const uint32_t*>(&h);
    }
}

template <typename QT>
__device__ __forceinline__ uint32_t pack2_bits(float a, float b) {
    if constexpr (std::is_same<QT, BF16>::value) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<const uint32_t*>(&h);
    } else {
        const __half2 h = __floats2half2_rn(a, b);
        return *reinterpret_cast<const uint32_t*>(&h);
    }
}

// One 32-byte store (sm_100 family); dst 32-byte aligned.
__device__ __forceinline__ void st_global_v8(void* dst, const uint32_t* w) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
                 ::"l"(dst), "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]),
                 "r"(w[6]), "r"(w[7])
                 : "memory");
}

// Packed fp32 pairs (sm_100 family): one instruction for two lanes of work.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
    return ((uint64_t)__float_as_uint(hi) << 32) | __float_as_uint(lo);
}
__device__ __forceinline__ float f2_lo(uint64_t x) { return __uint_as_float((uint32_t)x); }
__device__ __forceinline__ float f2_hi(uint64_t x) { return __uint_as_float((uint32_t)(x >> 32)); }
// x * s + m, element-wise, rounded once (as fmaf)
__device__ __forceinline__ uint64_t f2_fma(uint64_t x, uint64_t s, uint64_t m) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(x), "l"(s), "l"(m));
    return r;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
// max of three (a NaN operand is ignored, as by fmaxf)
__device__ __forceinline__ float max3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// Items: per sequence ceil(n * G / 256) row pairs times Hkv, the sequences taken
// longest context first (up to kMqSortSeqs sequences; beyond, in index order) so
// that the persistent CTAs take the longest items first; exclusive prefix.  The
// CTAs' item counter starts at zero.
constexpr int kMqSortSeqs = 1024;

__global__ void __launch_bounds__(1024) mq_plan_kernel(MqParams p) {
    const int total_q = p.total_q;
    __shared__ int wsum[32];
    __shared__ int carry;
    __shared__ int ctx_s[kMqSortSeqs];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) {
        carry = 0;
        if (p.query_start[p.num_seqs] != total_q || p.query_start[0] != 0)
            set_status(p.status, PKV_DEV_BAD_CONTEXT);
    }
    const int cap = min(p.max_context_len, p.max_blocks * p.block_size);
    // seq_order[k] = the sequence launched k-th: by context length, descending, ties
    // by index (a rank sort)
    if (p.num_seqs <= kMqSortSeqs) {
        for (int s = tid; s < p.num_seqs; s += blockDim.x) ctx_s[s] = p.context_lens[s];
        __syncthreads();
        for (int s = tid; s < p.num_seqs; s += blockDim.x) {
            const int c = ctx_s[s];
            int rank = 0;
            for (int t = 0; t < p.num_seqs; ++t) {
                const int ct = ctx_s[t];
                rank += (ct > c) || (ct == c && t < s);
            }
            p.seq_order[rank] = s;
        }
    } else {
        for (int s = tid; s < p.num_seqs; s += blockDim.x) p.seq_order[s] = s;
    }
    __syncthreads();
    for (int base = 0; base < p.num_seqs; base += blockDim.x) {
        const int k = base + tid;
        const int s = k < p.num_seqs ? p.seq_order[k] : 0;
        int items = 0;
        if (k < p.num_seqs) {
            const int n = p.query_start[s + 1] - p.query_start[s];
            const int ctx = p.context_lens[s];
            if (n < 0 || ctx < n || ctx > cap || p.query_start[s] < 0 ||
                p.query_start[s + 1] > total_q || (p.tree && n > kMaxTree)) {
                set_status(p.status, PKV_DEV_BAD_CONTEXT);
            } else {
                items = (n * p.group + kMqRows - 1) / kMqRows * p.num_kv_heads;
            }
        }
        int x = items;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, off);
            if (lane >= off) x += y;
        }
        if (lane == 31) wsum[warp] = x;
        __syncthreads();
        if (warp == 0) {
            int v = wsum[lane];
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, v, off);
                if (lane >= off) v += y;
            }
            wsum[lane] = v;
        }
        __syncthreads();
        const int incl = x + (warp > 0 ? wsum[warp - 1] : 0);
        if (k < p.num_seqs) p.item_prefix[k] = carry + incl - items;
        __syncthreads();
        if (tid == blockDim.x - 1) carry += incl;
        __syncthreads();
    }
    if (tid == 0) {
        p.item_prefix[p.num_seqs] = carry;
        *p.work_next = 0;                        // the attention CTAs' item counter
    }
}

// ---- one work item: a sequence, a kv head and a pair of 128-row tiles ----
struct MqItem {
    int s, kvh, q_begin, n, ctx, q0;
    int qn_a, qn_b;                // query tokens of row tiles A and B (B may have none)
    int kv_end_a, kv_end_b;        // tokens [0, kv_end_X) are read for tile X
    int T_a, T_b, T;               // 128-token K/V tiles of A, of B, of the item
    int kv_end;                    // tokens the item stages
};

// An entry of the CTA's item ring: the item decoded by the producer warp, so that the
// MMA and row warps start the next item without a chain of global loads of their own.
struct __align__(16) MqSlot {
    MqItem it;
    int idx;                       // the item's index in launch order; -1: no items left
    int pad;
};
static_assert(sizeof(MqSlot) == 64, "two item slots fill 128 bytes");

// Item `idx` in launch order (called by a whole warp; every lane gets the item): the
// last sequence (in launch order) whose first item is <= idx, found by a 32-way search
// (one load per lane and round: one round up to 32 sequences, two up to 1024), then its
// row pair (later, longer pairs first) and its kv head.
__device__ __forceinline__ MqItem mq_item(const MqParams& p, int idx) {
    const int lane = threadIdx.x & 31;
    int lo = 0, len = p.num_seqs;                 // item_prefix[lo] <= idx; answer in [lo, lo + len)
    while (len > 1) {
        const int step = (len + 31) >> 5;
        const int pos = lo + lane * step;
        const bool le = pos < lo + len && __ldg(&p.item_prefix[pos]) <= idx;
        const int last = 31 - __clz(__ballot_sync(0xffffffffu, le));   // lane 0 always holds
        lo += last * step;
        len = min(step, len - last * step);
    }
    MqItem it;
    it.s = __ldg(&p.seq_order[lo]);
    const int local = idx - __ldg(&p.item_prefix[lo]);
    const int G = p.group, qpt = kTile / G;
    it.q_begin = __ldg(&p.query_start[it.s]);
    it.n = __ldg(&p.query_start[it.s + 1]) - it.q_begin;
    it.ctx = __ldg(&p.context_lens[it.s]);
    const int pairs = (it.n * G + kMqRows - 1) / kMqRows;
    const int ct = pairs - 1 - local / p.num_kv_heads;
    it.kvh = local % p.num_kv_heads;
    it.q0 = 2 * ct * qpt;
    it.qn_a = min(qpt, it.n - it.q0);
    it.qn_b = max(0, min(qpt, it.n - it.q0 - qpt));
    it.kv_end_a = it.ctx - it.n + it.q0 + it.qn_a;
    it.kv_end_b = it.qn_b > 0 ? it.ctx - it.n + it.q0 + qpt + it.qn_b : 0;
    it.T_a = (it.kv_end_a + kTile - 1) / kTile;
    it.T_b = (it.kv_end_b + kTile - 1) / kTile;
    it.T = max(it.T_a, it.T_b);
    it.kv_end = max(it.kv_end_a, it.kv_end_b);
    return it;
}

// The CTA's k-th item (index -1: none left), published by the producer warp in a
// two-slot ring; each reading warp releases the slot with one arrival (lane 0).
__device__ __forceinline__ int mq_take_item(const MqSlot* items_s, uint64_t* item_full,
                                            uint64_t* item_empty, int k, MqItem& it,
                                            volatile int* abort_flag, unsigned* status) {
    const int slot = k & 1;
    int idx = -1;
    if (mbar_wait(&item_full[slot], (k >> 1) & 1)) {
        idx = items_s[slot].idx;
        if (idx >= 0) it = items_s[slot].it;
    } else {
        set_status(status, PKV_DEV_WAIT_TIMEOUT);
        *abort_flag = 1;
    }
    __syncwarp(__activemask());
    if ((threadIdx.x & 31) == 0) mbar_arrive(&item_empty[slot]);
    return idx;
}

// ---- the TMA producer warp: per item, ring entries 2j (K_j) and 2j + 1 (V_j) ----
__device__ __forceinline__ void mq_producer(const MqParams& p, const CUtensorMap* tmK,
                                            const CUtensorMap* tmV, const CUtensorMap* tmQ,
                                            uint8_t* smem, uint64_t* full, uint64_t* empty,
                                            uint64_t* q_full, uint64_t* q_free,
                                            MqSlot* items_s, uint64_t* item_full,
                                            uint64_t* item_empty, volatile int* abort_flag) {
    const int lane = threadIdx.x & 31;
    if (lane == 0) {
        prefetch_tensormap(tmK);
        prefetch_tensormap(tmV);
        prefetch_tensormap(tmQ);
    }
    const uint64_t policy = l2_evict_last_policy();   // other CTAs re-read K/V
    const uint64_t q_policy = l2_evict_first_policy();   // each query row is read once
    const int B = p.block_size;
    const int total = __ldg(&p.item_prefix[p.num_seqs]);
    uint32_t rbase = 0;                               // ring entries of earlier items
    for (int k = 0;; ++k) {
        // the next item, taken from the launch-wide counter once this warp has issued
        // every load of the previous one: CTAs take items in launch order, longest
        // first, about two tile pairs before they finish their current item
        const int slot = k & 1;
        int idx = -1;
        if (lane == 0) {
            if (!mbar_wait(&item_empty[slot], ((k >> 1) & 1) ^ 1u)) {
                set_status(p.status, PKV_DEV_WAIT_TIMEOUT);
                *abort_flag = 1;
            } else if (!*abort_flag) {
                idx = atomicAdd(p.work_next, 1);
                if (idx >= total) idx = -1;
            }
        }
        idx = __shfl_sync(0xffffffffu, idx, 0);
        MqItem it{};
        if (idx >= 0) it = mq_item(p, idx);
        if (lane == 0) {
            items_s[slot].it = it;
            items_s[slot].idx = idx;
            mbar_arrive(&item_full[slot]);
        }
        if (idx < 0) break;
        const int32_t* trow = p.block_tables + (int64_t)it.s * p.max_blocks;
        const int nb_all = (it.kv_end + B - 1) / B;   // table entries this item reads
        // block-table window: lane l holds entry wb + l (cur) and wb + 32 + l (nxt); the
        // next window loads as soon as the current one is entered, so a tile's entries
        // are in registers when its stage frees (a tile spans <= 16 entries)
        int wb = 0;
        int cur = lane < nb_all ? trow[lane] : 0;
        int nxt = lane + 32 < nb_all ? trow[lane + 32] : 0;
        bool ok = true;
        for (int i = 0; i < 2 * it.T; ++i) {
            if (i == 1 && lane == 0) {
                // the item's Q rows, once the previous item's S MMAs no longer read Q
                // (after its first K tile, so that K/V streaming starts first): per row
                // tile with rows, two boxes of 64 elements x G heads x 128 / G tokens
                if (k > 0 && !mbar_wait(q_free, (k - 1) & 1)) {
                    set_status(p.status, PKV_DEV_WAIT_TIMEOUT);
                    *abort_flag = 1;
                }
                const int nx = it.qn_b > 0 ? 2 : 1, G = p.group;
                mbar_arrive_expect_tx(q_full, (uint32_t)(nx * kTileBytes));
                for (int X = 0; X < nx; ++X)
                    for (int h = 0; h < 2; ++h)
                        tc5::tma_load_3d(smem + kOffQ + X * kTileBytes + h * kHalfBytes, tmQ, 64 * h,
                                         it.kvh * G, it.q_begin + it.q0 + X * (kTile / G), q_full,
                                         q_policy);
            }
            const uint32_t g = rbase + (uint32_t)i;
            const int j = i >> 1, st = (int)(g % kStages);
            const bool isV = i & 1;
            if (!mbar_wait(&empty[st], ((g / kStages) & 1) ^ 1u)) {
                set_status(p.status, PKV_DEV_WAIT_TIMEOUT);
                *abort_flag = 1;
                ok = false;
                break;
            }
            const int t0 = j * kTile, t1 = min(t0 + kTile, it.kv_end);
            const int fb = t0 / B, nblk = (t1 - 1) / B - fb + 1;   // <= 128 / B <= 16
            if (fb >= wb + 32) {                          // warp-uniform: enter the next window
                wb += 32;
                cur = nxt;
                nxt = wb + 32 + lane < nb_all ? trow[wb + 32 + lane] : 0;
            }
            if (lane == 0) mbar_arrive_expect_tx(&full[st], (uint32_t)(nblk * B) * 256u);
            __syncwarp();
            const int src = fb + lane - wb;               // fb - wb < 32, lane < nblk <= 16
            int phys = __shfl_sync(0xffffffffu, cur, src & 31);
            if (fb + nblk > wb + 32) {                    // warp-uniform: the tile straddles
                const int hi = __shfl_sync(0xffffffffu, nxt, src & 31);
                if (src >= 32) phys = hi;
            }
            if (lane < nblk) {
                if (phys < 0 || phys >= p.num_blocks) {
                    if (!isV) set_status(p.status, PKV_DEV_BAD_BLOCK_ID);
                    phys = 0;
                }
                // one box per block: both 128-byte halves of its B rows, landing as
                // [group of 8 rows][half][8 rows][128 B] at the block's place in the tile
                const int y = (phys * p.num_kv_heads + it.kvh) * B;
                uint8_t* dst = smem + kOffRing + st * kTileBytes + lane * B * 256;
                tc5::tma_load_4d(dst, isV ? tmV : tmK, 0, 0, 0, y >> 3, &full[st], policy);
            }
        }
        if (!ok) break;
        rbase += 2u * (uint32_t)it.T;
    }
}

// ---- the MMA issuer (one thread): per item PV_A(j), S_A(j+1), PV_B(j), S_B(j+1) ----
template <typename QT>
__device__ __forceinline__ void mq_mma(const MqParams& p, uint8_t* smem, uint32_t tmem,
                                       uint64_t* full, uint64_t* empty, uint64_t* s_full,
                                       uint64_t* p_full, uint64_t* q_full, uint64_t* q_free,
                                       uint64_t* drain, uint64_t* o_free, uint64_t* fin,
                                       const MqSlot* items_s, uint64_t* item_full,
                                       uint64_t* item_empty, volatile int* abort_flag) {
    constexpr bool kBF16 = std::is_same<QT, BF16>::value;
    constexpr uint32_t idqk = tc5::idesc_f16(kBF16, kTile, kTile, false, false);
    constexpr uint32_t idpv = tc5::idesc_f16(kBF16, kTile, kHD, false, true);
    const uint32_t aQ = smem_addr(smem + kOffQ), aR = smem_addr(smem + kOffRing);
    // The tcgen05.mma queue is about one instruction deep: the MMAs of a group go
    // out back to back, their descriptors differing from the group's first only
    // by constants added to the low word.
    constexpr uint32_t q_hi = tc5::desc_hi_sw128(1024), k_hi = tc5::desc_hi_sw128(kGroupBytes),
                       v_hi = tc5::desc_hi_sw128(kGroupBytes);
    const uint32_t q_lo0 = tc5::desc_lo_sw128(aQ, 16), r_lo0 = tc5::desc_lo_sw128(aR, 16),
                   v_lo0 = tc5::desc_lo_sw128(aR, kGroupHalf);
    // S_X = Q_X K^T from the K tile in ring stage `st`; published on s_full[X]
    auto issue_s = [&](int X, int st) {
        const uint32_t qx = q_lo0 + (uint32_t)(X * (kTileBytes >> 4));
        const uint32_t kx = r_lo0 + (uint32_t)(st * (kTileBytes >> 4));
        const uint32_t d = tmem + kColS + (uint32_t)(X * kTile);
#pragma unroll
        for (int k = 0; k < 8; ++k)
            tc5::mma_ss_w(d, qx + (uint32_t)(((k >> 2) * kHalfBytes + (k & 3) * 32) >> 4), q_hi,
                          kx + (uint32_t)(((k >> 2) * kGroupHalf + (k & 3) * 32) >> 4), k_hi, idqk,
                          k > 0);
        tc5::commit(&s_full[X]);
    };
    // O_X += P_X V from the V tile in ring stage `st`
    auto issue_pv = [&](int X, int st, bool acc) {
        const uint32_t vx = v_lo0 + (uint32_t)(st * (kTileBytes >> 4));
        const uint32_t d = tmem + kColO + (uint32_t)(X * kTile);
        const uint32_t a = tmem + kColS + (uint32_t)(X * kTile);
#pragma unroll
        for (int k = 0; k < 8; ++k)
            tc5::mma_ts_w(d, a + (uint32_t)(8 * k), vx + (uint32_t)((k * 2 * kGroupBytes) >> 4), v_hi,
                          idpv, acc || k > 0);
    };
    auto wait_entry = [&](uint32_t g) {
        const bool r = mbar_wait(&full[g % kStages], (g / kStages) & 1);
        tc5::fence_after_sync();
        return r;
    };
    auto wait_bar = [&](uint64_t* bar, uint32_t parity) {
        const bool r = mbar_wait(bar, parity);
        tc5::fence_after_sync();
        return r;
    };
    bool ok = true;
    uint32_t rbase = 0, np_a = 0, np_b = 0;              // ring entries; P tiles consumed
    for (int k = 0; ok; ++k) {
        MqItem it{};
        const int idx = mq_take_item(items_s, item_full, item_empty, k, it, abort_flag, p.status);
        if (idx < 0 || *abort_flag) break;
        if (!wait_bar(q_full, k & 1) || !wait_entry(rbase)) { ok = false; break; }
        issue_s(0, (int)(rbase % kStages));
        if (it.T_b > 0) issue_s(1, (int)(rbase % kStages));
        tc5::commit(&empty[rbase % kStages]);
        if (it.T == 1) tc5::commit(q_free);              // the item's last S MMAs
        // the previous item's epilogue has read O_A and O_B before P.V overwrites them
        if (k > 0 && (!wait_bar(&o_free[0], (k - 1) & 1) || !wait_bar(&o_free[1], (k - 1) & 1))) {
            ok = false;
            break;
        }
        for (int j = 0; j < it.T && ok; ++j) {
            const uint32_t gv = rbase + 2u * j + 1u, gk = gv + 1u;
            const int vs = (int)(gv % kStages), ks = (int)(gk % kStages);
            const bool next = j + 1 < it.T;
            // V_j and K_j+1 have normally landed long before; the fence that orders the
            // MMAs after these waits comes once per burst, after the wait for P
            if (!mbar_wait(&full[vs], (gv / kStages) & 1) ||
                (next && !mbar_wait(&full[ks], (gk / kStages) & 1))) {
                ok = false;
                break;
            }
            if (j < it.T_a) {
                if (!mbar_wait(&p_full[0], np_a++ & 1)) { ok = false; break; }
                tc5::fence_after_sync();
                issue_pv(0, vs, j > 0);
                if (j + 1 < it.T_a) issue_s(0, ks);
            }
            if (j < it.T_b) {
                if (!mbar_wait(&p_full[1], np_b++ & 1)) { ok = false; break; }
                tc5::fence_after_sync();
                issue_pv(1, vs, j > 0);
            }
            tc5::commit(&empty[vs]);
            if (j + 1 < it.T_b) issue_s(1, ks);
            if (next) tc5::commit(&empty[ks]);
            if (j == it.T - 2) tc5::commit(q_free);      // the item's last S MMAs: Q is free
        }
        // the item's O is complete once every MMA issued so far has completed
        tc5::commit(drain);
        rbase += 2u * (uint32_t)it.T;
    }
    // every MMA issued above completes before the TMEM is released
    tc5::commit(fin);
    if (!mbar_wait(fin, 0)) ok = false;
    if (!ok) {
        set_status(p.status, PKV_DEV_WAIT_TIMEOUT);
        *abort_flag = 1;
    }
}

// TREE: draft-tree verification (the ancestor masks of p.tree) instead of causal attention.
// OUT32: the output is 32-byte aligned, and each row's 256 bytes go out as 32-byte stores
// (one whole sector each) instead of 16-byte ones.
template <typename QT, bool TREE, bool OUT32>
__global__ void __launch_bounds__(kThreads, 1) mq_attention_kernel(
    MqParams p, const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
    const __grid_constant__ CUtensorMap tmQ) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBars);
    uint64_t* full = bars;                       // [kStages] TMA bytes of a ring stage landed
    uint64_t* empty = full + kStages;            // [kStages] the MMAs reading it completed
    uint64_t* s_full = empty + kStages;          // [2] S_X computed (and PV_X of the tile before)
    uint64_t* p_full = s_full + 2;               // [2] P_X written, O_X rescaled (128 arrivals)
    uint64_t* q_full = p_full + 2;               // an item's Q rows landed (TMA bytes)
    uint64_t* q_free = q_full + 1;               // an item's S MMAs completed: Q may be replaced
    uint64_t* drain = q_free + 1;                // an item's MMAs completed
    uint64_t* o_free = drain + 1;                // [2] an item's O_X read by its epilogue (128)
    uint64_t* item_full = o_free + 2;            // [2] an item index published
    uint64_t* item_empty = item_full + 2;        // [2] read by the MMA and row warps
    uint64_t* fin = item_empty + 2;              // every MMA of the CTA completed
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(fin + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    MqSlot* items_s = reinterpret_cast<MqSlot*>(smem + kOffItems);   // [2] the item ring

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&p_full[i], kTile);
            mbar_init(&o_free[i], kTile);
            mbar_init(&item_full[i], 1);
            mbar_init(&item_empty[i], kItemReaders);
        }
        mbar_init(q_full, 1);
        mbar_init(q_free, 1);
        mbar_init(drain, 1);
        mbar_init(fin, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 9) tc5::tmem_alloc(tmem_slot, kTmemCols);
    tc5::fence_before_sync();
    __syncthreads();
    tc5::fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp >= 8) {
        tc5::setmaxnreg_dec<kAuxRegs>();
        if (warp == 8) {
            mq_producer(p, &tmK, &tmV, &tmQ, smem, full, empty, q_full, q_free, items_s,
                        item_full, item_empty, abort_flag);
        } else if (warp == 9) {
            if (lane == 0)
                mq_mma<QT>(p, smem, tmem, full, empty, s_full, p_full, q_full, q_free, drain, o_free,
                           fin, items_s, item_full, item_empty, abort_flag);
            __syncwarp();
        } else if (warp == 10) {
            // each item's Q rows into L2 as soon as the item is published, about two tile
            // pairs before the Q buffer frees (with the previous item's last S MMAs)
            for (int k = 0;; ++k) {
                MqItem it{};
                const int idx = mq_take_item(items_s, item_full, item_empty, k, it, abort_flag,
                                             p.status);
                if (idx < 0) break;
                if (lane < 4 && (lane < 2 || it.qn_b > 0))
                    tc5::tma_prefetch_3d(&tmQ, 64 * (lane & 1), it.kvh * p.group,
                                         it.q_begin + it.q0 + (lane >> 1) * (kTile / p.group));
            }
        }
        // the TMEM is released once every thread is past its last use
        tc5::fence_before_sync();
        named_bar_sync(1, kThreads);
        if (warp == 9) {
            tc5::fence_after_sync();
            tc5::tmem_dealloc(tmem, kTmemCols);
        }
        return;
    }
    tc5::setmaxnreg_inc<kRowRegs>();
    {
        // ========== rows: Q, softmax, O rescale, epilogue; one thread per row ==========
        const int X = warp >> 2;
        const int r = threadIdx.x & (kTile - 1);          // TMEM lane = row
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t colS = tmem + lane_base + kColS + (uint32_t)(X * kTile),
                       colO = tmem + lane_base + kColO + (uint32_t)(X * kTile);
        const int G = p.group, qpt = kTile / G;
        bool ok = true;
        uint32_t rbase = 0, ns = 0;                       // ring entries; S_X tiles seen
        MqItem it{};
        int idx = mq_take_item(items_s, item_full, item_empty, 0, it, abort_flag, p.status);
        for (int k = 0; idx >= 0 && ok; ++k) {
            const int Tx = X ? it.T_b : it.T_a;
            const int qi = it.q0 + X * qpt + r / G;
            const bool row_valid = r < (X ? it.qn_b : it.qn_a) * G;
            const int64_t qrow = ((int64_t)(it.q_begin + qi) * p.num_q_heads + it.kvh * G + r % G) * kHD;
            // the last token the row sees (rows past the last query see no further)
            const int lim_row = min(it.ctx - it.n + qi, (X ? it.kv_end_b : it.kv_end_a) - 1);
            // draft trees: the row sees tree token u < qi (position c0 + u; u < 64) only
            // when bit u of its ancestor mask is set; tiles reaching the tree need the mask
            constexpr bool has_tree = TREE;
            const int c0 = it.ctx - it.n;
            const uint64_t tree_w = has_tree && row_valid ? __ldg(&p.tree[it.q_begin + qi]) : 0ull;
            // the V rows past the item's last token hold poison or stale data (0 x NaN
            // would reach O through P = 0): the row tile whose P.V reads the last V tile
            // first zeroes them once their copy has landed
            const bool zeroes = (X == 0) == (it.T_a == it.T);
            float m_run = -INFINITY, l_run = 0.f;
            for (int j = 0; j < Tx; ++j) {
                // wait decisions are warp-uniform: the tcgen05 loads and stores below
                // need the whole warp converged
                const bool got = !*abort_flag && mbar_wait(&s_full[X], ns++ & 1);
                if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
                tc5::fence_after_sync();
                // local tokens <= lim are visible; a tile every row of the warp sees whole
                // needs no mask
                const int lim = lim_row - j * kTile;
                const bool masked = !__all_sync(0xffffffffu, lim >= kTile - 1) ||
                                    (has_tree && (j + 1) * kTile > c0);
                uint32_t sv[2][64];
                tc5::ld_32x32b_x64(colS, sv[0]);
                tc5::ld_32x32b_x64(colS + 64u, sv[1]);
                tc5::wait_ld();
                if (masked) {
                    const int u0 = j * kTile - c0;        // tree index of column 0
#pragma unroll
                    for (int c = 0; c < kTile; ++c) {
                        const int u = u0 + c;
                        const bool hidden =
                            c > lim || (has_tree && u >= 0 && u < qi && !((tree_w >> u) & 1ull));
                        if (hidden) sv[c >> 6][c & 63] = __float_as_uint(-INFINITY);
                    }
                }
                // row max of the raw scores (the scale is positive: same order): four
                // independent partial maxima, two scores per three-input max
                float pmx[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) pmx[i] = -INFINITY;
#pragma unroll
                for (int c = 0; c < kTile; c += 2)
                    pmx[(c >> 1) & 3] = max3(pmx[(c >> 1) & 3], __uint_as_float(sv[c >> 6][c & 63]),
                                             __uint_as_float(sv[c >> 6][(c + 1) & 63]));
                const float mx = max3(pmx[0], pmx[1], fmaxf(pmx[2], pmx[3])) * p.qk_scale_log2;
                const float m_new = mx > m_run + kMaxSlack ? mx : m_run;
                const bool resc = j > 0 && m_new != m_run;
                if (__any_sync(0xffffffffu, resc)) {
                    // PV_X(j-1) has completed (the commit of S_X(j) covers it)
                    const float f = resc ? fast_exp2(m_run - m_new) : 1.f;
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4) {
                        uint32_t o[32];
                        tc5::ld_32x32b_x32(colO + (uint32_t)(c4 * 32), o);
                        tc5::wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * f);
                        tc5::st_32x32b_x32(colO + (uint32_t)(c4 * 32), o);
                    }
                    l_run *= f;
                }
                m_run = m_new;
                // P = 2^(scale * s - m) (one FMA and one ex2 per score; the FMAs and the
                // sums two scores per packed instruction), rounded to the operand type,
                // over the first 64 columns of S_X; l sums the weights
                const float neg_m = m_run == -INFINITY ? 0.f : -m_run;
                const uint64_t scale2 = f2_pack(p.qk_scale_log2, p.qk_scale_log2),
                               negm2 = f2_pack(neg_m, neg_m);
                uint64_t pls[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) pls[i] = 0ull;
                uint32_t pw[64];                          // the row's 128 weights, packed
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const int c = 64 * hh + 2 * e;
                        const uint64_t x = f2_fma(f2_pack(__uint_as_float(sv[c >> 6][c & 63]),
                                                          __uint_as_float(sv[c >> 6][(c + 1) & 63])),
                                                  scale2, negm2);
                        const float a = fast_exp2(f2_lo(x)), bb = fast_exp2(f2_hi(x));
                        pw[32 * hh + e] = pack2_bits<QT>(a, bb);
                        pls[e & 3] = f2_add(pls[e & 3], f2_pack(a, bb));
                    }
                }
                tc5::st_32x32b_x64(colS, pw);
                const uint64_t l2 = f2_add(f2_add(pls[0], pls[1]), f2_add(pls[2], pls[3]));
                l_run += f2_lo(l2) + f2_hi(l2);
                if (zeroes && j == it.T - 1 && it.kv_end - j * kTile < kTile) {
                    const uint32_t gv = rbase + 2u * j + 1u;
                    if (!__all_sync(0xffffffffu,
                                    mbar_wait(&full[gv % kStages], (gv / kStages) & 1))) {
                        ok = false;
                        break;
                    }
                    if (r >= it.kv_end - j * kTile) {
                        uint8_t* vrow = smem + kOffRing + (gv % kStages) * kTileBytes +
                                        (r >> 3) * kGroupBytes + (r & 7) * 128;
#pragma unroll
                        for (int c = 0; c < 8; ++c) {
                            *reinterpret_cast<uint4*>(vrow + c * 16) = make_uint4(0u, 0u, 0u, 0u);
                            *reinterpret_cast<uint4*>(vrow + kGroupHalf + c * 16) =
                                make_uint4(0u, 0u, 0u, 0u);
                        }
                    }
                    fence_proxy_async_smem();
                }
                tc5::wait_st();
                tc5::fence_before_sync();
                mbar_arrive(&p_full[X]);
            }
            if (!ok) break;
            rbase += 2u * (uint32_t)it.T;
            // the next item (its Q arrives by TMA: the MMAs of the next item may start
            // while this one's epilogue runs)
            MqItem nx{};
            idx = mq_take_item(items_s, item_full, item_empty, k + 1, nx, abort_flag, p.status);
            // epilogue: every MMA of this item has completed (every thread waits, so the
            // drain barrier's phases stay in step with the items)
            ok = __all_sync(0xffffffffu, !*abort_flag && mbar_wait(drain, k & 1));
            if (!ok) break;
            tc5::fence_after_sync();
            uint32_t ov[4][32];
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) tc5::ld_32x32b_x32(colO + (uint32_t)(c4 * 32), ov[c4]);
            tc5::wait_ld();
            tc5::fence_before_sync();
            mbar_arrive(&o_free[X]);                      // the next item's P.V may overwrite O_X
            if (Tx > 0 && row_valid) {
                const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4) {
                    // packed in place: pair e of the chunk overwrites word e (<= 2e)
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        float ra, rb;
                        ov[c4][e] = pack2<QT>(__uint_as_float(ov[c4][2 * e]) * inv,
                                              __uint_as_float(ov[c4][2 * e + 1]) * inv, ra, rb);
                    }
                    uint16_t* dst = static_cast<uint16_t*>(p.out) + qrow + c4 * 32;
                    if constexpr (OUT32) {
                        st_global_v8(dst, ov[c4]);
                        st_global_v8(dst + 16, ov[c4] + 8);
                    } else {
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            reinterpret_cast<uint4*>(dst)[e] = make_uint4(
                                ov[c4][4 * e], ov[c4][4 * e + 1], ov[c4][4 * e + 2], ov[c4][4 * e + 3]);
                    }
                }
            }
            it = nx;
        }
        if (!ok) {
            set_status(p.status, PKV_DEV_WAIT_TIMEOUT);
            *abort_flag = 1;
        }
    }
    tc5::fence_before_sync();
    named_bar_sync(1, kThreads);
}

template <typename QT>
cudaError_t launch_typed(const MqParams& p, int64_t max_items, int num_ctas, cudaStream_t stream) {
    static bool attr_set[64] = {};
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    const bool out32 = (reinterpret_cast<uintptr_t>(p.out) & 31) == 0;
    auto kernel = p.tree ? (out32 ? mq_attention_kernel<QT, true, true> : mq_attention_kernel<QT, true, false>)
                         : (out32 ? mq_attention_kernel<QT, false, true> : mq_attention_kernel<QT, false, false>);
    if (!attr_set[dev]) {
        for (auto f : {mq_attention_kernel<QT, false, false>, mq_attention_kernel<QT, false, true>,
                       mq_attention_kernel<QT, true, false>, mq_attention_kernel<QT, true, true>}) {
            err = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
            if (err != cudaSuccess) return err;
        }
        attr_set[dev] = true;
    }
    CUtensorMap tk, tv;
    const long long rows = (long long)p.num_blocks * p.num_kv_heads * p.block_size;
    CUtensorMap tq;
    if (!encode_pool_map_grouped(&tk, p.k_cache, rows, p.block_size) ||
        !encode_pool_map_grouped(&tv, p.v_cache, rows, p.block_size) ||
        !encode_q_map(&tq, p.q, p.total_q, p.num_q_heads, p.group))
        return cudaErrorInvalidValue;
    mq_plan_kernel<<<1, 1024, 0, stream>>>(p);
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    const unsigned grid = (unsigned)(max_items < num_ctas ? max_items : (int64_t)num_ctas);
    kernel<<<grid, kThreads, kSmem, stream>>>(p, tk, tv, tq);
    return cudaGetLastError();
}

}  // namespace

int64_t mq_max_items(int num_seqs, int total_q, int group, int num_kv_heads) {
    return (int64_t)num_kv_heads * (((int64_t)total_q * group + kMqRows - 1) / kMqRows + num_seqs);
}

cudaError_t launch_mq_attention(const MqParams& p, pkv_dtype q_dtype, int64_t max_items,
                                int num_sms, cudaStream_t stream) {
    if (max_items <= 0) return cudaSuccess;
    if (max_items > 0x7fffffffLL || num_sms <= 0) return cudaErrorInvalidValue;
    switch (q_dtype) {
    case PKV_F16: return launch_typed<F16>(p, max_items, num_sms, stream);
    case PKV_BF16: return launch_typed<BF16>(p, max_items, num_sms, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace pkv
