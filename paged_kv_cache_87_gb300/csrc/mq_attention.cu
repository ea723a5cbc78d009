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
// Organisation: one CTA per (sequence, kv head, 256 rows), a row being a
// (query token, query head of the kv head's group) pair, so the G heads that
// share a kv head share every K/V tile.  The 256 rows are two tiles A and B of
// 128 (TMEM lanes); every K/V tile staged in shared memory feeds both.  Twelve
// warps (the third warpgroup hands most of its registers to the first two):
//   warps 0-3  tile A, one thread per row: Q row to shared memory, the softmax
//              of each S tile, the rescale of O, the epilogue;
//   warps 4-7  the same for tile B;
//   warp 8     TMA producer: K_0, V_0, K_1, V_1, ... into a 5-stage ring, one
//              4-D box per (block, kv head) row of the pool;
//   warp 9     TMEM allocation; one lane issues the MMAs; warps 10-11 idle.
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
constexpr int kSmem = kOffBars + 256 + 1024;          // barriers, TMEM slot, flag; alignment
constexpr int kThreads = 384;                         // 8 row warps; producer, MMA, 2 idle
// registers per thread after the split: the row warpgroups take what the third
// warpgroup gives back (216 x 256 + 64 x 128 <= 168 x 384, the launch's budget)
constexpr int kRowRegs = 216;
constexpr int kAuxRegs = 64;
// TMEM columns (lane = row): S_X (fp32) at 128 X, its first 64 columns reused
// for P_X (16-bit, two per column); O_X (fp32) at 256 + 128 X
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;
constexpr uint32_t kColO = 256;
constexpr float kMaxSlack = 8.0f;                     // log2-domain headroom before the max moves

static_assert(kMqRows == 2 * kTile, "a CTA holds two row tiles");
static_assert(kRowRegs * 256 + kAuxRegs * 128 <= (65536 / kThreads) / 8 * 8 * kThreads,
              "the register split fits the launch's registers");
static_assert(kSmem <= 227 * 1024, "shared memory per CTA");
constexpr int kNumBars = 2 * kStages + 2 + 2 + 1 + 1;
static_assert(kNumBars * 8 + 8 <= 256, "barriers, TMEM slot and flag fit their region");

// 16-byte chunk c (0..7) of row r of a 128B-swizzled [rows x 128 B] region.
__device__ __forceinline__ uint32_t sw128(int r, int c) {
    return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4));
}

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

// Items: per sequence ceil(n * G / 256) row pairs times Hkv, the sequences taken
// longest context first (up to kMqSortSeqs sequences; beyond, in index order) so
// that the block scheduler hands out the longest CTAs first; exclusive prefix.
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
                p.query_start[s + 1] > total_q) {
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
    if (tid == 0) p.item_prefix[p.num_seqs] = carry;
}

// ---- the TMA producer warp: ring item 2j is K_j, item 2j + 1 is V_j ----
__device__ __forceinline__ void mq_producer(const MqParams& p, const CUtensorMap* tmK,
                                            const CUtensorMap* tmV, uint8_t* smem,
                                            uint64_t* full, uint64_t* empty,
                                            volatile int* abort_flag, int s, int kvh, int kv_end,
                                            int T) {
    const int lane = threadIdx.x & 31;
    if (lane == 0) {
        prefetch_tensormap(tmK);
        prefetch_tensormap(tmV);
    }
    const uint64_t policy = l2_evict_last_policy();   // other CTAs re-read K/V
    const int B = p.block_size;
    const int32_t* trow = p.block_tables + (int64_t)s * p.max_blocks;
    const int nb_all = (kv_end + B - 1) / B;          // table entries this CTA reads
    // block-table window: lane l holds entry wb + l (cur) and wb + 32 + l (nxt); the
    // next window loads as soon as the current one is entered, so a tile's entries
    // are in registers when its stage frees (a tile spans <= 16 entries)
    int wb = 0;
    int cur = lane < nb_all ? trow[lane] : 0;
    int nxt = lane + 32 < nb_all ? trow[lane + 32] : 0;
    for (int i = 0; i < 2 * T; ++i) {
        const int j = i >> 1, st = i % kStages;
        const bool isV = i & 1;
        if (!mbar_wait(&empty[st], ((i / kStages) & 1) ^ 1u)) {
            set_status(p.status, PKV_DEV_WAIT_TIMEOUT);
            *abort_flag = 1;
            break;
        }
        const int t0 = j * kTile, t1 = min(t0 + kTile, kv_end);
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
            const int y = (phys * p.num_kv_heads + kvh) * B;
            uint8_t* dst = smem + kOffRing + st * kTileBytes + lane * B * 256;
            tc5::tma_load_4d(dst, isV ? tmV : tmK, 0, 0, 0, y >> 3, &full[st], policy);
        }
    }
}

// ---- the MMA issuer (one thread): PV_A(j), S_A(j+1), PV_B(j), S_B(j+1) ----
template <typename QT>
__device__ __forceinline__ void mq_mma(uint8_t* smem, uint32_t tmem, uint64_t* full,
                                       uint64_t* empty, uint64_t* s_full, uint64_t* p_full,
                                       uint64_t* q_full, uint64_t* drain, unsigned* status,
                                       volatile int* abort_flag, int T, int T_a, int T_b) {
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
    auto wait_item = [&](int i) {
        const bool r = mbar_wait(&full[i % kStages], (i / kStages) & 1);
        tc5::fence_after_sync();
        return r;
    };
    auto wait_p = [&](int X, int j) {
        const bool r = mbar_wait(&p_full[X], j & 1);
        tc5::fence_after_sync();
        return r;
    };
    bool ok = mbar_wait(q_full, 0) && wait_item(0);
    if (ok) {
        issue_s(0, 0);
        if (T_b > 0) issue_s(1, 0);
        tc5::commit(&empty[0]);
    }
    for (int j = 0; j < T && ok; ++j) {
        const int vs = (2 * j + 1) % kStages, ks = (2 * j + 2) % kStages;
        const bool next = j + 1 < T;
        if (!wait_item(2 * j + 1)) { ok = false; break; }
        if (j < T_a) {
            if (!wait_p(0, j)) { ok = false; break; }
            issue_pv(0, vs, j > 0);
        }
        if (next && !wait_item(2 * j + 2)) { ok = false; break; }
        if (j + 1 < T_a) issue_s(0, ks);
        if (j < T_b) {
            if (!wait_p(1, j)) { ok = false; break; }
            issue_pv(1, vs, j > 0);
        }
        tc5::commit(&empty[vs]);
        if (j + 1 < T_b) issue_s(1, ks);
        if (next) tc5::commit(&empty[ks]);
    }
    // every MMA issued above completes before O is read and the TMEM released
    tc5::commit(drain);
    if (!mbar_wait(drain, 0)) ok = false;
    if (!ok) {
        set_status(status, PKV_DEV_WAIT_TIMEOUT);
        *abort_flag = 1;
    }
}

template <typename QT>
__global__ void __launch_bounds__(kThreads, 1) mq_attention_kernel(
    MqParams p, const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBars);
    uint64_t* full = bars;                       // [kStages] TMA bytes of a ring stage landed
    uint64_t* empty = full + kStages;            // [kStages] the MMAs reading it completed
    uint64_t* s_full = empty + kStages;          // [2] S_X computed (and PV_X of the tile before)
    uint64_t* p_full = s_full + 2;               // [2] P_X written, O_X rescaled (128 arrivals)
    uint64_t* q_full = p_full + 2;               // Q rows written (256 arrivals)
    uint64_t* drain = q_full + 1;                // every MMA of the CTA completed
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // ---- this CTA's item: in launch order, the last sequence whose first item is
    // <= blockIdx.x ----
    const int b = blockIdx.x;
    if (b >= p.item_prefix[p.num_seqs]) return;   // whole CTA, before any allocation
    int lo = 0, hi = p.num_seqs - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (p.item_prefix[mid] <= b) lo = mid;
        else hi = mid - 1;
    }
    const int s = p.seq_order[lo];
    const int local = b - p.item_prefix[lo];
    const int G = p.group;
    const int q_begin = p.query_start[s];
    const int n = p.query_start[s + 1] - q_begin;
    const int ctx = p.context_lens[s];
    const int qpt = kTile / G;                            // query tokens per row tile
    const int ctas = (n * G + kMqRows - 1) / kMqRows;
    const int ct = ctas - 1 - local / p.num_kv_heads;     // later (longer) row pairs first
    const int kvh = local % p.num_kv_heads;
    // row tile X (A = 0, B = 1) covers queries [q0 + X qpt, .. + qn_X) and reads
    // tokens [0, kv_end_X); tile A is never empty, tile B may be
    const int q0 = 2 * ct * qpt;
    const int qn_a = min(qpt, n - q0), qn_b = max(0, min(qpt, n - q0 - qpt));
    const int kv_end_a = ctx - n + q0 + qn_a;
    const int kv_end_b = qn_b > 0 ? ctx - n + q0 + qpt + qn_b : 0;
    const int T_a = (kv_end_a + kTile - 1) / kTile, T_b = (kv_end_b + kTile - 1) / kTile;
    const int kv_end = max(kv_end_a, kv_end_b);           // tokens the CTA stages
    const int T = max(T_a, T_b);                          // K/V tiles; T_a >= 1

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&p_full[i], kTile);
        }
        mbar_init(q_full, 2 * kTile);
        mbar_init(drain, 1);
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
            mq_producer(p, &tmK, &tmV, smem, full, empty, abort_flag, s, kvh, kv_end, T);
        } else if (warp == 9) {
            if (lane == 0)
                mq_mma<QT>(smem, tmem, full, empty, s_full, p_full, q_full, drain, p.status,
                           abort_flag, T, T_a, T_b);
            __syncwarp();
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
        const int Tx = X ? T_b : T_a, kv_end_r = X ? kv_end_b : kv_end_a;
        const int qi = q0 + X * qpt + r / G, hq = kvh * G + r % G;
        const bool row_valid = r < (X ? qn_b : qn_a) * G;
        const int64_t qrow = ((int64_t)(q_begin + qi) * p.num_q_heads + hq) * kHD;
        {
            // the row's q into Q_X: [half][row][128 B], 16-byte chunks swizzled by row
            const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.q) +
                                                              (row_valid ? qrow : 0));
            uint8_t* qs = smem + kOffQ + X * kTileBytes;
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                const uint4 v = row_valid ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
                *reinterpret_cast<uint4*>(qs + (c >> 3) * kHalfBytes + sw128(r, c & 7)) = v;
            }
            fence_proxy_async_smem();
            mbar_arrive(q_full);
        }
        // the V rows past the CTA's last token hold poison or stale data (0 x NaN would
        // reach O through P = 0): the row tile whose P.V reads the last V tile first
        // zeroes them once their copy has landed
        const bool zeroes = (X == 0) == (T_a == T);
        const int pos_r = ctx - n + qi;                   // this row's query position
        const uint32_t colS = tmem + lane_base + kColS + (uint32_t)(X * kTile),
                       colO = tmem + lane_base + kColO + (uint32_t)(X * kTile);
        float m_run = -INFINITY, l_run = 0.f;
        bool ok = true;
        for (int j = 0; j < Tx; ++j) {
            // wait decisions are warp-uniform: the tcgen05 loads and stores below need
            // the whole warp converged
            const bool got = !*abort_flag && mbar_wait(&s_full[X], j & 1);
            if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
            tc5::fence_after_sync();
            // local tokens <= lim are visible (rows past the last query see no further);
            // a tile every row of the warp sees whole needs no mask
            const int lim = min(pos_r, kv_end_r - 1) - j * kTile;
            const bool masked = !__all_sync(0xffffffffu, lim >= kTile - 1);
            uint32_t sv[4][32];
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) tc5::ld_32x32b_x32(colS + (uint32_t)(32 * c4), sv[c4]);
            tc5::wait_ld();
            if (masked) {
#pragma unroll
                for (int c = 0; c < kTile; ++c)
                    if (c > lim) sv[c >> 5][c & 31] = __float_as_uint(-INFINITY);
            }
            // row max of the raw scores (the scale is positive: same order), with 8
            // independent partial maxima
            float pmx[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) pmx[i] = -INFINITY;
#pragma unroll
            for (int c = 0; c < kTile; ++c)
                pmx[c & 7] = fmaxf(pmx[c & 7], __uint_as_float(sv[c >> 5][c & 31]));
#pragma unroll
            for (int i = 1; i < 8; ++i) pmx[0] = fmaxf(pmx[0], pmx[i]);
            const float mx = pmx[0] * p.qk_scale_log2;
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
            // P = 2^(scale * s - m) (one FMA and one ex2 per score), rounded to the
            // operand type, over the first 64 columns of S_X; l sums the weights
            const float neg_m = m_run == -INFINITY ? 0.f : -m_run;
            float pls[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) pls[i] = 0.f;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                uint32_t pw[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const int c = 64 * hh + 2 * e;
                    const float a = fast_exp2(fmaf(__uint_as_float(sv[c >> 5][c & 31]),
                                                   p.qk_scale_log2, neg_m));
                    const float bb = fast_exp2(fmaf(__uint_as_float(sv[(c + 1) >> 5][(c + 1) & 31]),
                                                    p.qk_scale_log2, neg_m));
                    pw[e] = pack2_bits<QT>(a, bb);
                    pls[(2 * e) & 7] += a;
                    pls[(2 * e + 1) & 7] += bb;
                }
                tc5::st_32x32b_x32(colS + (uint32_t)(32 * hh), pw);
            }
            float lsum = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) lsum += pls[i];
            l_run += lsum;
            if (zeroes && j == T - 1 && kv_end - j * kTile < kTile) {
                const int iv = 2 * j + 1;
                if (!__all_sync(0xffffffffu,
                                mbar_wait(&full[iv % kStages], (iv / kStages) & 1))) {
                    ok = false;
                    break;
                }
                if (r >= kv_end - j * kTile) {
                    uint8_t* vrow = smem + kOffRing + (iv % kStages) * kTileBytes +
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
        if (Tx > 0) {
            if (ok) ok = __all_sync(0xffffffffu, !*abort_flag && mbar_wait(drain, 0));
            if (ok) {
                tc5::fence_after_sync();
                const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4) {
                    uint32_t o[32];
                    tc5::ld_32x32b_x32(colO + (uint32_t)(c4 * 32), o);
                    tc5::wait_ld();
                    if (row_valid) {
                        uint32_t w[16];
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            float ra, rb;
                            w[e] = pack2<QT>(__uint_as_float(o[2 * e]) * inv,
                                             __uint_as_float(o[2 * e + 1]) * inv, ra, rb);
                        }
                        uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) +
                                                              qrow + c4 * 32);
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            dst[e] = make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
                    }
                }
            } else {
                set_status(p.status, PKV_DEV_WAIT_TIMEOUT);
                *abort_flag = 1;
            }
        }
    }
    tc5::fence_before_sync();
    named_bar_sync(1, kThreads);
}

template <typename QT>
cudaError_t launch_typed(const MqParams& p, int64_t max_items, cudaStream_t stream) {
    static bool attr_set[64] = {};
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    auto kernel = mq_attention_kernel<QT>;
    if (!attr_set[dev]) {
        err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
        if (err != cudaSuccess) return err;
        attr_set[dev] = true;
    }
    CUtensorMap tk, tv;
    const long long rows = (long long)p.num_blocks * p.num_kv_heads * p.block_size;
    if (!encode_pool_map_grouped(&tk, p.k_cache, rows, p.block_size) ||
        !encode_pool_map_grouped(&tv, p.v_cache, rows, p.block_size))
        return cudaErrorInvalidValue;
    mq_plan_kernel<<<1, 1024, 0, stream>>>(p);
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    kernel<<<(unsigned)max_items, kThreads, kSmem, stream>>>(p, tk, tv);
    return cudaGetLastError();
}

}  // namespace

int64_t mq_max_items(int num_seqs, int total_q, int group, int num_kv_heads) {
    return (int64_t)num_kv_heads * (((int64_t)total_q * group + kMqRows - 1) / kMqRows + num_seqs);
}

cudaError_t launch_mq_attention(const MqParams& p, pkv_dtype q_dtype, int64_t max_items,
                                cudaStream_t stream) {
    if (max_items <= 0) return cudaSuccess;
    if (max_items > 0x7fffffffLL) return cudaErrorInvalidValue;
    switch (q_dtype) {
    case PKV_F16: return launch_typed<F16>(p, max_items, stream);
    case PKV_BF16: return launch_typed<BF16>(p, max_items, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace pkv
