// mq_attention.cu -- multi-query causal paged attention on the 5th-generation
// tensor cores (tcgen05: operands in shared memory, accumulators in TMEM).
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
// Organisation: one CTA per (sequence, kv head, tile of 128 rows), a row being
// a (query token, query head of the kv head's group) pair, so the G heads that
// share a kv head share every K/V tile.  Six warps:
//   warps 0-3  one thread per row (TMEM lane): Q rows to shared memory, the
//              softmax of each S tile, the rescale of O, the epilogue;
//   warp 4     TMA producer: the K and V blocks of each 128-token tile, whole
//              (block, kv head) rows of the pool, into a 2-stage ring;
//   warp 5     TMEM allocation; one lane issues the MMAs.
// Per 128-token tile j:  S_j = Q K_j^T (M 128, N 128, K 128; TMEM, double
// buffered so S_{j+1} runs while tile j's softmax does), then
// O += P_j V_j (P from shared memory, V as an MN-major operand; O in TMEM).
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
constexpr int kHalfBytes = 128 * 128;                 // 128 rows x 128 B (64 elements)
constexpr int kTileBytes = 2 * kHalfBytes;            // 128 rows x 256 B
// K and V tiles arrive as [group of 8 tokens][half of d][8 tokens][128 B]
constexpr int kGroupHalf = 8 * 128;                   // one half of d of an 8-token group
constexpr int kGroupBytes = 2 * kGroupHalf;           // an 8-token group
constexpr int kKStages = 4;                           // K ring: freed when S_j completes
constexpr int kVStages = 3;                           // V ring: freed when P_j V_j completes
constexpr int kOffK = 0;
constexpr int kOffV = kOffK + kKStages * kTileBytes;
constexpr int kOffX = kOffV + kVStages * kTileBytes;  // the rows' softmax sums, exchanged
constexpr int kOffBars = kOffX + 1024;
constexpr int kSmem = kOffBars + 256 + 1024;          // barriers, TMEM slot, flag; alignment
constexpr int kThreads = 352;                         // 8 row warps, K and V producers, MMA
// TMEM columns (lane = row): S double-buffered (fp32), O (fp32), and the MMA A
// operands Q and P (16-bit, two elements per column)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;                         // S_j at kColS + 128 (j % 2)
constexpr uint32_t kColO = 256;
constexpr uint32_t kColQ = 384;
constexpr uint32_t kColP = 448;
constexpr float kMaxSlack = 8.0f;                     // log2-domain headroom before the max moves

static_assert(kOffBars + 256 + 1024 <= 227 * 1024, "shared memory per CTA");
constexpr int kNumBars = 2 * kKStages + 2 * kVStages + 2 + 2 + 2 + 1 + 1;
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

// Items: per sequence ceil(n * G / 128) row tiles times Hkv; exclusive prefix.
__global__ void __launch_bounds__(1024) mq_plan_kernel(MqParams p) {
    const int total_q = p.total_q;
    __shared__ int wsum[32];
    __shared__ int carry;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) {
        carry = 0;
        if (p.query_start[p.num_seqs] != total_q || p.query_start[0] != 0)
            set_status(p.status, PKV_DEV_BAD_CONTEXT);
    }
    const int cap = min(p.max_context_len, p.max_blocks * p.block_size);
    __syncthreads();
    for (int base = 0; base < p.num_seqs; base += blockDim.x) {
        const int s = base + tid;
        int items = 0;
        if (s < p.num_seqs) {
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
        if (s < p.num_seqs) p.item_prefix[s] = carry + incl - items;
        __syncthreads();
        if (tid == blockDim.x - 1) carry += incl;
        __syncthreads();
    }
    if (tid == 0) p.item_prefix[p.num_seqs] = carry;
}

template <typename QT>
__global__ void __launch_bounds__(kThreads, 1) mq_attention_kernel(
    MqParams p, const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBars);
    uint64_t* k_full = bars;                     // [kKStages] TMA bytes of a K stage landed
    uint64_t* k_empty = k_full + kKStages;       // [kKStages] the S MMA reading it completed
    uint64_t* v_full = k_empty + kKStages;       // [kVStages] TMA bytes of a V stage landed
    uint64_t* v_empty = v_full + kVStages;       // [kVStages] the P.V MMA reading it completed
    uint64_t* s_full = v_empty + kVStages;       // [2] S buffer computed
    uint64_t* p_full = s_full + 2;               // [2] P tile written, O rescaled (256 arrivals)
    uint64_t* o_done = p_full + 2;               // [2] P_j V_j completed (by tile parity)
    uint64_t* q_full = o_done + 2;               // Q rows written (256 arrivals)
    uint64_t* drain = q_full + 1;                // every MMA of the CTA completed
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // ---- this CTA's item: the last sequence whose first item is <= blockIdx.x ----
    const int b = blockIdx.x;
    if (b >= p.item_prefix[p.num_seqs]) return;   // whole CTA, before any allocation
    int lo = 0, hi = p.num_seqs - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (p.item_prefix[mid] <= b) lo = mid;
        else hi = mid - 1;
    }
    const int s = lo;
    const int local = b - p.item_prefix[s];
    const int G = p.group;
    const int q_begin = p.query_start[s];
    const int n = p.query_start[s + 1] - q_begin;
    const int ctx = p.context_lens[s];
    const int qpt = kMqRows / G;                          // query tokens per row tile
    const int tiles = (n * G + kMqRows - 1) / kMqRows;
    const int qt = tiles - 1 - local / p.num_kv_heads;    // later (longer) tiles first
    const int kvh = local % p.num_kv_heads;
    const int q0 = qt * qpt;
    const int qn = min(qpt, n - q0);
    const int rows_valid = qn * G;
    const int pos0 = ctx - n + q0;                        // position of query q0
    const int kv_end = pos0 + qn;                         // tokens [0, kv_end) are read
    const int T = (kv_end + kMqTokens - 1) / kMqTokens;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kKStages; ++i) {
            mbar_init(&k_full[i], 1);
            mbar_init(&k_empty[i], 1);
        }
        for (int i = 0; i < kVStages; ++i) {
            mbar_init(&v_full[i], 1);
            mbar_init(&v_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&p_full[i], 256);
            mbar_init(&o_done[i], 1);
        }
        mbar_init(q_full, 256);
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 10) tc5::tmem_alloc(tmem_slot, kTmemCols);
    tc5::fence_before_sync();
    __syncthreads();
    tc5::fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp == 8 || warp == 9) {
        // ===================== TMA producers: warp 8 K, warp 9 V =====================
        const bool isK = warp == 8;
        const CUtensorMap* map = isK ? &tmK : &tmV;
        if (lane == 0) prefetch_tensormap(map);
        const uint64_t policy = l2_evict_last_policy();   // other row tiles re-read K/V
        const int B = p.block_size;
        const int nst = isK ? kKStages : kVStages;
        uint64_t* full = isK ? k_full : v_full;
        uint64_t* empty = isK ? k_empty : v_empty;
        uint8_t* ring = smem + (isK ? kOffK : kOffV);
        const int32_t* trow = p.block_tables + (int64_t)s * p.max_blocks;
        const int nb_all = (kv_end + B - 1) / B;          // table entries this CTA reads
        // block-table window: lane l holds entry wb + l (cur) and wb + 32 + l (nxt); the
        // next window loads as soon as the current one is entered, so a tile's entries
        // are in registers when its stage frees (a tile spans <= 16 entries)
        int wb = 0;
        int cur = lane < nb_all ? trow[lane] : 0;
        int nxt = lane + 32 < nb_all ? trow[lane + 32] : 0;
        for (int j = 0; j < T; ++j) {
            const int st = j % nst;
            if (!mbar_wait(&empty[st], ((j / nst) & 1) ^ 1u)) {
                set_status(p.status, PKV_DEV_WAIT_TIMEOUT);
                *abort_flag = 1;
                break;
            }
            const int t0 = j * kMqTokens, t1 = min(t0 + kMqTokens, kv_end);
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
                    if (isK) set_status(p.status, PKV_DEV_BAD_BLOCK_ID);
                    phys = 0;
                }
                // one box per block: both 128-byte halves of its B rows, landing as
                // [group of 8 rows][half][8 rows][128 B] at the block's place in the tile
                const int y = (phys * p.num_kv_heads + kvh) * B;
                uint8_t* dst = ring + st * kTileBytes + lane * B * 256;
                tc5::tma_load_4d(dst, map, 0, 0, 0, y >> 3, &full[st], policy);
            }
        }
    } else if (warp == 10) {
        // ============================ MMA issuer =============================
        if (lane == 0) {
            constexpr bool kBF16 = std::is_same<QT, BF16>::value;
            constexpr uint32_t idqk = tc5::idesc_f16(kBF16, 128, 128, false, false);
            constexpr uint32_t idpv = tc5::idesc_f16(kBF16, 128, 128, false, true);

            bool ok = mbar_wait(q_full, 0);
            tc5::fence_after_sync();
            for (int j = 0; j <= T && ok; ++j) {
                if (j < T) {
                    // S_j = Q K_j^T into S buffer j % 2 (its previous reader, tile j - 2's
                    // softmax, finished before P_{j-2} was published)
                    const int st = j & 1, ks = j % kKStages;
                    if (!mbar_wait(&k_full[ks], (j / kKStages) & 1)) { ok = false; break; }
                    tc5::fence_after_sync();
                    const uint32_t aK = smem_addr(smem + kOffK + ks * kTileBytes);
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const uint32_t offk = (uint32_t)((k >> 2) * kGroupHalf + (k & 3) * 32);
                        tc5::mma_ts(tmem + kColS + (uint32_t)(st * 128),
                                    tmem + kColQ + (uint32_t)(8 * k),
                                    tc5::smem_desc_sw128(aK + offk, 16, kGroupBytes), idqk, k > 0);
                    }
                    tc5::commit(&s_full[st]);
                    tc5::commit(&k_empty[ks]);
                }
                if (j > 0) {
                    // O += P_{j-1} V_{j-1}
                    const int pj = j - 1, vs = pj % kVStages;
                    if (!mbar_wait(&p_full[pj & 1], (pj >> 1) & 1) ||
                        !mbar_wait(&v_full[vs], (pj / kVStages) & 1)) { ok = false; break; }
                    tc5::fence_after_sync();
                    const uint32_t aV = smem_addr(smem + kOffV + vs * kTileBytes);
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        tc5::mma_ts(tmem + kColO, tmem + kColP + (uint32_t)(8 * k),
                                    tc5::smem_desc_sw128(aV + (uint32_t)(k * 2 * kGroupBytes),
                                                         kGroupHalf, kGroupBytes),
                                    idpv, pj > 0 || k > 0);
                    }
                    tc5::commit(&o_done[pj & 1]);
                    tc5::commit(&v_empty[vs]);
                }
            }
            // every MMA issued above completes before the TMEM is released
            tc5::commit(drain);
            if (!mbar_wait(drain, 0)) ok = false;
            if (!ok) {
                set_status(p.status, PKV_DEV_WAIT_TIMEOUT);
                *abort_flag = 1;
            }
        }
        __syncwarp();
    } else {
        // ======= rows: Q, softmax, O rescale, epilogue; two threads per row =======
        // warps 4h .. 4h+3 take columns [64 h, 64 h + 64) of every S tile, of P and of
        // O (and half h of d for Q and the output); both threads of a row read all 128
        // scores for the row max, so they agree on it without exchanging anything
        const int half = warp >> 2;
        const int r = threadIdx.x & (kMqRows - 1);        // TMEM lane = row
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        const int qi = q0 + r / G, hq = kvh * G + r % G;
        const bool row_valid = r < rows_valid;
        const int64_t qrow = ((int64_t)(q_begin + qi) * p.num_q_heads + hq) * kHD;
        {
            // this thread's half of the row's q, packed two per column, into TMEM
            const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.q) +
                                                              (row_valid ? qrow : 0)) + 8 * half;
            uint32_t qw[32];
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const uint4 v = row_valid ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
                qw[4 * c] = v.x;
                qw[4 * c + 1] = v.y;
                qw[4 * c + 2] = v.z;
                qw[4 * c + 3] = v.w;
            }
            tc5::st_32x32b_x32(lane_base + tmem + kColQ + (uint32_t)(32 * half), qw);
            tc5::wait_st();
            tc5::fence_before_sync();
            mbar_arrive(q_full);
        }
        const int pos_r = pos0 + r / G;                   // this row's query position
        const uint32_t colS0 = tmem + lane_base + kColS,
                       colOh = tmem + lane_base + kColO + (uint32_t)(64 * half);
        float m_run = -INFINITY, l_run = 0.f;
        bool ok = true;
        for (int j = 0; j < T; ++j) {
            // wait decisions are warp-uniform: the tcgen05 loads and stores below need
            // the whole warp converged
            const bool got = !*abort_flag && mbar_wait(&s_full[j & 1], (j >> 1) & 1);
            if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
            tc5::fence_after_sync();
            const uint32_t colS = colS0 + (uint32_t)((j & 1) * 128);
            // local tokens <= lim are visible (rows past the last query see no further);
            // a tile every row of the warp sees whole needs no mask
            const int lim = min(pos_r, kv_end - 1) - j * kMqTokens;
            const bool masked = !__all_sync(0xffffffffu, lim >= kMqTokens - 1);
            // this thread's 64 scores, kept for P
            uint32_t sv[2][32];
            tc5::ld_32x32b_x32(colS + (uint32_t)(64 * half), sv[0]);
            tc5::ld_32x32b_x32(colS + (uint32_t)(64 * half + 32), sv[1]);
            // the other half's 64, only for the row max
            uint32_t so[2][32];
            tc5::ld_32x32b_x32(colS + (uint32_t)(64 * (1 - half)), so[0]);
            tc5::ld_32x32b_x32(colS + (uint32_t)(64 * (1 - half) + 32), so[1]);
            tc5::wait_ld();
            if (masked) {
#pragma unroll
                for (int c = 0; c < 64; ++c) {
                    if (64 * half + c > lim) sv[c >> 5][c & 31] = __float_as_uint(-INFINITY);
                    if (64 * (1 - half) + c > lim) so[c >> 5][c & 31] = __float_as_uint(-INFINITY);
                }
            }
            // row max of the raw scores (the scale is positive: same order), with 8
            // independent partial maxima
            float pmx[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) pmx[i] = -INFINITY;
#pragma unroll
            for (int c = 0; c < 64; ++c) {
                pmx[c & 7] = fmaxf(pmx[c & 7], __uint_as_float(sv[c >> 5][c & 31]));
                pmx[c & 7] = fmaxf(pmx[c & 7], __uint_as_float(so[c >> 5][c & 31]));
            }
#pragma unroll
            for (int i = 1; i < 8; ++i) pmx[0] = fmaxf(pmx[0], pmx[i]);
            const float mx = pmx[0] * p.qk_scale_log2;
            const float m_new = mx > m_run + kMaxSlack ? mx : m_run;
            const bool resc = j > 0 && m_new != m_run;
            if (__any_sync(0xffffffffu, resc)) {
                // O may be rescaled once the previous tile's P.V has completed
                if (!__all_sync(0xffffffffu, mbar_wait(&o_done[(j - 1) & 1], ((j - 1) >> 1) & 1))) {
                    ok = false;
                    break;
                }
                tc5::fence_after_sync();
                const float f = resc ? fast_exp2(m_run - m_new) : 1.f;
#pragma unroll
                for (int c4 = 0; c4 < 2; ++c4) {
                    uint32_t o[32];
                    tc5::ld_32x32b_x32(colOh + (uint32_t)(c4 * 32), o);
                    tc5::wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * f);
                    tc5::st_32x32b_x32(colOh + (uint32_t)(c4 * 32), o);
                }
                tc5::wait_st();
                l_run *= f;
            }
            m_run = m_new;
            // the P columns are free once P_{j-1} V_{j-1} has completed: the weights
            // are computed into registers first, the wait comes just before the store
            // P = 2^(scale * s - m) (one FMA and one ex2 per score), rounded to the
            // operand type; l sums this thread's weights, 8 partial sums
            const float neg_m = m_run == -INFINITY ? 0.f : -m_run;
            float pls[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) pls[i] = 0.f;
            uint32_t pw[32];                              // this thread's 64 weights, packed
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                const int c = 2 * e;
                const float a = fast_exp2(fmaf(__uint_as_float(sv[c >> 5][c & 31]),
                                               p.qk_scale_log2, neg_m));
                const float bb = fast_exp2(fmaf(__uint_as_float(sv[(c + 1) >> 5][(c + 1) & 31]),
                                                p.qk_scale_log2, neg_m));
                pw[e] = pack2_bits<QT>(a, bb);
                pls[(2 * e) & 7] += a;
                pls[(2 * e + 1) & 7] += bb;
            }
            if (j > 0 &&
                !__all_sync(0xffffffffu, mbar_wait(&o_done[(j - 1) & 1], ((j - 1) >> 1) & 1))) {
                ok = false;
                break;
            }
            tc5::fence_after_sync();
            tc5::st_32x32b_x32(tmem + lane_base + kColP + (uint32_t)(32 * half), pw);
            float lsum = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) lsum += pls[i];
            l_run += lsum;
            if (j == T - 1 && kv_end - j * kMqTokens < kMqTokens) {
                // V rows past the last token hold poison or stale data: 0 x NaN would
                // reach O through P = 0.  Zero them (this thread's half of d) once their
                // TMA copy has landed.
                if (!__all_sync(0xffffffffu,
                                mbar_wait(&v_full[j % kVStages], (j / kVStages) & 1))) {
                    ok = false;
                    break;
                }
                if (r >= kv_end - j * kMqTokens) {
                    uint8_t* vrow = smem + kOffV + (j % kVStages) * kTileBytes +
                                    (r >> 3) * kGroupBytes + half * kGroupHalf + (r & 7) * 128;
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        *reinterpret_cast<uint4*>(vrow + c * 16) = make_uint4(0u, 0u, 0u, 0u);
                }
            }
            tc5::wait_st();
            fence_proxy_async_smem();                     // the V rows zeroed above
            tc5::fence_before_sync();
            mbar_arrive(&p_full[j & 1]);
        }
        if (ok)
            ok = __all_sync(0xffffffffu, !*abort_flag &&
                                             mbar_wait(&o_done[(T - 1) & 1], ((T - 1) >> 1) & 1));
        // the row's softmax denominator: the two threads' sums, exchanged through
        // shared memory; all 256 row threads take part
        float* xl = reinterpret_cast<float*>(smem + kOffX);
        xl[half * kMqRows + r] = l_run;
        named_bar_sync(1, 2 * kMqRows);
        const float l_row = xl[r] + xl[kMqRows + r];
        if (ok) {
            tc5::fence_after_sync();
            const float inv = l_row > 0.f ? 1.f / l_row : 0.f;
#pragma unroll
            for (int c4 = 0; c4 < 2; ++c4) {
                uint32_t o[32];
                tc5::ld_32x32b_x32(colOh + (uint32_t)(c4 * 32), o);
                tc5::wait_ld();
                if (row_valid) {
                    uint32_t w[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        float ra, rb;
                        w[e] = pack2<QT>(__uint_as_float(o[2 * e]) * inv,
                                         __uint_as_float(o[2 * e + 1]) * inv, ra, rb);
                    }
                    uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) + qrow +
                                                          64 * half + c4 * 32);
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
    tc5::fence_before_sync();
    __syncthreads();
    if (warp == 10) {
        tc5::fence_after_sync();
        tc5::tmem_dealloc(tmem, kTmemCols);
    }
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
