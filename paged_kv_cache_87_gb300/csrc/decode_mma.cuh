// decode_mma.cuh -- paged decode attention for grouped query heads on tensor cores.
//
// Same result as decode.cuh ("PagedAttention: Mathematical Foundations ..."
// §3, §7), for kv groups of 3-8 query heads with 16-bit q and K/V.  With G
// heads per K/V load the CUDA-core kernel spends 2G FMAs per loaded element
// and becomes issue-bound; here the grouped scores and the P.V product are
// small dense contractions done with warp-level mma.sync (m16n8k16, fp32
// accumulate), FA2-style, with P kept in registers:
//
//   S^T[16 tokens x 8 heads]  = K_t[16 x d] . Q^T[d x 8]        (A = K from smem)
//   O^T[d x 8 heads]         += V_t^T[d x 16] . P^T[16 x 8]     (A = V^T from smem)
//
// P^T leaves the first product as a C fragment (tokens by lane/4) and enters
// the second as a B fragment (tokens by lane%4): one movmatrix.trans per 8x8
// block turns one into the other.  K/V tiles arrive through TMA tensor copies
// with the 128-byte swizzle, so every ldmatrix is free of bank conflicts.
//
// Organisation: a CTA is one producer warp and one consumer warp, several
// CTAs per SM.  The work -- every (sequence, kv head, head subgroup) unit cut
// into 64-token tiles -- is split evenly over the CTAs (stream-K style): CTA b
// owns tiles [b*Q, (b+1)*Q) of the flattened (unit, tile) sequence, so every
// CTA streams the same number of K/V bytes and a long unit is cut into a few
// segments instead of many fixed chunks.  The producer walks its range in
// windows of at most 64 blocks of one unit, loading the next window's block-
// table entries while it streams the current one, and fills a small ring of
// 32-token stages (one 2-D tensor copy per (block, kv head, 64-column half) of
// K and of V, plus the segment's query rows).  The consumer keeps two 16-token
// m-tiles in flight per stage.  The end of a segment is warp-local: a unit
// held by one CTA writes `out`; otherwise the segment's (m, l, acc) goes to
// the workspace and the CTA that finishes the unit's last segment merges the
// segments in order (deterministic), all heads in parallel.  Rows past the
// context (poisoned or stale) are masked in S and zeroed in V before P.V.
#pragma once

#include <cuda.h>

#include <type_traits>

#include "decode.cuh"

namespace pkv {

// ------------------------------------------------------------ PTX wrappers --

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

template <typename T>
struct Mma;

template <>
struct Mma<BF16> {
    __device__ __forceinline__ static void run(float (&d)[4], const uint32_t (&a)[4],
                                               uint32_t b0, uint32_t b1) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, "
            "{%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
    // round (lo, hi) to the operand type; also return the rounded values
    __device__ __forceinline__ static uint32_t pack(float lo, float hi, float& flo, float& fhi) {
        __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
        flo = __low2float(v);
        fhi = __high2float(v);
        return *reinterpret_cast<uint32_t*>(&v);
    }
};

template <>
struct Mma<F16> {
    __device__ __forceinline__ static void run(float (&d)[4], const uint32_t (&a)[4],
                                               uint32_t b0, uint32_t b1) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, "
            "{%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
    __device__ __forceinline__ static uint32_t pack(float lo, float hi, float& flo, float& fhi) {
        __half2 v = __floats2half2_rn(lo, hi);
        flo = __low2float(v);
        fhi = __high2float(v);
        return *reinterpret_cast<uint32_t*>(&v);
    }
};

// ------------------------------------------------------------------ config --

template <typename QT, typename KT, int HD, int NT = 1>
struct MmaCfg {
    static constexpr bool FP8 = std::is_same<KT, E4M3>::value;
    using MT = typename std::conditional<FP8, F16, KT>::type;   // mma operand type
    static constexpr int TPS = 32;                // tokens per stage: two 16-token m-tiles
    static constexpr int ROWB = HD * KT::bytes;   // bytes of one K/V row
    static constexpr int HALVES = ROWB / 128;     // 128-byte column slices of a row
    static constexpr int ELEMS_PER_SLICE = 128 / KT::bytes;
    static constexpr int KSTEPS = HD / 16;        // mma k-steps of Q.K^T
    static constexpr int MTILES = HD / 16;        // mma m-tiles of P.V (over d)
    static constexpr int HALF_BYTES = TPS * 128;  // one 128-byte slice of a stage
    static constexpr int KV_BYTES = HALVES * HALF_BYTES;
    // each segment's query rows (up to 8 heads, or 16 in the prefix kernel) arrive
    // with its first stage; only the 16-head kernel over 16-bit K/V at head_dim 128,
    // whose 16 KB stages leave no room, reads them from global memory instead
    static constexpr bool QSTAGE = NT == 1 || FP8 || HD == 64;
    static constexpr int Q_BYTES = QSTAGE ? NT * kMmaHeadsPerItem * HD * 2 : 0;
    static constexpr int STAGE_BYTES = (2 * KV_BYTES + Q_BYTES + 1023) / 1024 * 1024;
    static constexpr int NSTAGE = HD == 128 ? (FP8 ? (NT == 1 ? 5 : 4) : 3) : (NT == 1 ? 5 : 5);
    // consumer warps: each takes MTC of a stage's two 16-token m-tiles for all NT
    // n-tiles; the producer is warp NC.  Two consumers put a CTA at three warps, which
    // the SM spreads over all four sub-partitions (two-warp CTAs leave the consumers
    // on two of them).
    static constexpr int NC = NT;
    static constexpr int MTC = 2 / NC;
    static constexpr int THREADS = 32 * (NC + 1);
    // end of a segment with two consumers: consumer 1 hands its state to consumer 0
    // one n-tile at a time (per lane: MTILES x 4 accumulators, then m0, m1, l0, l1)
    static constexpr int XCH_FLOATS = MTILES * 4 + 4;
    static constexpr size_t OFF_METAS = (size_t)NSTAGE * STAGE_BYTES;
    static constexpr size_t OFF_BARS = OFF_METAS + NSTAGE * sizeof(StageMeta);
    static constexpr size_t OFF_XCH = OFF_BARS + (2 * NSTAGE + 2) * sizeof(uint64_t);
    static constexpr size_t SMEM =
        OFF_XCH + (NC > 1 ? (size_t)XCH_FLOATS * 32 * sizeof(float) : 0) + 1024;
    static_assert(HD == 64 || HD == 128, "head_dim");
    static_assert(!FP8 || HD == 128, "FP8 rows must be 128 bytes");
    static_assert(std::is_same<QT, F16>::value || std::is_same<QT, BF16>::value, "q type");
};

// Two e4m3 codes (low byte first) -> f16x2 (exact).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_codes) {
    __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two_codes),
                                               __NV_E4M3);
    return *reinterpret_cast<uint32_t*>(&h);
}

// Two 16-bit q values (low first) as the mma operand type MT.
template <typename QT, typename MT>
__device__ __forceinline__ uint32_t q_pair(uint32_t raw) {
    if constexpr (std::is_same<QT, MT>::value) {
        return raw;
    } else {   // bf16 q with an f16 mma (FP8 KV): exact for |q| in f16's normal range
        __nv_bfloat162 b = *reinterpret_cast<__nv_bfloat162*>(&raw);
        __half2 h = __floats2half2_rn(__low2float(b), __high2float(b));
        return *reinterpret_cast<uint32_t*>(&h);
    }
}

// Byte offset of 16-byte chunk `chunk` (0..7) of row `r` in a 128-byte-row,
// 128-byte-swizzled region whose base is 1024-byte aligned.
__device__ __forceinline__ uint32_t swz(int r, int chunk) {
    return (uint32_t)(r * 128 + ((chunk ^ (r & 7)) << 4));
}

// ---------------------------------------------------------------- planning --

// Block-wide exclusive scan of two counters (1024 threads); returns this
// thread's prefixes, and the block totals in *tot_a / *tot_b.
__device__ __forceinline__ void scan2(int a, int b, int* ex_a, int* ex_b, int* tot_a, int* tot_b,
                                      int* wa, int* wb) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int xa = a, xb = b;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int ya = __shfl_up_sync(0xffffffffu, xa, off);
        const int yb = __shfl_up_sync(0xffffffffu, xb, off);
        if (lane >= off) { xa += ya; xb += yb; }
    }
    if (lane == 31) { wa[warp] = xa; wb[warp] = xb; }
    __syncthreads();
    if (warp == 0) {
        int va = wa[lane], vb = wb[lane];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int ya = __shfl_up_sync(0xffffffffu, va, off);
            const int yb = __shfl_up_sync(0xffffffffu, vb, off);
            if (lane >= off) { va += ya; vb += yb; }
        }
        wa[lane] = va;
        wb[lane] = vb;
    }
    __syncthreads();
    *ex_a = xa - a + (warp > 0 ? wa[warp - 1] : 0);
    *ex_b = xb - b + (warp > 0 ? wb[warp - 1] : 0);
    *tot_a = wa[31];
    *tot_b = wb[31];
    __syncthreads();   // wa / wb are reused by the next call
}

// Balanced-split planning (1 CTA x 1024 threads, sequences in tiles of 1024).
//  1. Clamp context lengths.
//  2. Shared-prefix groups ("...Mathematical Foundations" §5 Parallel Sampling
//     and System Prompt Prefix Sharing): consecutive sequences whose tables
//     start with the same physical block form runs; a run is cut into groups
//     of at most kMaxGroupHeads / G members.  A group's shared prefix is the
//     leading blocks every member's table has in common with the leader's,
//     cut to the shortest member context and rounded down to 64 tokens; a
//     group with at least 64 shared tokens gets one shared unit per kv head.
//  3. Work records in sequence order -- a group's shared record before its
//     leader's private record -- each unit cut into 64-token tiles; prefix
//     sums over records; the per-worker quota Q; each worker's first record.
//  4. Per (sequence, unit): the number of partial states its result merges
//     (shared segments first, then private ones) and where the private ones
//     start.  Unit counters reset; outputs of empty sequences zeroed.
// Shared-prefix detection for the prefix-aware decode (one warp per sequence s,
// many CTAs, before the planner): common[s] = the number of leading block-table
// entries row s has in common with row s - 1, within the blocks both contexts use
// (0 for the first sequence of each planner tile of 1024, and whenever either
// context is empty).  Coalesced loads, 512 entries per round, ballots for the
// first difference.  Spreading the rows' loads over many SMs keeps the planner's
// single CTA off this latency-bound work.
template <typename QT>
__global__ void __launch_bounds__(256) prefix_common_kernel(DecodeParams p) {
    pdl_launch_dependents();   // the planner's launch overlaps this kernel
    const int s = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (s >= p.num_seqs) return;
    const int B = p.block_size;
    const int cap = min(p.max_context_len, p.max_blocks * B);
    auto clamp = [&](int c) { return c < 0 ? 0 : (c > cap ? cap : c); };
    int common = 0;
    if (s % 1024 != 0) {
        const int ca = clamp(__ldg(p.context_lens + s - 1)), cb = clamp(__ldg(p.context_lens + s));
        const int lim = min((ca + B - 1) / B, (cb + B - 1) / B);
        const int32_t* ra = p.block_tables + (int64_t)(s - 1) * p.max_blocks;
        const int32_t* rb = p.block_tables + (int64_t)s * p.max_blocks;
        common = lim;
        for (int j0 = 0; j0 < lim; j0 += 512) {
            bool diff[16];
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                const int j = j0 + 32 * u + lane;
                diff[u] = j < lim && __ldg(ra + j) != __ldg(rb + j);
            }
            int first = -1;
#pragma unroll
            for (int u = 15; u >= 0; --u) {
                const unsigned m = __ballot_sync(0xffffffffu, diff[u]);
                if (m) first = j0 + 32 * u + __ffs(m) - 1;
            }
            if (first >= 0) {
                common = first;
                break;
            }
        }
    }
    if (lane == 0) p.ws.common[s] = common;
}

// Record-prefix entries the planner keeps in shared memory for the workers'
// binary search (larger plans search the global copy).
constexpr int kPlanSmemRecords = 4096;

template <typename QT>
__global__ void __launch_bounds__(1024) plan_split_kernel(DecodeParams p) {
    pdl_launch_dependents();   // the decode kernel's prologue overlaps this plan
    pdl_wait();                // prefix-aware launches: prefix_common_kernel has completed
    __shared__ int s_ctx[1024], s_first[1024], s_run[1024], s_mem[1024], s_sh[1024];
    __shared__ int s_rp[kPlanSmemRecords + 1];      // record prefix (first tile of each record)
    __shared__ int wa[32], wb[32];
    __shared__ int carry_rec, carry_tiles;
    const int tid = threadIdx.x;
    const int upi = p.num_kv_heads * p.nsub;
    const bool can_group = p.allow_groups && p.nsub == 1 && p.group <= kMmaHeadsPerItem;
    const int maxm = can_group ? kMaxGroupHeads / p.group : 1;
    const int B = p.block_size;
    if (tid == 0) carry_rec = carry_tiles = 0;
    for (int i = tid; i < p.num_seqs * upi; i += blockDim.x) p.ws.unit_done[i] = 0u;
    const int cap = min(p.max_context_len, p.max_blocks * B);
    __syncthreads();
    for (int base = 0; base < p.num_seqs; base += blockDim.x) {
        const int s = base + tid;
        const bool valid = s < p.num_seqs;
        int ctx = 0;
        // entries this sequence's row has in common with its predecessor's (written by
        // prefix_common_kernel); it loads beside the context length
        const int common = can_group && valid ? __ldcg(p.ws.common + s) : 0;
        if (valid) {
            ctx = p.context_lens[s];
            if (ctx < 0 || ctx > cap) {
                set_status(p.status, PKV_DEV_BAD_CONTEXT);
                ctx = ctx < 0 ? 0 : cap;
            }
            p.ws.ctx_eff[s] = ctx;
        }
        s_ctx[tid] = ctx;
        s_sh[tid] = common;
        __syncthreads();
        // run start: inclusive max-scan of (same first block as the previous ? -1 : tid);
        // a run never crosses a tile of 1024 sequences
        const bool same = can_group && valid && tid > 0 && ctx > 0 && s_ctx[tid - 1] > 0 &&
                          common > 0;
        int run = same ? -1 : tid;
        {
            const int lane = tid & 31, warp = tid >> 5;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, run, off);
                if (lane >= off) run = max(run, y);
            }
            if (lane == 31) wa[warp] = run;
            __syncthreads();
            if (warp == 0) {
                int v = wa[lane];
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const int y = __shfl_up_sync(0xffffffffu, v, off);
                    if (lane >= off) v = max(v, y);
                }
                wa[lane] = v;
            }
            __syncthreads();
            if (warp > 0) run = max(run, wa[warp - 1]);
            s_run[tid] = run;
            __syncthreads();
        }
        // group leaders: every maxm-th position of a run
        const int k = tid - run;
        const bool is_lead = can_group && valid && k % maxm == 0 && ctx > 0;
        // a group's shared prefix: the minimum over its members of the entries each has
        // in common with its predecessor -- equal, by transitivity, to the minimum of
        // each member's common entries with the leader
        int members = 0, shared = 0;
        if (is_lead) {
            int m = 1;
            while (m < maxm && tid + m < (int)blockDim.x && base + tid + m < p.num_seqs &&
                   s_run[tid + m] == run && s_ctx[tid + m] > 0)
                ++m;
            if (m >= 2) {
                int sh = (ctx + B - 1) / B, minctx = ctx;
                for (int i = 1; i < m; ++i) {
                    minctx = min(minctx, s_ctx[tid + i]);
                    sh = min(sh, s_sh[tid + i]);
                }
                shared = min(sh * B, minctx) / kTileTokens * kTileTokens;
                if (shared >= kTileTokens) members = m;
                else shared = 0;
            }
        }
        __syncthreads();                                      // s_sh is rewritten below
        s_mem[tid] = members;
        s_sh[tid] = shared;
        __syncthreads();
        int leader = -1, start = 0;
        if (can_group && valid) {
            const int lp = run + (k / maxm) * maxm;
            if (s_mem[lp] >= 2) {
                leader = base + lp;
                start = s_sh[lp];
            }
        }
        const int priv_tiles = valid ? (ctx - start + kTileTokens - 1) / kTileTokens : 0;
        const int nrec = valid ? 1 + (members >= 2) : 0;
        const int ntiles = upi * priv_tiles + (members >= 2 ? p.num_kv_heads * shared / kTileTokens : 0);
        int rb, tb, trec, ttiles;
        scan2(nrec, ntiles, &rb, &tb, &trec, &ttiles, wa, wb);
        const int r0 = carry_rec + rb, t0 = carry_tiles + tb;
        const int gtiles = members >= 2 ? shared / kTileTokens : 0;   // leader only
        const int pbase = t0 + p.num_kv_heads * gtiles;                  // first private tile
        if (valid && members >= 2) {
            p.ws.rec[r0] = make_int4(s | kGroupRecord, 0, shared, members);
            p.ws.rec_prefix[r0] = t0;
            if (r0 < kPlanSmemRecords) s_rp[r0] = t0;
        }
        s_first[tid] = members >= 2 ? t0 : -1;                 // reuse: group tile base
        __syncthreads();
        // members read their leader's entries: into registers before the rewrite
        const int lp = leader - base;
        const int my_gbase = leader >= 0 ? s_first[lp] : -1;
        const int my_gst = leader >= 0 ? s_sh[lp] / kTileTokens : 0;
        if (valid) {
            const int r = r0 + (members >= 2);
            p.ws.rec[r] = make_int4(s, start, ctx, my_gbase);
            p.ws.rec_prefix[r] = pbase;
            if (r < kPlanSmemRecords) s_rp[r] = pbase;
            p.ws.seq_info[s] = make_int4(priv_tiles, pbase, my_gbase, my_gst);
        }
        __syncthreads();
        // a batch of <= 1024 sequences keeps its per-sequence entries in shared memory
        s_run[tid] = priv_tiles;
        s_ctx[tid] = pbase;
        s_mem[tid] = my_gbase;
        s_sh[tid] = my_gst;
        __syncthreads();
        if (tid == 0) {
            carry_rec += trec;
            carry_tiles += ttiles;
        }
        __syncthreads();
    }
    const int nrec = carry_rec, total = carry_tiles;
    const int q = max(p.chunk_tokens / kTileTokens, (total + p.num_workers - 1) / p.num_workers);
    if (tid == 0) {
        p.ws.rec_prefix[nrec] = total;
        if (nrec <= kPlanSmemRecords) s_rp[nrec] = total;
        p.ws.quota[0] = q;
        p.ws.quota[1] = total;
    }
    const bool in_smem = p.num_seqs <= (int)blockDim.x;
    __syncthreads();
    // each worker's first record: the last record starting at or before its first
    // tile (binary search over the record prefix, in shared memory when it fits)
    const int* rp = nrec <= kPlanSmemRecords ? s_rp : p.ws.rec_prefix;
    for (int b = tid; b < p.num_workers; b += blockDim.x) {
        const int pos = b * q;
        if (pos >= total) break;
        int lo = 0, hi = nrec - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (rp[mid] <= pos) lo = mid;
            else hi = mid - 1;
        }
        p.ws.worker_first[2 * b] = make_int4(lo, rp[lo], rp[lo + 1], 0);
        p.ws.worker_first[2 * b + 1] = p.ws.rec[lo];
    }
    // sequences without context: zero output (no private and no shared tiles)
    const int rowlen = p.num_q_heads * p.head_dim;
    for (int s = tid >> 5; s < p.num_seqs; s += blockDim.x >> 5) {
        const bool empty = in_smem ? s_run[s] == 0 && s_sh[s] == 0 : p.ws.ctx_eff[s] == 0;
        if (!empty) continue;
        for (int i = tid & 31; i < rowlen; i += 32)
            store_from_float<QT>(p.out, (int64_t)s * rowlen + i, 0.f);
    }
}

// Merge of the partial states of up to 32 / LPR (sequence, query head) rows,
// LPR lanes per row (lane LPR*h + k holds slice k of d of row h): M = max m_c,
// L = sum l_c 2^(m_c - M), out = sum acc_c 2^(m_c - M) / L over the row's nseg
// states, in state order.  Lanes with row < 0 idle.  The states sit in L2,
// written by other CTAs: a batch of states is loaded at once, and a row with
// more states than a batch carries M forward batch by batch (the earlier sums
// rescaled by 2^(M_old - M_new)).
template <typename QT, int HD, int LPR>
__device__ __noinline__ void merge_rows_warp(const DecodeParams& p, int64_t row, int nseg,
                                             int lane) {
    constexpr int DQ = HD / LPR;               // dims per lane
    constexpr int NV = DQ / 4;                 // float4 per lane and state
    constexpr int NB = NV >= 8 ? 2 : 16 / NV;  // states per batch (<= 16 float4 in flight)
    if (row < 0) return;
    const int k = lane % LPR;
    const float* pm = p.ws.pm + row * p.part_stride;
    const float* pl = p.ws.pl + row * p.part_stride;
    const float4* pa = reinterpret_cast<const float4*>(p.ws.pacc + row * p.part_stride * HD) +
                       k * NV;
    float M = -INFINITY, L = 0.f;
    float4 A[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) A[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int c0 = 0; c0 < nseg; c0 += NB) {
        float mb[NB], lb[NB];
        float4 v[NB][NV];
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            const bool in = c0 + b < nseg;
            mb[b] = in ? __ldcg(pm + c0 + b) : -INFINITY;
            lb[b] = in ? __ldcg(pl + c0 + b) : 0.f;
#pragma unroll
            for (int i = 0; i < NV; ++i)
                v[b][i] = in ? __ldcg(pa + (int64_t)(c0 + b) * (HD / 4) + i)
                             : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        float Mn = M;
#pragma unroll
        for (int b = 0; b < NB; ++b) Mn = fmaxf(Mn, mb[b]);
        if (Mn == -INFINITY) continue;
        if (M != Mn && M != -INFINITY) {
            const float r = fast_exp2(M - Mn);
            L *= r;
#pragma unroll
            for (int i = 0; i < NV; ++i) {
                A[i].x *= r; A[i].y *= r; A[i].z *= r; A[i].w *= r;
            }
        }
        M = Mn;
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            const float f = mb[b] == -INFINITY ? 0.f : fast_exp2(mb[b] - M);
            L = fmaf(lb[b], f, L);
#pragma unroll
            for (int i = 0; i < NV; ++i) {
                A[i].x = fmaf(v[b][i].x, f, A[i].x);
                A[i].y = fmaf(v[b][i].y, f, A[i].y);
                A[i].z = fmaf(v[b][i].z, f, A[i].z);
                A[i].w = fmaf(v[b][i].w, f, A[i].w);
            }
        }
    }
    const float inv = L > 0.f ? p.out_scale / L : 0.f;
    const int64_t o0 = row * HD + k * DQ;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        store_from_float<QT>(p.out, o0 + 4 * i + 0, A[i].x * inv);
        store_from_float<QT>(p.out, o0 + 4 * i + 1, A[i].y * inv);
        store_from_float<QT>(p.out, o0 + 4 * i + 2, A[i].z * inv);
        store_from_float<QT>(p.out, o0 + 4 * i + 3, A[i].w * inv);
    }
}

// The merge of the nh (<= 8) heads of one unit by a warp: 8 lanes per row when
// the unit has at most 4 heads, else 4.
template <typename QT, int HD>
__device__ __forceinline__ void merge_unit_warp(const DecodeParams& p, int64_t row0, int nh,
                                                int nseg, int lane) {
    if (nh <= 4) {
        const int h = lane >> 3;
        merge_rows_warp<QT, HD, 8>(p, h < nh ? row0 + h : -1, nseg, lane);
    } else {
        const int h = lane >> 2;
        merge_rows_warp<QT, HD, 4>(p, h < nh ? row0 + h : -1, nseg, lane);
    }
}

// Grouped (prefix-aware) launches: after the decode kernel, one warp per
// (sequence, unit) merges the unit's partial states -- its group's shared
// segments, then its private ones, in that order -- all units in parallel.
// Ungrouped units whose context fits one segment were written directly.
template <typename QT, int HD>
__global__ void __launch_bounds__(256) merge_units_kernel(DecodeParams p) {
    pdl_wait();                                           // every partial state is written
    const int upi = p.num_kv_heads * p.nsub;
    const int w = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (w >= p.num_seqs * upi) return;
    const int s = w / upi, u = w % upi;
    const int q = p.ws.quota[0];
    const int4 si = p.ws.seq_info[s];   // {private tiles, first private tile, group base, group tiles}
    int np = 0, ns = 0;
    if (si.x > 0) {
        const int us = si.y + u * si.x;
        np = (us + si.x - 1) / q - us / q + 1;
    }
    if (si.z >= 0) {
        const int gs = si.z + u * si.w;
        ns = (gs + si.w - 1) / q - gs / q + 1;
    }
    const int nseg = ns + np;
    if (nseg == 0 || (si.z < 0 && nseg == 1)) return;
    const int kvh = u / p.nsub, qsub = u % p.nsub;
    const int nh = min(kMmaHeadsPerItem, p.group - qsub * kMmaHeadsPerItem);
    merge_unit_warp<QT, HD>(p, (int64_t)s * p.num_q_heads + kvh * p.group +
                                   qsub * kMmaHeadsPerItem, nh, nseg, lane);
}

// ------------------------------------------------------------ work windows --

// One window of a worker's range: at most 64 blocks of one unit.
struct Window {
    int valid;
    int group;                  // a shared-prefix unit (else a private one)
    int s;                      // sequence whose table row is read (a group's leader)
    int kvh, qsub, nh;          // kv head, head subgroup, query heads served
    int members;                // sequences served (1 for a private unit)
    int seg;                    // segment index within the unit
    int expect, segoff;         // private unit: partial states merged, first private one
    int t0, t1;                 // logical tokens [t0, t1)
    int first, last;            // first / last window of the segment
};

// The record a producer is currently walking.
struct RecCursor {
    int r, lo, hi;              // record index, its tile range [lo, hi)
    int group, id, start, end;  // kind, sequence / leader, token range [start, end)
    int members;                // sequences served
    int gbase;                  // private record: first tile of its group's record, or -1
};

__device__ __forceinline__ void rec_set(RecCursor& rc, int lo, int hi, int4 e) {
    rc.lo = lo;
    rc.hi = hi;
    rc.group = (e.x & kGroupRecord) != 0;
    rc.id = e.x & (kGroupRecord - 1);
    rc.start = e.y;
    rc.end = e.z;
    rc.members = rc.group ? e.w : 1;
    rc.gbase = rc.group ? -1 : e.w;
}

__device__ __forceinline__ void rec_load(const DecodeParams& p, RecCursor& rc) {
    rec_set(rc, __ldcg(&p.ws.rec_prefix[rc.r]), __ldcg(&p.ws.rec_prefix[rc.r + 1]),
            __ldcg(&p.ws.rec[rc.r]));
}

// The window starting at flattened tile `pos` of a worker whose range is
// [a, end); `rc` advances in place to the record holding `pos` (global loads
// only when the record changes).
__device__ __forceinline__ Window make_window(const DecodeParams& p, int worker, int a, int end,
                                              int q, int pos, RecCursor& rc) {
    Window w{};
    if (pos >= end) return w;
    while (rc.hi <= pos) {
        ++rc.r;
        rec_load(p, rc);
    }
    const int tiles = (rc.end - rc.start + kTileTokens - 1) / kTileTokens;
    const int rel = pos - rc.lo;
    const int u = rel / tiles, tile = rel % tiles;
    const int ustart = pos - tile, uend = ustart + tiles;
    const int wt = min(min(p.block_size, uend - pos), end - pos);   // <= 64 blocks
    w.valid = 1;
    w.group = rc.group;
    w.s = rc.id;
    w.members = rc.members;
    if (rc.group) {
        w.kvh = u;
        w.qsub = 0;
        w.nh = rc.members * p.group;
        w.expect = -1;                           // per member: read at the segment's end
        w.segoff = 0;                            // shared segments come first
    } else {
        w.kvh = u / p.nsub;
        w.qsub = u % p.nsub;
        w.nh = min(kMmaHeadsPerItem, p.group - w.qsub * kMmaHeadsPerItem);
        // segments of this unit's group record (one unit per kv head), then its own
        int ns = 0;
        if (rc.gbase >= 0) {
            const int gst = rc.start / kTileTokens;
            const int gs = rc.gbase + u * gst;
            ns = (gs + gst - 1) / q - gs / q + 1;
        }
        w.segoff = ns;
        w.expect = ns + (uend - 1) / q - ustart / q + 1;
    }
    w.seg = worker - ustart / q;
    w.t0 = rc.start + tile * kTileTokens;
    w.t1 = min(rc.start + (tile + wt) * kTileTokens, rc.end);
    w.first = pos == a || pos == ustart;
    w.last = pos + wt == end || pos + wt == uend;
    return w;
}

// Sequence and query head of head slot j of a window's unit.
__device__ __forceinline__ void slot_head(const DecodeParams& p, int group, int s, int kvh,
                                          int qsub, int j, int* seq, int* qhead) {
    if (group) {
        *seq = s + j / p.group;
        *qhead = kvh * p.group + j % p.group;
    } else {
        *seq = s;
        *qhead = kvh * p.group + qsub * kMmaHeadsPerItem + j;
    }
}

// --------------------------------------------------------------------- kernel --

template <typename QT, typename KT, int HD, int NT>
__global__ void __launch_bounds__(32 * (NT + 1), 4) decode_mma_kernel(DecodeParams p,
                                                        const __grid_constant__ CUtensorMap tmK,
                                                        const __grid_constant__ CUtensorMap tmV) {
    using Cfg = MmaCfg<QT, KT, HD, NT>;
    using MT = typename Cfg::MT;
    constexpr int TPS = Cfg::TPS;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    StageMeta* metas = reinterpret_cast<StageMeta*>(smem + Cfg::OFF_METAS);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + Cfg::OFF_BARS);
    uint64_t* empty = full + Cfg::NSTAGE;
    uint64_t* xfull = empty + Cfg::NSTAGE;    // consumer 1's state is in the exchange buffer
    uint64_t* xempty = xfull + 1;             // consumer 0 has read it
    float* xbuf = reinterpret_cast<float*>(smem + Cfg::OFF_XCH);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < Cfg::NSTAGE; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], Cfg::NC);
        }
        mbar_init(xfull, 1);
        mbar_init(xempty, 1);
        fence_mbar_init();
        mbar_arrive(xempty);                  // the buffer starts free (phase 0 complete)
    }
    __syncthreads();

    const int B = p.block_size;
    pdl_wait();                                           // the planning kernel has completed
    const int q = p.ws.quota[0], total = p.ws.quota[1];   // written by the planning kernel
    const int a = blockIdx.x * q, end = min(a + q, total);

    if (warp == Cfg::NC) {
        // ======================= producer warp =======================
        if (lane == 0) {
            prefetch_tensormap(&tmK);
            prefetch_tensormap(&tmV);
        }
        const uint64_t policy = l2_evict_first_policy();
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        RecCursor rc{};
        if (a < end) {
            // the planner stored this worker's first record beside its index
            const int4 wf = __ldcg(&p.ws.worker_first[2 * blockIdx.x]);
            const int4 e = __ldcg(&p.ws.worker_first[2 * blockIdx.x + 1]);
            rc.r = wf.x;
            rec_set(rc, wf.y, wf.z, e);
        }
        Window win = make_window(p, blockIdx.x, a, end, q, a, rc);
        int pos = a;
        int e0 = 0, e1 = 0;
        if (win.valid) {
            const int32_t* trow = p.block_tables + (int64_t)win.s * p.max_blocks;
            const int jb0 = win.t0 / B, nb = (win.t1 + B - 1) / B - jb0;
            e0 = lane < nb ? trow[jb0 + lane] : 0;
            e1 = lane + 32 < nb ? trow[jb0 + lane + 32] : 0;
        }
        while (win.valid && ok) {
            const int wtiles = (win.t1 - win.t0 + kTileTokens - 1) / kTileTokens;
            Window nxt{};
            int n0 = 0, n1 = 0;
            const int jb0 = win.t0 / B, nb = (win.t1 + B - 1) / B - jb0;
            if ((lane < nb && (e0 < 0 || e0 >= p.num_blocks)) ||
                (lane + 32 < nb && (e1 < 0 || e1 >= p.num_blocks))) {
                set_status(p.status, PKV_DEV_BAD_BLOCK_ID);
                if (e0 < 0 || e0 >= p.num_blocks) e0 = 0;
                if (e1 < 0 || e1 >= p.num_blocks) e1 = 0;
            }
            const int nstages = (win.t1 - win.t0 + TPS - 1) / TPS;
            for (int st = 0; st < nstages; ++st) {
                const int ts = win.t0 + st * TPS, te = min(ts + TPS, win.t1);
                const bool first = win.first && st == 0;
                if (!mbar_wait(&empty[stage], phase ^ 1u)) {
                    set_status(p.status, PKV_DEV_WAIT_TIMEOUT);
                    ok = false;
                    break;
                }
                uint8_t* sbase = smem + (size_t)stage * Cfg::STAGE_BYTES;
                const int fb = ts / B, nblk = (te - 1) / B - fb + 1;   // whole blocks
                const uint32_t qbytes = Cfg::QSTAGE && first ? (uint32_t)(win.nh * HD * 2) : 0u;
                if (lane == 0) {
                    StageMeta& m = metas[stage];
                    m.s = win.s; m.kvh = win.kvh; m.qsub = win.qsub; m.nh = win.nh;
                    m.chunk = win.seg; m.nchunks = win.members; m.ts = ts; m.te = te;
                    m.expect = win.expect; m.segoff = win.segoff;
                    m.flags = (first ? kFirst : 0) | (win.last && st == nstages - 1 ? kLast : 0) |
                              (win.group ? kGroup : 0);
                    mbar_arrive_expect_tx(&full[stage],
                                          2u * (uint32_t)(nblk * B) * Cfg::ROWB + qbytes);
                }
                __syncwarp();
                const int rel = fb + lane - jb0;
                const int pa = __shfl_sync(0xffffffffu, e0, rel & 31);
                const int pb = __shfl_sync(0xffffffffu, e1, rel & 31);
                if (lane < nblk) {
                    const int phys = rel < 32 ? pa : pb;
                    const int y = (phys * p.num_kv_heads + win.kvh) * B;
                    const int row0 = lane * B;                       // stage row of the block
#pragma unroll
                    for (int h = 0; h < Cfg::HALVES; ++h) {
                        const int x = h * Cfg::ELEMS_PER_SLICE;
                        tma_load_2d(sbase + h * Cfg::HALF_BYTES + row0 * 128, &tmK, x, y,
                                    &full[stage], policy);
                        tma_load_2d(sbase + Cfg::KV_BYTES + h * Cfg::HALF_BYTES + row0 * 128,
                                    &tmV, x, y, &full[stage], policy);
                    }
                }
                if (qbytes) {
                    // the segment's query rows in head-slot order: a private unit's heads
                    // are one contiguous run; a group's are G rows of each member
                    if (win.group) {
                        if (lane < win.members) {
                            const int64_t qoff =
                                ((int64_t)(win.s + lane) * p.num_q_heads + win.kvh * p.group) * HD * 2;
                            bulk_g2s(sbase + 2 * Cfg::KV_BYTES + lane * p.group * HD * 2,
                                     (const uint8_t*)p.q + qoff, (uint32_t)(p.group * HD * 2),
                                     &full[stage]);
                        }
                    } else if (lane == 31) {
                        const int h0 = win.kvh * p.group + win.qsub * kMmaHeadsPerItem;
                        const int64_t qoff = ((int64_t)win.s * p.num_q_heads + h0) * HD * 2;
                        bulk_g2s(sbase + 2 * Cfg::KV_BYTES, (const uint8_t*)p.q + qoff, qbytes,
                                 &full[stage]);
                    }
                }
                if (++stage == Cfg::NSTAGE) { stage = 0; phase ^= 1u; }
                if (st == 0) {
                    // look one window ahead once this window's first stage is in flight:
                    // its block-table entries load while this window streams
                    nxt = make_window(p, blockIdx.x, a, end, q, pos + wtiles, rc);
                    if (nxt.valid) {
                        const int32_t* trow = p.block_tables + (int64_t)nxt.s * p.max_blocks;
                        const int nj0 = nxt.t0 / B, nnb = (nxt.t1 + B - 1) / B - nj0;
                        n0 = lane < nnb ? trow[nj0 + lane] : 0;
                        n1 = lane + 32 < nnb ? trow[nj0 + lane + 32] : 0;
                    }
                }
            }
            pos += wtiles;
            win = nxt;
            e0 = n0;
            e1 = n1;
        }
        if (ok) {
            if (mbar_wait(&empty[stage], phase ^ 1u)) {
                if (lane == 0) {
                    metas[stage].flags = kDone;
                    mbar_arrive(&full[stage]);
                }
            } else {
                set_status(p.status, PKV_DEV_WAIT_TIMEOUT);
            }
        }
        return;
    }

    // ========================= consumer warps =========================
    // Consumer cw takes m-tiles cw*MTC .. cw*MTC+MTC-1 (16 tokens each) of every stage
    // for all n-tiles, with its own running state; with two consumers, consumer 1
    // hands its state to consumer 0 at the end of each segment and consumer 0 merges
    // the two (the rescale of the running-max recurrence) and finishes the segment.
    constexpr int MTC = Cfg::MTC;
    const int cw = warp;
    const bool grp_launch = p.allow_groups != 0;   // merges left to the merge kernel
    const int g = lane >> 2, c = lane & 3;
    uint32_t qf[NT][Cfg::KSTEPS][2];   // Q^T B fragments, n-tile nt = head slots 8nt..8nt+7
    float o[Cfg::MTILES][NT][4];       // O^T C fragments, rows mapped to d by d_row()
    float m0[NT], m1[NT], l0[NT], l1[NT];
    int stage = 0;
    uint32_t phase = 0;
    uint32_t xphase = 0;               // exchange barrier parity (each consumer its own)
    int nt_live = 1;
    bool ok = true;
    // d index of C-fragment row g (half 0) or g + 8 (half 1) of P.V m-tile mt
    auto d_row = [&](int mt, int half) -> int {
        if constexpr (Cfg::FP8) return 32 * (mt >> 1) + 2 * g + (mt & 1) + 16 * half;
        else return 16 * mt + g + 8 * half;
    };

    while (ok) {
        if (!mbar_wait(&full[stage], phase)) {
            set_status(p.status, PKV_DEV_WAIT_TIMEOUT);
            break;
        }
        const StageMeta meta = metas[stage];
        if (meta.flags & kDone) break;
        uint8_t* sbase = smem + (size_t)stage * Cfg::STAGE_BYTES;
        const uint32_t sK = smem_addr(sbase);
        const uint32_t sV = sK + Cfg::KV_BYTES;

        if (meta.flags & kFirst) {
            // Q^T fragments: from the stage (rows staged by the producer) or, in the
            // 16-head kernel over 16-bit K/V at head_dim 128, from global memory
            const uint32_t* qg = static_cast<const uint32_t*>(p.q);
            if constexpr (Cfg::QSTAGE) qg = reinterpret_cast<const uint32_t*>(sbase + 2 * Cfg::KV_BYTES);
            nt_live = meta.nh > 8 ? 2 : 1;
            const bool grp = (meta.flags & kGroup) != 0;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int hs = nt * 8 + g;                 // head slot of this lane's n column
                const bool live = hs < meta.nh;
                int seq = 0, qh = 0;
                slot_head(p, grp, meta.s, meta.kvh, meta.qsub, live ? hs : 0, &seq, &qh);
                const int64_t rowq = Cfg::QSTAGE ? (int64_t)hs * HD                  // staged rows
                                                 : ((int64_t)seq * p.num_q_heads + qh) * HD;
#pragma unroll
                for (int t = 0; t < Cfg::KSTEPS; ++t) {
                    if constexpr (Cfg::FP8) {
                        qf[nt][t][0] = live ? q_pair<QT, MT>(qg[(rowq + 16 * t + 4 * c) >> 1]) : 0u;
                        qf[nt][t][1] = live ? q_pair<QT, MT>(qg[(rowq + 16 * t + 4 * c + 2) >> 1]) : 0u;
                    } else {
                        qf[nt][t][0] = live ? qg[(rowq + 16 * t + 2 * c) >> 1] : 0u;
                        qf[nt][t][1] = live ? qg[(rowq + 16 * t + 8 + 2 * c) >> 1] : 0u;
                    }
                }
#pragma unroll
                for (int mt = 0; mt < Cfg::MTILES; ++mt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) o[mt][nt][e] = 0.f;
                m0[nt] = m1[nt] = -INFINITY;
                l0[nt] = l1[nt] = 0.f;
            }
        }

        const int nvalid = meta.te - meta.ts;            // 1..32
        const int r_lo = cw * MTC * 16;                  // this consumer's stage rows
        const int r_hi = r_lo + MTC * 16;
        const bool mine = nvalid > r_lo;                 // its m-tiles hold tokens
        if (mine && nvalid < r_hi) {
            // its rows past the context: stale or poisoned -> zero V (P is 0 there)
            const int zrows = r_hi - nvalid;
            for (int i = lane; i < zrows * Cfg::HALVES * 8; i += 32) {
                const int r = nvalid + i / (Cfg::HALVES * 8);
                const int h = (i / 8) % Cfg::HALVES, ch = i % 8;
                *reinterpret_cast<uint4*>(sbase + Cfg::KV_BYTES + h * Cfg::HALF_BYTES + r * 128 +
                                          ch * 16) = make_uint4(0u, 0u, 0u, 0u);
            }
            fence_proxy_async_smem();
            __syncwarp();
        }
        if (mine) {
        // ---- S^T = K . Q^T: this consumer's (up to) MTC 16-token m-tiles x NT n-tiles ----
        float sa[MTC][NT][4];
#pragma unroll
        for (int mi = 0; mi < MTC; ++mi)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) sa[mi][nt][e] = 0.f;
        {
            const int rl = (lane & 7) + ((lane >> 3) & 1) * 8;
            if constexpr (Cfg::FP8) {
#pragma unroll
                for (int pr = 0; pr < Cfg::KSTEPS / 2; ++pr) {
                    const int chunk = 2 * pr + (lane >> 4);
#pragma unroll
                    for (int mi = 0; mi < MTC; ++mi) {
                        const int mt = cw * MTC + mi;
                        if (mi > 0 && mt * 16 >= nvalid) break;
                        uint32_t r[4];
                        ldsm_x4(sK + swz(16 * mt + rl, chunk), r);
#pragma unroll
                        for (int k = 0; k < 2; ++k) {
                            const uint32_t lo = r[2 * k], hi = r[2 * k + 1];
                            const uint32_t a[4] = {e4m3x2_to_f16x2(lo & 0xffffu),
                                                   e4m3x2_to_f16x2(hi & 0xffffu),
                                                   e4m3x2_to_f16x2(lo >> 16),
                                                   e4m3x2_to_f16x2(hi >> 16)};
#pragma unroll
                            for (int nt = 0; nt < NT; ++nt)
                                if (NT == 1 || nt < nt_live)
                                    Mma<MT>::run(sa[mi][nt], a, qf[nt][2 * pr + k][0],
                                                 qf[nt][2 * pr + k][1]);
                        }
                    }
                }
            } else {
#pragma unroll
                for (int t = 0; t < Cfg::KSTEPS; ++t) {
                    const int half = t >> 2, chunk = (t & 3) * 2 + (lane >> 4);
                    const uint32_t base = sK + half * Cfg::HALF_BYTES;
#pragma unroll
                    for (int mi = 0; mi < MTC; ++mi) {
                        const int mt = cw * MTC + mi;
                        if (mi > 0 && mt * 16 >= nvalid) break;
                        uint32_t a[4];
                        ldsm_x4(base + swz(16 * mt + rl, chunk), a);
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt)
                            if (NT == 1 || nt < nt_live) Mma<MT>::run(sa[mi][nt], a, qf[nt][t][0], qf[nt][t][1]);
                    }
                }
            }
        }
        // ---- online softmax over the stage's tokens, per n-tile ----
        uint32_t pb[MTC][NT][2];   // P^T B fragments: k-step (this consumer's m-tiles) x n-tile
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            if (NT > 1 && nt >= nt_live) break;
            float x[MTC][4];
#pragma unroll
            for (int mi = 0; mi < MTC; ++mi) {
                const int mt = cw * MTC + mi;
                const bool va = mt * 16 + g < nvalid, vb = mt * 16 + g + 8 < nvalid;
                x[mi][0] = va ? sa[mi][nt][0] * p.qk_scale_log2 : -INFINITY;
                x[mi][1] = va ? sa[mi][nt][1] * p.qk_scale_log2 : -INFINITY;
                x[mi][2] = vb ? sa[mi][nt][2] * p.qk_scale_log2 : -INFINITY;
                x[mi][3] = vb ? sa[mi][nt][3] * p.qk_scale_log2 : -INFINITY;
            }
            float mx0 = fmaxf(x[0][0], x[0][2]);
            float mx1 = fmaxf(x[0][1], x[0][3]);
#pragma unroll
            for (int mi = 1; mi < MTC; ++mi) {
                mx0 = fmaxf(mx0, fmaxf(x[mi][0], x[mi][2]));
                mx1 = fmaxf(mx1, fmaxf(x[mi][1], x[mi][3]));
            }
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
            }
            const bool n0 = mx0 > m0[nt] + kRescaleSlack, n1 = mx1 > m1[nt] + kRescaleSlack;
            if (__any_sync(0xffffffffu, n0 || n1)) {
                const float r0 = n0 ? fast_exp2(m0[nt] - mx0) : 1.f;
                const float r1 = n1 ? fast_exp2(m1[nt] - mx1) : 1.f;
                if (n0) m0[nt] = mx0;
                if (n1) m1[nt] = mx1;
                l0[nt] *= r0;
                l1[nt] *= r1;
#pragma unroll
                for (int mt = 0; mt < Cfg::MTILES; ++mt) {
                    o[mt][nt][0] *= r0;
                    o[mt][nt][2] *= r0;
                    o[mt][nt][1] *= r1;
                    o[mt][nt][3] *= r1;
                }
            }
#pragma unroll
            for (int mi = 0; mi < MTC; ++mi) {
                float f0, f1, f2, f3;
                const uint32_t p01 = Mma<MT>::pack(fast_exp2(x[mi][0] - m0[nt]),
                                                   fast_exp2(x[mi][1] - m1[nt]), f0, f1);
                const uint32_t p23 = Mma<MT>::pack(fast_exp2(x[mi][2] - m0[nt]),
                                                   fast_exp2(x[mi][3] - m1[nt]), f2, f3);
                l0[nt] += f0 + f2;
                l1[nt] += f1 + f3;
                pb[mi][nt][0] = movmatrix_trans(p01);
                pb[mi][nt][1] = movmatrix_trans(p23);
            }
        }
        // ---- O^T += V^T . P^T ----
        {
            const int mi_ = lane >> 3;
            const int rv = (lane & 7) + (mi_ >> 1) * 8;
            if constexpr (Cfg::FP8) {
#pragma unroll
                for (int pr = 0; pr < Cfg::MTILES / 2; ++pr) {
                    const int chunk = 2 * pr + (mi_ & 1);
#pragma unroll
                    for (int ki = 0; ki < MTC; ++ki) {
                        const int ks = cw * MTC + ki;
                        if (ki > 0 && ks * 16 >= nvalid) break;
                        uint32_t r[4];
                        ldsm_x4_trans(sV + swz(16 * ks + rv, chunk), r);
                        uint32_t ev[4], od[4];
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            ev[k] = e4m3x2_to_f16x2(__byte_perm(r[k], 0u, 0x0020));
                            od[k] = e4m3x2_to_f16x2(__byte_perm(r[k], 0u, 0x0031));
                        }
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            if (NT > 1 && nt >= nt_live) break;
                            Mma<MT>::run(o[2 * pr][nt], ev, pb[ki][nt][0], pb[ki][nt][1]);
                            Mma<MT>::run(o[2 * pr + 1][nt], od, pb[ki][nt][0], pb[ki][nt][1]);
                        }
                    }
                }
            } else {
#pragma unroll
                for (int mt = 0; mt < Cfg::MTILES; ++mt) {
                    const int half = mt >> 2, chunk = (mt & 3) * 2 + (mi_ & 1);
                    const uint32_t base = sV + half * Cfg::HALF_BYTES;
#pragma unroll
                    for (int ki = 0; ki < MTC; ++ki) {
                        const int ks = cw * MTC + ki;
                        if (ki > 0 && ks * 16 >= nvalid) break;
                        uint32_t a[4];
                        ldsm_x4_trans(base + swz(16 * ks + rv, chunk), a);
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt)
                            if (NT == 1 || nt < nt_live)
                                Mma<MT>::run(o[mt][nt], a, pb[ki][nt][0], pb[ki][nt][1]);
                    }
                }
            }
        }
        }   // mine
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[stage]);
        if (++stage == Cfg::NSTAGE) { stage = 0; phase ^= 1u; }

        if (!(meta.flags & kLast)) continue;

        // ---------------- end of the segment ----------------
        if constexpr (Cfg::NC > 1) {
            // consumer 1 -> consumer 0, one n-tile per round, through the exchange buffer
            // (lane-interleaved: value i of lane l at xbuf[32 i + l], no bank conflicts)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                if (nt >= nt_live) break;
                if (!mbar_wait(cw == 1 ? xempty : xfull, xphase)) {
                    set_status(p.status, PKV_DEV_WAIT_TIMEOUT);
                    ok = false;
                    break;
                }
                xphase ^= 1u;
                if (cw == 1) {
#pragma unroll
                    for (int mt = 0; mt < Cfg::MTILES; ++mt)
#pragma unroll
                        for (int e = 0; e < 4; ++e) xbuf[32 * (4 * mt + e) + lane] = o[mt][nt][e];
                    xbuf[32 * (Cfg::MTILES * 4 + 0) + lane] = m0[nt];
                    xbuf[32 * (Cfg::MTILES * 4 + 1) + lane] = m1[nt];
                    xbuf[32 * (Cfg::MTILES * 4 + 2) + lane] = l0[nt];
                    xbuf[32 * (Cfg::MTILES * 4 + 3) + lane] = l1[nt];
                    __syncwarp();
                    if (lane == 0) mbar_arrive(xfull);
                } else {
                    const float mb0 = xbuf[32 * (Cfg::MTILES * 4 + 0) + lane];
                    const float mb1 = xbuf[32 * (Cfg::MTILES * 4 + 1) + lane];
                    const float lb0 = xbuf[32 * (Cfg::MTILES * 4 + 2) + lane];
                    const float lb1 = xbuf[32 * (Cfg::MTILES * 4 + 3) + lane];
                    // every lane of a head column holds the same m; a side that saw no
                    // token of the segment has m = -inf and contributes nothing
                    const float M0 = fmaxf(m0[nt], mb0), M1 = fmaxf(m1[nt], mb1);
                    const float ra0 = m0[nt] == -INFINITY ? 0.f : fast_exp2(m0[nt] - M0);
                    const float rb0 = mb0 == -INFINITY ? 0.f : fast_exp2(mb0 - M0);
                    const float ra1 = m1[nt] == -INFINITY ? 0.f : fast_exp2(m1[nt] - M1);
                    const float rb1 = mb1 == -INFINITY ? 0.f : fast_exp2(mb1 - M1);
#pragma unroll
                    for (int mt = 0; mt < Cfg::MTILES; ++mt) {
                        o[mt][nt][0] = o[mt][nt][0] * ra0 + xbuf[32 * (4 * mt + 0) + lane] * rb0;
                        o[mt][nt][1] = o[mt][nt][1] * ra1 + xbuf[32 * (4 * mt + 1) + lane] * rb1;
                        o[mt][nt][2] = o[mt][nt][2] * ra0 + xbuf[32 * (4 * mt + 2) + lane] * rb0;
                        o[mt][nt][3] = o[mt][nt][3] * ra1 + xbuf[32 * (4 * mt + 3) + lane] * rb1;
                    }
                    l0[nt] = l0[nt] * ra0 + lb0 * rb0;
                    l1[nt] = l1[nt] * ra1 + lb1 * rb1;
                    m0[nt] = M0;
                    m1[nt] = M1;
                    __syncwarp();
                    if (lane == 0) mbar_arrive(xempty);
                }
            }
            if (!ok || cw != 0) continue;
        }
        const bool grp = (meta.flags & kGroup) != 0;
        const int upi = p.num_kv_heads * p.nsub;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            if (NT > 1 && nt >= nt_live) break;
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                l0[nt] += __shfl_xor_sync(0xffffffffu, l0[nt], off);
                l1[nt] += __shfl_xor_sync(0xffffffffu, l1[nt], off);
            }
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int j = nt * 8 + 2 * c + hh;        // head slot of this lane's column
                if (j >= meta.nh) continue;
                int seq, qh;
                slot_head(p, grp, meta.s, meta.kvh, meta.qsub, j, &seq, &qh);
                const int expect = grp ? 0 : meta.expect;   // grouped: always a partial state
                const int64_t sh = (int64_t)seq * p.num_q_heads + qh;
                const float lsum = hh ? l1[nt] : l0[nt];
                const float msum = hh ? m1[nt] : m0[nt];
                if (expect == 1) {
                    // this segment is the head's whole context: write the output
                    const float inv = lsum > 0.f ? p.out_scale / lsum : 0.f;
#pragma unroll
                    for (int mt = 0; mt < Cfg::MTILES; ++mt) {
                        store_from_float<QT>(p.out, sh * HD + d_row(mt, 0), o[mt][nt][hh] * inv);
                        store_from_float<QT>(p.out, sh * HD + d_row(mt, 1),
                                             o[mt][nt][2 + hh] * inv);
                    }
                } else {
                    const int idx = meta.segoff + meta.chunk;
                    const int64_t pi = sh * p.part_stride + idx;
#pragma unroll
                    for (int mt = 0; mt < Cfg::MTILES; ++mt) {
                        p.ws.pacc[pi * HD + d_row(mt, 0)] = o[mt][nt][hh];
                        p.ws.pacc[pi * HD + d_row(mt, 1)] = o[mt][nt][2 + hh];
                    }
                    if (g == 0) {
                        p.ws.pm[pi] = msum;
                        p.ws.pl[pi] = lsum;
                    }
                }
            }
        }
        if constexpr (Cfg::NC == 1) {
            // split units: lane i (< units served) arrives on unit i's counter once the
            // warp barrier has ordered every lane's partial-state stores before it;
            // units the segment covers whole need neither.  Grouped launches leave
            // every merge to the merge kernel (the two-consumer kernel serves only those).
            __syncwarp();
            if (grp_launch) continue;
            const int my_expect = meta.expect;
            bool last = false;
            if (lane == 0 && my_expect > 1) {
                const int unit = meta.s * upi + meta.kvh * p.nsub + meta.qsub;
                last = atom_add_acq_rel_gpu(&p.ws.unit_done[unit], 1u) == (unsigned)(my_expect - 1);
            }
            unsigned last_mask = __ballot_sync(0xffffffffu, last);
            if (last_mask) __syncwarp();   // the acquiring lane's view reaches the warp
            // the merge of the unit this warp finished last
            if (last_mask)
                merge_unit_warp<QT, HD>(p, (int64_t)meta.s * p.num_q_heads + meta.kvh * p.group +
                                               meta.qsub * kMmaHeadsPerItem, meta.nh, my_expect, lane);
        }
    }
}

}  // namespace pkv
