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

// 2-D TMA tile load global -> shared, completing on `bar`; (x, y) = (column, row).
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;"
        ::"r"(smem_addr(smem_dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y),
        "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Order this thread's generic-proxy shared-memory writes before later
// async-proxy (TMA) writes to the same bytes.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------------ config --

template <typename QT, typename KT, int HD>
struct MmaCfg {
    static constexpr bool FP8 = std::is_same<KT, E4M3>::value;
    using MT = typename std::conditional<FP8, F16, KT>::type;   // mma operand type
    static constexpr int HPI = kMmaHeadsPerItem;  // query heads per item (mma N = 8)
    static constexpr int TPS = 32;                // tokens per stage: two 16-token m-tiles
    static constexpr int ROWB = HD * KT::bytes;   // bytes of one K/V row
    static constexpr int HALVES = ROWB / 128;     // 128-byte column slices of a row
    static constexpr int ELEMS_PER_SLICE = 128 / KT::bytes;
    static constexpr int KSTEPS = HD / 16;        // mma k-steps of Q.K^T
    static constexpr int MTILES = HD / 16;        // mma m-tiles of P.V (over d)
    static constexpr int HALF_BYTES = TPS * 128;  // one 128-byte slice of a stage
    static constexpr int KV_BYTES = HALVES * HALF_BYTES;
    static constexpr int Q_BYTES = HPI * HD * 2;
    static constexpr int STAGE_BYTES = (2 * KV_BYTES + Q_BYTES + 1023) / 1024 * 1024;
    static constexpr int NSTAGE = FP8 ? 5 : (HD == 128 ? 3 : 5);
    static constexpr int THREADS = 64;            // consumer warp + producer warp
    static constexpr size_t OFF_METAS = (size_t)NSTAGE * STAGE_BYTES;
    static constexpr size_t OFF_BARS = OFF_METAS + NSTAGE * sizeof(StageMeta);
    static constexpr size_t SMEM = OFF_BARS + 2 * NSTAGE * sizeof(uint64_t) + 1024;
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

// Balanced-split planning (1 CTA x 1024 threads): clamp the context lengths,
// count tiles = ceil(ctx / 64) x (kv heads x subgroups) per sequence, prefix-
// sum them, pick the per-worker quota Q (at least one chunk of tokens), record
// each worker's first sequence, reset the unit counters and zero the outputs
// of empty sequences.
template <typename QT>
__global__ void __launch_bounds__(1024) plan_split_kernel(DecodeParams p) {
    __shared__ int warp_sums[32];
    __shared__ int carry;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int upi = p.num_kv_heads * p.nsub;
    if (tid == 0) carry = 0;
    for (int i = tid; i < p.num_seqs * upi; i += blockDim.x) p.ws.unit_done[i] = 0u;
    const int cap = min(p.max_context_len, p.max_blocks * p.block_size);
    __syncthreads();
    for (int base = 0; base < p.num_seqs; base += blockDim.x) {
        const int s = base + tid;
        int n = 0;
        if (s < p.num_seqs) {
            int ctx = p.context_lens[s];
            if (ctx < 0 || ctx > cap) {
                set_status(p.status, PKV_DEV_BAD_CONTEXT);
                ctx = ctx < 0 ? 0 : cap;
            }
            p.ws.ctx_eff[s] = ctx;
            n = (ctx + kTileTokens - 1) / kTileTokens * upi;
        }
        int x = n;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, off);
            if (lane >= off) x += y;
        }
        if (lane == 31) warp_sums[warp] = x;
        __syncthreads();
        if (warp == 0) {
            int v = lane < (int)(blockDim.x >> 5) ? warp_sums[lane] : 0;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, v, off);
                if (lane >= off) v += y;
            }
            warp_sums[lane] = v;
        }
        __syncthreads();
        const int incl = x + (warp > 0 ? warp_sums[warp - 1] : 0);
        if (s < p.num_seqs) p.ws.tile_prefix[s] = carry + incl - n;
        __syncthreads();
        if (tid == blockDim.x - 1) carry += incl;
        __syncthreads();
    }
    const int total = carry;
    const int min_q = p.chunk_tokens / kTileTokens;
    const int q = max(min_q, (total + p.num_workers - 1) / p.num_workers);
    if (tid == 0) {
        p.ws.tile_prefix[p.num_seqs] = total;
        *p.ws.quota = q;
    }
    // worker b starts at tile b*q: record the sequence holding that tile
    for (int s = tid; s < p.num_seqs; s += blockDim.x) {
        const int lo = p.ws.tile_prefix[s], hi = lo + (p.ws.ctx_eff[s] + kTileTokens - 1) /
                                                      kTileTokens * upi;
        for (int b = (lo + q - 1) / q; b * q < hi && b < p.num_workers; ++b)
            p.ws.worker_seq[b] = s;
    }
    const int row = p.num_q_heads * p.head_dim;
    for (int s = warp; s < p.num_seqs; s += blockDim.x >> 5) {
        if (p.ws.ctx_eff[s] != 0) continue;
        for (int i = lane; i < row; i += 32) store_from_float<QT>(p.out, (int64_t)s * row + i, 0.f);
    }
}

// The warp that finished the last segment of (sequence s, heads hq0..hq0+nh-1)
// merges the segment states in order: M = max m_c, L = sum l_c 2^(m_c - M),
// out = sum acc_c 2^(m_c - M) / L.  Lane i owns head i/4 and a quarter of d.
template <typename QT, int HD>
__device__ __noinline__ void merge_segments_warp(const DecodeParams& p, int s, int hq0, int nh,
                                                 int nseg, int lane) {
    constexpr int DQ = HD / 4;     // dims per lane: 32 or 16
    const int h = lane >> 2, q4 = lane & 3;
    if (h >= nh) return;
    const int64_t sh = (int64_t)s * p.num_q_heads + hq0 + h;
    const float* pm = p.ws.pm + sh * p.part_stride;
    const float* pl = p.ws.pl + sh * p.part_stride;
    const float4* pa = reinterpret_cast<const float4*>(p.ws.pacc + sh * p.part_stride * HD + q4 * DQ);
    float M = -INFINITY;
    for (int c = 0; c < nseg; ++c) M = fmaxf(M, __ldcg(pm + c));
    float L = 0.f;
    float4 A[DQ / 4];
#pragma unroll
    for (int k = 0; k < DQ / 4; ++k) A[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int c = 0; c < nseg; ++c) {
        const float mc = __ldcg(pm + c);
        const float f = mc == -INFINITY ? 0.f : fast_exp2(mc - M);
        L = fmaf(__ldcg(pl + c), f, L);
        float4 v[DQ / 4];
#pragma unroll
        for (int k = 0; k < DQ / 4; ++k) v[k] = __ldcg(pa + (int64_t)c * (HD / 4) + k);
#pragma unroll
        for (int k = 0; k < DQ / 4; ++k) {
            A[k].x = fmaf(v[k].x, f, A[k].x);
            A[k].y = fmaf(v[k].y, f, A[k].y);
            A[k].z = fmaf(v[k].z, f, A[k].z);
            A[k].w = fmaf(v[k].w, f, A[k].w);
        }
    }
    const float inv = L > 0.f ? p.out_scale / L : 0.f;
    const int64_t o0 = sh * HD + q4 * DQ;
#pragma unroll
    for (int k = 0; k < DQ / 4; ++k) {
        store_from_float<QT>(p.out, o0 + 4 * k + 0, A[k].x * inv);
        store_from_float<QT>(p.out, o0 + 4 * k + 1, A[k].y * inv);
        store_from_float<QT>(p.out, o0 + 4 * k + 2, A[k].z * inv);
        store_from_float<QT>(p.out, o0 + 4 * k + 3, A[k].w * inv);
    }
}

// One window of a worker's range: at most 64 blocks of one unit.
struct Window {
    int valid;
    int s, kvh, qsub, nh;
    int seg, nseg;              // segment index within the unit, segments of the unit
    int t0, t1;                 // logical tokens [t0, t1)
    int first, last;            // first / last window of the segment
};

// The sequence a producer is currently walking: its tile range [lo, hi) in
// the flattened (unit, tile) order and its context length.
struct SeqCursor {
    int s, lo, hi, ctx;
};

__device__ __forceinline__ void seq_load(const DecodeParams& p, SeqCursor& sc) {
    sc.lo = __ldcg(&p.ws.tile_prefix[sc.s]);
    sc.hi = __ldcg(&p.ws.tile_prefix[sc.s + 1]);
    sc.ctx = __ldcg(&p.ws.ctx_eff[sc.s]);
}

// The window starting at flattened tile `pos` of a worker whose range is
// [a, end); `sc` advances in place to the sequence holding `pos` (global
// loads only when the sequence changes).
__device__ __forceinline__ Window make_window(const DecodeParams& p, int worker, int a, int end,
                                              int q, int pos, SeqCursor& sc) {
    Window w{};
    if (pos >= end) return w;
    while (sc.hi <= pos) {
        ++sc.s;
        seq_load(p, sc);
    }
    const int tiles = (sc.ctx + kTileTokens - 1) / kTileTokens;
    const int rel = pos - sc.lo;
    const int u = rel / tiles, tile = rel % tiles;
    const int ustart = pos - tile, uend = ustart + tiles;
    const int wt = min(min(p.block_size, uend - pos), end - pos);   // <= 64 blocks
    w.valid = 1;
    w.s = sc.s;
    w.kvh = u / p.nsub;
    w.qsub = u % p.nsub;
    w.nh = min(kMmaHeadsPerItem, p.group - w.qsub * kMmaHeadsPerItem);
    w.seg = worker - ustart / q;
    w.nseg = (uend - 1) / q - ustart / q + 1;
    w.t0 = tile * kTileTokens;
    w.t1 = min((tile + wt) * kTileTokens, sc.ctx);
    w.first = pos == a || pos == ustart;
    w.last = pos + wt == end || pos + wt == uend;
    return w;
}

template <typename QT, typename KT, int HD>
__global__ void __launch_bounds__(64, 4) decode_mma_kernel(DecodeParams p,
                                                        const __grid_constant__ CUtensorMap tmK,
                                                        const __grid_constant__ CUtensorMap tmV) {
    using Cfg = MmaCfg<QT, KT, HD>;
    using MT = typename Cfg::MT;
    constexpr int HPI = Cfg::HPI, TPS = Cfg::TPS;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    StageMeta* metas = reinterpret_cast<StageMeta*>(smem + Cfg::OFF_METAS);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + Cfg::OFF_BARS);
    uint64_t* empty = full + Cfg::NSTAGE;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < Cfg::NSTAGE; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        fence_mbar_init();
    }
    __syncthreads();

    const int B = p.block_size;
    const int q = *p.ws.quota;
    const int total = p.ws.tile_prefix[p.num_seqs];
    const int a = blockIdx.x * q, end = min(a + q, total);

    if (warp == 1) {
        // ======================= producer warp =======================
        if (lane == 0) {
            prefetch_tensormap(&tmK);
            prefetch_tensormap(&tmV);
        }
        const uint64_t policy = l2_evict_first_policy();
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        SeqCursor sc{a < end ? p.ws.worker_seq[blockIdx.x] : 0, 0, 0, 0};
        if (a < end) seq_load(p, sc);
        Window win = make_window(p, blockIdx.x, a, end, q, a, sc);
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
            const int h0 = win.kvh * p.group + win.qsub * HPI;
            const int nstages = (win.t1 - win.t0 + TPS - 1) / TPS;
            for (int st = 0; st < nstages; ++st) {
                const int ts = win.t0 + st * TPS, te = min(ts + TPS, win.t1);
                if (!mbar_wait(&empty[stage], phase ^ 1u)) {
                    set_status(p.status, PKV_DEV_WAIT_TIMEOUT);
                    ok = false;
                    break;
                }
                uint8_t* sbase = smem + (size_t)stage * Cfg::STAGE_BYTES;
                const int fb = ts / B, nblk = (te - 1) / B - fb + 1;   // whole blocks
                const bool qstage = win.first && st == 0;
                const uint32_t qbytes = qstage ? (uint32_t)(win.nh * HD * 2) : 0u;
                if (lane == 0) {
                    StageMeta& m = metas[stage];
                    m.s = win.s; m.kvh = win.kvh; m.qsub = win.qsub; m.nh = win.nh;
                    m.chunk = win.seg; m.nchunks = win.nseg; m.ts = ts; m.te = te;
                    m.flags = (qstage ? kFirst : 0) |
                              (win.last && st == nstages - 1 ? kLast : 0);
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
                if (qstage && lane == 31) {
                    const int64_t qoff = ((int64_t)win.s * p.num_q_heads + h0) * HD * 2;
                    bulk_g2s(sbase + 2 * Cfg::KV_BYTES, (const uint8_t*)p.q + qoff, qbytes,
                             &full[stage]);
                }
                if (++stage == Cfg::NSTAGE) { stage = 0; phase ^= 1u; }
                if (st == 0) {
                    // look one window ahead once this window's first stage is in flight:
                    // its block-table entries load while this window streams
                    nxt = make_window(p, blockIdx.x, a, end, q, pos + wtiles, sc);
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

    // ========================= consumer warp =========================
    const int g = lane >> 2, c = lane & 3;
    uint32_t qf[Cfg::KSTEPS][2];      // Q^T B fragments
    float o[Cfg::MTILES][4];          // O^T C fragments, rows mapped to d by d_row()
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    int stage = 0;
    uint32_t phase = 0;
    // d index of C-fragment row g (half 0) or g + 8 (half 1) of P.V m-tile mt
    auto d_row = [&](int mt, int half) -> int {
        if constexpr (Cfg::FP8) return 32 * (mt >> 1) + 2 * g + (mt & 1) + 16 * half;
        else return 16 * mt + g + 8 * half;
    };

    while (true) {
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
            const uint32_t* sQ = reinterpret_cast<const uint32_t*>(sbase + 2 * Cfg::KV_BYTES);
            const bool live = g < meta.nh;
#pragma unroll
            for (int t = 0; t < Cfg::KSTEPS; ++t) {
                if constexpr (Cfg::FP8) {
                    // k-slots (2c, 2c+1) <-> dims 16t+4c, +1; (8+2c, 9+2c) <-> 16t+4c+2, +3
                    qf[t][0] = live ? q_pair<QT, MT>(sQ[(g * HD + 16 * t + 4 * c) >> 1]) : 0u;
                    qf[t][1] = live ? q_pair<QT, MT>(sQ[(g * HD + 16 * t + 4 * c + 2) >> 1]) : 0u;
                } else {
                    qf[t][0] = live ? sQ[(g * HD + 16 * t + 2 * c) >> 1] : 0u;
                    qf[t][1] = live ? sQ[(g * HD + 16 * t + 8 + 2 * c) >> 1] : 0u;
                }
            }
#pragma unroll
            for (int mt = 0; mt < Cfg::MTILES; ++mt)
#pragma unroll
                for (int e = 0; e < 4; ++e) o[mt][e] = 0.f;
            m0 = m1 = -INFINITY;
            l0 = l1 = 0.f;
        }

        const int nvalid = meta.te - meta.ts;            // 1..32
        if (nvalid < TPS) {
            // rows past the context: stale or poisoned -> zero V (P is 0 there)
            const int zrows = TPS - nvalid;
            for (int i = lane; i < zrows * Cfg::HALVES * 8; i += 32) {
                const int r = nvalid + i / (Cfg::HALVES * 8);
                const int h = (i / 8) % Cfg::HALVES, ch = i % 8;
                *reinterpret_cast<uint4*>(sbase + Cfg::KV_BYTES + h * Cfg::HALF_BYTES + r * 128 +
                                          ch * 16) = make_uint4(0u, 0u, 0u, 0u);
            }
            fence_proxy_async_smem();
            __syncwarp();
        }
        const bool two = nvalid > 16;                    // second m-tile holds tokens
        // ---- S^T = K . Q^T for the stage's (up to) two 16-token m-tiles ----
        float sa[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        {
            const int rl = (lane & 7) + ((lane >> 3) & 1) * 8;
            if constexpr (Cfg::FP8) {
                // one 16-byte chunk = 16 e4m3 dims = one k-step; a lane's 4 bytes of a
                // row feed its k-slots (2c, 2c+1) and (8+2c, 9+2c)
#pragma unroll
                for (int pr = 0; pr < Cfg::KSTEPS / 2; ++pr) {
                    const int chunk = 2 * pr + (lane >> 4);
#pragma unroll
                    for (int mt = 0; mt < 2; ++mt) {
                        if (mt == 1 && !two) break;
                        uint32_t r[4];
                        ldsm_x4(sK + swz(16 * mt + rl, chunk), r);
#pragma unroll
                        for (int k = 0; k < 2; ++k) {
                            const uint32_t lo = r[2 * k], hi = r[2 * k + 1];
                            const uint32_t a[4] = {e4m3x2_to_f16x2(lo & 0xffffu),
                                                   e4m3x2_to_f16x2(hi & 0xffffu),
                                                   e4m3x2_to_f16x2(lo >> 16),
                                                   e4m3x2_to_f16x2(hi >> 16)};
                            Mma<MT>::run(sa[mt], a, qf[2 * pr + k][0], qf[2 * pr + k][1]);
                        }
                    }
                }
            } else {
#pragma unroll
                for (int t = 0; t < Cfg::KSTEPS; ++t) {
                    const int half = t >> 2, chunk = (t & 3) * 2 + (lane >> 4);
                    const uint32_t base = sK + half * Cfg::HALF_BYTES;
                    uint32_t a[4];
                    ldsm_x4(base + swz(rl, chunk), a);
                    Mma<MT>::run(sa[0], a, qf[t][0], qf[t][1]);
                    if (two) {
                        uint32_t b[4];
                        ldsm_x4(base + swz(16 + rl, chunk), b);
                        Mma<MT>::run(sa[1], b, qf[t][0], qf[t][1]);
                    }
                }
            }
        }
        // ---- online softmax over the stage's tokens ----
        float x[2][4];
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
            const bool va = mt * 16 + g < nvalid, vb = mt * 16 + g + 8 < nvalid;
            x[mt][0] = va ? sa[mt][0] * p.qk_scale_log2 : -INFINITY;
            x[mt][1] = va ? sa[mt][1] * p.qk_scale_log2 : -INFINITY;
            x[mt][2] = vb ? sa[mt][2] * p.qk_scale_log2 : -INFINITY;
            x[mt][3] = vb ? sa[mt][3] * p.qk_scale_log2 : -INFINITY;
        }
        float mx0 = fmaxf(fmaxf(x[0][0], x[0][2]), fmaxf(x[1][0], x[1][2]));
        float mx1 = fmaxf(fmaxf(x[0][1], x[0][3]), fmaxf(x[1][1], x[1][3]));
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
        }
        const bool n0 = mx0 > m0 + kRescaleSlack, n1 = mx1 > m1 + kRescaleSlack;
        if (__any_sync(0xffffffffu, n0 || n1)) {
            const float r0 = n0 ? fast_exp2(m0 - mx0) : 1.f;
            const float r1 = n1 ? fast_exp2(m1 - mx1) : 1.f;
            if (n0) m0 = mx0;
            if (n1) m1 = mx1;
            l0 *= r0;
            l1 *= r1;
#pragma unroll
            for (int mt = 0; mt < Cfg::MTILES; ++mt) {
                o[mt][0] *= r0;
                o[mt][2] *= r0;
                o[mt][1] *= r1;
                o[mt][3] *= r1;
            }
        }
        uint32_t pb[2][2];   // P^T B fragments of the two k-steps (tokens 0-15, 16-31)
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
            float f0, f1, f2, f3;
            const uint32_t p01 =
                Mma<MT>::pack(fast_exp2(x[mt][0] - m0), fast_exp2(x[mt][1] - m1), f0, f1);
            const uint32_t p23 =
                Mma<MT>::pack(fast_exp2(x[mt][2] - m0), fast_exp2(x[mt][3] - m1), f2, f3);
            l0 += f0 + f2;
            l1 += f1 + f3;
            pb[mt][0] = movmatrix_trans(p01);
            pb[mt][1] = movmatrix_trans(p23);
        }
        // ---- O^T += V^T . P^T ----
        {
            const int mi = lane >> 3;
            const int rv = (lane & 7) + (mi >> 1) * 8;
            if constexpr (Cfg::FP8) {
                // a transposed 8x8 b16 block of e4m3 rows gives each lane V[2c][2g, 2g+1]
                // and V[2c+1][2g, 2g+1]; byte permutes split them into an even-d and an
                // odd-d A fragment (m-tiles 2pr and 2pr+1 over dims 32pr .. 32pr+31)
#pragma unroll
                for (int pr = 0; pr < Cfg::MTILES / 2; ++pr) {
                    const int chunk = 2 * pr + (mi & 1);
#pragma unroll
                    for (int ks = 0; ks < 2; ++ks) {
                        if (ks == 1 && !two) break;
                        uint32_t r[4];
                        ldsm_x4_trans(sV + swz(16 * ks + rv, chunk), r);
                        uint32_t ev[4], od[4];
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            ev[k] = e4m3x2_to_f16x2(__byte_perm(r[k], 0u, 0x0020));
                            od[k] = e4m3x2_to_f16x2(__byte_perm(r[k], 0u, 0x0031));
                        }
                        Mma<MT>::run(o[2 * pr], ev, pb[ks][0], pb[ks][1]);
                        Mma<MT>::run(o[2 * pr + 1], od, pb[ks][0], pb[ks][1]);
                    }
                }
            } else {
#pragma unroll
                for (int mt = 0; mt < Cfg::MTILES; ++mt) {
                    const int half = mt >> 2, chunk = (mt & 3) * 2 + (mi & 1);
                    const uint32_t base = sV + half * Cfg::HALF_BYTES;
                    uint32_t a[4];
                    ldsm_x4_trans(base + swz(rv, chunk), a);
                    Mma<MT>::run(o[mt], a, pb[0][0], pb[0][1]);
                    if (two) {
                        uint32_t b[4];
                        ldsm_x4_trans(base + swz(16 + rv, chunk), b);
                        Mma<MT>::run(o[mt], b, pb[1][0], pb[1][1]);
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[stage]);
        if (++stage == Cfg::NSTAGE) { stage = 0; phase ^= 1u; }

        if (!(meta.flags & kLast)) continue;

        // ---------------- end of the segment (warp-local) ----------------
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            l0 += __shfl_xor_sync(0xffffffffu, l0, off);
            l1 += __shfl_xor_sync(0xffffffffu, l1, off);
        }
        const int hq0 = meta.kvh * p.group + meta.qsub * HPI;
        const int ha = 2 * c, hb = 2 * c + 1;
        const int64_t sha = (int64_t)meta.s * p.num_q_heads + hq0 + ha;
        const int64_t shb = sha + 1;
        if (meta.nchunks == 1) {
            const float ia = l0 > 0.f ? p.out_scale / l0 : 0.f;
            const float ib = l1 > 0.f ? p.out_scale / l1 : 0.f;
#pragma unroll
            for (int mt = 0; mt < Cfg::MTILES; ++mt) {
                const int d0 = d_row(mt, 0), d1 = d_row(mt, 1);
                if (ha < meta.nh) {
                    store_from_float<QT>(p.out, sha * HD + d0, o[mt][0] * ia);
                    store_from_float<QT>(p.out, sha * HD + d1, o[mt][2] * ia);
                }
                if (hb < meta.nh) {
                    store_from_float<QT>(p.out, shb * HD + d0, o[mt][1] * ib);
                    store_from_float<QT>(p.out, shb * HD + d1, o[mt][3] * ib);
                }
            }
            continue;
        }
        const int64_t pa_i = sha * p.part_stride + meta.chunk;
        const int64_t pb_i = shb * p.part_stride + meta.chunk;
#pragma unroll
        for (int mt = 0; mt < Cfg::MTILES; ++mt) {
            const int d0 = d_row(mt, 0), d1 = d_row(mt, 1);
            if (ha < meta.nh) {
                p.ws.pacc[pa_i * HD + d0] = o[mt][0];
                p.ws.pacc[pa_i * HD + d1] = o[mt][2];
            }
            if (hb < meta.nh) {
                p.ws.pacc[pb_i * HD + d0] = o[mt][1];
                p.ws.pacc[pb_i * HD + d1] = o[mt][3];
            }
        }
        if (g == 0) {
            if (ha < meta.nh) { p.ws.pm[pa_i] = m0; p.ws.pl[pa_i] = l0; }
            if (hb < meta.nh) { p.ws.pm[pb_i] = m1; p.ws.pl[pb_i] = l1; }
        }
        __syncwarp();
        int last = 0;
        if (lane == 0) {
            // the warp barrier above orders the lanes' stores before this lane's
            // gpu-scope fence, which publishes them before the arrival
            __threadfence();
            const int unit = (meta.s * p.num_kv_heads + meta.kvh) * p.nsub + meta.qsub;
            last = atomicAdd(&p.ws.unit_done[unit], 1u) == (unsigned)(meta.nchunks - 1);
            if (last) __threadfence();
        }
        last = __shfl_sync(0xffffffffu, last, 0);
        if (last) merge_segments_warp<QT, HD>(p, meta.s, hq0, meta.nh, meta.nchunks, lane);
    }
}

}  // namespace pkv
