// decode.cuh -- paged single-query decode attention (CUDA cores, sm_103a).
//
// "PagedAttention: Mathematical Foundations ..." §3 defines the result
// (a_ij = softmax_j(q_i.k_j / sqrt d), o_i = sum_j a_ij v_j over blocks K_j,
// V_j reached through a block table) and §7 describes the kernel family: a
// warp walks the physical block pointers, takes partial q.K_j dot products,
// keeps online-softmax normalisers and accumulates V_j in registers.  The
// decode pseudocode of §7 gives the running max / rescale / sum recurrence.
//
// Structure here (our design for sm_103a, not the pages'):
//  * One planning CTA turns context_lens into a work list of (sequence,
//    chunk) items, chunk = `chunk_tokens` consecutive logical tokens, and
//    resets the arrival counters.  Work item = (item, kv head, head subgroup).
//  * The decode kernel is persistent: every CTA pulls work items from an
//    atomic counter.  Warp 4 is the producer: it reads the item's block-table
//    entries and streams each (physical block, kv head) tile of K and V -- one
//    contiguous run in the [blocks][kv heads][B][d] layout -- into a ring of
//    shared-memory stages with 1-D bulk copies (cp.async.bulk) completing on
//    mbarriers.  K and V of a stage arrive together: a single pass over the
//    table.  The producer runs ahead across item boundaries.
//  * Warps 0-3 consume.  A lane group of LPT lanes owns one token at a time
//    and d/LPT dims of it; every lane keeps q and the running state (m, l,
//    acc) of all heads of the kv group for its dims in registers, so one K/V
//    load serves every query head of the group (GQA).  Scores are reduced
//    with warp shuffles.  The running max is only moved when a score exceeds
//    it by more than 2^8 (log2 domain), so the rescale of acc is rare; the
//    result is exact because (m, l, acc) always share the same reference m.
//  * At the end of an item the lane groups and warps merge their states
//    (rescale to a common max, add).  A single-chunk sequence writes the
//    output directly.  Otherwise the chunk's (m, l, acc) goes to the
//    workspace and the last CTA to finish a (sequence, kv head, subgroup)
//    merges all its chunks in chunk order (deterministic) and writes out.
#pragma once

#include "common.cuh"

namespace pkv {

constexpr int kMaxMergeChunks = 256;   // chunk states merged per (sequence, head)
constexpr int kMaxItemBlocks = 64;     // table entries a producer holds per item
constexpr float kRescaleSlack = 8.0f;  // log2-domain headroom before moving the max
constexpr int kMmaHeadsPerItem = 8;    // query heads per item of the tensor-core variant
constexpr int kMaxWorkers = 4096;      // CTAs of the balanced-split decode, at most
constexpr int kGroupRecord = 1 << 30;  // record code flag: a shared-prefix group
constexpr int kMaxGroupHeads = 16;     // query heads a shared-prefix unit serves
constexpr int kTileTokens = 64;        // split granularity of the balanced split

struct DecodeWork {
    unsigned* counter;    // next work index (dynamic items)
    unsigned* total;      // number of work indices (dynamic items)
    int* quota;           // tiles per worker (balanced split)
    int* ctx_eff;         // [S] context length after clamping
    int2* items;          // [S * max_chunks] (sequence, chunk)            (dynamic items)
    // balanced split with shared-prefix groups (tensor-core kernel)
    int* rec_prefix;      // [2S + 1] tile prefix over work records
    int4* rec;            // [2S] record {sequence | kGroupRecord for a group's shared
                          //   record, first token, end token, members (group) or
                          //   first tile of its group's shared record (-1: none)}
    int4* worker_first;   // [2 * kMaxWorkers] per worker: {record holding its first tile,
                          //   that record's tile range [lo, hi)}, then the record itself
    int4* seq_info;       // [S] {private tiles per unit, first private tile, first tile
                          //   of its group's shared record (-1: none), group tiles per unit}
    int* common;          // [S] leading table entries shared with the previous sequence
    int* unit_expect;     // [S * Hkv * nsub] partial states a grouped unit merges
    unsigned* unit_done;  // [S * Hkv * nsub] chunks / segments finished
    float* pm;            // [S * Hq * part_stride]
    float* pl;            // [S * Hq * part_stride]
    float* pacc;          // [S * Hq * part_stride * d]
};

struct DecodeParams {
    const void* q;
    const void* k_cache;
    const void* v_cache;
    const int32_t* block_tables;
    const int32_t* context_lens;
    void* out;
    DecodeWork ws;
    unsigned* status;
    int num_seqs, num_q_heads, num_kv_heads, group, nsub;
    int head_dim, block_size, num_blocks, max_blocks, max_context_len;
    int chunk_tokens, max_chunks;
    int part_stride;      // partial states per (sequence, query head) in the workspace
    int num_workers;      // CTAs of the balanced-split decode
    int allow_groups;     // group sequences that share leading blocks (prefix-aware decode);
                          // its split units are merged by a separate merge kernel
    int self_plan;        // CUDA-core path, every context within one chunk: no planning
                          // kernel; work item w is (sequence w / units, unit w % units)
    float qk_scale_log2;  // scale * log2(e) (* kv_scale for FP8)
    float out_scale;      // kv_scale for FP8, else 1
};

// ------------------------------------------------------------- planning --

template <typename QT>
__global__ void __launch_bounds__(1024) plan_kernel(DecodeParams p) {
    pdl_launch_dependents();   // the decode kernel's launch overlaps this plan
    __shared__ int warp_sums[32];
    __shared__ int carry;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) carry = 0;
    const int nunits = p.num_seqs * p.num_kv_heads * p.nsub;
    for (int i = tid; i < nunits; i += blockDim.x) p.ws.unit_done[i] = 0u;
    const int cap = min(p.max_context_len, p.max_blocks * p.block_size);
    const int C = p.chunk_tokens;
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
            n = (ctx + C - 1) / C;
        }
        int x = n;  // inclusive scan over the block
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, x, off);
            if (lane >= off) x += y;
        }
        if (lane == 31) warp_sums[warp] = x;
        __syncthreads();
        if (warp == 0) {
            int v = lane < (int)(blockDim.x >> 5) ? warp_sums[lane] : 0;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                int y = __shfl_up_sync(0xffffffffu, v, off);
                if (lane >= off) v += y;
            }
            warp_sums[lane] = v;
        }
        __syncthreads();
        const int incl = x + (warp > 0 ? warp_sums[warp - 1] : 0);
        const int first = carry + incl - n;
        for (int c = 0; c < n; ++c) p.ws.items[first + c] = make_int2(s, c);
        __syncthreads();
        if (tid == blockDim.x - 1) carry += incl;
        __syncthreads();
    }
    // sequences with no context: all-zero output
    const int row = p.num_q_heads * p.head_dim;
    for (int s = warp; s < p.num_seqs; s += blockDim.x >> 5) {
        if (p.ws.ctx_eff[s] != 0) continue;
        for (int i = lane; i < row; i += 32) store_from_float<QT>(p.out, (int64_t)s * row + i, 0.f);
    }
    if (tid == 0) {
        *p.ws.counter = 0u;
        *p.ws.total = (unsigned)carry * (unsigned)(p.num_kv_heads * p.nsub);
    }
}

// ---------------------------------------------------------------- decode --

template <typename QT, typename KT, int HD, int HPI>
struct SimtCfg {
    static constexpr int E = KT::bytes;
    static constexpr int ROWB = HD * E;               // bytes of one token row
    static constexpr int NCH = ROWB / 16;             // 16-byte chunks per row
    static constexpr int LPT = NCH < 8 ? NCH : 8;     // lanes per token
    static constexpr int CPL = NCH / LPT;             // chunks per lane
    static constexpr int EPC = 16 / E;                // elements per chunk
    static constexpr int DPL = CPL * EPC;             // dims per lane
    static constexpr int NCW = 4;                     // consumer warps
    static constexpr int GPW = 32 / LPT;              // lane groups per warp
    static constexpr int NG = NCW * GPW;              // lane groups per CTA
    static constexpr int TPS_RAW = 8192 / ROWB;
    static constexpr int TPS = TPS_RAW < 16 ? 16 : (TPS_RAW > 64 ? 64 : TPS_RAW);
    static constexpr int TPG = TPS / NG;              // tokens per group per stage
    static constexpr int NSTAGE = 5;
    static constexpr int QB = QT::bytes;
    static constexpr int STAGE_KV = TPS * ROWB;
    static constexpr int STAGE_Q = HPI * HD * QB;
    static constexpr int STAGE_BYTES = (2 * STAGE_KV + STAGE_Q + 127) / 128 * 128;
    static constexpr int THREADS = (NCW + 1) * 32;
    static constexpr int SCRATCH_FLOATS =
        (NCW * HPI * (HD + 2) > 2 * HPI * kMaxMergeChunks + 2 * HPI)
            ? NCW * HPI * (HD + 2)
            : 2 * HPI * kMaxMergeChunks + 2 * HPI;
    static_assert(TPS % NG == 0 && TPG >= 1, "stage must split evenly over lane groups");
    static_assert(HD % (LPT * EPC) == 0, "head_dim must split evenly over a lane group");
};

struct StageMeta {
    int s, kvh, qsub, nh;       // sequence, kv head, head subgroup, valid heads
    int chunk, nchunks;         // chunk index, chunks of this sequence
    int ts, te;                 // logical tokens [ts, te) held by this stage
    int flags;                  // kFirst | kLast | kDone
    int expect, segoff;         // private unit: partial states merged, first private one
    int pad[5];
};
constexpr int kFirst = 1, kLast = 2, kDone = 4, kGroup = 8;

template <typename Cfg>
struct SimtSmem {
    static constexpr size_t stages = 0;
    static constexpr size_t metas = stages + (size_t)Cfg::NSTAGE * Cfg::STAGE_BYTES;
    static constexpr size_t bars = metas + (size_t)Cfg::NSTAGE * sizeof(StageMeta);
    static constexpr size_t scratch = bars + 2 * Cfg::NSTAGE * sizeof(uint64_t);
    static constexpr size_t misc = scratch + (size_t)Cfg::SCRATCH_FLOATS * sizeof(float);
    static constexpr size_t total = misc + 16;
};

// Merge state b into a (both relative to their own reference max).
__device__ __forceinline__ void merge_factor(float ma, float mb, float& fa, float& fb,
                                             float& M) {
    M = fmaxf(ma, mb);
    fa = ma == -INFINITY ? 0.f : fast_exp2(ma - M);
    fb = mb == -INFINITY ? 0.f : fast_exp2(mb - M);
}

// End of a work item, after every consumer warp has put its state in `scratch`
// ([NCW][HPI][HD] acc, then [NCW][HPI] m, then [NCW][HPI] l; all relative to
// the warp's own reference max, log2 domain).  Merges the warps by the
// rescale rule; a single-chunk sequence writes `out`, otherwise the chunk's
// state goes to the workspace and the last CTA to finish this (sequence, kv
// head, subgroup) merges all chunks in chunk order and writes `out`.
// Called by all NCW*32 consumer threads; leaves `scratch` free for reuse.
template <typename QT, int HD, int HPI, int NCW>
__device__ __forceinline__ void finish_item(const DecodeParams& p, const StageMeta& meta,
                                            float* scratch, int* misc, int ctid) {
    constexpr int NT = NCW * 32;
    float* s_acc = scratch;
    float* s_m = scratch + NCW * HPI * HD;
    float* s_l = s_m + NCW * HPI;
    named_bar_sync(1, NT);
    const bool single = meta.nchunks == 1;
    const int hq0 = meta.kvh * p.group + meta.qsub * HPI;
    for (int idx = ctid; idx < HPI * HD; idx += NT) {
        const int h = idx / HD, dim = idx % HD;
        if (h >= meta.nh) continue;
        float M = -INFINITY;
#pragma unroll
        for (int w2 = 0; w2 < NCW; ++w2) M = fmaxf(M, s_m[w2 * HPI + h]);
        float L = 0.f, A = 0.f;
#pragma unroll
        for (int w2 = 0; w2 < NCW; ++w2) {
            const float mw = s_m[w2 * HPI + h];
            const float f = mw == -INFINITY ? 0.f : fast_exp2(mw - M);
            L = fmaf(s_l[w2 * HPI + h], f, L);
            A = fmaf(s_acc[(w2 * HPI + h) * HD + dim], f, A);
        }
        const int64_t sh = (int64_t)meta.s * p.num_q_heads + hq0 + h;
        if (single) {
            store_from_float<QT>(p.out, sh * HD + dim, L > 0.f ? A / L * p.out_scale : 0.f);
        } else {
            const int64_t pi = sh * p.part_stride + meta.chunk;
            p.ws.pacc[pi * HD + dim] = A;
            if (dim == 0) {
                p.ws.pm[pi] = M;
                p.ws.pl[pi] = L;
            }
        }
    }
    named_bar_sync(1, NT);   // scratch reads done; partial stores issued by every thread
    if (single) return;
    if (ctid == 0) {
        // the barrier above orders every thread's partial stores before this
        // thread's gpu-scope fence, which publishes them before the arrival
        __threadfence();
        const int unit = (meta.s * p.num_kv_heads + meta.kvh) * p.nsub + meta.qsub;
        const unsigned done = atomicAdd(&p.ws.unit_done[unit], 1u);
        misc[0] = done == (unsigned)(meta.nchunks - 1);
        if (misc[0]) __threadfence();
    }
    named_bar_sync(1, NT);
    if (misc[0]) {
        // last chunk of this (sequence, kv head, subgroup) to finish: merge all chunks
        const int nc = meta.nchunks;
        float* f_tab = scratch;                        // [HPI][kMaxMergeChunks] factors
        float* lsum = scratch + HPI * kMaxMergeChunks; // [HPI] merged l
        for (int idx = ctid; idx < HPI * nc; idx += NT) {
            const int h = idx / nc, c = idx % nc;
            if (h >= meta.nh) continue;
            const int64_t pi = ((int64_t)meta.s * p.num_q_heads + hq0 + h) * p.part_stride + c;
            f_tab[h * kMaxMergeChunks + c] = __ldcg(&p.ws.pm[pi]);
        }
        named_bar_sync(1, NT);
        if (ctid < HPI && ctid < meta.nh) {
            const int h = ctid;
            float M = -INFINITY;
            for (int c = 0; c < nc; ++c) M = fmaxf(M, f_tab[h * kMaxMergeChunks + c]);
            float L = 0.f;
            for (int c = 0; c < nc; ++c) {
                const int64_t pi = ((int64_t)meta.s * p.num_q_heads + hq0 + h) * p.part_stride + c;
                const float mc = f_tab[h * kMaxMergeChunks + c];
                const float f = mc == -INFINITY ? 0.f : fast_exp2(mc - M);
                f_tab[h * kMaxMergeChunks + c] = f;
                L = fmaf(__ldcg(&p.ws.pl[pi]), f, L);
            }
            lsum[h] = L;
        }
        named_bar_sync(1, NT);
        for (int idx = ctid; idx < HPI * HD; idx += NT) {
            const int h = idx / HD, dim = idx % HD;
            if (h >= meta.nh) continue;
            const int64_t sh = (int64_t)meta.s * p.num_q_heads + hq0 + h;
            float A = 0.f;
            for (int c = 0; c < nc; ++c)
                A = fmaf(__ldcg(&p.ws.pacc[(sh * p.part_stride + c) * HD + dim]),
                         f_tab[h * kMaxMergeChunks + c], A);
            const float L = lsum[h];
            store_from_float<QT>(p.out, sh * HD + dim, L > 0.f ? A / L * p.out_scale : 0.f);
        }
    }
    named_bar_sync(1, NT);   // scratch and misc are reused by the next item
}

template <typename QT, typename KT, int HD, int HPI>
__global__ void __launch_bounds__(SimtCfg<QT, KT, HD, HPI>::THREADS, 2)
    decode_simt_kernel(DecodeParams p) {
    using Cfg = SimtCfg<QT, KT, HD, HPI>;
    using Smem = SimtSmem<Cfg>;
    extern __shared__ __align__(128) uint8_t smem[];
    StageMeta* metas = reinterpret_cast<StageMeta*>(smem + Smem::metas);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + Smem::bars);
    uint64_t* empty = full + Cfg::NSTAGE;
    float* scratch = reinterpret_cast<float*>(smem + Smem::scratch);
    int* misc = reinterpret_cast<int*>(smem + Smem::misc);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < Cfg::NSTAGE; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], Cfg::NCW);
        }
        fence_mbar_init();
    }
    __syncthreads();
    pdl_wait();   // the preceding kernel (planner, or the cache write) has completed

    const int B = p.block_size, C = p.chunk_tokens;
    const int units_per_item = p.num_kv_heads * p.nsub;
    const unsigned total = p.self_plan ? (unsigned)(p.num_seqs * units_per_item) : *p.ws.total;

    if (warp == Cfg::NCW) {
        // ======================= producer warp =======================
        const uint64_t policy = l2_evict_first_policy();
        int stage = 0;
        uint32_t phase = 0;
        unsigned w = blockIdx.x;
        if (!p.self_plan) {
            if (lane == 0) w = atomicAdd(p.ws.counter, 1u);
            w = __shfl_sync(0xffffffffu, w, 0);
        }
        bool ok = true;
        while (w < total && ok) {
            unsigned wn = w + gridDim.x;
            if (!p.self_plan && lane == 0) wn = atomicAdd(p.ws.counter, 1u);   // overlaps the item
            const int it = (int)(w / units_per_item), rem = (int)(w % units_per_item);
            const int kvh = rem / p.nsub, qsub = rem % p.nsub;
            int s, chunk, ctx, e0, e1;
            if (p.self_plan) {
                // one chunk per sequence: the table's first entries load beside the length
                s = it;
                chunk = 0;
                const int32_t* trow = p.block_tables + (int64_t)s * p.max_blocks;
                e0 = lane < p.max_blocks ? trow[lane] : 0;
                e1 = lane + 32 < p.max_blocks ? trow[lane + 32] : 0;
                ctx = p.context_lens[s];
                const int cap = min(p.max_context_len, p.max_blocks * B);
                if (ctx < 0 || ctx > cap) {
                    if (rem == 0) set_status(p.status, PKV_DEV_BAD_CONTEXT);
                    ctx = ctx < 0 ? 0 : cap;
                }
                if (ctx == 0) {
                    // no context: this unit's heads of the output are zero
                    const int h0z = kvh * p.group + qsub * HPI;
                    const int nhz = min(HPI, p.group - qsub * HPI);
                    const int64_t o0 = ((int64_t)s * p.num_q_heads + h0z) * HD;
                    for (int i = lane; i < nhz * HD; i += 32) store_from_float<QT>(p.out, o0 + i, 0.f);
                    w = wn;
                    continue;
                }
            } else {
                const int2 sc = p.ws.items[it];
                s = sc.x;
                chunk = sc.y;
                ctx = p.ws.ctx_eff[s];
            }
            const int nchunks = (ctx + C - 1) / C;
            const int t0 = chunk * C, t1 = min(t0 + C, ctx);
            const int jb0 = t0 / B, nb = (t1 + B - 1) / B - jb0;
            if (!p.self_plan) {
                const int32_t* trow = p.block_tables + (int64_t)s * p.max_blocks;
                e0 = lane < nb ? trow[jb0 + lane] : 0;
                e1 = lane + 32 < nb ? trow[jb0 + lane + 32] : 0;
            }
            if ((lane < nb && (e0 < 0 || e0 >= p.num_blocks)) ||
                (lane + 32 < nb && (e1 < 0 || e1 >= p.num_blocks))) {
                set_status(p.status, PKV_DEV_BAD_BLOCK_ID);
                if (e0 < 0 || e0 >= p.num_blocks) e0 = 0;
                if (e1 < 0 || e1 >= p.num_blocks) e1 = 0;
            }
            const int h0 = kvh * p.group + qsub * HPI;
            const int nh = min(HPI, p.group - qsub * HPI);
            const int nstages = (t1 - t0 + Cfg::TPS - 1) / Cfg::TPS;
            for (int st = 0; st < nstages; ++st) {
                const int ts = t0 + st * Cfg::TPS, te = min(ts + Cfg::TPS, t1);
                if (!mbar_wait(&empty[stage], phase ^ 1u)) {
                    set_status(p.status, PKV_DEV_WAIT_TIMEOUT);
                    ok = false;
                    break;
                }
                uint8_t* sbase = smem + Smem::stages + (size_t)stage * Cfg::STAGE_BYTES;
                const int fb = ts / B, nseg = (te - 1) / B - fb + 1;
                const uint32_t qbytes = st == 0 ? (uint32_t)(nh * HD * Cfg::QB) : 0u;
                if (lane == 0) {
                    StageMeta& m = metas[stage];
                    m.s = s; m.kvh = kvh; m.qsub = qsub; m.nh = nh;
                    m.chunk = chunk; m.nchunks = nchunks; m.ts = ts; m.te = te;
                    m.flags = (st == 0 ? kFirst : 0) | (st == nstages - 1 ? kLast : 0);
                    mbar_arrive_expect_tx(&full[stage],
                                          2u * (uint32_t)(te - ts) * Cfg::ROWB + qbytes);
                }
                __syncwarp();
                const int rel = fb + lane - jb0;
                const int pa = __shfl_sync(0xffffffffu, e0, rel & 31);
                const int pb = __shfl_sync(0xffffffffu, e1, rel & 31);
                if (lane < nseg) {
                    const int jblk = fb + lane;
                    const int phys = rel < 32 ? pa : pb;
                    const int r0 = max(ts, jblk * B) - jblk * B;
                    const int r1 = min(te, (jblk + 1) * B) - jblk * B;
                    const size_t soff = (size_t)(jblk * B + r0 - ts) * Cfg::ROWB;
                    const int64_t goff =
                        (((int64_t)phys * p.num_kv_heads + kvh) * B + r0) * Cfg::ROWB;
                    const uint32_t bytes = (uint32_t)(r1 - r0) * Cfg::ROWB;
                    bulk_g2s_hint(sbase + soff, (const uint8_t*)p.k_cache + goff, bytes,
                                  &full[stage], policy);
                    bulk_g2s_hint(sbase + Cfg::STAGE_KV + soff, (const uint8_t*)p.v_cache + goff,
                                  bytes, &full[stage], policy);
                }
                if (qbytes && lane == 31) {
                    const int64_t qoff = ((int64_t)s * p.num_q_heads + h0) * HD * Cfg::QB;
                    bulk_g2s(sbase + 2 * Cfg::STAGE_KV, (const uint8_t*)p.q + qoff, qbytes,
                             &full[stage]);
                }
                if (++stage == Cfg::NSTAGE) { stage = 0; phase ^= 1u; }
            }
            w = p.self_plan ? wn : __shfl_sync(0xffffffffu, wn, 0);
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
    constexpr int LPT = Cfg::LPT, CPL = Cfg::CPL, EPC = Cfg::EPC, DPL = Cfg::DPL;
    constexpr int TPG = Cfg::TPG, NG = Cfg::NG, NCW = Cfg::NCW;
    const int gid = warp * Cfg::GPW + lane / LPT;   // lane group within the CTA
    const int j = lane % LPT;                       // position within the group
    const int ctid = threadIdx.x;                   // 0 .. NCW*32-1

    float q[HPI][DPL];
    float acc[HPI][DPL];
    float m[HPI], l[HPI];
    int stage = 0;
    uint32_t phase = 0;

    while (true) {
        if (!mbar_wait(&full[stage], phase)) {
            set_status(p.status, PKV_DEV_WAIT_TIMEOUT);
            break;
        }
        const StageMeta meta = metas[stage];
        if (meta.flags & kDone) break;
        const uint8_t* sK = smem + Smem::stages + (size_t)stage * Cfg::STAGE_BYTES;
        const uint8_t* sV = sK + Cfg::STAGE_KV;

        if (meta.flags & kFirst) {
            const void* sQ = sK + 2 * Cfg::STAGE_KV;
#pragma unroll
            for (int h = 0; h < HPI; ++h) {
#pragma unroll
                for (int k = 0; k < CPL; ++k)
#pragma unroll
                    for (int e = 0; e < EPC; ++e) {
                        const int dim = (j + k * LPT) * EPC + e;
                        q[h][k * EPC + e] =
                            h < meta.nh ? load_as_float<QT>(sQ, h * HD + dim) * p.qk_scale_log2
                                        : 0.f;
                        acc[h][k * EPC + e] = 0.f;
                    }
                m[h] = -INFINITY;
                l[h] = 0.f;
            }
        }

        const int ntok = meta.te - meta.ts;
        float sc[TPG][HPI];
#pragma unroll
        for (int i = 0; i < TPG; ++i) {
            const int tl = i * NG + gid;
            float kf[DPL];
#pragma unroll
            for (int k = 0; k < CPL; ++k) {
                uint4 raw = make_uint4(0u, 0u, 0u, 0u);
                if (tl < ntok)
                    raw = *reinterpret_cast<const uint4*>(sK + (size_t)tl * Cfg::ROWB +
                                                          (j + k * LPT) * 16);
                Chunk<KT>::to_float(raw, &kf[k * EPC]);
            }
#pragma unroll
            for (int h = 0; h < HPI; ++h) {
                float d = 0.f;
#pragma unroll
                for (int x = 0; x < DPL; ++x) d = fmaf(q[h][x], kf[x], d);
                sc[i][h] = d;
            }
        }
#pragma unroll
        for (int off = LPT / 2; off >= 1; off >>= 1)
#pragma unroll
            for (int i = 0; i < TPG; ++i)
#pragma unroll
                for (int h = 0; h < HPI; ++h)
                    sc[i][h] += __shfl_xor_sync(0xffffffffu, sc[i][h], off);

        // online softmax over this stage's tokens (lazy max movement)
        bool need = false;
        float smax[HPI];
#pragma unroll
        for (int h = 0; h < HPI; ++h) {
            float v = -INFINITY;
#pragma unroll
            for (int i = 0; i < TPG; ++i)
                if (i * NG + gid < ntok) v = fmaxf(v, sc[i][h]);
            smax[h] = v;
            need |= v > m[h] + kRescaleSlack;
        }
        if (__any_sync(0xffffffffu, need)) {
#pragma unroll
            for (int h = 0; h < HPI; ++h) {
                if (smax[h] > m[h] + kRescaleSlack) {
                    const float r = fast_exp2(m[h] - smax[h]);   // m = -inf gives 0
                    l[h] *= r;
#pragma unroll
                    for (int x = 0; x < DPL; ++x) acc[h][x] *= r;
                    m[h] = smax[h];
                }
            }
        }
#pragma unroll
        for (int i = 0; i < TPG; ++i) {
            const int tl = i * NG + gid;
            if (tl < ntok) {
                float pr[HPI];
#pragma unroll
                for (int h = 0; h < HPI; ++h) {
                    pr[h] = fast_exp2(sc[i][h] - m[h]);
                    l[h] += pr[h];
                }
                float vf[DPL];
#pragma unroll
                for (int k = 0; k < CPL; ++k) {
                    const uint4 raw = *reinterpret_cast<const uint4*>(
                        sV + (size_t)tl * Cfg::ROWB + (j + k * LPT) * 16);
                    Chunk<KT>::to_float(raw, &vf[k * EPC]);
                }
#pragma unroll
                for (int h = 0; h < HPI; ++h)
#pragma unroll
                    for (int x = 0; x < DPL; ++x) acc[h][x] = fmaf(pr[h], vf[x], acc[h][x]);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[stage]);
        if (++stage == Cfg::NSTAGE) { stage = 0; phase ^= 1u; }

        if (!(meta.flags & kLast)) continue;

        // ---------------- finish the item: merge lane groups, warps ----------------
#pragma unroll
        for (int off = LPT; off < 32; off <<= 1) {
#pragma unroll
            for (int h = 0; h < HPI; ++h) {
                const float mo = __shfl_xor_sync(0xffffffffu, m[h], off);
                const float lo = __shfl_xor_sync(0xffffffffu, l[h], off);
                float fa, fb, M;
                merge_factor(m[h], mo, fa, fb, M);
                l[h] = l[h] * fa + lo * fb;
#pragma unroll
                for (int x = 0; x < DPL; ++x) {
                    const float ao = __shfl_xor_sync(0xffffffffu, acc[h][x], off);
                    acc[h][x] = acc[h][x] * fa + ao * fb;
                }
                m[h] = M;
            }
        }
        // scratch: acc [NCW][HPI][HD], then m [NCW][HPI], l [NCW][HPI]
        float* s_acc = scratch;
        float* s_m = scratch + NCW * HPI * HD;
        float* s_l = s_m + NCW * HPI;
        if (lane < LPT) {
#pragma unroll
            for (int h = 0; h < HPI; ++h)
#pragma unroll
                for (int k = 0; k < CPL; ++k)
#pragma unroll
                    for (int e = 0; e < EPC; ++e)
                        s_acc[(warp * HPI + h) * HD + (j + k * LPT) * EPC + e] = acc[h][k * EPC + e];
            if (lane == 0) {
#pragma unroll
                for (int h = 0; h < HPI; ++h) {
                    s_m[warp * HPI + h] = m[h];
                    s_l[warp * HPI + h] = l[h];
                }
            }
        }
        finish_item<QT, HD, HPI, NCW>(p, meta, scratch, misc, ctid);
    }
}

}  // namespace pkv
