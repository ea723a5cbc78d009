/*
 * oracle.c -- plain, slow, fp64 CPU oracle for the paged-KV-cache hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or
 * calls this file: only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header, table or helper with the
 * CUDA library; it is written from the pages' definitions, step by step, with
 * no blocking, fusion or reordering beyond what those definitions state.
 *
 * Sources (page title, section):
 *   [P1] "PagedAttention: Mathematical Foundations, Virtual Memory Block
 *        Allocation, and Zero-Waste KV Cache Serving" (llms.blog)
 *        §1 KV Cache Memory Footprint, §3 Mathematical Formulation,
 *        §4 Virtual Memory Architecture and Block Tables, §5 Parallel Sampling,
 *        §7 Custom GPU Kernel Optimization (kernels 1-3, decode pseudocode).
 *   [P2] "Pytorch implementation of paper: Efficient Memory Management for
 *        Large Language Model Serving with PagedAttention" (aishastr.live),
 *        §2 PagedAttentionExecutor.forward (gather by table, then dense).
 *   [P3] "PagedAttention ... 为什么走到了尽头" (10100.com), §4 (FP8 e4m3 KV is
 *        stored as fp8 and converted to a wider type on load, times a scale).
 *
 * Readings where the pages are silent (each is also listed in the design notes):
 *   - KV cache layout: k_cache and v_cache are both [num_blocks, num_kv_heads,
 *     block_size, head_dim], head_dim contiguous.  The pages contradict each
 *     other on the layout ([P2] §2 vs [P3] §2); this is the library's contract.
 *   - GQA: query head h reads kv head h / (num_q_heads / num_kv_heads).
 *   - context_len == 0 gives an all-zero output.
 *   - FP8 is OCP E4M3 ("e4m3fn"): bias 7, no infinities, S.1111.111 = NaN,
 *     max finite 448.  Dequantised value = decode(code) * kv_scale.  Encode
 *     divides the fp32 value by kv_scale in fp32 (IEEE, correctly rounded),
 *     then rounds to nearest-even with saturation to +-448; NaN -> 0x7F.
 *   - slot_mapping < 0 means "padding token, write nothing".
 *   - copy_blocks requires a dst set with no repeats and no dst that is also a src.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* element types; the numbering matches the Python wrapper (oracle/__init__.py) */
enum { OR_F32 = 0, OR_F16 = 1, OR_BF16 = 2, OR_E4M3 = 3 };

static int elem_bytes(int t) {
    switch (t) {
    case OR_F32: return 4;
    case OR_F16: return 2;
    case OR_BF16: return 2;
    case OR_E4M3: return 1;
    default: return 0;
    }
}

/* ---------------------------------------------------------------- codecs -- */

/* IEEE 754 binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits. */
double oracle_f16_to_double(uint16_t h) {
    int s = (h >> 15) & 1, e = (h >> 10) & 31, f = h & 1023;
    double v;
    if (e == 0) v = ldexp((double)f, -24);              /* subnormal: 2^-14 * f/1024 */
    else if (e == 31) v = f ? NAN : INFINITY;
    else v = ldexp(1.0 + f / 1024.0, e - 15);
    return s ? -v : v;
}

/* bfloat16 is the upper half of an IEEE binary32. */
double oracle_bf16_to_double(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* OCP E4M3: 1 sign, 4 exponent (bias 7), 3 mantissa bits.  Exponent field 0 is
 * subnormal (2^-6 * m/8); 0bS1111111 is NaN; there is no infinity. */
double oracle_e4m3_to_double(uint8_t c) {
    int s = (c >> 7) & 1, e = (c >> 3) & 15, m = c & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m, -9);
    else v = ldexp(1.0 + m / 8.0, e - 7);
    return s ? -v : v;
}

/* Round-to-nearest-even into E4M3 with saturation to the largest finite value. */
uint8_t oracle_e4m3_from_float(float x) {
    if (isnan(x)) return 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs((double)x);
    if (a >= 448.0) return sign | 0x7E;                  /* satfinite (inf included) */
    if (a < ldexp(1.0, -6)) {
        /* subnormal range: spacing 2^-9; rint() rounds half to even */
        double q = rint(ldexp(a, 9));                    /* 0..8; 8 is 2^-6 = code 0x08 */
        return sign | (uint8_t)q;
    }
    int e2;
    double fr = frexp(a, &e2);                           /* a = fr * 2^e2, fr in [0.5,1) */
    int e = e2 - 1;                                      /* a = (2 fr) * 2^e, 2fr in [1,2) */
    double m = rint((2.0 * fr - 1.0) * 8.0);             /* 0..8 */
    if (m == 8.0) { m = 0.0; e += 1; }
    int field = e + 7;                                   /* 1..15 */
    int code = (field << 3) | (int)m;
    if (code > 0x7E) code = 0x7E;                        /* cannot happen below 448 */
    return sign | (uint8_t)code;
}

/* Value of element i of a buffer of type t, exactly, in fp64. */
static double load_elem(const void* base, int t, int64_t i) {
    switch (t) {
    case OR_F32: return (double)((const float*)base)[i];
    case OR_F16: return oracle_f16_to_double(((const uint16_t*)base)[i]);
    case OR_BF16: return oracle_bf16_to_double(((const uint16_t*)base)[i]);
    case OR_E4M3: return oracle_e4m3_to_double(((const uint8_t*)base)[i]);
    default: return NAN;
    }
}

/* ----------------------------------------------- closed form ([P1] §1) -- */

/* Bytes of K and V held per token across all layers: two vectors (K, V) of
 * d_model elements per layer.  With 2-byte elements this is 4 L d_model. */
int64_t oracle_kv_bytes_per_token(int64_t num_layers, int64_t d_model, int64_t elem_size) {
    return 2 * num_layers * d_model * elem_size;
}

/* --------------------------------- reshape_and_cache ([P1] §7 kernel 1) -- */

/* Offset (in elements) of element `dim` of token row `off` of kv head `h` in
 * physical block `blk`, for the layout [num_blocks, num_kv_heads, B, d]. */
static int64_t cache_index(int64_t blk, int64_t h, int64_t off, int64_t dim,
                           int num_kv_heads, int block_size, int head_dim) {
    return ((blk * num_kv_heads + h) * block_size + off) * head_dim + dim;
}

/* For each token t with slot_mapping[t] >= 0: block = slot / B, offset = slot % B;
 * write key[t][h][:] and value[t][h][:] into that block's row for every kv head.
 * Same element type: copy the bytes.  kv_dtype E4M3: encode(x / kv_scale).
 * Returns 0, or -1 on a bad argument / a slot outside the pool. */
int oracle_reshape_and_cache(const void* key, const void* value, void* k_cache, void* v_cache,
                             const int64_t* slot_mapping, int num_tokens, int num_kv_heads,
                             int head_dim, int block_size, int num_blocks, int src_dtype,
                             int kv_dtype, float kv_scale) {
    int se = elem_bytes(src_dtype), ke = elem_bytes(kv_dtype);
    if (!se || !ke || src_dtype == OR_E4M3) return -1;
    if (kv_dtype != src_dtype && kv_dtype != OR_E4M3) return -1;
    for (int t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        int64_t blk = slot / block_size, off = slot % block_size;
        if (blk >= num_blocks) return -1;
        for (int h = 0; h < num_kv_heads; ++h) {
            for (int i = 0; i < head_dim; ++i) {
                int64_t src = ((int64_t)t * num_kv_heads + h) * head_dim + i;
                int64_t dst = cache_index(blk, h, off, i, num_kv_heads, block_size, head_dim);
                if (kv_dtype == src_dtype) {
                    memcpy((char*)k_cache + dst * ke, (const char*)key + src * se, (size_t)se);
                    memcpy((char*)v_cache + dst * ke, (const char*)value + src * se, (size_t)se);
                } else {
                    float xk = (float)load_elem(key, src_dtype, src);     /* exact */
                    float xv = (float)load_elem(value, src_dtype, src);
                    ((uint8_t*)k_cache)[dst] = oracle_e4m3_from_float(xk / kv_scale);
                    ((uint8_t*)v_cache)[dst] = oracle_e4m3_from_float(xv / kv_scale);
                }
            }
        }
    }
    return 0;
}

/* ------------------------------ copy_blocks ([P1] §5 step 4, §7 kernel 3) -- */

/* For each pair (src, dst): physical block dst of both caches becomes a byte
 * copy of block src (all kv heads).  Returns -1 if an id is out of range, a
 * dst repeats, or a dst is also a src. */
int oracle_copy_blocks(void* k_cache, void* v_cache, const int32_t* pairs, int num_pairs,
                       int num_kv_heads, int head_dim, int block_size, int num_blocks,
                       int kv_dtype) {
    int e = elem_bytes(kv_dtype);
    if (!e) return -1;
    for (int i = 0; i < num_pairs; ++i) {
        int32_t s = pairs[2 * i], d = pairs[2 * i + 1];
        if (s < 0 || s >= num_blocks || d < 0 || d >= num_blocks) return -1;
        for (int j = 0; j < num_pairs; ++j) {
            if (j != i && pairs[2 * j + 1] == d) return -1;
            if (pairs[2 * j] == d) return -1;
        }
    }
    size_t block_bytes = (size_t)num_kv_heads * block_size * head_dim * e;
    for (int i = 0; i < num_pairs; ++i) {
        int64_t s = pairs[2 * i], d = pairs[2 * i + 1];
        memcpy((char*)k_cache + d * block_bytes, (const char*)k_cache + s * block_bytes, block_bytes);
        memcpy((char*)v_cache + d * block_bytes, (const char*)v_cache + s * block_bytes, block_bytes);
    }
    return 0;
}

/* ------------------------- paged decode attention ([P1] §3, [P2] §2) ------ */

typedef struct {
    const void* query; const void* k_cache; const void* v_cache;
    const int32_t* block_tables; const int32_t* context_lens;
    int num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, max_blocks;
    double scale; int q_dtype, kv_dtype; double kv_scale;
} dec_args;

/* k_t / v_t of sequence s, kv head g, logical token t, dequantised to fp64,
 * fetched through the block table: block = table[s][t / B], row = t % B. */
static int fetch_row(const dec_args* a, const void* cache, int s, int g, int t, double* row) {
    int32_t blk = a->block_tables[(int64_t)s * a->max_blocks + t / a->block_size];
    int off = t % a->block_size;
    if (blk < 0 || blk >= a->num_blocks) return -1;
    double mult = a->kv_dtype == OR_E4M3 ? a->kv_scale : 1.0;
    for (int i = 0; i < a->head_dim; ++i) {
        int64_t idx = cache_index(blk, g, off, i, a->num_kv_heads, a->block_size, a->head_dim);
        row[i] = load_elem(cache, a->kv_dtype, idx) * mult;
    }
    return 0;
}

/* Unnormalised attention state over logical tokens [t0, t1) of sequence s for
 * query head h of query row `qrow` (the sequence's own row for decode):
 *   z_t = scale * q.k_t,  m = max z_t,  l = sum exp(z_t - m),
 *   acc = sum exp(z_t - m) v_t.
 * The full output is acc / l ([P1] §3: a_ij = exp(z_j) / sum_t exp(z_t),
 * o_i = sum_j a_ij v_j; subtracting m from every logit leaves a_ij unchanged).
 * An empty range gives m = -inf, l = 0, acc = 0. */
static int partial_state(const dec_args* a, int s, int qrow, int h, int t0, int t1,
                         double* m_out, double* l_out, double* acc) {
    int d = a->head_dim;
    int g = h / (a->num_q_heads / a->num_kv_heads);
    int n = t1 - t0;
    for (int i = 0; i < d; ++i) acc[i] = 0.0;
    *m_out = -INFINITY;
    *l_out = 0.0;
    if (n <= 0) return 0;
    double* q = malloc(sizeof(double) * d);
    double* row = malloc(sizeof(double) * d);
    double* z = malloc(sizeof(double) * n);
    int rc = 0;
    for (int i = 0; i < d; ++i)
        q[i] = load_elem(a->query, a->q_dtype, ((int64_t)qrow * a->num_q_heads + h) * d + i);
    /* pass 1: logits, [P1] §3 S_ij = q^T K_j^T / sqrt(d) (scale passed in) */
    double m = -INFINITY;
    for (int t = t0; t < t1 && !rc; ++t) {
        rc = fetch_row(a, a->k_cache, s, g, t, row);
        double dot = 0.0;
        for (int i = 0; i < d; ++i) dot += q[i] * row[i];
        z[t - t0] = a->scale * dot;
        if (z[t - t0] > m) m = z[t - t0];
    }
    /* pass 2: weights and the weighted sum of values, [P1] §3 o_i = sum_j A_ij V_j */
    double l = 0.0;
    for (int t = t0; t < t1 && !rc; ++t) {
        double w = exp(z[t - t0] - m);
        l += w;
        rc = fetch_row(a, a->v_cache, s, g, t, row);
        for (int i = 0; i < d; ++i) acc[i] += w * row[i];
    }
    *m_out = m;
    *l_out = l;
    free(q); free(row); free(z);
    return rc;
}

static void fill_args(dec_args* a, const void* query, const void* k_cache, const void* v_cache,
                      const int32_t* block_tables, const int32_t* context_lens,
                      int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                      int num_blocks, int max_blocks, double scale, int q_dtype,
                      int kv_dtype, double kv_scale) {
    a->query = query; a->k_cache = k_cache; a->v_cache = v_cache;
    a->block_tables = block_tables; a->context_lens = context_lens;
    a->num_q_heads = num_q_heads; a->num_kv_heads = num_kv_heads; a->head_dim = head_dim;
    a->block_size = block_size; a->num_blocks = num_blocks; a->max_blocks = max_blocks;
    a->scale = scale; a->q_dtype = q_dtype; a->kv_dtype = kv_dtype; a->kv_scale = kv_scale;
}

/*
 * Paged decode attention for the (seq, q head) pairs listed in `sel`
 * (sel[2k] = seq, sel[2k+1] = q head); out[k][:] receives the fp64 output
 * o = softmax(scale * q K^T) V over the sequence's context_lens[seq] tokens,
 * gathered block by block through its block-table row.  context_len 0 gives
 * zeros.  `nthreads` > 1 runs independent pairs on several threads; every
 * pair's arithmetic is the same sequential loop either way.
 * Returns 0, or -1 on a bad argument / an out-of-range block id.
 */
int oracle_paged_decode_attention(const void* query, const void* k_cache, const void* v_cache,
                                  const int32_t* block_tables, const int32_t* context_lens,
                                  int num_q_heads, int num_kv_heads, int head_dim,
                                  int block_size, int num_blocks, int max_blocks, double scale,
                                  int q_dtype, int kv_dtype, double kv_scale,
                                  const int32_t* sel, int num_sel, double* out, int nthreads) {
    if (num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0) return -1;
    if (!elem_bytes(q_dtype) || q_dtype == OR_E4M3 || !elem_bytes(kv_dtype)) return -1;
    dec_args a;
    fill_args(&a, query, k_cache, v_cache, block_tables, context_lens, num_q_heads,
              num_kv_heads, head_dim, block_size, num_blocks, max_blocks, scale, q_dtype,
              kv_dtype, kv_scale);
    int bad = 0;
    (void)nthreads;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads > 0 ? nthreads : 1) reduction(| : bad)
    for (int k = 0; k < num_sel; ++k) {
        int s = sel[2 * k], h = sel[2 * k + 1];
        int ctx = context_lens[s];
        double m, l;
        double* o = out + (int64_t)k * head_dim;
        if (ctx > max_blocks * block_size) { bad = 1; continue; }
        if (partial_state(&a, s, s, h, 0, ctx, &m, &l, o)) { bad = 1; continue; }
        if (ctx == 0) continue;                          /* zeros */
        for (int i = 0; i < head_dim; ++i) o[i] /= l;
    }
    return bad ? -1 : 0;
}

/*
 * Split-KV partial state of (seq, q head) over tokens [t0, t1): m, l and the
 * unnormalised acc[head_dim] (see partial_state).  The pages do not split the
 * context; this and oracle_merge_partials state the merge that the running
 * rescale of the [P1] §7 decode pseudocode implies.
 */
int oracle_attention_partial(const void* query, const void* k_cache, const void* v_cache,
                             const int32_t* block_tables, int num_q_heads, int num_kv_heads,
                             int head_dim, int block_size, int num_blocks, int max_blocks,
                             double scale, int q_dtype, int kv_dtype, double kv_scale, int seq,
                             int q_head, int t0, int t1, double* m, double* l, double* acc) {
    dec_args a;
    fill_args(&a, query, k_cache, v_cache, block_tables, NULL, num_q_heads, num_kv_heads,
              head_dim, block_size, num_blocks, max_blocks, scale, q_dtype, kv_dtype, kv_scale);
    return partial_state(&a, seq, seq, q_head, t0, t1, m, l, acc);
}

/*
 * Merge n partial states in the given order, as the rescale step of the
 * [P1] §7 pseudocode does block by block: with M = max m_k,
 *   l = sum_k l_k exp(m_k - M),  acc = sum_k acc_k exp(m_k - M),  o = acc / l.
 * Partials with m_k = -inf (empty ranges) contribute nothing.  All empty -> 0.
 */
void oracle_merge_partials(int n, const double* ms, const double* ls, const double* accs,
                           int head_dim, double* out) {
    double M = -INFINITY;
    for (int k = 0; k < n; ++k)
        if (ms[k] > M) M = ms[k];
    for (int i = 0; i < head_dim; ++i) out[i] = 0.0;
    if (M == -INFINITY) return;
    double l = 0.0;
    for (int k = 0; k < n; ++k) {
        if (ms[k] == -INFINITY) continue;
        double f = exp(ms[k] - M);
        l += ls[k] * f;
        for (int i = 0; i < head_dim; ++i) out[i] += accs[(int64_t)k * head_dim + i] * f;
    }
    for (int i = 0; i < head_dim; ++i) out[i] /= l;
}

/* ------------------- multi-query paged attention ([P1] §1, §3) ----------- */

/*
 * Causal attention of several query tokens per sequence over the paged cache
 * (prefill, chunked prefill, or verifying a chain of draft tokens).  Sequence s
 * owns query rows query_start[s] .. query_start[s+1]-1 of `query`
 * ([total_q, num_q_heads, head_dim]); its cache holds context_lens[s] >= n_s
 * tokens, the last n_s of them being these queries' own keys and values.
 * Query i of the sequence is the token at logical position p = ctx - n_s + i
 * and, like every generated token in [P1] §1, attends to all tokens before it
 * and to itself: o = softmax(scale * q K[0..p]^T) V[0..p] ([P1] §3), i.e. the
 * decode attention of that row over the first p + 1 tokens.
 * `sel` lists (query row, query head) pairs; out[k][:] gets pair k's output.
 * Returns 0, or -1 on a bad argument, n_s > ctx_s, or a block id out of range.
 */
int oracle_paged_prefill_attention(const void* query, const void* k_cache, const void* v_cache,
                                   const int32_t* block_tables, const int32_t* context_lens,
                                   const int32_t* query_start, int num_seqs, int num_q_heads,
                                   int num_kv_heads, int head_dim, int block_size, int num_blocks,
                                   int max_blocks, double scale, int q_dtype, int kv_dtype,
                                   double kv_scale, const int32_t* sel, int num_sel, double* out,
                                   int nthreads) {
    if (num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0 || num_seqs < 0) return -1;
    if (!elem_bytes(q_dtype) || q_dtype == OR_E4M3 || !elem_bytes(kv_dtype)) return -1;
    dec_args a;
    fill_args(&a, query, k_cache, v_cache, block_tables, context_lens, num_q_heads,
              num_kv_heads, head_dim, block_size, num_blocks, max_blocks, scale, q_dtype,
              kv_dtype, kv_scale);
    int bad = 0;
    (void)nthreads;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads > 0 ? nthreads : 1) reduction(| : bad)
    for (int k = 0; k < num_sel; ++k) {
        int row = sel[2 * k], h = sel[2 * k + 1];
        double* o = out + (int64_t)k * head_dim;
        /* the sequence owning this query row */
        int s = -1;
        for (int j = 0; j < num_seqs; ++j)
            if (query_start[j] <= row && row < query_start[j + 1]) { s = j; break; }
        if (s < 0) { bad = 1; continue; }
        int n = query_start[s + 1] - query_start[s];
        int ctx = context_lens[s];
        if (n > ctx || ctx > max_blocks * block_size) { bad = 1; continue; }
        int p = ctx - n + (row - query_start[s]);        /* logical position of the query */
        double m, l;
        if (partial_state(&a, s, row, h, 0, p + 1, &m, &l, o)) { bad = 1; continue; }
        for (int i = 0; i < head_dim; ++i) o[i] /= l;
    }
    return bad ? -1 : 0;
}

/*
 * Verification of a tree of draft tokens (speculative decoding trees, [P1] §9):
 * the last n_s <= 64 tokens of sequence s are the tree's tokens, laid out so that
 * every token comes after its ancestors.  Query i of the sequence sees every
 * token of the prior context (positions < c0 = ctx - n_s), itself (position
 * c0 + i), and each earlier tree token j < i whose bit j is set in
 * tree[query_start[s] + i] (its ancestors); bits j >= i are ignored.  With
 * bits 0 .. i-1 set this is the causal attention above.  The output is the
 * softmax-weighted sum over exactly that set of tokens ([P1] §3), in fp64.
 */
int oracle_paged_tree_attention(const void* query, const void* k_cache, const void* v_cache,
                                const int32_t* block_tables, const int32_t* context_lens,
                                const int32_t* query_start, const uint64_t* tree, int num_seqs,
                                int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                int num_blocks, int max_blocks, double scale, int q_dtype,
                                int kv_dtype, double kv_scale, const int32_t* sel, int num_sel,
                                double* out, int nthreads) {
    if (num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0 || num_seqs < 0 || !tree) return -1;
    if (!elem_bytes(q_dtype) || q_dtype == OR_E4M3 || !elem_bytes(kv_dtype)) return -1;
    dec_args a;
    fill_args(&a, query, k_cache, v_cache, block_tables, context_lens, num_q_heads,
              num_kv_heads, head_dim, block_size, num_blocks, max_blocks, scale, q_dtype,
              kv_dtype, kv_scale);
    int bad = 0;
    (void)nthreads;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads > 0 ? nthreads : 1) reduction(| : bad)
    for (int k = 0; k < num_sel; ++k) {
        int row = sel[2 * k], h = sel[2 * k + 1];
        double* o = out + (int64_t)k * head_dim;
        int s = -1;
        for (int j = 0; j < num_seqs; ++j)
            if (query_start[j] <= row && row < query_start[j + 1]) { s = j; break; }
        if (s < 0) { bad = 1; continue; }
        int n = query_start[s + 1] - query_start[s];
        int ctx = context_lens[s];
        if (n > 64 || n > ctx || ctx > max_blocks * block_size) { bad = 1; continue; }
        int c0 = ctx - n, i = row - query_start[s];
        uint64_t bits = tree[row];
        /* the visible positions: the prior context, then ancestors and the token itself */
        int* pos = malloc(sizeof(int) * (size_t)(c0 + i + 1));
        int np = 0;
        for (int t = 0; t < c0; ++t) pos[np++] = t;
        for (int j = 0; j < i; ++j)
            if ((bits >> j) & 1u) pos[np++] = c0 + j;
        pos[np++] = c0 + i;
        /* softmax over the visible logits, the weighted sum of their values */
        int d = head_dim, g = h / (num_q_heads / num_kv_heads), rc = 0;
        double* q = malloc(sizeof(double) * d);
        double* krow = malloc(sizeof(double) * d);
        double* z = malloc(sizeof(double) * np);
        for (int e = 0; e < d; ++e)
            q[e] = load_elem(a.query, a.q_dtype, ((int64_t)row * num_q_heads + h) * d + e);
        double m = -INFINITY;
        for (int u = 0; u < np && !rc; ++u) {
            rc = fetch_row(&a, a.k_cache, s, g, pos[u], krow);
            double dot = 0.0;
            for (int e = 0; e < d; ++e) dot += q[e] * krow[e];
            z[u] = a.scale * dot;
            if (z[u] > m) m = z[u];
        }
        double l = 0.0;
        for (int e = 0; e < d; ++e) o[e] = 0.0;
        for (int u = 0; u < np && !rc; ++u) {
            double w = exp(z[u] - m);
            l += w;
            rc = fetch_row(&a, a.v_cache, s, g, pos[u], krow);
            for (int e = 0; e < d; ++e) o[e] += w * krow[e];
        }
        for (int e = 0; e < d; ++e) o[e] /= l;
        free(pos); free(q); free(krow); free(z);
        if (rc) bad = 1;
    }
    return bad ? -1 : 0;
}

/* Threads the OpenMP runtime would give a parallel region (1 without OpenMP). */
int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
