/*
 * attn_oracle.c -- plain, slow FP64 reference for grouped-query attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file: only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header or constant with the
 * CUDA library.
 *
 * What it computes (the definition, written out, no blocking or fusion):
 *
 *   scale  = 1 / sqrt(D)
 *   g(h)   = floor(h * H_kv / H_q)                         (GQA head map)
 *   s_j    = scale * sum_d q[d] * k_j[d]                    (scores)
 *   M      = max_j s_j
 *   w_j    = exp(s_j - M) / sum_k exp(s_k - M)              (softmax)
 *   o[d]   = sum_j w_j * v_j[d]
 *   lse    = M + log(sum_j exp(s_j - M))
 *
 * Sources:
 *  - "Tutorial: Adding a New Kernel to RL.cu" (add-cuda-kernel page),
 *    header include/kernels/attention.cuh, "Flash Attention 2 -- Prefill":
 *    [B,S,H,D] layouts, kv_head = q_head*H_kv/H_q, causal "token i attends
 *    only to positions <= i", FP16 I/O.
 *  - same page, "Paged Attention -- Decode": q [num_seqs,H_q,D], caches
 *    [num_blocks,H_kv,block_size,D], block_tables [num_seqs,max_blocks_per_seq]
 *    mapping logical to physical blocks, seq_lens = context length including
 *    the new token.
 *  - same page, tests/test_attention.cu, ref_attention / ref_decode_attention:
 *    the two-pass, max-subtracted softmax on FP16-quantised inputs; scale
 *    1/sqrt(D).  Here it is done in double instead of float.
 *  - Kimi-K2.6 KernelBench trace (fused cross-attention page), the derivation
 *    that o_N / l_N of the online recurrence equals sum v e^s / sum e^s: the
 *    basis of oracle_lse_combine (merging partial results by their lse).
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *  - an empty key set (seq_len == 0) gives o = 0 and lse = -inf;
 *  - causal=0 attends to all S keys;
 *  - NaN/Inf inputs propagate with no special handling;
 *  - RoPE pairs element i with element i + D/2 (the split-half form the
 *    Qwen3 notes name) and pair i turns by pos * base^(-2i/D); the base is a
 *    parameter (the pages print none).
 *
 * Every function here is pinned by tests against torch float64 SDPA and
 * rms_norm on tiny shapes, a complex-number form of the rotation, closed forms
 * and invariants; see tests/test_oracle_pins.py.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* IEEE 754 binary16 -> double, exact (every half is a double).
 * Layout: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double oracle_half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int exp = (h >> 10) & 0x1f;
    int frac = h & 0x3ff;
    double v;
    if (exp == 0) {
        v = ldexp((double)frac, -24); /* subnormal: frac * 2^-14 * 2^-10 */
    } else if (exp == 31) {
        v = frac ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + frac), exp - 25); /* (1 + frac/1024) * 2^(exp-15) */
    }
    return sign ? -v : v;
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Threads for the calls that follow (n >= 1); used to time the oracle on one core. */
void oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n >= 1)
        omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/*
 * Attention of one query vector over n keys.
 * q: D halves.  key(j) / val(j): pointers to the j-th key / value row (D halves).
 * scores: caller scratch of n doubles.  Writes o[D] and *lse.
 */
typedef const uint16_t *(*row_fn)(const void *ctx, int j);

static void attend_one(const uint16_t *q, int D, int n, row_fn key, row_fn val,
                       const void *ctx, double *scores, double *o, double *lse)
{
    const double scale = 1.0 / sqrt((double)D);
    for (int d = 0; d < D; d++)
        o[d] = 0.0;
    if (n <= 0) {
        *lse = -INFINITY;
        return;
    }
    /* pass 1: scores and their maximum */
    double M = -INFINITY;
    for (int j = 0; j < n; j++) {
        const uint16_t *k = key(ctx, j);
        double dot = 0.0;
        for (int d = 0; d < D; d++)
            dot += oracle_half_to_double(q[d]) * oracle_half_to_double(k[d]);
        scores[j] = dot * scale;
        if (scores[j] > M)
            M = scores[j];
    }
    /* pass 2: normaliser */
    double sum = 0.0;
    for (int j = 0; j < n; j++)
        sum += exp(scores[j] - M);
    /* pass 3: weighted sum of values */
    for (int j = 0; j < n; j++) {
        const double w = exp(scores[j] - M) / sum;
        const uint16_t *v = val(ctx, j);
        for (int d = 0; d < D; d++)
            o[d] += w * oracle_half_to_double(v[d]);
    }
    *lse = M + log(sum);
}

/* ---------------------------------------------------------------- prefill */

typedef struct {
    const uint16_t *K, *V;
    long row_stride; /* halves between consecutive sequence positions */
    long base;       /* offset of (b, position 0, kv head g) */
} contig_ctx;

static const uint16_t *contig_key(const void *c, int j)
{
    const contig_ctx *x = (const contig_ctx *)c;
    return x->K + x->base + (long)j * x->row_stride;
}
static const uint16_t *contig_val(const void *c, int j)
{
    const contig_ctx *x = (const contig_ctx *)c;
    return x->V + x->base + (long)j * x->row_stride;
}

static void prefill_row(const uint16_t *Q, const uint16_t *K, const uint16_t *V, int S,
                        int H_q, int H_kv, int D, int causal, int b, int i, int h,
                        double *scores, double *o, double *lse)
{
    const int g = (int)(((long)h * H_kv) / H_q);
    contig_ctx c;
    c.K = K;
    c.V = V;
    c.row_stride = (long)H_kv * D;
    c.base = ((long)b * S * H_kv + g) * D;
    const uint16_t *q = Q + (((long)b * S + i) * H_q + h) * D;
    const int n = causal ? i + 1 : S;
    attend_one(q, D, n, contig_key, contig_val, &c, scores, o, lse);
}

/*
 * Full prefill.  Q,O: [B,S,H_q,D]; K,V: [B,S,H_kv,D]; lse: [B,S,H_q] (may be NULL).
 * O is unrounded double.
 */
void oracle_prefill(const uint16_t *Q, const uint16_t *K, const uint16_t *V, int B, int S,
                    int H_q, int H_kv, int D, int causal, double *O, double *lse)
{
    const long rows = (long)B * S * H_q;
#pragma omp parallel
    {
        double *scores = (double *)malloc(sizeof(double) * (S > 0 ? S : 1));
#pragma omp for schedule(dynamic, 16)
        for (long r = 0; r < rows; r++) {
            const int h = (int)(r % H_q);
            const int i = (int)((r / H_q) % S);
            const int b = (int)(r / ((long)H_q * S));
            double l;
            prefill_row(Q, K, V, S, H_q, H_kv, D, causal, b, i, h, scores, O + r * D, &l);
            if (lse)
                lse[r] = l;
        }
        free(scores);
    }
}

/*
 * Selected prefill rows.  rows: n_rows triples (b, i, h).  O_rows: [n_rows, D].
 */
void oracle_prefill_rows(const uint16_t *Q, const uint16_t *K, const uint16_t *V, int B,
                         int S, int H_q, int H_kv, int D, int causal, const int32_t *rows,
                         int n_rows, double *O_rows, double *lse_rows)
{
    (void)B;
#pragma omp parallel
    {
        double *scores = (double *)malloc(sizeof(double) * (S > 0 ? S : 1));
#pragma omp for schedule(dynamic, 1)
        for (int r = 0; r < n_rows; r++) {
            double l;
            prefill_row(Q, K, V, S, H_q, H_kv, D, causal, rows[3 * r], rows[3 * r + 1],
                        rows[3 * r + 2], scores, O_rows + (long)r * D, &l);
            if (lse_rows)
                lse_rows[r] = l;
        }
        free(scores);
    }
}

/* ----------------------------------------------------------- paged decode */

typedef struct {
    const uint16_t *kc, *vc;
    const int32_t *table; /* this sequence's row of block_tables */
    int H_kv, bs, D, g;
} paged_ctx;

/* logical key t lives in physical block table[t / bs], slot t % bs */
static long paged_offset(const paged_ctx *x, int t)
{
    const long phys = x->table[t / x->bs];
    return ((phys * x->H_kv + x->g) * x->bs + (t % x->bs)) * (long)x->D;
}
static const uint16_t *paged_key(const void *c, int t)
{
    const paged_ctx *x = (const paged_ctx *)c;
    return x->kc + paged_offset(x, t);
}
static const uint16_t *paged_val(const void *c, int t)
{
    const paged_ctx *x = (const paged_ctx *)c;
    return x->vc + paged_offset(x, t);
}

static void decode_row(const uint16_t *q, const uint16_t *kc, const uint16_t *vc,
                       const int32_t *block_tables, const int32_t *seq_lens, int H_q,
                       int H_kv, int D, int max_blocks_per_seq, int block_size, int n, int h,
                       double *scores, double *o, double *lse)
{
    paged_ctx c;
    c.kc = kc;
    c.vc = vc;
    c.table = block_tables + (long)n * max_blocks_per_seq;
    c.H_kv = H_kv;
    c.bs = block_size;
    c.D = D;
    c.g = (int)(((long)h * H_kv) / H_q);
    attend_one(q + ((long)n * H_q + h) * D, D, seq_lens[n], paged_key, paged_val, &c, scores,
               o, lse);
}

static int max_len(const int32_t *seq_lens, int num_seqs)
{
    int m = 1;
    for (int n = 0; n < num_seqs; n++)
        if (seq_lens[n] > m)
            m = seq_lens[n];
    return m;
}

/*
 * Paged decode.  q,out: [num_seqs,H_q,D]; lse: [num_seqs,H_q] (may be NULL).
 */
void oracle_decode_paged(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                         const int32_t *block_tables, const int32_t *seq_lens, int num_seqs,
                         int H_q, int H_kv, int D, int max_blocks_per_seq, int block_size,
                         double *out, double *lse)
{
    const int L = max_len(seq_lens, num_seqs);
    const long rows = (long)num_seqs * H_q;
#pragma omp parallel
    {
        double *scores = (double *)malloc(sizeof(double) * L);
#pragma omp for schedule(dynamic, 1)
        for (long r = 0; r < rows; r++) {
            double l;
            decode_row(q, k_cache, v_cache, block_tables, seq_lens, H_q, H_kv, D,
                       max_blocks_per_seq, block_size, (int)(r / H_q), (int)(r % H_q),
                       scores, out + r * D, &l);
            if (lse)
                lse[r] = l;
        }
        free(scores);
    }
}

/* Selected decode rows.  rows: n_rows pairs (n, h).  out_rows: [n_rows, D]. */
void oracle_decode_paged_rows(const uint16_t *q, const uint16_t *k_cache,
                              const uint16_t *v_cache, const int32_t *block_tables,
                              const int32_t *seq_lens, int num_seqs, int H_q, int H_kv, int D,
                              int max_blocks_per_seq, int block_size, const int32_t *rows,
                              int n_rows, double *out_rows, double *lse_rows)
{
    const int L = max_len(seq_lens, num_seqs);
#pragma omp parallel
    {
        double *scores = (double *)malloc(sizeof(double) * L);
#pragma omp for schedule(dynamic, 1)
        for (int r = 0; r < n_rows; r++) {
            double l;
            decode_row(q, k_cache, v_cache, block_tables, seq_lens, H_q, H_kv, D,
                       max_blocks_per_seq, block_size, rows[2 * r], rows[2 * r + 1], scores,
                       out_rows + (long)r * D, &l);
            if (lse_rows)
                lse_rows[r] = l;
        }
        free(scores);
    }
}

/*
 * Merge partial results of the same query over disjoint key segments.
 * Partial i is (o_i, lse_i) with o_i the normalised attention over segment i.
 * Since o_i = sum_{j in i} v_j e^{s_j} / e^{lse_i}, the full result is
 *   L = log sum_i e^{lse_i},  o = sum_i e^{lse_i - L} o_i.
 * Segments with lse_i = -inf (empty) contribute nothing; if all are empty the
 * result is o = 0, L = -inf.
 * O_part: [R, n_split, D]; lse_part: [R, n_split]; out: [R, D]; lse: [R] or NULL.
 */
void oracle_lse_combine(const double *O_part, const double *lse_part, int R, int n_split,
                        int D, double *out, double *lse)
{
    for (int r = 0; r < R; r++) {
        const double *lp = lse_part + (long)r * n_split;
        double M = -INFINITY;
        for (int i = 0; i < n_split; i++)
            if (lp[i] > M)
                M = lp[i];
        double *o = out + (long)r * D;
        for (int d = 0; d < D; d++)
            o[d] = 0.0;
        if (M == -INFINITY) {
            if (lse)
                lse[r] = -INFINITY;
            continue;
        }
        double sum = 0.0;
        for (int i = 0; i < n_split; i++)
            sum += exp(lp[i] - M);
        const double L = M + log(sum);
        for (int i = 0; i < n_split; i++) {
            const double w = exp(lp[i] - L);
            const double *oi = O_part + ((long)r * n_split + i) * D;
            for (int d = 0; d < D; d++)
                o[d] += w * oi[d];
        }
        if (lse)
            lse[r] = L;
    }
}

/*
 * Write new K/V rows into their paged slots ("GRPO-CUDA Project Memory" page,
 * "KV Cache design": slot = physical_block * block_size + offset; slot -1 is a
 * padding token and is skipped).  Raw 16-bit copies, so the result is exact.
 * k_new, v_new: [T, H_kv, D]; caches: [num_blocks, H_kv, bs, D] updated in place.
 * Slots outside [0, num_blocks*bs) are skipped; returns how many were.
 */
int oracle_kv_append(const uint16_t *k_new, const uint16_t *v_new, uint16_t *k_cache,
                     uint16_t *v_cache, const int64_t *slot_mapping, int T, int H_kv, int D,
                     int bs, long num_blocks)
{
    int skipped = 0;
    for (int t = 0; t < T; t++) {
        const int64_t slot = slot_mapping[t];
        if (slot < 0 || slot >= (int64_t)num_blocks * bs) {
            if (slot != -1)
                skipped++;
            continue;
        }
        const long block = (long)(slot / bs);
        const int pos = (int)(slot % bs);
        for (int g = 0; g < H_kv; g++)
            for (int d = 0; d < D; d++) {
                const long dst = (((block * H_kv) + g) * bs + pos) * (long)D + d;
                const long src = ((long)t * H_kv + g) * (long)D + d;
                k_cache[dst] = k_new[src];
                v_cache[dst] = v_new[src];
            }
    }
    return skipped;
}

/*
 * Prefill of new query chunks against a paged KV cache (varlen, with cached
 * prefix).  Sequence b has L_q = cu_seqlens_q[b+1] - cu_seqlens_q[b] new
 * queries, packed at rows cu_seqlens_q[b].. of Q and O ([total_q, H_q, D]),
 * and a context of L_kv = seq_lens_kv[b] keys in the paged cache (its last
 * L_q keys belong to the new queries, L_kv >= L_q).  Query i of sequence b
 * sits at absolute position L_kv - L_q + i; with the causal mask it attends to
 * keys t <= L_kv - L_q + i, otherwise to all L_kv keys.  The key placement is
 * the paged layout of the "Paged Attention -- Decode" header; the causal rule
 * is the prefill one, shifted by the cached prefix.
 */
/* One output row (query i of sequence b, head h) of the paged prefill. */
static void prefill_paged_row(const uint16_t *Q, const uint16_t *k_cache,
                              const uint16_t *v_cache, const int32_t *cu_seqlens_q,
                              const int32_t *seq_lens_kv, const int32_t *block_tables, int H_q,
                              int H_kv, int D, int max_blocks_per_seq, int block_size,
                              int causal, int b, int i, int h, double *scores, double *o,
                              double *lse)
{
    const int Lq = cu_seqlens_q[b + 1] - cu_seqlens_q[b];
    const int Lkv = seq_lens_kv[b];
    paged_ctx c;
    c.kc = k_cache;
    c.vc = v_cache;
    c.table = block_tables + (long)b * max_blocks_per_seq;
    c.H_kv = H_kv;
    c.bs = block_size;
    c.D = D;
    c.g = (int)(((long)h * H_kv) / H_q);
    const int n = causal ? Lkv - Lq + i + 1 : Lkv;
    const long row = (long)cu_seqlens_q[b] + i;
    attend_one(Q + (row * H_q + h) * D, D, n, paged_key, paged_val, &c, scores, o, lse);
}

void oracle_prefill_paged(const uint16_t *Q, const uint16_t *k_cache, const uint16_t *v_cache,
                          const int32_t *cu_seqlens_q, const int32_t *seq_lens_kv,
                          const int32_t *block_tables, int B, int H_q, int H_kv, int D,
                          int max_blocks_per_seq, int block_size, int causal, double *O,
                          double *lse)
{
    const int total_q = cu_seqlens_q[B];
    const int L = max_len(seq_lens_kv, B);
    const long rows = (long)total_q * H_q;
#pragma omp parallel
    {
        double *scores = (double *)malloc(sizeof(double) * L);
#pragma omp for schedule(dynamic, 4)
        for (long r = 0; r < rows; r++) {
            const int h = (int)(r % H_q);
            const int row = (int)(r / H_q);
            int b = 0;
            while (cu_seqlens_q[b + 1] <= row)
                b++;
            double l;
            prefill_paged_row(Q, k_cache, v_cache, cu_seqlens_q, seq_lens_kv, block_tables, H_q,
                              H_kv, D, max_blocks_per_seq, block_size, causal, b,
                              row - cu_seqlens_q[b], h, scores, O + r * D, &l);
            if (lse)
                lse[r] = l;
        }
        free(scores);
    }
}

/*
 * Selected rows of the paged prefill.  rows: n_rows triples (b, i, h), query i
 * of sequence b's chunk; O_rows: [n_rows, D]; lse_rows: [n_rows] or NULL.
 */
void oracle_prefill_paged_rows(const uint16_t *Q, const uint16_t *k_cache,
                               const uint16_t *v_cache, const int32_t *cu_seqlens_q,
                               const int32_t *seq_lens_kv, const int32_t *block_tables, int B,
                               int H_q, int H_kv, int D, int max_blocks_per_seq, int block_size,
                               int causal, const int32_t *rows, int n_rows, double *O_rows,
                               double *lse_rows)
{
    const int L = max_len(seq_lens_kv, B);
#pragma omp parallel
    {
        double *scores = (double *)malloc(sizeof(double) * L);
#pragma omp for schedule(dynamic, 1)
        for (int r = 0; r < n_rows; r++) {
            double l;
            prefill_paged_row(Q, k_cache, v_cache, cu_seqlens_q, seq_lens_kv, block_tables, H_q,
                              H_kv, D, max_blocks_per_seq, block_size, causal, rows[3 * r],
                              rows[3 * r + 1], rows[3 * r + 2], scores, O_rows + (long)r * D, &l);
            if (lse_rows)
                lse_rows[r] = l;
        }
        free(scores);
    }
}

/*
 * Per-head QK-norm followed by rotary position embedding: the prologue that
 * turns projected q/k rows into the attention inputs.
 *
 *  - "GRPO-CUDA Project Memory" page, "Qwen3-Specific Notes": RMSNorm over
 *    each head's D = 128 values, applied before RoPE, eps 1e-6; "Model forward
 *    pass": QK-norm -> RoPE -> KV append -> attention.
 *  - same page, "RoPE design": NeoX split-half pairing, element i rotates with
 *    element i + D/2 for i < D/2; rotation arithmetic in full precision.
 *  - Kimi-K2.6 KernelBench trace (fused cross-attention page): pair i turns by
 *    the angle pos * base^(-2i/D).
 *
 *   r            = sqrt(mean_d x[d]^2 + eps)
 *   y[d]         = w[d] * x[d] / r          (y = x when w is NULL: RoPE only)
 *   a_i          = pos * base^(-2i/D),       i in [0, D/2)
 *   out[i]       = y[i] cos a_i - y[i + D/2] sin a_i
 *   out[i + D/2] = y[i + D/2] cos a_i + y[i] sin a_i
 *
 * x: [T, H, D] fp16 bits; w: [D] fp16 bits or NULL; positions: [T] int32, the
 * absolute position of each token; out: [T, H, D] double.
 */
void oracle_qk_norm_rope(const uint16_t *x, const uint16_t *w, const int32_t *positions, int T,
                         int H, int D, double base, double eps, double *out)
{
    const int half = D / 2;
#pragma omp parallel for schedule(dynamic, 16)
    for (long r = 0; r < (long)T * H; r++) {
        const int t = (int)(r / H);
        const uint16_t *xr = x + r * D;
        double *o = out + r * D;
        double y[1024];
        double ss = 0.0;
        for (int d = 0; d < D; d++) {
            y[d] = oracle_half_to_double(xr[d]);
            ss += y[d] * y[d];
        }
        if (w) {
            const double rms = sqrt(ss / D + eps);
            for (int d = 0; d < D; d++)
                y[d] = oracle_half_to_double(w[d]) * y[d] / rms;
        }
        for (int i = 0; i < half; i++) {
            const double a = (double)positions[t] * pow(base, -2.0 * i / D);
            const double c = cos(a), s = sin(a);
            o[i] = y[i] * c - y[i + half] * s;
            o[i + half] = y[i + half] * c + y[i] * s;
        }
    }
}
