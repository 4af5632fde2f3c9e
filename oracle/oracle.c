/*
 * oracle.c -- plain, slow fp64 CPU reference for single-token decode attention
 * over a paged KV cache (and the cache append, the rolling sliding-window cache,
 * Quest page selection, the FP8 indexer and the gated delta-rule decode step).
 *
 * TEST INFRASTRUCTURE ONLY. Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library. It shares no code,
 * header or table with the CUDA path, and the CUDA path never calls it.
 *
 * Every result is the plain definition written out: scores, one softmax over
 * the visible tokens, a weighted sum of values. No online softmax, no split,
 * no tiling. Inputs are read as stored (bf16 or fp32) and widened exactly to
 * double; all arithmetic is double (except where a function says it follows the
 * kernel's float32 to decide an integer, as the e4m3 quantizer does); outputs are
 * double.
 *
 * Sources (page title, section):
 *  - "Overview of Attention Mechanism", GQA / Code (repeat_kv and
 *    eager_attention_forward): scores q.k * scaling, softmax, times V; KV head
 *    j serves query heads j*n_rep .. j*n_rep + n_rep-1.
 *  - "All the attentions", section 4 (Sliding Window): key j is visible to
 *    query i iff j <= i and j > i - W.
 *  - "Long context, KV eviction and sparse attention", KV eviction:
 *    StreamingLLM: the first n_sink tokens are kept alongside the window.
 *  - "Attention Optimizations", Attention sinks; "Overview of Attention
 *    Mechanism", StreamingLLM (softmax-off-by-one): a learned sink is one more
 *    logit in the softmax denominator whose value vector is zero.
 *  - "All the attentions", section 8 (PagedAttention): logical page n of
 *    sequence b lives at physical page block_table[b][n]; output unchanged.
 *  - "Attention Optimizations", DSA / Computation Path: MLA caches one
 *    576-wide row per token (512 latent + 64 RoPE key); the first 512 entries
 *    are the value part. Indexer score I_t = sum_h w_h * ReLU(q_h . k_t);
 *    indices = the k largest scores.
 *  - "Attention Optimizations", KV cache size: bytes = S * 2 * layers *
 *    kv_heads * d_head * bytes_per_element.
 *  - "All the attentions", section 4: a sliding window's cache is a rolling
 *    buffer of W entries, the newest replacing the oldest; "Attention
 *    Optimizations", DSA / Computation Path: the new token's row goes into the
 *    cache before attention (update_cache).
 *  - "Long context, KV eviction and sparse attention", Sparse attention (Quest):
 *    per page of keys the elementwise minimum and maximum; the upper bound of
 *    a query's scores in a page is sum_d max(q_d kmin_d, q_d kmax_d); each
 *    query head attends over the pages with the largest bounds plus the
 *    trailing partial page.
 *  - "All the attentions", sections 6 (Gated DeltaNet) and 7 (KDA); "Attention
 *    Optimizations", KDA: one decode step of the gated delta rule per head on
 *    a dv x dk state: fade, correction write, read.
 *
 * Conventions: seq_lens[b] counts cached tokens including the token being
 * decoded, so the query sits at position i = L_b - 1 and every cached token
 * t <= i. dtype 0 = float32, 1 = bfloat16 (stored as uint16).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static double widen(const void *base, int dtype, size_t i) {
    if (dtype == 0) return (double)((const float *)base)[i];
    uint32_t u = (uint32_t)((const uint16_t *)base)[i] << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Physical row of logical token t of sequence b; rows are page-major with
 * `heads_per_page` head slots per page (the GQA pool stores [page][head][slot]). */
static size_t pool_row(const int32_t *block_table, int max_pages, int page_size,
                       int heads_per_page, int b, int head, long t) {
    int page = block_table[(size_t)b * max_pages + t / page_size];
    return ((size_t)page * heads_per_page + head) * page_size + (size_t)(t % page_size);
}

/* KV cache size: tokens * 2 (K and V) * layers * kv heads * head dim * bytes. */
double oracle_kv_cache_bytes(double tokens, double layers, double kv_heads, double d_head,
                             double bytes_per_elem) {
    return tokens * 2.0 * layers * kv_heads * d_head * bytes_per_elem;
}

/* MLA cache size: one (latent + RoPE key) row per token per layer, no K/V pair. */
double oracle_mla_cache_bytes(double tokens, double layers, double d_latent, double d_rope,
                              double bytes_per_elem) {
    return tokens * layers * (d_latent + d_rope) * bytes_per_elem;
}

/* Attention FLOPs for one token that sees S tokens: 4 * S * heads * head_dim per
 * layer (half for q.k, half for p.v), times layers. */
double oracle_attention_flops(double S, double layers, double heads, double head_dim) {
    return 4.0 * S * heads * head_dim * layers;
}

/* Is token t visible to the query at position L-1?
 * window <= 0 means no window (all t < L). */
static int visible(long t, long L, long window, long n_sink) {
    if (t < 0 || t >= L) return 0;
    if (t < n_sink) return 1;
    if (window <= 0) return 1;
    long i = L - 1;
    return t <= i && t > i - window;
}

/*
 * Grouped-query attention for one decode token per sequence.
 * q [B,Hq,D]; k_pool, v_pool [num_pages,Hkv,P,D]; out [B,Hq,D]; lse [B,Hq]
 * (natural log of the softmax denominator, with the max folded back in).
 * sink_logit: NULL or [Hq] (logit in the same units as scale*q.k).
 * pairs: NULL (all (b,h)) or n_pairs (b,h) pairs; out/lse are then indexed by pair.
 */
/* Cache slot of token t: t itself in a paged cache (ring_window == 0); in a rolling cache of
 * ring_sink + ring_window slots the sinks keep theirs and later tokens cycle through the rest. */
static long cache_slot(long t, long ring_window, long ring_sink) {
    if (ring_window <= 0 || t < ring_sink) return t;
    return ring_sink + (t - ring_sink) % ring_window;
}

static void gqa_impl(const void *q, const void *k_pool, const void *v_pool, int dtype,
                     const int32_t *block_table, const int32_t *seq_lens, int B, int Hq,
                     int Hkv, int D, int page_size, int max_pages, double scale, long window,
                     long n_sink, const double *sink_logit, const int32_t *pairs, int n_pairs,
                     double *out, double *lse, long ring_window, long ring_sink) {
    int n_rep = Hq / Hkv;
    int n = pairs ? n_pairs : B * Hq;
#pragma omp parallel for schedule(dynamic, 1)
    for (int p = 0; p < n; p++) {
        int b = pairs ? pairs[2 * p] : p / Hq;
        int h = pairs ? pairs[2 * p + 1] : p % Hq;
        int g = h / n_rep;
        long L = seq_lens[b];
        double *s = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
        double m = -INFINITY;
        for (long t = 0; t < L; t++) {
            if (!visible(t, L, window, n_sink)) continue;
            size_t row = pool_row(block_table, max_pages, page_size, Hkv, b, g,
                                  cache_slot(t, ring_window, ring_sink));
            double dot = 0.0;
            for (int d = 0; d < D; d++)
                dot += widen(q, dtype, ((size_t)b * Hq + h) * D + d) *
                       widen(k_pool, dtype, row * D + d);
            s[t] = scale * dot;
            if (s[t] > m) m = s[t];
        }
        double sig = sink_logit ? sink_logit[h] : -INFINITY;
        if (sig > m) m = sig;
        double denom = 0.0;
        double *o = out + (size_t)p * D;
        for (int d = 0; d < D; d++) o[d] = 0.0;
        for (long t = 0; t < L; t++) {
            if (!visible(t, L, window, n_sink)) continue;
            size_t row = pool_row(block_table, max_pages, page_size, Hkv, b, g,
                                  cache_slot(t, ring_window, ring_sink));
            double e = exp(s[t] - m);
            denom += e;
            for (int d = 0; d < D; d++) o[d] += e * widen(v_pool, dtype, row * D + d);
        }
        if (sink_logit) denom += exp(sig - m); /* sink: denominator only, zero value */
        for (int d = 0; d < D; d++) o[d] /= denom;
        lse[p] = m + log(denom);
        free(s);
    }
}

void oracle_gqa(const void *q, const void *k_pool, const void *v_pool, int dtype,
                const int32_t *block_table, const int32_t *seq_lens, int B, int Hq, int Hkv,
                int D, int page_size, int max_pages, double scale, long window, long n_sink,
                const double *sink_logit, const int32_t *pairs, int n_pairs, double *out,
                double *lse) {
    gqa_impl(q, k_pool, v_pool, dtype, block_table, seq_lens, B, Hq, Hkv, D, page_size,
             max_pages, scale, window, n_sink, sink_logit, pairs, n_pairs, out, lse, 0, 0);
}

/*
 * Sliding window + sinks read from a rolling cache: the visible positions are those of
 * oracle_gqa with the same window and n_sink (L = seq_lens[b], the true length), and the
 * K/V of position t are read from cache slot n_sink + (t - n_sink) mod window (t itself for
 * a sink), where cache append put them.
 */
void oracle_gqa_ring(const void *q, const void *k_ring, const void *v_ring, int dtype,
                     const int32_t *block_table, const int32_t *seq_lens, int B, int Hq,
                     int Hkv, int D, int page_size, int max_pages, double scale, long window,
                     long n_sink, const double *sink_logit, const int32_t *pairs, int n_pairs,
                     double *out, double *lse) {
    gqa_impl(q, k_ring, v_ring, dtype, block_table, seq_lens, B, Hq, Hkv, D, page_size,
             max_pages, scale, window, n_sink, sink_logit, pairs, n_pairs, out, lse, window,
             n_sink);
}

/*
 * Absorbed-latent MLA decode (one shared 576-wide row per token).
 * q [B,H,d_qk]; c_pool [num_pages,P,d_qk] (dtype 0 float32 / 1 bf16);
 * out [B,H,d_v]; lse [B,H].
 * idx: NULL (dense: tokens 0..L_b-1) or [B, idx_stride] logical token indices
 * with idx_count[b] valid entries (sparse, the DSA selection).
 * Score s_t = scale * sum_{j<d_qk} q_j c_t[j]; value = c_t[0:d_v].
 */
void oracle_mla(const void *q, const void *c_pool, int dtype, const int32_t *block_table,
                const int32_t *seq_lens, const int32_t *idx, const int32_t *idx_count,
                int idx_stride, int B, int H, int d_qk, int d_v, int page_size, int max_pages,
                double scale, const int32_t *pairs, int n_pairs, double *out, double *lse) {
    int n = pairs ? n_pairs : B * H;
#pragma omp parallel for schedule(dynamic, 1)
    for (int p = 0; p < n; p++) {
        int b = pairs ? pairs[2 * p] : p / H;
        int h = pairs ? pairs[2 * p + 1] : p % H;
        long L = seq_lens[b];
        long cnt = idx ? idx_count[b] : L;
        double *s = (double *)malloc(sizeof(double) * (size_t)(cnt > 0 ? cnt : 1));
        double m = -INFINITY;
        for (long j = 0; j < cnt; j++) {
            long t = idx ? idx[(size_t)b * idx_stride + j] : j;
            size_t row = pool_row(block_table, max_pages, page_size, 1, b, 0, t);
            double dot = 0.0;
            for (int d = 0; d < d_qk; d++)
                dot += widen(q, dtype, ((size_t)b * H + h) * d_qk + d) *
                       widen(c_pool, dtype, row * d_qk + d);
            s[j] = scale * dot;
            if (s[j] > m) m = s[j];
        }
        double denom = 0.0;
        double *o = out + (size_t)p * d_v;
        for (int d = 0; d < d_v; d++) o[d] = 0.0;
        for (long j = 0; j < cnt; j++) {
            long t = idx ? idx[(size_t)b * idx_stride + j] : j;
            size_t row = pool_row(block_table, max_pages, page_size, 1, b, 0, t);
            double e = exp(s[j] - m);
            denom += e;
            for (int d = 0; d < d_v; d++) o[d] += e * widen(c_pool, dtype, row * d_qk + d);
        }
        for (int d = 0; d < d_v; d++) o[d] /= denom;
        lse[p] = m + log(denom);
        free(s);
    }
}

/*
 * Lightning-indexer scores: I_t = sum_h w_h * max(0, sum_j q_h[j] k_t[j]).
 * q [B,Hi,Di] bf16; k_pool [num_pages,P,Di] bf16; w [B,Hi] float32;
 * scores [n_b, out_stride] for the listed batch rows (t < L_b written).
 */
void oracle_indexer_scores(const void *q, const void *k_pool, const float *w,
                           const int32_t *block_table, const int32_t *seq_lens, int Hi, int Di,
                           int page_size, int max_pages, const int32_t *b_list, int n_b,
                           long out_stride, double *scores) {
    for (int bi = 0; bi < n_b; bi++) {
        int b = b_list[bi];
        long L = seq_lens[b];
#pragma omp parallel for schedule(static)
        for (long t = 0; t < L; t++) {
            size_t row = pool_row(block_table, max_pages, page_size, 1, b, 0, t);
            double total = 0.0;
            for (int h = 0; h < Hi; h++) {
                double dot = 0.0;
                for (int j = 0; j < Di; j++)
                    dot += widen(q, 1, ((size_t)b * Hi + h) * Di + j) *
                           widen(k_pool, 1, row * Di + j);
                total += (double)w[(size_t)b * Hi + h] * (dot > 0.0 ? dot : 0.0);
            }
            scores[(size_t)bi * out_stride + t] = total;
        }
    }
}

typedef struct {
    double score;
    int32_t index;
} scored_t;

/* larger score first; equal scores: lower index first */
static int by_score_then_index(const void *a, const void *b) {
    const scored_t *x = (const scored_t *)a, *y = (const scored_t *)b;
    if (x->score > y->score) return -1;
    if (x->score < y->score) return 1;
    return (x->index > y->index) - (x->index < y->index);
}

static int ascending_i32(const void *a, const void *b) {
    int32_t x = *(const int32_t *)a, y = *(const int32_t *)b;
    return (x > y) - (x < y);
}

/*
 * Top-k selection: the indices of the min(k, L) largest scores, ties going to
 * the lower index; written in ascending index order to idx_out[0..count-1].
 * Returns count.
 */
int oracle_topk(const double *scores, long L, int k, int32_t *idx_out) {
    scored_t *all = (scored_t *)malloc(sizeof(scored_t) * (size_t)(L > 0 ? L : 1));
    for (long t = 0; t < L; t++) {
        all[t].score = scores[t];
        all[t].index = (int32_t)t;
    }
    qsort(all, (size_t)L, sizeof(scored_t), by_score_then_index);
    int count = (long)k < L ? k : (int)L;
    for (int j = 0; j < count; j++) idx_out[j] = all[j].index;
    qsort(idx_out, (size_t)count, sizeof(int32_t), ascending_i32);
    free(all);
    return count;
}

/*
 * FP8 lightning indexer ("Long context, KV eviction and sparse attention", section on
 * exact selection with a fast scorer: the indexer scores every past token with few heads
 * in FP8). The pages give neither the code format nor the scaling; the readings used:
 *  - codes are e4m3: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits; exponent field
 *    0 holds subnormals (m/8 * 2^-6); S.1111.111 is NaN; no infinities; largest finite
 *    value 448;
 *  - one float32 scale per key row (token) and per query row (head): amax / 448, so that
 *    the largest magnitude lands on the largest finite code (a row of zeros: scale 1);
 *  - a value is encoded as the nearest code to x / scale (ties: the code with the even
 *    last bit), magnitudes above 448 saturating to 448.
 */
double oracle_e4m3_decode(int code) {
    int sign = (code >> 7) & 1, e = (code >> 3) & 15, m = code & 7;
    if (e == 15 && m == 7) return NAN;
    double v = (e == 0) ? ldexp(m / 8.0, -6) : ldexp(1.0 + m / 8.0, e - 7);
    return sign ? -v : v;
}

/* Nearest e4m3 code to the float32 x, by comparison with every finite code. */
int oracle_e4m3_encode(float xf) {
    double x = (double)xf;
    if (isnan(x)) return 0x7F;
    int sign = x < 0 || (x == 0 && signbit(x));
    double a = fabs(x);
    if (a >= 448.0) return (sign << 7) | 0x7E;
    int best = 0;
    double best_d = a;  /* distance to code 0 (value 0) */
    for (int c = 1; c <= 0x7E; c++) {
        double d = fabs(oracle_e4m3_decode(c) - a);
        if (d < best_d || (d == best_d && (c & 1) == 0)) {
            best = c;
            best_d = d;
        }
    }
    return (sign << 7) | best;
}

/* Row-wise quantization of bf16 x [rows, cols] to e4m3 codes and one float32 scale per row.
 * The scale and the quotients are computed in float32, as the kernel does, so that both
 * sides round the same values. */
void oracle_quantize_e4m3_rows(const void *x, long rows, int cols, uint8_t *codes,
                               float *scales) {
    for (long r = 0; r < rows; r++) {
        float amax = 0.0f;
        for (int c = 0; c < cols; c++) {
            float v = (float)widen(x, 1, (size_t)r * cols + c);
            if (fabsf(v) > amax) amax = fabsf(v);
        }
        float s = amax > 0.0f ? amax / 448.0f : 1.0f;
        scales[r] = s;
        for (int c = 0; c < cols; c++) {
            float v = (float)widen(x, 1, (size_t)r * cols + c);
            codes[(size_t)r * cols + c] = (uint8_t)oracle_e4m3_encode(v / s);
        }
    }
}

/*
 * FP8 indexer scores: I_t = sum_h w_h * max(0, sum_j (sq_h q8_h[j]) (sk_t k8_t[j])) with
 * every code decoded exactly. q8 [B,Hi,Di], q_scale [B,Hi]; k8_pool [num_pages,P,Di],
 * k_scale [num_pages*P] (per physical row); w [B,Hi].
 */
void oracle_indexer_scores_fp8(const uint8_t *q8, const float *q_scale, const uint8_t *k8_pool,
                               const float *k_scale, const float *w,
                               const int32_t *block_table, const int32_t *seq_lens, int Hi,
                               int Di, int page_size, int max_pages, const int32_t *b_list,
                               int n_b, long out_stride, double *scores) {
    for (int bi = 0; bi < n_b; bi++) {
        int b = b_list[bi];
        long L = seq_lens[b];
#pragma omp parallel for schedule(static)
        for (long t = 0; t < L; t++) {
            size_t row = pool_row(block_table, max_pages, page_size, 1, b, 0, t);
            double sk = (double)k_scale[row];
            double total = 0.0;
            for (int h = 0; h < Hi; h++) {
                double sq = (double)q_scale[(size_t)b * Hi + h];
                double dot = 0.0;
                for (int j = 0; j < Di; j++)
                    dot += (sq * oracle_e4m3_decode(q8[((size_t)b * Hi + h) * Di + j])) *
                           (sk * oracle_e4m3_decode(k8_pool[row * Di + j]));
                total += (double)w[(size_t)b * Hi + h] * (dot > 0.0 ? dot : 0.0);
            }
            scores[(size_t)bi * out_stride + t] = total;
        }
    }
}

/*
 * One decode step of the gated delta rule, for n independent heads ("All the attentions",
 * section 6 Gated DeltaNet and section 7 KDA). Per head, with state S (dv rows x dk
 * columns, row-major), key k and query q (dk), value v (dv), write strength beta:
 *   fade:        S[i][j] *= a[j]   (KDA: one decay per key channel j; Gated DeltaNet: one
 *                                   value for the whole head, a_per_channel = 0)
 *   correction:  e[i] = v[i] - sum_j S[i][j] k[j]      (recall error of the faded state for k)
 *   write:       S[i][j] += beta e[i] k[j]
 *   read:        o[i] = sum_j S[i][j] q[j]             (with the updated S)
 * S (float32 in) is widened to double; S_out and o are double. a holds n*dk values when
 * a_per_channel, else n.
 */
void oracle_delta_step(const float *S, const float *q, const float *k, const float *v,
                       const float *a, const float *beta, int n, int dk, int dv,
                       int a_per_channel, double *S_out, double *o) {
#pragma omp parallel for schedule(static)
    for (int h = 0; h < n; h++) {
        const float *Sh = S + (size_t)h * dv * dk;
        double *Th = S_out + (size_t)h * dv * dk;
        const float *qh = q + (size_t)h * dk, *kh = k + (size_t)h * dk;
        for (int i = 0; i < dv; i++) {
            for (int j = 0; j < dk; j++) {
                double decay = a_per_channel ? (double)a[(size_t)h * dk + j] : (double)a[h];
                Th[(size_t)i * dk + j] = decay * (double)Sh[(size_t)i * dk + j];
            }
            double pred = 0.0;
            for (int j = 0; j < dk; j++) pred += Th[(size_t)i * dk + j] * (double)kh[j];
            double e = (double)v[(size_t)h * dv + i] - pred;
            for (int j = 0; j < dk; j++)
                Th[(size_t)i * dk + j] += (double)beta[h] * e * (double)kh[j];
            double out = 0.0;
            for (int j = 0; j < dk; j++) out += Th[(size_t)i * dk + j] * (double)qh[j];
            o[(size_t)h * dv + i] = out;
        }
    }
}

/*
 * Cache append: the newest token of sequence b, position t = L_b - 1, is written to logical
 * slot r of its cache and so to physical row (block_table[b][r / P], r % P). A paged cache
 * keeps every token (r = t). A rolling cache (window > 0) has n_sink + window slots: the
 * first n_sink tokens keep their own slots, and every later token takes the slot of the
 * token window positions before it (r = n_sink + (t - n_sink) mod window), so the ring
 * always holds the sinks and the newest window tokens. Rows are copied byte for byte.
 * pool [num_pages, H, P, row_bytes] (updated), src [B, H, row_bytes].
 */
void oracle_cache_append(uint8_t *pool, const uint8_t *src, const int32_t *block_table,
                         const int32_t *seq_lens, int B, int H, long row_bytes, int page_size,
                         int max_pages, int window, int n_sink) {
    for (int b = 0; b < B; b++) {
        long t = (long)seq_lens[b] - 1;
        long r = t;
        if (window > 0 && t >= n_sink) r = n_sink + (t - n_sink) % window;
        long page = block_table[(size_t)b * max_pages + r / page_size];
        long slot = r % page_size;
        for (int h = 0; h < H; h++) {
            uint8_t *dst = pool + (((size_t)page * H + h) * page_size + slot) * row_bytes;
            const uint8_t *from = src + ((size_t)b * H + h) * row_bytes;
            for (long i = 0; i < row_bytes; i++) dst[i] = from[i];
        }
    }
}

/*
 * Quest page summaries: for each listed physical page and KV head, the elementwise minimum
 * and maximum of the page's P keys. k_pool [num_pages, Hkv, P, D] (dtype 0/1);
 * kmin, kmax [n_list, Hkv, D] double.
 */
void oracle_quest_minmax(const void *k_pool, int dtype, const int32_t *pages, int n_list,
                         int Hkv, int P, int D, double *kmin, double *kmax) {
    for (int i = 0; i < n_list; i++)
        for (int g = 0; g < Hkv; g++)
            for (int d = 0; d < D; d++) {
                double lo = INFINITY, hi = -INFINITY;
                for (int t = 0; t < P; t++) {
                    double x = widen(k_pool, dtype, (((size_t)pages[i] * Hkv + g) * P + t) * D + d);
                    if (x < lo) lo = x;
                    if (x > hi) hi = x;
                }
                kmin[((size_t)i * Hkv + g) * D + d] = lo;
                kmax[((size_t)i * Hkv + g) * D + d] = hi;
            }
}

/*
 * Quest decode step for query head h of sequence b (L = seq_lens[b], P tokens a page):
 *   full pages n < L / P get the bound U_n = sum_d max(q_d kmin_{n,d}, q_d kmax_{n,d}) from
 *   the keys of KV head h / (Hq / Hkv) (summaries computed here from the cache);
 *   the n_sel pages with the largest U (ties: the lower page index) are chosen, all of them
 *   when there are no more than n_sel; the tokens past the last full page are always kept;
 *   attention (scores q.k * scale, one softmax, weighted sum of V) runs over the chosen
 *   pages' tokens and the kept tail.
 * Outputs: out [n, D] and lse [n] for the n listed (b, h) pairs (all when pairs is NULL),
 * sel [n, n_sel] the chosen logical pages in ascending order (-1 padded), ub [n, max_pages]
 * the bounds (NaN for pages that are not full).
 */
void oracle_quest(const void *q, const void *k_pool, const void *v_pool, int dtype,
                  const int32_t *block_table, const int32_t *seq_lens, int B, int Hq, int Hkv,
                  int D, int page_size, int max_pages, double scale, int n_sel,
                  const int32_t *pairs, int n_pairs, double *out, double *lse, int32_t *sel,
                  double *ub) {
    int n_rep = Hq / Hkv;
    int n = pairs ? n_pairs : B * Hq;
#pragma omp parallel for schedule(dynamic, 1)
    for (int p = 0; p < n; p++) {
        int b = pairs ? pairs[2 * p] : p / Hq;
        int h = pairs ? pairs[2 * p + 1] : p % Hq;
        int g = h / n_rep;
        long L = seq_lens[b];
        long full = L / page_size;
        double *U = ub + (size_t)p * max_pages;
        for (long m = 0; m < max_pages; m++) U[m] = NAN;
        for (long m = 0; m < full; m++) {
            double u = 0.0;
            for (int d = 0; d < D; d++) {
                double lo = INFINITY, hi = -INFINITY;
                for (int t = 0; t < page_size; t++) {
                    size_t row = pool_row(block_table, max_pages, page_size, Hkv, b, g,
                                          m * page_size + t);
                    double x = widen(k_pool, dtype, row * D + d);
                    if (x < lo) lo = x;
                    if (x > hi) hi = x;
                }
                double qd = widen(q, dtype, ((size_t)b * Hq + h) * D + d);
                double a = qd * lo, c = qd * hi;
                u += a > c ? a : c;
            }
            U[m] = u;
        }
        /* choose: repeatedly the largest remaining bound, the lower index on ties */
        char *taken = (char *)calloc((size_t)(full > 0 ? full : 1), 1);
        long n_take = full < n_sel ? full : n_sel;
        for (long r = 0; r < n_take; r++) {
            long best = -1;
            for (long m = 0; m < full; m++)
                if (!taken[m] && (best < 0 || U[m] > U[best])) best = m;
            taken[best] = 1;
        }
        int32_t *sp = sel + (size_t)p * n_sel;
        long k = 0;
        for (long m = 0; m < full; m++)
            if (taken[m]) sp[k++] = (int32_t)m;
        for (; k < n_sel; k++) sp[k] = -1;
        /* attention over the chosen pages and the tail */
        double *s = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
        double m_ = -INFINITY;
        for (long t = 0; t < L; t++) {
            long pg = t / page_size;
            if (pg < full && !taken[pg]) continue;
            size_t row = pool_row(block_table, max_pages, page_size, Hkv, b, g, t);
            double dot = 0.0;
            for (int d = 0; d < D; d++)
                dot += widen(q, dtype, ((size_t)b * Hq + h) * D + d) *
                       widen(k_pool, dtype, row * D + d);
            s[t] = scale * dot;
            if (s[t] > m_) m_ = s[t];
        }
        double denom = 0.0;
        double *o = out + (size_t)p * D;
        for (int d = 0; d < D; d++) o[d] = 0.0;
        for (long t = 0; t < L; t++) {
            long pg = t / page_size;
            if (pg < full && !taken[pg]) continue;
            size_t row = pool_row(block_table, max_pages, page_size, Hkv, b, g, t);
            double e = exp(s[t] - m_);
            denom += e;
            for (int d = 0; d < D; d++) o[d] += e * widen(v_pool, dtype, row * D + d);
        }
        for (int d = 0; d < D; d++) o[d] /= denom;
        lse[p] = m_ + log(denom);
        free(s);
        free(taken);
    }
}
