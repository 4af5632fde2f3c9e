/*
 * kvdecode.h -- C ABI of libkvdecode.so: single-token decode attention over a
 * long, paged KV cache on one GB300 GPU (sm_103a).
 *
 * Operations (each names the passage that defines it):
 *  - attn_decode_gqa_paged: grouped-query attention of one new token per
 *    sequence over its paged cache. "Overview of Attention Mechanism", GQA /
 *    Code (query head h reads KV head h / (Hq/Hkv), scores q.k * scaling,
 *    softmax, weighted sum of V); "All the attentions", section 8
 *    (PagedAttention: a block table maps each sequence's logical pages to
 *    physical pages and the output does not change).
 *  - attn_decode_swa_sink: the same over a sliding window plus attention
 *    sinks. "All the attentions", section 4 (key j visible to query i iff
 *    j <= i and j > i - W); "Long context, KV eviction and sparse attention",
 *    KV eviction: StreamingLLM (the first tokens are always kept);
 *    "Attention Optimizations", Attention sinks (a learned per-head sink
 *    logit in the softmax denominator, with no value).
 *  - attn_decode_mla: absorbed-latent MLA decode over one shared 576-wide
 *    row per token (512 latent + 64 RoPE key; value = the first 512).
 *    "Attention Optimizations", DSA / Computation Path and KV cache size;
 *    "Overview of Attention Mechanism", MLA (absorption of W^UK and W^UV).
 *  - dsa_indexer_topk: lightning-indexer scores of every cached token,
 *    I_t = sum_h w_h * ReLU(q_h . k_t), then the indices of the k largest.
 *    "Attention Optimizations", DSA / Computation Path; "All the
 *    attentions", section 5 (DSA).
 *  - dsa_topk: the selection step alone, over scores the caller provides.
 *  - attn_decode_mla_sparse: MLA over only the selected tokens.
 *    "Attention Optimizations", DSA / Computation Path (gather of the
 *    selected cache rows, then attention).
 *  - dsa_indexer_topk_fp8, kvd_quantize_e4m3_rows, dsa_indexer_cache_append_fp8:
 *    the indexer on e4m3 codes with row scales and the quantizer that fills its
 *    cache. "Long context, KV eviction and sparse attention", exact selection
 *    with a fast scorer (the indexer runs in FP8).
 *  - kvd_cache_append, attn_decode_swa_ring, attn_decode_swa_ring_append: the
 *    new token's K/V (or latent row) written into a paged or rolling cache, and
 *    sliding-window attention read from the rolling cache (the last one does
 *    both in one call). "Attention Optimizations", DSA / Computation Path
 *    (update_cache before attention) and Sliding-window (a rolling buffer of W
 *    entries); "All the attentions", section 4.
 *  - quest_page_minmax, quest_select_pages, attn_decode_quest (and the split
 *    quest_page_bounds + attn_decode_quest_from_bounds): query-aware page
 *    selection. "Long context, KV eviction and sparse attention", Sparse attention
 *    (Quest: per-page key bounds, the best pages, attention over them).
 *  - kvd_delta_decode_step: one Gated DeltaNet / KDA decode step on each head's
 *    fixed-size state. "All the attentions", sections 6 and 7.
 *
 * Common conventions
 *  - Every tensor pointer is a DEVICE pointer owned by the caller; the library
 *    never allocates or frees memory and keeps no pointer past a call. Tensors
 *    are dense, row-major, 16-byte aligned.
 *  - seq_lens[b] (device, int32) counts cached tokens INCLUDING the token
 *    being decoded: its K/V (or latent row) were appended before the call, so
 *    the query sits at position L_b - 1. 1 <= L_b <= max_pages * page_size.
 *  - block_table[b][n] (device, int32, [B, max_pages]) is the physical page of
 *    logical page n of sequence b, 0 <= page < num_pages. Entries past the
 *    last page of a sequence are not read.
 *  - GQA pools are [num_pages, Hkv, page_size, D]; the MLA latent pool is
 *    [num_pages, page_size, 576]; the indexer key pool [num_pages,
 *    page_size, Di]. page_size is a power of two, 16 <= page_size <= 256.
 *  - scale multiplies q.k before the softmax (1/sqrt(D) for GQA, 1/sqrt(192)
 *    for DeepSeek-V3 MLA: the un-absorbed 128 + 64 query width).
 *  - Every call is asynchronous on `stream`. Split-KV partial results live in
 *    the caller's workspace `ws` of at least kvd_workspace_size(...) bytes,
 *    zero-filled once before its first use; the kernels leave it ready for
 *    the next call of the same operation family with the same shape arguments
 *    (the workspace's layout follows B, the head counts, the lengths and k).
 *    Zero-fill it again before a call of the family with other shape
 *    arguments. Calls that share a workspace must be ordered on one stream.
 *  - A workspace serves one operation family at a time: (1) GQA / SWA decode,
 *    (2) MLA decode (dense or sparse), (3) DSA indexer / top-k. A family
 *    keeps zero only the parts it relies on (completion counters, top-k
 *    histograms and counters, the selection bitmap), and another family's
 *    kernels leave other data there. Zero-fill the buffer again before
 *    handing it to another family. A top-k that finds non-zero state stays in
 *    bounds and records KVD_ERR_DEVICE_STATE; a GQA / SWA call may then
 *    return wrong outputs.
 *  - Return value: KVD_OK, or a negative KVD_ERR_* code. Argument checks run
 *    on the host before any launch; on failure nothing is launched and the
 *    outputs are untouched. Faults the host cannot see (a block-table entry or
 *    sequence length out of range, a bounded device wait that gave up) are
 *    recorded in the workspace and read with kvd_check_device_error(); an
 *    out-of-range page or length is clamped (never dereferenced).
 */
#ifndef KVDECODE_H
#define KVDECODE_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

enum kvd_status {
    KVD_OK = 0,
    KVD_ERR_INVALID_ARG = -1,         /* null pointer, bad size or alignment */
    KVD_ERR_UNSUPPORTED = -2,         /* shape or dtype this build does not handle */
    KVD_ERR_CUDA = -3,                /* a CUDA call or launch failed */
    KVD_ERR_TIMEOUT = -4,             /* (device) a bounded wait gave up */
    KVD_ERR_WORKSPACE_TOO_SMALL = -5, /* ws_bytes below kvd_workspace_size() */
    KVD_ERR_DEVICE_OOB = -6,          /* (device) page index or length out of range */
    KVD_ERR_DEVICE_STATE = -7         /* (device) workspace was not in its zeroed state */
};

enum kvd_dtype { KVD_F32 = 0, KVD_BF16 = 1 };

enum kvd_op {
    KVD_OP_GQA = 0,
    KVD_OP_SWA = 1,
    KVD_OP_MLA = 2,
    KVD_OP_DSA_TOPK = 3,
    KVD_OP_MLA_SPARSE = 4
};

/*
 * Dense GQA / MHA / MQA decode over a paged cache.
 *  q       [B, Hq, D]                      dtype
 *  k_pool  [num_pages, Hkv, page_size, D]  dtype
 *  v_pool  [num_pages, Hkv, page_size, D]  dtype
 *  out     [B, Hq, D]                      dtype (bf16 in -> bf16 out, f32 -> f32)
 *  lse_out [B, Hq] float32, nullable: natural-log softmax normaliser
 *          log(sum_t exp(scale q.k_t)).
 * Supported: Hq % Hkv == 0, D in {64, 128}, dtype KVD_BF16 or KVD_F32,
 * Hq/Hkv <= 128.
 */
int attn_decode_gqa_paged(const void *q, const void *k_pool, const void *v_pool,
                          const int32_t *block_table, const int32_t *seq_lens, void *out,
                          float *lse_out, int B, int Hq, int Hkv, int D, int page_size,
                          int max_pages, int num_pages, float scale, int dtype, void *ws,
                          size_t ws_bytes, cudaStream_t stream);

/*
 * attn_decode_gqa_paged without a workspace argument. The pages have no counterpart to
 * this entry point: it exists for callers that cannot allocate device memory (a plugin
 * whose host engine owns all device memory and hands out only input and output buffers,
 * or a decode loop that must not pay the device-wide synchronisation of cudaMalloc /
 * cudaFree). It allocates nothing and calls no allocating routine.
 *  - Scratch: a library-owned device array of 32 MiB (every GPU that loads the library
 *    holds it until the process exits). Shapes whose split plan needs more scratch than
 *    that return KVD_ERR_WORKSPACE_TOO_SMALL; the Llama-3-8B-shaped decode (B=32,
 *    Hq=32, Hkv=8, D=128, up to 8192 tokens) needs about 11-21 MiB.
 *  - The first call on each device looks up the array's device address (a
 *    cudaGetSymbolAddress on the current device); make that first call before any
 *    stream capture.
 *  - Every call shares the one array and clears its counters and error flag (an
 *    asynchronous memset on `stream`) before launching. Calls that overlap on the GPU
 *    (different streams without ordering, or concurrent host threads) race on it.
 *  - Device-side faults are still contained (out-of-range pages and lengths are
 *    clamped, waits are bounded), but their error flag is cleared by the next call and
 *    cannot be read with kvd_check_device_error.
 * Arguments, layouts and supported shapes as attn_decode_gqa_paged.
 */
int attn_decode_gqa_paged_static_ws(const void *q, const void *k_pool, const void *v_pool,
                                    const int32_t *block_table, const int32_t *seq_lens,
                                    void *out, float *lse_out, int B, int Hq, int Hkv, int D,
                                    int page_size, int max_pages, int num_pages, float scale,
                                    int dtype, cudaStream_t stream);

/*
 * Sliding-window + sink decode. Visible tokens of sequence b:
 *   { t < min(n_sink_tokens, L_b) }  U  { L_b - window <= t < L_b }
 * (the window counts the decoded token itself; sink tokens that fall inside
 * the window are counted once). sink_logit [Hq] float32, nullable: a learned
 * per-query-head logit, in the units of scale*q.k, added once to the softmax
 * denominator with a zero value vector (sink_logit = 0 is softmax-off-by-one;
 * -inf is no sink). Other arguments as attn_decode_gqa_paged; window >= 1,
 * n_sink_tokens >= 0.
 */
int attn_decode_swa_sink(const void *q, const void *k_pool, const void *v_pool,
                         const int32_t *block_table, const int32_t *seq_lens, void *out,
                         float *lse_out, int B, int Hq, int Hkv, int D, int page_size,
                         int max_pages, int num_pages, float scale, int dtype, int window,
                         int n_sink_tokens, const float *sink_logit, void *ws, size_t ws_bytes,
                         cudaStream_t stream);

/*
 * Sliding-window + sink decode over a ROLLING cache ("All the attentions", section 4: the
 * window's cache is a buffer of W entries, each new entry replacing the oldest; "Attention
 * Optimizations", Sliding-window: Mistral's rolling buffer, O(W) cache). Sequence b's cache
 * has n_sink_tokens + window slots (logical positions of its block table): the first
 * n_sink_tokens hold the sink tokens, and token t >= n_sink_tokens lives in slot
 * n_sink_tokens + (t - n_sink_tokens) mod window (as kvd_cache_append writes it). seq_lens
 * holds the TRUE sequence lengths L_b (tokens decoded so far, >= 1, unbounded); the visible
 * set is every filled slot, the first min(L_b, n_sink_tokens + window), which is exactly
 * the set attn_decode_swa_sink sees on a full cache. sink_logit as attn_decode_swa_sink.
 * Requires window >= 1, n_sink_tokens >= 0 and n_sink_tokens + window <= max_pages *
 * page_size; other arguments, workspace (as KVD_OP_GQA with max_len = max_pages *
 * page_size) and errors as attn_decode_gqa_paged.
 */
int attn_decode_swa_ring(const void *q, const void *k_ring, const void *v_ring,
                         const int32_t *block_table, const int32_t *seq_lens, void *out,
                         float *lse_out, int B, int Hq, int Hkv, int D, int page_size,
                         int max_pages, int num_pages, float scale, int dtype, int window,
                         int n_sink_tokens, const float *sink_logit, void *ws, size_t ws_bytes,
                         cudaStream_t stream);

/*
 * One decode step on a rolling cache: exactly kvd_cache_append of the newest token's rows
 * (k_new, v_new [B, Hkv, D], device, 16-byte aligned, the cache's dtype) into k_ring / v_ring
 * with this window and n_sink_tokens, followed by attn_decode_swa_ring on the updated ring
 * ("Attention Optimizations", DSA / Computation Path: the new token's cache row is written
 * before attention runs; "All the attentions", section 4: the newest entry of the rolling
 * buffer replaces the oldest). k_ring and v_ring are updated in place. For bf16 rings the
 * attention launch writes the rows itself (each chunk of the ring that holds the newest
 * slot writes them before reading it: one launch instead of two); float32 rings take the
 * append's launch, then the attention's. A length below 1 or an out-of-range page id of the
 * newest slot records KVD_ERR_DEVICE_OOB in the workspace's error flag (read it with
 * kvd_check_device_error) and that sequence's rows are not written. Other arguments,
 * workspace and host-side errors as attn_decode_swa_ring; every check runs before anything
 * is written.
 */
int attn_decode_swa_ring_append(const void *q, const void *k_new, const void *v_new,
                                void *k_ring, void *v_ring, const int32_t *block_table,
                                const int32_t *seq_lens, void *out, float *lse_out, int B,
                                int Hq, int Hkv, int D, int page_size, int max_pages,
                                int num_pages, float scale, int dtype, int window,
                                int n_sink_tokens, const float *sink_logit, void *ws,
                                size_t ws_bytes, cudaStream_t stream);

/*
 * Cache append ("Attention Optimizations", DSA / Computation Path: the new token's cache
 * row is written before attention runs): for each sequence b, the rows of its newest token,
 * position t = seq_lens[b] - 1, are copied into the cache slot
 *   r = t                                      (window == 0: paged cache), or
 *   r = t if t < n_sink, else n_sink + (t - n_sink) mod window   (window > 0: rolling cache)
 * at page block_table[b][r / page_size], offset r % page_size.
 *  k_new, v_new  [B, H, D] (dtype KVD_F32 or KVD_BF16), device; v_new and v_pool both null
 *                for a single pool (the MLA latent cache: H = 1, D = 576)
 *  k_pool, v_pool [num_pages, H, page_size, D], device, updated in place
 *  err           int32 on the device: set to KVD_ERR_DEVICE_OOB when a length or page id is
 *                out of range (that sequence's rows are then not written); never cleared
 * Bytes are copied unchanged. Requires D * element size a multiple of 16 (and at most
 * 1 MiB), 16-byte aligned rows, and for a rolling cache n_sink + window <= max_pages *
 * page_size; a paged cache needs 1 <= L_b <= max_pages * page_size. Host-side errors:
 * KVD_ERR_INVALID_ARG, KVD_ERR_UNSUPPORTED. No workspace.
 */
int kvd_cache_append(const void *k_new, const void *v_new, void *k_pool, void *v_pool,
                     const int32_t *block_table, const int32_t *seq_lens, int B, int H, int D,
                     int page_size, int max_pages, int num_pages, int dtype, int window,
                     int n_sink, int *err, cudaStream_t stream);

/*
 * Quest page summaries ("Long context, KV eviction and sparse attention", Sparse attention:
 * each page of keys is summarised by its elementwise minimum and maximum). For each listed
 * physical page (pages [n_list] int32, device; null = every page 0..num_pages-1) and KV head:
 *   kmin[page][g][d] = min_t k_pool[page][g][t][d],  kmax likewise (t < page_size)
 *  k_pool [num_pages, Hkv, page_size, D], kmin / kmax [num_pages, Hkv, D], all of dtype
 *  (KVD_BF16 or KVD_F32; the extremes of stored values are stored exactly), device.
 * Compute a page's summary once it is full (only full pages are scored). err: int32 on the
 * device, set to KVD_ERR_DEVICE_OOB for a listed page out of range (skipped). Supported:
 * D in {64, 128}. No workspace.
 */
int quest_page_minmax(const void *k_pool, void *kmin, void *kmax, const int32_t *pages,
                      int n_list, int num_pages, int Hkv, int page_size, int D, int dtype,
                      int *err, cudaStream_t stream);

/*
 * Quest page choice for every query head (same passage): sequence b has full = L_b /
 * page_size full pages (logical); query head h (KV head g = h / (Hq / Hkv)) bounds its
 * scores on page n by U = sum_d max(q_d kmin_d, q_d kmax_d) (the summaries of the page's
 * physical page, head g; products and sums in float32) and keeps the n_sel pages with the
 * largest U, ties to the lower page (all full pages when there are no more than n_sel).
 *  sel    [B, Hq, n_sel] int32 output: the chosen logical pages in ascending order, -1 padded
 *  ub_out [B, Hq, max_pages] float32 output (required; the bounds are computed there, then
 *         chosen from): U, NaN past the full pages
 * Other arguments as attn_decode_gqa_paged. Supported: D in {64, 128}, Hq / Hkv <= 16,
 * 1 <= n_sel <= 64, max_pages <= 6400. err as quest_page_minmax (KVD_ERR_DEVICE_OOB for a
 * length or page id out of range, clamped). Two launches; no workspace.
 */
int quest_select_pages(const void *q, const void *kmin, const void *kmax,
                       const int32_t *block_table, const int32_t *seq_lens, int32_t *sel,
                       float *ub_out, int B, int Hq, int Hkv, int D, int page_size, int max_pages,
                       int num_pages, int n_sel, int dtype, int *err, cudaStream_t stream);

/*
 * Attention of each query head over its chosen pages and the tokens past the last full page
 * (same passage): scores scale * q.k, one softmax, weighted sum of V, over the tokens of the
 * pages listed in sel (as quest_select_pages writes it; entries past min(full, n_sel) are
 * not read) plus positions full * page_size .. L_b - 1. out [B, Hq, D] (dtype of q),
 * lse_out [B, Hq] float32 natural log (nullable). Other arguments as
 * attn_decode_gqa_paged; err as quest_select_pages (a listed page outside 0..full-1 is
 * flagged and skipped). No workspace.
 */
int attn_decode_quest(const void *q, const void *k_pool, const void *v_pool,
                      const int32_t *block_table, const int32_t *seq_lens, const int32_t *sel,
                      void *out, float *lse_out, int B, int Hq, int Hkv, int D, int page_size,
                      int max_pages, int num_pages, int n_sel, float scale, int dtype, int *err,
                      cudaStream_t stream);

/*
 * The bound step of quest_select_pages alone: ub [B, Hq, max_pages] float32 (device,
 * caller-owned) receives each query head's page bounds U (NaN past the full pages).
 * Arguments, support and errors as quest_select_pages. One launch.
 */
int quest_page_bounds(const void *q, const void *kmin, const void *kmax,
                      const int32_t *block_table, const int32_t *seq_lens, float *ub, int B,
                      int Hq, int Hkv, int D, int page_size, int max_pages, int num_pages,
                      int dtype, int *err, cudaStream_t stream);

/*
 * Choice and attention in one launch: each query head takes the n_sel largest of its bounds
 * ub (as quest_page_bounds writes them; ties to the lower page), writes them to sel_out
 * [B, Hq, n_sel] (ascending, -1 padded, exactly as quest_select_pages would), and attends
 * over those pages and the tail as attn_decode_quest does. Supported: as attn_decode_quest,
 * max_pages <= 25600. One launch.
 */
int attn_decode_quest_from_bounds(const void *q, const void *k_pool, const void *v_pool,
                                  const int32_t *block_table, const int32_t *seq_lens,
                                  const float *ub, int32_t *sel_out, void *out, float *lse_out,
                                  int B, int Hq, int Hkv, int D, int page_size, int max_pages,
                                  int num_pages, int n_sel, float scale, int dtype, int *err,
                                  cudaStream_t stream);

/*
 * Absorbed MLA decode over all cached tokens.
 *  q       [B, H, d_qk] bf16: per head [W_UK^T q_nope (512) ; rotated q_pe (64)]
 *  c_pool  [num_pages, page_size, d_qk] bf16: rows [c_KV (512) ; rotated k_pe (64)]
 *  out     [B, H, d_v] bf16 = sum_t softmax_t(scale q.c_t) c_t[0:d_v]
 *  lse_out [B, H] float32, nullable.
 * Supported: H == 128, d_qk == 576, d_v == 512.
 */
int attn_decode_mla(const void *q, const void *c_pool, const int32_t *block_table,
                    const int32_t *seq_lens, void *out, float *lse_out, int B, int H, int d_qk,
                    int d_v, int page_size, int max_pages, int num_pages, float scale, void *ws,
                    size_t ws_bytes, cudaStream_t stream);

/*
 * DSA indexer + top-k.
 *  q_idx      [B, Hi, Di] bf16 indexer queries
 *  k_idx_pool [num_pages, page_size, Di] bf16 indexer key cache
 *  w          [B, Hi] float32 per-head weights (any positive factor such as
 *             Hi^-0.5 may be folded in; it does not change the selection)
 *  topk_idx   [B, k] int32 out: logical token positions of the min(k, L_b)
 *             largest scores, ascending; ties go to the lower position; slots
 *             past the count hold -1
 *  topk_count [B] int32 out: min(k, L_b)
 *  scores_out [B, max_pages*page_size] float32, nullable: the fp32 scores
 *             (entries past L_b are not written)
 * Supported: Hi == 64, Di == 128, 1 <= k <= 4096.
 */
int dsa_indexer_topk(const void *q_idx, const void *k_idx_pool, const float *w,
                     const int32_t *block_table, const int32_t *seq_lens, int32_t *topk_idx,
                     int32_t *topk_count, float *scores_out, int B, int Hi, int Di, int page_size,
                     int max_pages, int num_pages, int k, void *ws, size_t ws_bytes,
                     cudaStream_t stream);

/*
 * FP8 lightning indexer + top-k. "Long context, KV eviction and sparse attention" (exact
 * selection with a fast scorer): the indexer scores every past token with few heads in FP8.
 * Codes are e4m3 (1 sign, 4 exponent bits with bias 7, 3 mantissa bits; no infinities; 448
 * the largest finite value) with one float32 scale per row:
 *  q8       [B, Hi, Di] e4m3 codes (uint8), device; q_scale [B, Hi] float32 (per head)
 *  k8_pool  [num_pages, page_size, Di] e4m3 codes; k_scale [num_pages, page_size] float32
 *           (per token, 16-byte aligned)
 *  w        [B, Hi] float32
 * Score of token t: I_t = k_scale(t) * sum_h w_h q_scale_h * ReLU(q8_h . k8_t), the codes
 * decoded exactly and the dot products accumulated in fp32. Outputs, tie rule, workspace
 * (kvd_workspace_size(KVD_OP_DSA_TOPK, ...)) and errors as dsa_indexer_topk.
 * Supported: Hi == 64, Di == 128, 1 <= k <= 4096.
 */
int dsa_indexer_topk_fp8(const void *q8, const float *q_scale, const void *k8_pool,
                         const float *k_scale, const float *w, const int32_t *block_table,
                         const int32_t *seq_lens, int32_t *topk_idx, int32_t *topk_count,
                         float *scores_out, int B, int Hi, int Di, int page_size, int max_pages,
                         int num_pages, int k, void *ws, size_t ws_bytes, cudaStream_t stream);

/*
 * Row quantization to e4m3 (the FP8 indexer's query and key format): for each row of
 * x [rows, cols] bf16 (device), scale = amax / 448 (1 for a row of zeros) and each code is
 * the nearest e4m3 value to x / scale computed in float32 (ties to even, magnitudes above 448
 * saturating). codes [rows, cols] uint8, scales [rows] float32, both device, caller-owned.
 * Supported: 1 <= cols <= 65536. No workspace.
 */
int kvd_quantize_e4m3_rows(const void *x, void *codes, float *scales, int rows, int cols,
                           cudaStream_t stream);

/*
 * FP8 indexer cache append ("Attention Optimizations", DSA / Computation Path: the new
 * token's indexer key is written to the indexer cache before scoring): quantizes each
 * sequence's new key k_new [B, Di] bf16 as kvd_quantize_e4m3_rows does and stores the codes
 * and the scale at the cache row of position seq_lens[b] - 1 (page block_table[b][t / P],
 * slot t % P) of k8_pool [num_pages, page_size, Di] / k_scale [num_pages, page_size].
 * err: a device int that receives KVD_ERR_DEVICE_OOB when a length or page index is out of
 * range (the write is then redirected to a clamped, valid row). Supported: Di <= 65536.
 */
int dsa_indexer_cache_append_fp8(const void *k_new, const int32_t *block_table,
                                 const int32_t *seq_lens, void *k8_pool, float *k_scale, int B,
                                 int Di, int page_size, int max_pages, int num_pages, int *err,
                                 cudaStream_t stream);

/*
 * Top-k selection alone over caller-provided scores.
 *  scores [B, score_stride] float32 (row b holds lens[b] scores; NaN not allowed)
 *  lens   [B] int32 device, 1 <= lens[b] <= score_stride
 *  outputs and tie rule as dsa_indexer_topk. Supported: 1 <= k <= 4096.
 */
int dsa_topk(const float *scores, const int32_t *lens, int32_t *topk_idx, int32_t *topk_count,
             int B, int score_stride, int k, void *ws, size_t ws_bytes, cudaStream_t stream);

/*
 * MLA over the selected tokens only.
 *  topk_idx [B, k] int32 logical positions (< L_b); topk_count [B] int32
 *  (1 <= count <= k); other arguments as attn_decode_mla. Order of the
 *  indices does not matter; each listed position is attended once.
 */
int attn_decode_mla_sparse(const void *q, const void *c_pool, const int32_t *block_table,
                           const int32_t *seq_lens, const int32_t *topk_idx,
                           const int32_t *topk_count, void *out, float *lse_out, int B, int H,
                           int d_qk, int d_v, int k, int page_size, int max_pages, int num_pages,
                           float scale, void *ws, size_t ws_bytes, cudaStream_t stream);

/*
 * Workspace bytes for one call of `op` (enum kvd_op). Arguments that do not
 * apply to the op are ignored: H is Hq for GQA/SWA and the head count for
 * MLA; D is the head dim (GQA/SWA) or d_v (MLA); max_len = max_pages *
 * page_size; window/n_sink for SWA; k for the DSA ops. Returns 0 for an
 * unknown op or an unsupported shape.
 */
size_t kvd_workspace_size(int op, int B, int H, int Hkv, int D, int max_len, int window,
                          int n_sink, int k);

/*
 * Synchronise `stream`, return (and clear) the first device-side error that
 * kernels using workspace `ws` recorded: KVD_OK, KVD_ERR_TIMEOUT,
 * KVD_ERR_DEVICE_OOB or KVD_ERR_DEVICE_STATE; KVD_ERR_CUDA if the
 * synchronisation itself failed.
 */
int kvd_check_device_error(void *ws, cudaStream_t stream);

/* Static, human-readable name of a status code. */
const char *kvd_status_string(int status);

/*
 * One decode step of the gated delta rule for n independent heads ("All the attentions",
 * section 6 Gated DeltaNet and section 7 KDA; "Attention Optimizations", KDA). Per head h,
 * with state S_h of dv rows and dk columns (row-major, float32, device, updated in place):
 *   fade        S[i][j] *= a[j]                (a_per_channel != 0: a [n, dk], one decay per
 *                                               key channel (KDA); else a [n], one per head)
 *   correction  e[i] = v[i] - sum_j S[i][j] k[j]
 *   write       S[i][j] += beta * e[i] * k[j]
 *   read        o[i] = sum_j S[i][j] q[j]       (the updated state)
 *  S     [n, dv, dk] float32, 16-byte aligned (8-byte when dk == 64)
 *  q, k  [n, dk] float32, same alignment; v [n, dv] float32; beta [n] float32
 *  o     [n, dv] float32 output, must not overlap S
 * q and k are used as given (any normalisation belongs to the caller). Each row's dot
 * products are accumulated in float32. All buffers are caller-owned device memory; no
 * workspace. Supported: dk in {64, 128, 256}, 1 <= dv <= 65536. Errors: KVD_ERR_INVALID_ARG
 * for null or misaligned pointers or n < 1; KVD_ERR_UNSUPPORTED for other dk or dv.
 */
int kvd_delta_decode_step(float *S, const float *q, const float *k, const float *v,
                          const float *a, const float *beta, float *o, int n, int dk, int dv,
                          int a_per_channel, cudaStream_t stream);

/*
 * Process-wide options, for measurement and for tests of the library itself; normal use
 * needs none of them (the pages have no counterpart). Each setting holds for calls made
 * after it, from any thread, until it is set again.
 *  KVD_OPT_PDL            1 (default): kernels are launched with programmatic dependent
 *                         launch, so that a kernel's set-up overlaps the tail of the
 *                         previous one on the stream; 0: plain launches. Before its
 *                         dependency wait a kernel touches no global memory, except that the
 *                         bf16 GQA / SWA kernel reads lengths and block-table entries
 *                         (L2-only) to prefetch its first tiles into L2, and issues its first
 *                         copies from them only if the same values are read after the wait.
 *                         That kernel also lets the next kernel on the stream be scheduled
 *                         once its copies are issued; a kernel launched after it with
 *                         programmatic dependent launch must wait for it (griddepcontrol.wait
 *                         / cudaGridDependencySynchronize) before reading its outputs, as
 *                         that launch mode requires in any case.
 *  KVD_OPT_GQA_CHUNK      0 (default): the GQA / SWA split plan picks the tokens per split;
 *                         >= 64: that many tokens (rounded down to a multiple of 64) per
 *                         split, raised if the plan would exceed its chunk limit.
 *  KVD_OPT_MLA_MIN_TILES  0 (default): the MLA plan gives each two-CTA cluster at least one
 *                         64-token tile (dense) or two (sparse); >= 1: at least that many.
 *  KVD_OPT_WAIT_TIMEOUT_TEST  1: the next bf16 GQA / SWA call (and only that call) runs
 *                         with a limit of about 1000 SM cycles on each bounded wait of its
 *                         copy ring, and its consumer warps first wait on a barrier that
 *                         nothing completes: the wait runs out, the call records
 *                         KVD_ERR_TIMEOUT (read with kvd_check_device_error), waits for the
 *                         copies it issued and returns; its outputs are undefined and its
 *                         workspace stays ready for the next call.
 *  KVD_OPT_GQA_CLUSTER    1 (default): a bf16 GQA / SWA call with few (sequence, KV head)
 *                         groups, whose groups need few chunks, runs each group's chunks as
 *                         one thread-block cluster that combines them in distributed shared
 *                         memory; 2: also with many groups, when each needs at most 8 chunks;
 *                         0: the chunk partials always go through the workspace and the last
 *                         CTA of each group combines them.
 * Returns KVD_OK, or KVD_ERR_INVALID_ARG for an unknown option or a value out of range.
 */
enum kvd_option {
    KVD_OPT_PDL = 0,
    KVD_OPT_GQA_CHUNK = 1,
    KVD_OPT_MLA_MIN_TILES = 2,
    KVD_OPT_WAIT_TIMEOUT_TEST = 3,
    KVD_OPT_GQA_CLUSTER = 4
};
int kvd_set_option(int option, long long value);

#ifdef __cplusplus
}
#endif
#endif /* KVDECODE_H */
