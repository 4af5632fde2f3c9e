// kvd_host.h -- internal interface between the C-ABI layer (api.cu) and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "kvdecode.h"

namespace kvd {

// The first 256 bytes of every workspace hold the device error flag (int32 at offset 0).
constexpr size_t kWsHeaderBytes = 256;

constexpr int kGqaMaxChunks = 256;  // split-KV chunks per (sequence, KV head, head block)

// Kernel arguments of the GQA / SWA decode (one struct for both dtypes).
struct GqaParams {
    const void* q;
    const void* k_pool;
    const void* v_pool;
    const int32_t* block_table;
    const int32_t* seq_lens;
    void* out;
    float* lse_out;
    const float* sink_logit;
    float* part_o;    // [units, max_chunks, 16, D]
    float* part_lse;  // [units, max_chunks, 16]   (log2 domain)
    int* counters;    // [units] completion counters (zero between calls)
    int* err;         // workspace error flag
    int B, Hq, Hkv, D, G, NHG, units;
    int page_size, max_pages, num_pages, max_len;
    int window, n_sink;  // window <= 0: dense
    int ring;            // > 0: a rolling cache of this many slots; visible = min(L, ring)
    int ring_sink;       // the ring's pinned sink slots (ring - ring_sink = the window)
    // ring mode, bf16: the newest token's K and V rows [B, Hkv, D], written into their ring
    // slot by the attention kernel before it reads the ring (null: the rows are in place)
    const void* k_new;
    const void* v_new;
    int chunk, max_chunks;
    int dtype;
    float scale_log2;  // scale * log2(e)
    long long wait_cycles;  // limit of each bounded wait of the bf16 kernel's ring
    int stall_test;         // test of the give-up path: the consumers first wait on a
                            // barrier that nothing completes, so their wait runs out
};

// Host-side split plan and workspace layout of one GQA / SWA call.
struct GqaPlan {
    int chunk;       // tokens per split (multiple of 64)
    int max_chunks;  // chunk slots per unit (grid.x)
    int hpt;         // KV heads per K/V tile (2: D = 64 pages of <= 64 tokens, G <= 8)
    int NHG;         // head blocks of <= 16 query heads per KV head
    int units;       // B * Hkv * NHG
    int cluster;     // > 0: the chunks of a group form a cluster of this many CTAs (= chunks)
    size_t off_counters, off_lse, off_o, total;
};

int gqa_plan(int B, int Hq, int Hkv, int D, int page_size, int max_len, int window, int n_sink,
             int dtype, GqaPlan* plan);
int gqa_launch(const GqaPlan& plan, const GqaParams& p, const CUtensorMap* tk,
               const CUtensorMap* tv, cudaStream_t stream);

// Host-side argument checks of one GQA / SWA decode (everything but the workspace).
int gqa_check(const void* q, const void* k_pool, const void* v_pool, const int32_t* block_table,
              const int32_t* seq_lens, const void* out, int B, int Hq, int Hkv, int D,
              int page_size, int max_pages, int num_pages, float scale, int dtype, int window,
              int n_sink, int ring);

// Validate, plan and launch one GQA / SWA decode (window <= 0: dense) using workspace ws.
int gqa_run(const void* q, const void* k_pool, const void* v_pool, const int32_t* block_table,
            const int32_t* seq_lens, void* out, float* lse_out, int B, int Hq, int Hkv, int D,
            int page_size, int max_pages, int num_pages, float scale, int dtype, int window,
            int n_sink, const float* sink_logit, void* ws, size_t ws_bytes, cudaStream_t stream,
            int ring = 0, int ring_sink = 0, const void* k_new = nullptr,
            const void* v_new = nullptr);

// 2-D bf16 tensor map over a row-major [rows, cols] matrix with a {64, box_rows} box and
// 128-byte swizzle (cols a multiple of 64). Returns KVD_OK or KVD_ERR_CUDA.
// ---------------------------------------------------------------------------------------
// DSA indexer + top-k
// ---------------------------------------------------------------------------------------
constexpr int kTopkMaxK = 4096;

struct IdxParams {
    const void* q;             // [B, 64, 128] bf16 or e4m3 (read through a tensor map)
    const float* w;            // [B, 64]
    const float* q_scale;      // FP8 indexer: [B, 64] per-head query scales
    const float* k_scale;      // FP8 indexer: [num_pages * page_size] per-token key scales
    const int32_t* block_table;
    const int32_t* seq_lens;
    float* scores;             // [B, score_stride]
    long long score_stride;
    uint32_t* hist;            // [B, 2048] top-11-bit key histogram
    int* counts;               // [B, 4] selection counters, zeroed here for the selection
    int* err;
    int B, page_size, max_pages, num_pages, max_len, tiles_per_b;
};

// Row quantization to e4m3 (dsa_indexer_fp8.cu). With a block table, row r is sequence r's
// newest token (position seq_lens[r] - 1) and lands on that token's row of the paged cache.
struct QuantParams {
    const void* x;             // [rows, cols] bf16
    void* codes;               // e4m3 codes, [rows or cache rows, cols]
    float* scales;             // one float32 scale per row
    const int32_t* block_table;  // null: row r to row r
    const int32_t* seq_lens;
    int* err;
    int rows, cols, page_size, max_pages, num_pages, max_len;
};

struct TopkParams {
    const float* scores;       // [B, score_stride]
    long long score_stride;
    const int32_t* lens;       // [B]
    uint32_t* hist;            // [B, 2048]
    uint32_t* hist2;           // [B, 256] next 8 key bits of the threshold bucket's keys
    int* counts;               // [B, 4]: selected, candidates, blocks done, (pad)
    int* sel;                  // [B, k] selected positions
    uint64_t* cand;            // [B, max_len] candidates' (score key, reversed position) keys
    uint32_t* bitmap;          // [B, ceil(max_len / 32)] chosen positions (kept zero)
    int32_t* topk_idx;         // [B, k]
    int32_t* topk_count;       // [B]
    int* err;
    int B, k, max_len;
};

// Workspace layout of the DSA selection (offsets from the workspace base).
struct TopkLayout {
    size_t off_hist, off_hist2, off_counts, off_sel, off_cand, off_bitmap, off_scores, total;
};
TopkLayout topk_layout(int B, int max_len, int k, bool with_scores);

int dsa_indexer_launch(const IdxParams& p, const CUtensorMap& tk, const CUtensorMap& tk128,
                       const CUtensorMap& tq, cudaStream_t stream);
int dsa_indexer_fp8_launch(const IdxParams& p, const CUtensorMap& tk, const CUtensorMap& tk128,
                           const CUtensorMap& tq, cudaStream_t stream);
int quantize_e4m3_launch(const QuantParams& p, cudaStream_t stream);

// Arguments of one gated delta-rule decode step over n independent heads.
struct DeltaParams {
    float* S;                  // [n, dv, dk] state, updated in place
    const float* q;            // [n, dk]
    const float* k;            // [n, dk]
    const float* v;            // [n, dv]
    const float* a;            // [n, dk] (per key channel) or [n] (per head)
    const float* beta;         // [n]
    float* o;                  // [n, dv]
    int n, dk, dv, a_per_channel;
};
int delta_step_launch(const DeltaParams& p, cudaStream_t stream);

// Arguments of the cache append: each sequence's newest token (position seq_lens[b] - 1)
// copied into its cache slot, for n_pools pools (K and V, or one latent pool).
struct AppendParams {
    const void* src[2];        // [B, H, row_bytes] each
    void* pool[2];             // [num_pages, H, page_size, row_bytes] each
    const int32_t* block_table;
    const int32_t* seq_lens;
    int* err;
    int n_pools, B, H, row_bytes, page_size, max_pages, num_pages;
    int window, n_sink;        // window > 0: rolling cache of n_sink + window slots
};
int append_launch(const AppendParams& p, cudaStream_t stream);

// Arguments of the Quest kernels (page summaries, page selection, attention over the pages).
struct QuestParams {
    const void* q;             // [B, Hq, D]
    const void* k_pool;        // [num_pages, Hkv, P, D]
    const void* v_pool;
    void* kmin;                // [num_pages, Hkv, D], the pool's dtype
    void* kmax;
    const int32_t* block_table;
    const int32_t* seq_lens;
    const int32_t* pages;      // summaries: the physical pages to (re)compute, null = all
    int32_t* sel;              // [B, Hq, n_sel] chosen logical pages, ascending, -1 padded
    float* ub_out;             // [B, Hq, max_pages] bounds (optional)
    void* out;                 // [B, Hq, D]
    float* lse_out;            // [B, Hq] (optional)
    int* err;
    int B, Hq, Hkv, D, page_size, max_pages, num_pages, max_len, n_sel, n_list, dtype;
    float scale;
};
int quest_minmax_launch(const QuestParams& p, cudaStream_t stream);
size_t quest_select_smem(int Hq, int Hkv, int max_pages);
int quest_bounds_launch(const QuestParams& p, cudaStream_t stream);
int quest_select_launch(const QuestParams& p, cudaStream_t stream);   // bounds, then choice
int quest_attn_launch(const QuestParams& p, bool choose, cudaStream_t stream);
int topk_launch(const TopkParams& p, bool need_hist, cudaStream_t stream);

// ---------------------------------------------------------------------------------------
// MLA (absorbed latent), dense or over selected tokens
// ---------------------------------------------------------------------------------------
struct MlaParams {
    const void* q;             // [B, 128, 576] bf16 absorbed queries
    const int32_t* block_table;
    const int32_t* seq_lens;
    const int32_t* idx;        // sparse: [B, idx_stride] logical positions
    const int32_t* idx_count;  // sparse: [B]
    const void* c_pool;        // [num_pages, P, 576] bf16 (gathered rows, sparse)
    float* part_o;             // [n_clusters + B - 1, 128, 512] one slot per piece
    float* part_lse;           // [n_clusters + B - 1, 128] (log2 domain)
    int* err;
    int B, page_size, max_pages, num_pages, max_len;
    int n_clusters, idx_stride, sparse;
    int tile;                  // tokens per tile of the kernel that wrote the partials
    int gap;                   // virtual tiles before each later sequence (piece_gap)
    float scale_log2;
};

// Persistent plan: n_clusters two-CTA clusters share all tiles in equal contiguous ranges;
// the pieces a range cuts out of the sequences get slots cluster + sequence.
struct MlaPlan {
    int n_clusters;
    size_t off_lse, off_o, total;
};
MlaPlan mla_plan(int B, int max_items, bool sparse);
int mla_run(const void* q, const void* c_pool, const int32_t* block_table,
            const int32_t* seq_lens, const int32_t* idx, const int32_t* idx_count, int k,
            void* out, float* lse_out, int B, int H, int d_qk, int d_v, int page_size,
            int max_pages, int num_pages, float scale, void* ws, size_t ws_bytes,
            cudaStream_t stream);
int mla_launch(const MlaParams& p, const CUtensorMap& tc0, const CUtensorMap& tc1,
               const CUtensorMap& tc2, const CUtensorMap& tq, void* out, float* lse_out,
               cudaStream_t stream);

int make_tmap_bf16_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                      uint32_t box_rows);

// 3-D bf16 tensor map over a row-major [rows, cols] matrix: box {64, box_rows, nblocks}
// fills shared memory as [block][row][64] with 128-byte swizzle (cols a multiple of 64).
int make_tmap_u8_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                    uint32_t box_rows);
int make_tmap_bf16_blocked(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                           uint32_t box_rows, uint32_t nblocks);

int num_sms();

// Programmatic dependent launch is on unless kvd_set_option(KVD_OPT_PDL, 0).
bool pdl_enabled();

// Launch with programmatic stream serialization: the kernel may be scheduled while its
// predecessor on the stream finishes (launch and set-up overlap that tail). Every kernel of
// the library waits for the predecessor (griddepcontrol.wait) before it touches memory, so
// the order of memory effects is that of a plain launch. With cluster_x > 0 the blocks form
// thread-block clusters of cluster_x blocks along x (grid.x a multiple of it).
template <typename... P, typename... A>
inline cudaError_t launch_kernel_cluster(void (*kernel)(P...), dim3 grid, dim3 block, size_t smem,
                                         int cluster_x, cudaStream_t stream, A&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int n = 0;
    if (pdl_enabled()) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    if (cluster_x > 0) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = static_cast<unsigned>(cluster_x);
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<A&&>(args)...);
}

template <typename... P, typename... A>
inline cudaError_t launch_kernel(void (*kernel)(P...), dim3 grid, dim3 block, size_t smem,
                                 cudaStream_t stream, A&&... args) {
    return launch_kernel_cluster(kernel, grid, block, smem, 0, stream, static_cast<A&&>(args)...);
}

}  // namespace kvd
