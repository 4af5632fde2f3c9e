// api.cu -- the C ABI of libkvdecode.so: argument validation, split planning,
// workspace layout, tensor-map encoding and kernel launches. See include/kvdecode.h.

#include <cmath>
#include <cstdint>
#include <cstring>
#include <algorithm>
#include <atomic>
#include <mutex>

#include <cudaTypedefs.h>

#include "kvd_host.h"

namespace kvd {

namespace {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }
inline int cdiv(long long a, long long b) { return static_cast<int>((a + b - 1) / b); }
inline size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

// Process-wide options (kvd_set_option); the defaults are what the library is tuned for.
std::atomic<int> g_opt_pdl{1};
std::atomic<long long> g_opt_gqa_chunk{0};
std::atomic<long long> g_opt_mla_min_tiles{0};
std::atomic<int> g_opt_wait_test{0};
std::atomic<int> g_opt_gqa_cluster{1};

}  // namespace

bool pdl_enabled() { return g_opt_pdl.load(std::memory_order_relaxed) != 0; }

int num_sms() {
    static int n = 0;
    if (n == 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 148;
    }
    return n;
}

int make_tmap_bf16_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                      uint32_t box_rows) {
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    if (!g_encode) return KVD_ERR_CUDA;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {64, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? KVD_OK : KVD_ERR_CUDA;
}

// Row-major [rows, cols] bytes (e4m3 codes): 128-byte boxes of box_rows rows, 128-byte swizzle.
int make_tmap_u8_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                    uint32_t box_rows) {
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    if (!g_encode) return KVD_ERR_CUDA;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols};
    cuuint32_t box[2] = {128, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? KVD_OK : KVD_ERR_CUDA;
}

// 3-D view of a row-major [rows, cols] bf16 matrix as (64-element column piece, row,
// column block); the block's stride (128 bytes) is smaller than the row pitch, so a box
// {64, box_rows, nblocks} lands in shared memory as [block][row][64] with 128-byte swizzle.
int make_tmap_bf16_blocked(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                           uint32_t box_rows, uint32_t nblocks) {
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    if (!g_encode || cols % 64 != 0) return KVD_ERR_CUDA;
    cuuint64_t dims[3] = {64, rows, cols / 64};
    cuuint64_t strides[2] = {cols * 2, 128};
    cuuint32_t box[3] = {64, box_rows, nblocks};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? KVD_OK : KVD_ERR_CUDA;
}

// Split plan. Every (sequence, group of KV heads, head block, chunk) is one CTA, two
// CTAs per SM for bf16. A CTA pays a fixed start-up (barrier set-up, block-table read,
// first TMA round trip) and a merge, and a second wave of CTAs pays them again, so:
//  * few groups (at most half the CTA slots): cut the visible range into as many chunks
//    as fit the slots in one wave;
//  * many groups: four chunks of the longest visible range, so that ragged lengths still
//    spread over the SMs.
// Measured on the Llama-3-8B-shaped and sliding-window workloads (chunk sweeps).
int gqa_plan(int B, int Hq, int Hkv, int D, int page_size, int max_len, int window, int n_sink,
             int dtype, GqaPlan* plan) {
    const int G = Hq / Hkv;
    plan->NHG = cdiv(G, 16);
    plan->units = B * Hkv * plan->NHG;
    // two KV heads per tile when a 64-dim page fits one TMA box twice (16 KB per copy)
    plan->hpt = (dtype == KVD_BF16 && D == 64 && Hkv % 2 == 0 && G <= 8 && page_size <= 64)
                    ? 2
                    : 1;
    const long long groups = static_cast<long long>(B) * (Hkv / plan->hpt) * plan->NHG;
    const long long vis = window > 0 ? std::min<long long>(max_len, (long long)window + n_sink)
                                     : max_len;
    long long chunk;
    if (dtype == KVD_F32) {
        chunk = (groups * vis) / std::max(1LL, 16LL * num_sms());
        chunk = std::max(128LL, std::min(1024LL, (chunk / 64) * 64));
    } else {
        const long long slots = 2LL * num_sms();
        const long long per_group = 2 * groups <= slots ? slots / groups : 4;
        chunk = std::max(256LL, (vis + per_group - 1) / per_group);
        chunk = (chunk + 63) / 64 * 64;
    }
    const long long forced = g_opt_gqa_chunk.load(std::memory_order_relaxed);
    if (forced >= 64) chunk = (forced / 64) * 64;  // fixed chunk (KVD_OPT_GQA_CHUNK)
    auto chunks_for = [&](long long C) -> int {
        if (window <= 0) return cdiv(max_len, C);
        const int a = (n_sink > 0 ? cdiv(std::min(n_sink, max_len), C) : 0) +
                      cdiv(std::min(window, max_len) + 63, C);
        const int m = cdiv(std::min<long long>(max_len, (long long)window + n_sink), C);
        return std::max(a, m);
    };
    while (chunks_for(chunk) > kGqaMaxChunks) chunk += 64;
    // Cluster combine (bf16): the chunks of a group form one thread-block cluster of at most
    // 8 CTAs and combine through distributed shared memory, with no global round trip after
    // the last chunk (measured: the workspace combine is ~3.5 us of a sliding-window step).
    // Taken when a group needs at most 8 chunks anyway, or when raising the chunk to get 8
    // still leaves at least three quarters of a wave of CTAs.
    // (KVD_OPT_GQA_CLUSTER = 2 also takes it for many groups when they need <= 8 chunks.)
    plan->cluster = 0;
    const int copt = g_opt_gqa_cluster.load(std::memory_order_relaxed);
    if (dtype == KVD_BF16 && forced < 64 && copt > 0) {
        const long long slots = 2LL * num_sms();
        long long cc = chunk;
        while (chunks_for(cc) > 8) cc += 64;
        const bool few = 2 * groups <= slots;
        if ((few && (chunks_for(chunk) <= 8 || 4 * groups * chunks_for(cc) >= 3 * slots)) ||
            (copt == 2 && chunks_for(chunk) <= 8)) {
            chunk = cc;
            plan->cluster = std::max(1, chunks_for(cc));
        }
    }
    plan->chunk = static_cast<int>(chunk);
    plan->max_chunks = std::max(1, chunks_for(chunk));
    size_t off = kWsHeaderBytes;
    plan->off_counters = off;
    off = round256(off + sizeof(int) * plan->units);
    plan->off_lse = off;
    off = round256(off + sizeof(float) * (size_t)plan->units * plan->max_chunks * 16);
    plan->off_o = off;
    off = round256(off + sizeof(float) * (size_t)plan->units * plan->max_chunks * 16 * D);
    plan->total = off;
    return KVD_OK;
}

TopkLayout topk_layout(int B, int max_len, int k, bool with_scores) {
    TopkLayout l;
    size_t off = kWsHeaderBytes;
    l.off_hist = off;
    off = round256(off + sizeof(uint32_t) * (size_t)B * 2048);
    l.off_hist2 = off;
    off = round256(off + sizeof(uint32_t) * (size_t)B * 256);
    l.off_counts = off;
    off = round256(off + sizeof(int) * (size_t)B * 4);
    l.off_sel = off;
    off = round256(off + sizeof(int) * (size_t)B * k);
    l.off_cand = off;
    off = round256(off + sizeof(uint64_t) * (size_t)B * max_len);
    l.off_bitmap = off;
    off = round256(off + sizeof(uint32_t) * (size_t)B * ((max_len + 31) / 32));
    l.off_scores = off;
    if (with_scores) off = round256(off + sizeof(float) * (size_t)B * max_len);
    l.total = off;
    return l;
}

// MLA split plan: dense units are (sequence, token chunk), about three per SM pair;
// sparse units are (sequence, chunk of the index list), about one per SM pair.
MlaPlan mla_plan(int B, int max_items, bool sparse) {
    MlaPlan pl;
    const long long max_tiles = (long long)B * ((max_items + 63) / 64);
    // Tiles a cluster takes at least (KVD_OPT_MLA_MIN_TILES overrides): 2 for the sparse
    // decode, whose few tiles would otherwise spread one per cluster and each cluster writes a
    // whole 128 x 512 partial (measured on the DSA workload: 61.6 -> 60.6 us a step; 3 was
    // slower), 1 for the dense decode.
    const long long opt = g_opt_mla_min_tiles.load(std::memory_order_relaxed);
    const long long min_tiles = opt >= 1 ? opt : (sparse ? 2 : 1);
    pl.n_clusters = static_cast<int>(std::max(
        1LL, std::min<long long>(num_sms() / 2, (max_tiles + min_tiles - 1) / min_tiles)));
    const size_t slots = (size_t)pl.n_clusters + B - 1;
    size_t off = kWsHeaderBytes;
    pl.off_lse = off;
    off = round256(off + sizeof(float) * slots * 128);
    pl.off_o = off;
    off = round256(off + sizeof(float) * slots * 128 * 512);
    pl.total = off;
    return pl;
}

int mla_run(const void* q, const void* c_pool, const int32_t* block_table,
            const int32_t* seq_lens, const int32_t* idx, const int32_t* idx_count, int k,
            void* out, float* lse_out, int B, int H, int d_qk, int d_v, int page_size,
            int max_pages, int num_pages, float scale, void* ws, size_t ws_bytes,
            cudaStream_t stream) {
    if (!q || !c_pool || !block_table || !seq_lens || !out || !ws) return KVD_ERR_INVALID_ARG;
    if (B < 1 || max_pages < 1 || num_pages < 1 || !std::isfinite(scale))
        return KVD_ERR_INVALID_ARG;
    if (H != 128 || d_qk != 576 || d_v != 512) return KVD_ERR_UNSUPPORTED;
    if (!pow2(page_size) || page_size < 16 || page_size > 256) return KVD_ERR_UNSUPPORTED;
    if ((long long)num_pages * page_size >= (1LL << 31) || (long long)B * 128 >= (1LL << 31))
        return KVD_ERR_UNSUPPORTED;
    if ((long long)max_pages * page_size >= (1LL << 30)) return KVD_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(c_pool) || !aligned16(out) || !aligned16(ws))
        return KVD_ERR_INVALID_ARG;
    const bool sparse = idx != nullptr;
    const int max_len = max_pages * page_size;
    const MlaPlan pl = mla_plan(B, sparse ? k : max_len, sparse);
    if (ws_bytes < pl.total) return KVD_ERR_WORKSPACE_TOO_SMALL;
    uint8_t* wb = static_cast<uint8_t*>(ws);
    MlaParams p;
    std::memset(&p, 0, sizeof p);
    p.q = q;
    p.block_table = block_table;
    p.seq_lens = seq_lens;
    p.idx = idx;
    p.idx_count = idx_count;
    p.c_pool = c_pool;
    p.part_o = reinterpret_cast<float*>(wb + pl.off_o);
    p.part_lse = reinterpret_cast<float*>(wb + pl.off_lse);
    p.err = reinterpret_cast<int*>(wb);
    p.B = B;
    p.page_size = page_size;
    p.max_pages = max_pages;
    p.num_pages = num_pages;
    p.max_len = max_len;
    p.n_clusters = pl.n_clusters;
    p.idx_stride = k;
    p.sparse = sparse ? 1 : 0;
    p.tile = 64;
    p.gap = 6;
    p.scale_log2 = scale * 1.4426950408889634f;
    // 3-D maps (rank 0: 4 blocks of 64 dims, rank 1: 5) for 64-token tiles within a page,
    // and a 2-D map for pages shorter than a tile
    CUtensorMap tc0, tc1, tc2;
    const uint64_t rows = (uint64_t)num_pages * page_size;
    if (make_tmap_bf16_blocked(&tc0, c_pool, rows, 576, 64, 4) != KVD_OK) return KVD_ERR_CUDA;
    if (make_tmap_bf16_blocked(&tc1, c_pool, rows, 576, 64, 5) != KVD_OK) return KVD_ERR_CUDA;
    if (make_tmap_bf16_2d(&tc2, c_pool, rows, 576, page_size < 64 ? page_size : 64) != KVD_OK)
        return KVD_ERR_CUDA;
    // the queries as [B * 128 rows, 576] (128-row boxes: one head block of one sequence)
    CUtensorMap tq;
    if (make_tmap_bf16_2d(&tq, q, static_cast<uint64_t>(B) * 128, 576, 128) != KVD_OK)
        return KVD_ERR_CUDA;
    return mla_launch(p, tc0, tc1, tc2, tq, out, lse_out, stream);
}

}  // namespace kvd

using namespace kvd;

namespace kvd {

int gqa_check(const void* q, const void* k_pool, const void* v_pool, const int32_t* block_table,
              const int32_t* seq_lens, const void* out, int B, int Hq, int Hkv, int D,
              int page_size, int max_pages, int num_pages, float scale, int dtype, int window,
              int n_sink, int ring) {
    if (!q || !k_pool || !v_pool || !block_table || !seq_lens || !out) return KVD_ERR_INVALID_ARG;
    if (ring < 0 || (ring > 0 && (window != 0 || n_sink != 0 ||
                                  (long long)ring > (long long)max_pages * page_size)))
        return KVD_ERR_INVALID_ARG;
    if (B < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || max_pages < 1 || num_pages < 1)
        return KVD_ERR_INVALID_ARG;
    if (!std::isfinite(scale) || window < 0 || n_sink < 0) return KVD_ERR_INVALID_ARG;
    if (!pow2(page_size) || page_size < 16 || page_size > 256) return KVD_ERR_UNSUPPORTED;
    if (D != 64 && D != 128) return KVD_ERR_UNSUPPORTED;
    if (dtype != KVD_F32 && dtype != KVD_BF16) return KVD_ERR_UNSUPPORTED;
    if (Hq / Hkv > 128) return KVD_ERR_UNSUPPORTED;
    if ((long long)num_pages * Hkv * page_size >= (1LL << 31)) return KVD_ERR_UNSUPPORTED;
    if ((long long)max_pages * page_size >= (1LL << 30)) return KVD_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(out))
        return KVD_ERR_INVALID_ARG;
    return KVD_OK;
}

int gqa_run(const void* q, const void* k_pool, const void* v_pool, const int32_t* block_table,
               const int32_t* seq_lens, void* out, float* lse_out, int B, int Hq, int Hkv, int D,
               int page_size, int max_pages, int num_pages, float scale, int dtype, int window,
               int n_sink, const float* sink_logit, void* ws, size_t ws_bytes,
               cudaStream_t stream, int ring, int ring_sink, const void* k_new,
               const void* v_new) {
    const int st = gqa_check(q, k_pool, v_pool, block_table, seq_lens, out, B, Hq, Hkv, D,
                             page_size, max_pages, num_pages, scale, dtype, window, n_sink, ring);
    if (st != KVD_OK) return st;
    if (!ws || !aligned16(ws)) return KVD_ERR_INVALID_ARG;
    const int max_len = max_pages * page_size;
    GqaPlan plan;
    if (gqa_plan(B, Hq, Hkv, D, page_size, max_len, window, n_sink, dtype, &plan) != KVD_OK)
        return KVD_ERR_UNSUPPORTED;
    if (ws_bytes < plan.total) return KVD_ERR_WORKSPACE_TOO_SMALL;

    GqaParams p;
    std::memset(&p, 0, sizeof p);
    p.q = q;
    p.k_pool = k_pool;
    p.v_pool = v_pool;
    p.block_table = block_table;
    p.seq_lens = seq_lens;
    p.out = out;
    p.lse_out = lse_out;
    p.sink_logit = sink_logit;
    uint8_t* w = static_cast<uint8_t*>(ws);
    p.err = reinterpret_cast<int*>(w);
    p.counters = reinterpret_cast<int*>(w + plan.off_counters);
    p.part_lse = reinterpret_cast<float*>(w + plan.off_lse);
    p.part_o = reinterpret_cast<float*>(w + plan.off_o);
    p.B = B;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.D = D;
    p.G = Hq / Hkv;
    p.NHG = plan.NHG;
    p.units = plan.units;
    p.page_size = page_size;
    p.max_pages = max_pages;
    p.num_pages = num_pages;
    p.max_len = max_len;
    p.window = window;
    p.n_sink = n_sink;
    p.ring = ring;
    p.ring_sink = ring_sink;
    p.k_new = k_new;
    p.v_new = v_new;
    p.chunk = plan.chunk;
    p.max_chunks = plan.max_chunks;
    p.dtype = dtype;
    p.scale_log2 = scale * 1.4426950408889634f;

    if (dtype == KVD_F32) return gqa_launch(plan, p, nullptr, nullptr, stream);
    // KVD_OPT_WAIT_TIMEOUT_TEST, taken by this call only: a short limit on every wait of the
    // ring and consumers that first wait on a barrier nothing completes
    if (g_opt_wait_test.exchange(0) != 0) {
        p.wait_cycles = 1000;
        p.stall_test = 1;
    }
    CUtensorMap tk, tv;
    const uint64_t rows = (uint64_t)num_pages * Hkv * page_size;
    const uint32_t box_rows = (page_size < 64 ? page_size : 64) * plan.hpt;
    if (make_tmap_bf16_blocked(&tk, k_pool, rows, D, box_rows, D / 64) != KVD_OK)
        return KVD_ERR_CUDA;
    if (make_tmap_bf16_blocked(&tv, v_pool, rows, D, box_rows, D / 64) != KVD_OK)
        return KVD_ERR_CUDA;
    return gqa_launch(plan, p, &tk, &tv, stream);
}

}  // namespace kvd

extern "C" {

int attn_decode_gqa_paged(const void* q, const void* k_pool, const void* v_pool,
                          const int32_t* block_table, const int32_t* seq_lens, void* out,
                          float* lse_out, int B, int Hq, int Hkv, int D, int page_size,
                          int max_pages, int num_pages, float scale, int dtype, void* ws,
                          size_t ws_bytes, cudaStream_t stream) {
    return gqa_run(q, k_pool, v_pool, block_table, seq_lens, out, lse_out, B, Hq, Hkv, D,
                      page_size, max_pages, num_pages, scale, dtype, 0, 0, nullptr, ws, ws_bytes,
                      stream);
}

int attn_decode_swa_sink(const void* q, const void* k_pool, const void* v_pool,
                         const int32_t* block_table, const int32_t* seq_lens, void* out,
                         float* lse_out, int B, int Hq, int Hkv, int D, int page_size,
                         int max_pages, int num_pages, float scale, int dtype, int window,
                         int n_sink_tokens, const float* sink_logit, void* ws, size_t ws_bytes,
                         cudaStream_t stream) {
    if (window < 1) return KVD_ERR_INVALID_ARG;
    return gqa_run(q, k_pool, v_pool, block_table, seq_lens, out, lse_out, B, Hq, Hkv, D,
                      page_size, max_pages, num_pages, scale, dtype, window, n_sink_tokens,
                      sink_logit, ws, ws_bytes, stream);
}

int attn_decode_swa_ring(const void* q, const void* k_ring, const void* v_ring,
                         const int32_t* block_table, const int32_t* seq_lens, void* out,
                         float* lse_out, int B, int Hq, int Hkv, int D, int page_size,
                         int max_pages, int num_pages, float scale, int dtype, int window,
                         int n_sink_tokens, const float* sink_logit, void* ws, size_t ws_bytes,
                         cudaStream_t stream) {
    if (window < 1 || n_sink_tokens < 0) return KVD_ERR_INVALID_ARG;
    const long long cap = (long long)n_sink_tokens + window;
    if (cap > (long long)max_pages * page_size) return KVD_ERR_INVALID_ARG;
    return gqa_run(q, k_ring, v_ring, block_table, seq_lens, out, lse_out, B, Hq, Hkv, D,
                   page_size, max_pages, num_pages, scale, dtype, 0, 0, sink_logit, ws, ws_bytes,
                   stream, static_cast<int>(cap));
}

int attn_decode_swa_ring_append(const void* q, const void* k_new, const void* v_new,
                                void* k_ring, void* v_ring, const int32_t* block_table,
                                const int32_t* seq_lens, void* out, float* lse_out, int B,
                                int Hq, int Hkv, int D, int page_size, int max_pages,
                                int num_pages, float scale, int dtype, int window,
                                int n_sink_tokens, const float* sink_logit, void* ws,
                                size_t ws_bytes, cudaStream_t stream) {
    if (!k_new || !v_new || !k_ring || !v_ring) return KVD_ERR_INVALID_ARG;
    if (!aligned16(k_new) || !aligned16(v_new)) return KVD_ERR_INVALID_ARG;
    if (window < 1 || n_sink_tokens < 0) return KVD_ERR_INVALID_ARG;
    const long long cap = (long long)n_sink_tokens + window;
    if (cap > (long long)max_pages * page_size) return KVD_ERR_INVALID_ARG;
    // every argument check (the attention's) before anything is written
    const int st = gqa_check(q, k_ring, v_ring, block_table, seq_lens, out, B, Hq, Hkv, D,
                             page_size, max_pages, num_pages, scale, dtype, 0, 0,
                             static_cast<int>(cap));
    if (st != KVD_OK) return st;
    if (!ws || !aligned16(ws)) return KVD_ERR_INVALID_ARG;
    if (dtype == KVD_F32) {
        // float32 rings: the append's own launch, then the attention (the bf16 kernel
        // writes the rows itself)
        AppendParams ap;
        std::memset(&ap, 0, sizeof ap);
        ap.src[0] = k_new;
        ap.pool[0] = k_ring;
        ap.src[1] = v_new;
        ap.pool[1] = v_ring;
        ap.n_pools = 2;
        ap.block_table = block_table;
        ap.seq_lens = seq_lens;
        ap.err = static_cast<int*>(ws);
        ap.B = B;
        ap.H = Hkv;
        ap.row_bytes = D * 4;
        ap.page_size = page_size;
        ap.max_pages = max_pages;
        ap.num_pages = num_pages;
        ap.window = window;
        ap.n_sink = n_sink_tokens;
        const int ea = append_launch(ap, stream);
        if (ea != KVD_OK) return ea;
        return gqa_run(q, k_ring, v_ring, block_table, seq_lens, out, lse_out, B, Hq, Hkv, D,
                       page_size, max_pages, num_pages, scale, dtype, 0, 0, sink_logit, ws,
                       ws_bytes, stream, static_cast<int>(cap), n_sink_tokens);
    }
    return gqa_run(q, k_ring, v_ring, block_table, seq_lens, out, lse_out, B, Hq, Hkv, D,
                   page_size, max_pages, num_pages, scale, dtype, 0, 0, sink_logit, ws, ws_bytes,
                   stream, static_cast<int>(cap), n_sink_tokens, k_new, v_new);
}

int kvd_cache_append(const void* k_new, const void* v_new, void* k_pool, void* v_pool,
                     const int32_t* block_table, const int32_t* seq_lens, int B, int H, int D,
                     int page_size, int max_pages, int num_pages, int dtype, int window,
                     int n_sink, int* err, cudaStream_t stream) {
    if (!k_new || !k_pool || !block_table || !seq_lens || !err) return KVD_ERR_INVALID_ARG;
    if (!v_new != !v_pool) return KVD_ERR_INVALID_ARG;
    if (B < 1 || H < 1 || D < 1 || page_size < 1 || max_pages < 1 || num_pages < 1 ||
        window < 0 || n_sink < 0)
        return KVD_ERR_INVALID_ARG;
    if (dtype != KVD_F32 && dtype != KVD_BF16) return KVD_ERR_UNSUPPORTED;
    const long long row_bytes = (long long)D * (dtype == KVD_F32 ? 4 : 2);
    if (row_bytes % 16 != 0 || row_bytes > (1 << 20)) return KVD_ERR_UNSUPPORTED;
    if ((long long)max_pages * page_size >= (1LL << 30)) return KVD_ERR_UNSUPPORTED;
    if (window > 0 && (long long)n_sink + window > (long long)max_pages * page_size)
        return KVD_ERR_INVALID_ARG;
    if (!aligned16(k_new) || !aligned16(k_pool) || (v_new && !aligned16(v_new)) ||
        (v_pool && !aligned16(v_pool)) || (reinterpret_cast<uintptr_t>(err) & 3))
        return KVD_ERR_INVALID_ARG;
    AppendParams ap;
    std::memset(&ap, 0, sizeof ap);
    ap.src[0] = k_new;
    ap.pool[0] = k_pool;
    ap.src[1] = v_new;
    ap.pool[1] = v_pool;
    ap.n_pools = v_new ? 2 : 1;
    ap.block_table = block_table;
    ap.seq_lens = seq_lens;
    ap.err = err;
    ap.B = B;
    ap.H = H;
    ap.row_bytes = static_cast<int>(row_bytes);
    ap.page_size = page_size;
    ap.max_pages = max_pages;
    ap.num_pages = num_pages;
    ap.window = window;
    ap.n_sink = n_sink;
    return append_launch(ap, stream);
}

// Checks shared by the three Quest entry points.
static int quest_common(QuestParams& qp, int B, int Hq, int Hkv, int D, int page_size,
                        int max_pages, int num_pages, int dtype, int* err) {
    if (!err || (reinterpret_cast<uintptr_t>(err) & 3)) return KVD_ERR_INVALID_ARG;
    if (B < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || page_size < 1 || max_pages < 1 ||
        num_pages < 1)
        return KVD_ERR_INVALID_ARG;
    if (D != 64 && D != 128) return KVD_ERR_UNSUPPORTED;
    if (dtype != KVD_F32 && dtype != KVD_BF16) return KVD_ERR_UNSUPPORTED;
    if (Hq / Hkv > 16) return KVD_ERR_UNSUPPORTED;
    if ((long long)num_pages * Hkv * page_size >= (1LL << 31) ||
        (long long)max_pages * page_size >= (1LL << 30))
        return KVD_ERR_UNSUPPORTED;
    std::memset(&qp, 0, sizeof qp);
    qp.B = B;
    qp.Hq = Hq;
    qp.Hkv = Hkv;
    qp.D = D;
    qp.page_size = page_size;
    qp.max_pages = max_pages;
    qp.num_pages = num_pages;
    qp.max_len = max_pages * page_size;
    qp.dtype = dtype;
    qp.err = err;
    return KVD_OK;
}

int quest_page_minmax(const void* k_pool, void* kmin, void* kmax, const int32_t* pages,
                      int n_list, int num_pages, int Hkv, int page_size, int D, int dtype,
                      int* err, cudaStream_t stream) {
    if (!k_pool || !kmin || !kmax) return KVD_ERR_INVALID_ARG;
    QuestParams qp;
    const int st = quest_common(qp, 1, Hkv, Hkv, D, page_size, 1, num_pages, dtype, err);
    if (st != KVD_OK) return st;
    if (!pages) n_list = num_pages;
    if (n_list < 1) return KVD_ERR_INVALID_ARG;
    if (!aligned16(k_pool) || !aligned16(kmin) || !aligned16(kmax) ||
        (pages && (reinterpret_cast<uintptr_t>(pages) & 3)))
        return KVD_ERR_INVALID_ARG;
    qp.k_pool = k_pool;
    qp.kmin = kmin;
    qp.kmax = kmax;
    qp.pages = pages;
    qp.n_list = n_list;
    return quest_minmax_launch(qp, stream);
}

int quest_select_pages(const void* q, const void* kmin, const void* kmax,
                       const int32_t* block_table, const int32_t* seq_lens, int32_t* sel,
                       float* ub_out, int B, int Hq, int Hkv, int D, int page_size, int max_pages,
                       int num_pages, int n_sel, int dtype, int* err, cudaStream_t stream) {
    if (!q || !kmin || !kmax || !block_table || !seq_lens || !sel || !ub_out)
        return KVD_ERR_INVALID_ARG;
    QuestParams qp;
    const int st = quest_common(qp, B, Hq, Hkv, D, page_size, max_pages, num_pages, dtype, err);
    if (st != KVD_OK) return st;
    if (n_sel < 1 || n_sel > 64) return KVD_ERR_UNSUPPORTED;
    if (quest_select_smem(Hq, Hkv, max_pages) > 200 * 1024) return KVD_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(kmin) || !aligned16(kmax) ||
        (reinterpret_cast<uintptr_t>(sel) & 3) || (reinterpret_cast<uintptr_t>(ub_out) & 3))
        return KVD_ERR_INVALID_ARG;
    qp.q = q;
    qp.kmin = const_cast<void*>(kmin);
    qp.kmax = const_cast<void*>(kmax);
    qp.block_table = block_table;
    qp.seq_lens = seq_lens;
    qp.sel = sel;
    qp.ub_out = ub_out;
    qp.n_sel = n_sel;
    return quest_select_launch(qp, stream);
}

int attn_decode_quest(const void* q, const void* k_pool, const void* v_pool,
                      const int32_t* block_table, const int32_t* seq_lens, const int32_t* sel,
                      void* out, float* lse_out, int B, int Hq, int Hkv, int D, int page_size,
                      int max_pages, int num_pages, int n_sel, float scale, int dtype, int* err,
                      cudaStream_t stream) {
    if (!q || !k_pool || !v_pool || !block_table || !seq_lens || !sel || !out)
        return KVD_ERR_INVALID_ARG;
    QuestParams qp;
    const int st = quest_common(qp, B, Hq, Hkv, D, page_size, max_pages, num_pages, dtype, err);
    if (st != KVD_OK) return st;
    if (n_sel < 1 || n_sel > 64) return KVD_ERR_UNSUPPORTED;
    if (!std::isfinite(scale)) return KVD_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(out) ||
        (reinterpret_cast<uintptr_t>(sel) & 3) || (reinterpret_cast<uintptr_t>(lse_out) & 3))
        return KVD_ERR_INVALID_ARG;
    qp.q = q;
    qp.k_pool = k_pool;
    qp.v_pool = v_pool;
    qp.block_table = block_table;
    qp.seq_lens = seq_lens;
    qp.sel = const_cast<int32_t*>(sel);
    qp.out = out;
    qp.lse_out = lse_out;
    qp.n_sel = n_sel;
    qp.scale = scale;
    return quest_attn_launch(qp, false, stream);
}

int quest_page_bounds(const void* q, const void* kmin, const void* kmax,
                      const int32_t* block_table, const int32_t* seq_lens, float* ub, int B,
                      int Hq, int Hkv, int D, int page_size, int max_pages, int num_pages,
                      int dtype, int* err, cudaStream_t stream) {
    if (!q || !kmin || !kmax || !block_table || !seq_lens || !ub) return KVD_ERR_INVALID_ARG;
    QuestParams qp;
    const int st = quest_common(qp, B, Hq, Hkv, D, page_size, max_pages, num_pages, dtype, err);
    if (st != KVD_OK) return st;
    if (!aligned16(q) || !aligned16(kmin) || !aligned16(kmax) ||
        (reinterpret_cast<uintptr_t>(ub) & 3))
        return KVD_ERR_INVALID_ARG;
    qp.q = q;
    qp.kmin = const_cast<void*>(kmin);
    qp.kmax = const_cast<void*>(kmax);
    qp.block_table = block_table;
    qp.seq_lens = seq_lens;
    qp.ub_out = ub;
    return quest_bounds_launch(qp, stream);
}

int attn_decode_quest_from_bounds(const void* q, const void* k_pool, const void* v_pool,
                                  const int32_t* block_table, const int32_t* seq_lens,
                                  const float* ub, int32_t* sel_out, void* out, float* lse_out,
                                  int B, int Hq, int Hkv, int D, int page_size, int max_pages,
                                  int num_pages, int n_sel, float scale, int dtype, int* err,
                                  cudaStream_t stream) {
    if (!q || !k_pool || !v_pool || !block_table || !seq_lens || !ub || !sel_out || !out)
        return KVD_ERR_INVALID_ARG;
    QuestParams qp;
    const int st = quest_common(qp, B, Hq, Hkv, D, page_size, max_pages, num_pages, dtype, err);
    if (st != KVD_OK) return st;
    if (n_sel < 1 || n_sel > 64) return KVD_ERR_UNSUPPORTED;
    if ((size_t)max_pages * 8 > 200 * 1024) return KVD_ERR_UNSUPPORTED;
    if (!std::isfinite(scale)) return KVD_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(out) ||
        (reinterpret_cast<uintptr_t>(ub) & 3) || (reinterpret_cast<uintptr_t>(sel_out) & 3) ||
        (reinterpret_cast<uintptr_t>(lse_out) & 3))
        return KVD_ERR_INVALID_ARG;
    qp.q = q;
    qp.k_pool = k_pool;
    qp.v_pool = v_pool;
    qp.block_table = block_table;
    qp.seq_lens = seq_lens;
    qp.ub_out = const_cast<float*>(ub);
    qp.sel = sel_out;
    qp.out = out;
    qp.lse_out = lse_out;
    qp.n_sel = n_sel;
    qp.scale = scale;
    return quest_attn_launch(qp, true, stream);
}

int attn_decode_mla(const void* q, const void* c_pool, const int32_t* block_table,
                    const int32_t* seq_lens, void* out, float* lse_out, int B, int H, int d_qk,
                    int d_v, int page_size, int max_pages, int num_pages, float scale, void* ws,
                    size_t ws_bytes, cudaStream_t stream) {
    return mla_run(q, c_pool, block_table, seq_lens, nullptr, nullptr, 0, out, lse_out, B, H,
                   d_qk, d_v, page_size, max_pages, num_pages, scale, ws, ws_bytes, stream);
}

// Both indexer precisions (fp8: e4m3 codes with row scales): validation, workspace layout,
// tensor maps, the indexer launch, then the selection.
static int indexer_topk(bool fp8, const void* q_idx, const float* q_scale, const void* k_idx_pool,
                        const float* k_scale, const float* w, const int32_t* block_table,
                        const int32_t* seq_lens, int32_t* topk_idx, int32_t* topk_count,
                        float* scores_out, int B, int Hi, int Di, int page_size, int max_pages,
                        int num_pages, int k, void* ws, size_t ws_bytes, cudaStream_t stream) {
    if (!q_idx || !k_idx_pool || !w || !block_table || !seq_lens || !topk_idx || !topk_count ||
        !ws)
        return KVD_ERR_INVALID_ARG;
    if (fp8 && (!q_scale || !k_scale || !aligned16(k_scale) ||
                (reinterpret_cast<uintptr_t>(q_scale) & 3)))
        return KVD_ERR_INVALID_ARG;
    if (B < 1 || max_pages < 1 || num_pages < 1 || k < 1) return KVD_ERR_INVALID_ARG;
    if (Hi != 64 || Di != 128 || k > kTopkMaxK) return KVD_ERR_UNSUPPORTED;
    if (!pow2(page_size) || page_size < 16 || page_size > 256) return KVD_ERR_UNSUPPORTED;
    if ((long long)num_pages * page_size >= (1LL << 31) || (long long)B * 64 >= (1LL << 31))
        return KVD_ERR_UNSUPPORTED;
    if ((long long)max_pages * page_size >= (1LL << 30)) return KVD_ERR_UNSUPPORTED;
    if (!aligned16(q_idx) || !aligned16(k_idx_pool) || !aligned16(ws) ||
        (reinterpret_cast<uintptr_t>(w) & 3) || (reinterpret_cast<uintptr_t>(scores_out) & 3))
        return KVD_ERR_INVALID_ARG;
    const int max_len = max_pages * page_size;
    const TopkLayout lay = topk_layout(B, max_len, k, scores_out == nullptr);
    if (ws_bytes < lay.total) return KVD_ERR_WORKSPACE_TOO_SMALL;
    uint8_t* wb = static_cast<uint8_t*>(ws);
    IdxParams ip;
    std::memset(&ip, 0, sizeof ip);
    ip.q = q_idx;
    ip.w = w;
    ip.q_scale = q_scale;
    ip.k_scale = k_scale;
    ip.block_table = block_table;
    ip.seq_lens = seq_lens;
    ip.scores = scores_out ? scores_out : reinterpret_cast<float*>(wb + lay.off_scores);
    ip.score_stride = max_len;
    ip.hist = reinterpret_cast<uint32_t*>(wb + lay.off_hist);
    ip.counts = reinterpret_cast<int*>(wb + lay.off_counts);
    ip.err = reinterpret_cast<int*>(wb);
    ip.B = B;
    ip.page_size = page_size;
    ip.max_pages = max_pages;
    ip.num_pages = num_pages;
    ip.max_len = max_len;
    ip.tiles_per_b = (max_len + 127) / 128;
    CUtensorMap tk, tk128, tq;
    const uint64_t rows = (uint64_t)num_pages * page_size;
    const uint32_t piece = page_size < 128 ? page_size : 128;
    int st;
    if (fp8) {
        // one-byte codes: a 128-dim row is one 128-byte box
        if (make_tmap_u8_2d(&tk, k_idx_pool, rows, 128, piece) != KVD_OK ||
            make_tmap_u8_2d(&tk128, k_idx_pool, rows, 128, 128) != KVD_OK ||
            make_tmap_u8_2d(&tq, q_idx, (uint64_t)B * 64, 128, 64) != KVD_OK)
            return KVD_ERR_CUDA;
        st = dsa_indexer_fp8_launch(ip, tk, tk128, tq, stream);
    } else {
        if (make_tmap_bf16_2d(&tk, k_idx_pool, rows, 128, piece) != KVD_OK) return KVD_ERR_CUDA;
        // one instruction per 128-token tile when its rows are contiguous in the pool
        if (make_tmap_bf16_blocked(&tk128, k_idx_pool, rows, 128, 128, 2) != KVD_OK)
            return KVD_ERR_CUDA;
        if (make_tmap_bf16_2d(&tq, q_idx, (uint64_t)B * 64, 128, 64) != KVD_OK)
            return KVD_ERR_CUDA;
        st = dsa_indexer_launch(ip, tk, tk128, tq, stream);
    }
    if (st != KVD_OK) return st;
    TopkParams tp;
    std::memset(&tp, 0, sizeof tp);
    tp.scores = ip.scores;
    tp.score_stride = max_len;
    tp.lens = seq_lens;
    tp.hist = ip.hist;
    tp.hist2 = reinterpret_cast<uint32_t*>(wb + lay.off_hist2);
    tp.counts = reinterpret_cast<int*>(wb + lay.off_counts);
    tp.sel = reinterpret_cast<int*>(wb + lay.off_sel);
    tp.cand = reinterpret_cast<uint64_t*>(wb + lay.off_cand);
    tp.bitmap = reinterpret_cast<uint32_t*>(wb + lay.off_bitmap);
    tp.topk_idx = topk_idx;
    tp.topk_count = topk_count;
    tp.err = ip.err;
    tp.B = B;
    tp.k = k;
    tp.max_len = max_len;
    return topk_launch(tp, false, stream);
}

int dsa_indexer_topk(const void* q_idx, const void* k_idx_pool, const float* w,
                     const int32_t* block_table, const int32_t* seq_lens, int32_t* topk_idx,
                     int32_t* topk_count, float* scores_out, int B, int Hi, int Di, int page_size,
                     int max_pages, int num_pages, int k, void* ws, size_t ws_bytes,
                     cudaStream_t stream) {
    return indexer_topk(false, q_idx, nullptr, k_idx_pool, nullptr, w, block_table, seq_lens,
                        topk_idx, topk_count, scores_out, B, Hi, Di, page_size, max_pages,
                        num_pages, k, ws, ws_bytes, stream);
}

int dsa_indexer_topk_fp8(const void* q8, const float* q_scale, const void* k8_pool,
                         const float* k_scale, const float* w, const int32_t* block_table,
                         const int32_t* seq_lens, int32_t* topk_idx, int32_t* topk_count,
                         float* scores_out, int B, int Hi, int Di, int page_size, int max_pages,
                         int num_pages, int k, void* ws, size_t ws_bytes, cudaStream_t stream) {
    return indexer_topk(true, q8, q_scale, k8_pool, k_scale, w, block_table, seq_lens, topk_idx,
                        topk_count, scores_out, B, Hi, Di, page_size, max_pages, num_pages, k, ws,
                        ws_bytes, stream);
}

int kvd_quantize_e4m3_rows(const void* x, void* codes, float* scales, int rows, int cols,
                           cudaStream_t stream) {
    if (!x || !codes || !scales) return KVD_ERR_INVALID_ARG;
    if (rows < 1 || cols < 1 || cols > 65536) return KVD_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(x) & 1) || (reinterpret_cast<uintptr_t>(scales) & 3))
        return KVD_ERR_INVALID_ARG;
    QuantParams qp;
    std::memset(&qp, 0, sizeof qp);
    qp.x = x;
    qp.codes = codes;
    qp.scales = scales;
    qp.rows = rows;
    qp.cols = cols;
    return quantize_e4m3_launch(qp, stream);
}

int kvd_delta_decode_step(float* S, const float* q, const float* k, const float* v,
                          const float* a, const float* beta, float* o, int n, int dk, int dv,
                          int a_per_channel, cudaStream_t stream) {
    if (!S || !q || !k || !v || !a || !beta || !o || n < 1) return KVD_ERR_INVALID_ARG;
    if (dk != 64 && dk != 128 && dk != 256) return KVD_ERR_UNSUPPORTED;
    if (dv < 1 || dv > 65536) return KVD_ERR_UNSUPPORTED;
    const uintptr_t vec = dk == 64 ? 7 : 15;  // the kernel's vector width in bytes, minus 1
    if ((reinterpret_cast<uintptr_t>(S) & vec) || (reinterpret_cast<uintptr_t>(q) & vec) ||
        (reinterpret_cast<uintptr_t>(k) & vec) ||
        (a_per_channel && (reinterpret_cast<uintptr_t>(a) & vec)) ||
        (reinterpret_cast<uintptr_t>(v) & 3) || (reinterpret_cast<uintptr_t>(a) & 3) ||
        (reinterpret_cast<uintptr_t>(beta) & 3) || (reinterpret_cast<uintptr_t>(o) & 3))
        return KVD_ERR_INVALID_ARG;
    // o must not overlap the state it is read from
    const uintptr_t s0 = reinterpret_cast<uintptr_t>(S), o0 = reinterpret_cast<uintptr_t>(o);
    const uintptr_t s1 = s0 + (uintptr_t)n * dv * dk * 4, o1 = o0 + (uintptr_t)n * dv * 4;
    if (o0 < s1 && s0 < o1) return KVD_ERR_INVALID_ARG;
    DeltaParams dp;
    std::memset(&dp, 0, sizeof dp);
    dp.S = S;
    dp.q = q;
    dp.k = k;
    dp.v = v;
    dp.a = a;
    dp.beta = beta;
    dp.o = o;
    dp.n = n;
    dp.dk = dk;
    dp.dv = dv;
    dp.a_per_channel = a_per_channel ? 1 : 0;
    return delta_step_launch(dp, stream);
}

int dsa_indexer_cache_append_fp8(const void* k_new, const int32_t* block_table,
                                 const int32_t* seq_lens, void* k8_pool, float* k_scale, int B,
                                 int Di, int page_size, int max_pages, int num_pages, int* err,
                                 cudaStream_t stream) {
    if (!k_new || !block_table || !seq_lens || !k8_pool || !k_scale || !err)
        return KVD_ERR_INVALID_ARG;
    if (B < 1 || Di < 1 || Di > 65536 || max_pages < 1 || num_pages < 1 || page_size < 1)
        return KVD_ERR_INVALID_ARG;
    if ((long long)num_pages * page_size >= (1LL << 31) ||
        (long long)max_pages * page_size >= (1LL << 30))
        return KVD_ERR_UNSUPPORTED;
    if ((reinterpret_cast<uintptr_t>(k_new) & 1) || (reinterpret_cast<uintptr_t>(k_scale) & 3) ||
        (reinterpret_cast<uintptr_t>(err) & 3))
        return KVD_ERR_INVALID_ARG;
    QuantParams qp;
    std::memset(&qp, 0, sizeof qp);
    qp.x = k_new;
    qp.codes = k8_pool;
    qp.scales = k_scale;
    qp.block_table = block_table;
    qp.seq_lens = seq_lens;
    qp.err = err;
    qp.rows = B;
    qp.cols = Di;
    qp.page_size = page_size;
    qp.max_pages = max_pages;
    qp.num_pages = num_pages;
    qp.max_len = max_pages * page_size;
    return quantize_e4m3_launch(qp, stream);
}

int dsa_topk(const float* scores, const int32_t* lens, int32_t* topk_idx, int32_t* topk_count,
             int B, int score_stride, int k, void* ws, size_t ws_bytes, cudaStream_t stream) {
    if (!scores || !lens || !topk_idx || !topk_count || !ws) return KVD_ERR_INVALID_ARG;
    if (B < 1 || score_stride < 1 || k < 1) return KVD_ERR_INVALID_ARG;
    if (k > kTopkMaxK) return KVD_ERR_UNSUPPORTED;
    if (!aligned16(ws) || (reinterpret_cast<uintptr_t>(scores) & 3)) return KVD_ERR_INVALID_ARG;
    const TopkLayout lay = topk_layout(B, score_stride, k, false);
    if (ws_bytes < lay.total) return KVD_ERR_WORKSPACE_TOO_SMALL;
    uint8_t* wb = static_cast<uint8_t*>(ws);
    TopkParams tp;
    std::memset(&tp, 0, sizeof tp);
    tp.scores = scores;
    tp.score_stride = score_stride;
    tp.lens = lens;
    tp.hist = reinterpret_cast<uint32_t*>(wb + lay.off_hist);
    tp.hist2 = reinterpret_cast<uint32_t*>(wb + lay.off_hist2);
    tp.counts = reinterpret_cast<int*>(wb + lay.off_counts);
    tp.sel = reinterpret_cast<int*>(wb + lay.off_sel);
    tp.cand = reinterpret_cast<uint64_t*>(wb + lay.off_cand);
    tp.bitmap = reinterpret_cast<uint32_t*>(wb + lay.off_bitmap);
    tp.topk_idx = topk_idx;
    tp.topk_count = topk_count;
    tp.err = reinterpret_cast<int*>(wb);
    tp.B = B;
    tp.k = k;
    tp.max_len = score_stride;
    return topk_launch(tp, true, stream);
}

int attn_decode_mla_sparse(const void* q, const void* c_pool, const int32_t* block_table,
                           const int32_t* seq_lens, const int32_t* topk_idx,
                           const int32_t* topk_count, void* out, float* lse_out, int B, int H,
                           int d_qk, int d_v, int k, int page_size, int max_pages, int num_pages,
                           float scale, void* ws, size_t ws_bytes, cudaStream_t stream) {
    if (!topk_idx || !topk_count) return KVD_ERR_INVALID_ARG;
    if (k < 1) return KVD_ERR_INVALID_ARG;
    return mla_run(q, c_pool, block_table, seq_lens, topk_idx, topk_count, k, out, lse_out, B, H,
                   d_qk, d_v, page_size, max_pages, num_pages, scale, ws, ws_bytes, stream);
}

size_t kvd_workspace_size(int op, int B, int H, int Hkv, int D, int max_len, int window,
                          int n_sink, int k) {
    if (B < 1 || H < 1 || max_len < 1) return 0;
    if (op == KVD_OP_DSA_TOPK) {
        if (k < 1 || k > kTopkMaxK) return 0;
        return topk_layout(B, max_len, k, true).total;
    }
    if (op == KVD_OP_MLA) return mla_plan(B, max_len, false).total;
    if (op == KVD_OP_MLA_SPARSE) return k >= 1 ? mla_plan(B, k, true).total : 0;
    if (op == KVD_OP_GQA || op == KVD_OP_SWA) {
        if (Hkv < 1 || H % Hkv != 0 || (D != 64 && D != 128)) return 0;
        // the plan's chunk length is smallest (most partials) for 16-token pages
        size_t need = 0;
        for (int dt = 0; dt < 2; ++dt) {
            GqaPlan plan;
            if (gqa_plan(B, H, Hkv, D, 16, max_len, op == KVD_OP_SWA ? std::max(window, 1) : 0,
                         op == KVD_OP_SWA ? std::max(n_sink, 0) : 0, dt, &plan) == KVD_OK)
                need = std::max(need, plan.total);
        }
        return need;
    }
    return 0;
}

int kvd_check_device_error(void* ws, cudaStream_t stream) {
    if (!ws) return KVD_ERR_INVALID_ARG;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return KVD_ERR_CUDA;
    int flag = 0;
    if (cudaMemcpy(&flag, ws, sizeof flag, cudaMemcpyDeviceToHost) != cudaSuccess)
        return KVD_ERR_CUDA;
    if (flag != 0) {
        if (cudaMemset(ws, 0, sizeof flag) != cudaSuccess) return KVD_ERR_CUDA;
    }
    return flag;
}

int kvd_set_option(int option, long long value) {
    switch (option) {
        case KVD_OPT_PDL:
            if (value != 0 && value != 1) return KVD_ERR_INVALID_ARG;
            g_opt_pdl.store(static_cast<int>(value));
            return KVD_OK;
        case KVD_OPT_GQA_CHUNK:
            if (value != 0 && (value < 64 || value > (1LL << 30))) return KVD_ERR_INVALID_ARG;
            g_opt_gqa_chunk.store(value);
            return KVD_OK;
        case KVD_OPT_MLA_MIN_TILES:
            if (value < 0 || value > (1LL << 30)) return KVD_ERR_INVALID_ARG;
            g_opt_mla_min_tiles.store(value);
            return KVD_OK;
        case KVD_OPT_WAIT_TIMEOUT_TEST:
            if (value != 0 && value != 1) return KVD_ERR_INVALID_ARG;
            g_opt_wait_test.store(static_cast<int>(value));
            return KVD_OK;
        case KVD_OPT_GQA_CLUSTER:
            if (value < 0 || value > 2) return KVD_ERR_INVALID_ARG;
            g_opt_gqa_cluster.store(static_cast<int>(value));
            return KVD_OK;
        default: return KVD_ERR_INVALID_ARG;
    }
}

const char* kvd_status_string(int status) {
    switch (status) {
        case KVD_OK: return "ok";
        case KVD_ERR_INVALID_ARG: return "invalid argument";
        case KVD_ERR_UNSUPPORTED: return "unsupported shape or dtype";
        case KVD_ERR_CUDA: return "CUDA error";
        case KVD_ERR_TIMEOUT: return "device wait timed out";
        case KVD_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
        case KVD_ERR_DEVICE_OOB: return "page index or sequence length out of range";
        case KVD_ERR_DEVICE_STATE: return "workspace not in its zeroed state";
        default: return "unknown status";
    }
}

}  // extern "C"
