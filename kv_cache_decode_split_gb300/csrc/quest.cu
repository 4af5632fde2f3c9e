// quest.cu -- query-aware page selection (Quest) for GQA decode over a paged cache.
//
// What is computed ("Long context, KV eviction and sparse attention", Sparse attention):
// every page of keys is summarised by its elementwise minimum and maximum; a query head's
// score for any key of the page is at most U = sum_d max(q_d kmin_d, q_d kmax_d); each query
// head keeps the n_sel full pages with the largest U (ties: the lower page) and the tokens
// past the last full page, and attends over those only.
//
// GB300: four small kernels, all bound by memory traffic or latency.
//  * quest_minmax_kernel: one warp per (page, KV head): the page's keys once, min and max in
//    the cache's own dtype (exact). Run once per page, when it fills.
//  * quest_bounds_kernel: one CTA per (sequence, KV head, 128 pages), a warp per 32 pages
//    (their page ids in one load, all their summaries copied into shared memory at once): a
//    lane holds its D/32 dims of kmin/kmax and of the group's queries, and warp sums give
//    every query head of the group its bound, written to the caller's bound array.
//  * quest_choose_kernel: one warp per (sequence, query head) picks the n_sel best bounds
//    (value, then lower index): each lane sorts its own pages once, then every round takes
//    the best of the lanes' heads by two warp max-reductions; written in ascending order.
//  * quest_attn_kernel: one CTA per (sequence, query head) over its chosen pages and tail:
//    warps take pages, eight rows in flight per warp, scores by warp sums, running max /
//    running sum softmax, then the four warps merge in shared memory.
// The selected rows are a few hundred per head, read with plain vector loads; there is no
// shared contraction across heads (each head reads its own pages) for the tensor cores.

#include <algorithm>
#include <cuda_bf16.h>

#include "kvd_device.cuh"
#include "kvd_host.h"

namespace kvd {

namespace {

constexpr float kQLog2e = 1.4426950408889634f;
constexpr int kAttnWarps = 4;
// Eight K and V rows in flight per warp, few enough registers for seven CTAs per SM: on the
// Llama-3-shaped workload all 1024 (sequence, head) CTAs are then resident at once instead of
// running in two waves (step 74 -> 62 us; with 16 rows and 128 registers, four per SM).
constexpr int kRowsInFlight = 8;
constexpr int kAttnCtasPerSm = 7;

// VEC consecutive elements of a row as float (bf16 or float32 storage).
template <int VEC, bool BF16>
__device__ __forceinline__ void load_vec(const void* base, size_t elem, float (&x)[VEC]) {
    if constexpr (BF16) {
        const __nv_bfloat16* p = static_cast<const __nv_bfloat16*>(base) + elem;
        if constexpr (VEC == 2) {
            const __nv_bfloat162 t = *reinterpret_cast<const __nv_bfloat162*>(p);
            x[0] = __low2float(t), x[1] = __high2float(t);
        } else {
#pragma unroll
            for (int i = 0; i < VEC; i += 4) {
                const uint2 raw = *reinterpret_cast<const uint2*>(p + i);
                const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&raw.x);
                const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&raw.y);
                x[i] = __low2float(a), x[i + 1] = __high2float(a);
                x[i + 2] = __low2float(b), x[i + 3] = __high2float(b);
            }
        }
    } else {
        const float* p = static_cast<const float*>(base) + elem;
        if constexpr (VEC == 2) {
            const float2 t = *reinterpret_cast<const float2*>(p);
            x[0] = t.x, x[1] = t.y;
        } else {
#pragma unroll
            for (int i = 0; i < VEC; i += 4) {
                const float4 t = *reinterpret_cast<const float4*>(p + i);
                x[i] = t.x, x[i + 1] = t.y, x[i + 2] = t.z, x[i + 3] = t.w;
            }
        }
    }
}

// A lane's VEC elements of a row kept as stored (bf16 pairs or floats) until used, so that
// many rows can be in flight in few registers.
template <int VEC, bool BF16>
struct Raw {
    static constexpr int kWords = BF16 ? VEC / 2 : VEC;
    uint32_t w[kWords];
    __device__ __forceinline__ void load(const void* base, size_t elem) {
        if constexpr (BF16) {
            const uint32_t* src =
                reinterpret_cast<const uint32_t*>(static_cast<const __nv_bfloat16*>(base) + elem);
            if constexpr (kWords == 1) {
                w[0] = *src;
            } else {
#pragma unroll
                for (int i = 0; i < kWords; i += 2) {
                    const uint2 t = *reinterpret_cast<const uint2*>(src + i);
                    w[i] = t.x, w[i + 1] = t.y;
                }
            }
        } else {
            const uint32_t* src =
                reinterpret_cast<const uint32_t*>(static_cast<const float*>(base) + elem);
#pragma unroll
            for (int i = 0; i < kWords; i += (kWords >= 4 ? 4 : 2)) {
                if constexpr (kWords >= 4) {
                    const uint4 t = *reinterpret_cast<const uint4*>(src + i);
                    w[i] = t.x, w[i + 1] = t.y, w[i + 2] = t.z, w[i + 3] = t.w;
                } else {
                    const uint2 t = *reinterpret_cast<const uint2*>(src + i);
                    w[i] = t.x, w[i + 1] = t.y;
                }
            }
        }
    }
    __device__ __forceinline__ float at(int i) const {
        if constexpr (BF16) {
            const uint32_t x = w[i / 2];
            return __uint_as_float((i & 1) ? (x & 0xffff0000u) : (x << 16));
        } else {
            return __uint_as_float(w[i]);
        }
    }
};

// ---------------------------------------------------------------------------- summaries
template <int VEC, bool BF16>
__global__ void __launch_bounds__(256) quest_minmax_kernel(const QuestParams p) {
    griddep_wait();
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) / 32, lane = threadIdx.x % 32;
    const int n_units = p.n_list * p.Hkv;
    if (warp >= n_units) return;
    const int i = warp / p.Hkv, g = warp % p.Hkv;
    const int pg = p.pages ? p.pages[i] : i;
    if (pg < 0 || pg >= p.num_pages) {
        if (lane == 0) record_error(p.err, KVD_ERR_DEVICE_OOB);
        return;
    }
    const int D = VEC * 32;
    const size_t row0 = (static_cast<size_t>(pg) * p.Hkv + g) * p.page_size;
    float lo[VEC], hi[VEC];
    load_vec<VEC, BF16>(p.k_pool, row0 * D + lane * VEC, lo);
#pragma unroll
    for (int j = 0; j < VEC; ++j) hi[j] = lo[j];
    // rows kRows at a time, all their loads issued before any is used (page sizes are powers
    // of two >= 16, so the batches divide the page)
    constexpr int kRows = 8;
    for (int t0 = 0; t0 < p.page_size; t0 += kRows) {
        float x[kRows][VEC];
#pragma unroll
        for (int r = 0; r < kRows; ++r)
            load_vec<VEC, BF16>(p.k_pool, (row0 + t0 + r) * D + lane * VEC, x[r]);
#pragma unroll
        for (int r = 0; r < kRows; ++r)
#pragma unroll
            for (int j = 0; j < VEC; ++j)
                lo[j] = fminf(lo[j], x[r][j]), hi[j] = fmaxf(hi[j], x[r][j]);
    }
    const size_t o = (static_cast<size_t>(pg) * p.Hkv + g) * D + lane * VEC;
#pragma unroll
    for (int j = 0; j < VEC; ++j) {
        // min and max of stored values are stored values: the conversion back is exact
        if constexpr (BF16) {
            static_cast<__nv_bfloat16*>(p.kmin)[o + j] = __float2bfloat16(lo[j]);
            static_cast<__nv_bfloat16*>(p.kmax)[o + j] = __float2bfloat16(hi[j]);
        } else {
            static_cast<float*>(p.kmin)[o + j] = lo[j];
            static_cast<float*>(p.kmax)[o + j] = hi[j];
        }
    }
}

// ---------------------------------------------------------------------------- bounds
// One CTA of kBoundWarps warps per (sequence, KV head, 32 * kBoundWarps pages); a warp takes
// 32 pages. The sequence's length and the warp's 32 page ids are read together, then all the
// warp's pages' summaries (the kmin and kmax rows) are copied into its shared-memory slot at
// once (cp.async, no registers held): one memory round trip for the summaries instead of one
// per batch of pages. The bounds are computed from shared memory: a lane holds D/32 dims of
// each page and of the group's queries, and 32 / KG pages' (page, head) partial sums at a
// time are reduced across the warp by a transposing butterfly (31 shuffles for all 32 sums,
// lane i ending with sum i) instead of five shuffle levels per sum.
constexpr int kBoundWarps = 4;

template <int VEC, bool BF16>
constexpr int bound_row_bytes() {  // one summary row (kmin or kmax) of a (page, KV head)
    return VEC * 32 * (BF16 ? 2 : 4);
}
template <int VEC, bool BF16>
constexpr int bound_smem_bytes() {
    return kBoundWarps * 32 * 2 * bound_row_bytes<VEC, BF16>();
}

template <int VEC, bool BF16, int KG>
__global__ void __launch_bounds__(kBoundWarps * 32) quest_bounds_kernel(const QuestParams p) {
    constexpr int D = VEC * 32;
    constexpr int kRow = bound_row_bytes<VEC, BF16>();
    constexpr int kPieces = 2 * kRow / 16;  // 16-byte pieces of a page's two rows
    extern __shared__ __align__(16) uint8_t bsm[];
    griddep_wait();
    const int b = blockIdx.x / p.Hkv, g = blockIdx.x % p.Hkv;
    const int G = p.Hq / p.Hkv;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int m0 = (blockIdx.y * kBoundWarps + warp) * 32;
    const int my = m0 + lane;
    // the length and this lane's block-table entry in flight together
    int L = p.seq_lens[b];
    const int pg_raw = my < p.max_pages ? p.block_table[static_cast<size_t>(b) * p.max_pages + my]
                                        : 0;
    if (L < 1 || L > p.max_len) {
        record_error(p.err, KVD_ERR_DEVICE_OOB);
        L = min(max(L, 1), p.max_len);
    }
    const int full = L / p.page_size;
    float* ub = p.ub_out + (static_cast<size_t>(b) * p.Hq + g * G) * p.max_pages;
    // pages that are not full have no bound
    for (int j = 0; j < G; ++j)
        if (my >= full && my < p.max_pages)
            ub[static_cast<size_t>(j) * p.max_pages + my] = __int_as_float(0x7fc00000);
    if (m0 >= full) return;
    int pg_lane = 0;
    if (my < full) {
        pg_lane = pg_raw;
        if (pg_lane < 0 || pg_lane >= p.num_pages) {
            record_error(p.err, KVD_ERR_DEVICE_OOB);
            pg_lane = 0;
        }
    }
    const int n_here = min(32, full - m0);
    // page k of the warp: its kmin row at ws + 2 k kRow, its kmax row after it
    uint8_t* ws = bsm + warp * 32 * 2 * kRow;
    for (int k = 0; k < n_here; ++k) {
        const int pg = __shfl_sync(0xffffffffu, pg_lane, k);
        const size_t row = (static_cast<size_t>(pg) * p.Hkv + g) * kRow;
        for (int pc = lane; pc < kPieces; pc += 32) {
            const bool upper = pc >= kRow / 16;
            const uint8_t* src = static_cast<const uint8_t*>(upper ? p.kmax : p.kmin) + row +
                                 (upper ? pc - kRow / 16 : pc) * 16;
            cp_async_16(smem_u32(ws + k * 2 * kRow + pc * 16), src, 16u);
        }
    }
    cp_async_commit();
    // the group's queries while the summaries are on their way
    float q[KG][VEC];
#pragma unroll
    for (int j = 0; j < KG; ++j)
        if (j < G)
            load_vec<VEC, BF16>(p.q, (static_cast<size_t>(b) * p.Hq + g * G + j) * D + lane * VEC,
                                q[j]);
    // bf16 summaries: max(q kmin, q kmax) = q+ kmax + q- kmin (q+ = max(q, 0), q- = min(q, 0),
    // kmin <= kmax), two fused multiply-adds a term. A bf16 x bf16 product is exact in fp32
    // and one of the two is zero, so every partial sum is rounded exactly as in the max form
    // (for finite summaries). float32 summaries keep the max form.
    float qp[KG][VEC], qn[KG][VEC];
#pragma unroll
    for (int j = 0; j < KG; ++j)
#pragma unroll
        for (int i = 0; i < VEC; ++i) {
            qp[j][i] = fmaxf(q[j][i], 0.f);
            qn[j][i] = fminf(q[j][i], 0.f);
        }
    cp_async_wait<0>();
    __syncwarp();
    constexpr int NP = 32 / KG;
    for (int c = 0; c < n_here; c += NP) {
        float v[32];  // v[k * KG + j]: page c + k, head j
#pragma unroll
        for (int k = 0; k < NP; ++k) {
            Raw<VEC, BF16> lo, hi;
            if (c + k < n_here) {
                lo.load(ws + (c + k) * 2 * kRow, lane * VEC);
                hi.load(ws + (c + k) * 2 * kRow + kRow, lane * VEC);
            }
#pragma unroll
            for (int j = 0; j < KG; ++j) {
                float a = 0.f;
                if (c + k < n_here)
#pragma unroll
                    for (int i = 0; i < VEC; ++i) {
                        if constexpr (BF16)
                            a = fmaf(qp[j][i], hi.at(i), fmaf(qn[j][i], lo.at(i), a));
                        else
                            a += fmaxf(q[j][i] * lo.at(i), q[j][i] * hi.at(i));
                    }
                v[k * KG + j] = a;
            }
        }
#pragma unroll
        for (int sft = 16; sft >= 1; sft >>= 1) {
            const bool upper = (lane & sft) != 0;
#pragma unroll
            for (int i = 0; i < sft; ++i) {
                const float send = upper ? v[i] : v[i + sft];
                const float keep = upper ? v[i + sft] : v[i];
                v[i] = keep + __shfl_xor_sync(0xffffffffu, send, sft);
            }
        }
        // lane i holds the sum of page c + i / KG, head i % KG
        const int k = lane / KG, j = lane % KG;
        if (c + k < n_here && j < G) ub[static_cast<size_t>(j) * p.max_pages + m0 + c + k] = v[0];
    }
}

// ---------------------------------------------------------------------------- choice
// One warp per (sequence, query head): the sort keys of its full pages' bounds into shared
// memory, then choose_pages.
constexpr int kChooseWarps = 4;

// Sort key of a bound: larger bound first, then the lower page (a NaN bound ranks below
// every number); 0 marks "no candidate".
__device__ __forceinline__ uint64_t bound_key(float v, int m);

// The sort keys of a head's full pages, key[m] for m < full, from its bound row (global):
// each lane's loads are issued kBatch at a time before any is used, so that the row costs a
// few memory round trips instead of one per page a lane holds.
__device__ __forceinline__ void load_bound_keys(const float* src, int full, uint64_t* key) {
    constexpr int kBatch = 8;
    const int lane = threadIdx.x % 32;
    for (int m0 = lane; m0 < full; m0 += 32 * kBatch) {
        float v[kBatch];
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            const int m = m0 + 32 * i;
            v[i] = m < full ? __ldcg(src + m) : 0.f;
        }
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            const int m = m0 + 32 * i;
            if (m < full) key[m] = bound_key(v[i], m);
        }
    }
}
__device__ __forceinline__ uint64_t bound_key(float v, int m) {
    uint32_t o = 0u;
    if (v == v) {
        const uint32_t b = __float_as_uint(v);
        o = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
    }
    return (static_cast<uint64_t>(o) << 32) | (0xffffffffu - static_cast<uint32_t>(m));
}

// One warp: the n_sel best of the pages 0..full-1, whose keys are in key[] (shared memory,
// consumed), written to out[0..n_sel) in ascending page order, -1 padded. Each lane sorts
// its own pages (m = lane mod 32) once; a round is then two warp max-reductions over the
// lanes' current heads and one step of the winning lane's list.
__device__ __forceinline__ void choose_pages(uint64_t* key, int full, int n_sel, int32_t* out) {
    const int lane = threadIdx.x % 32;
    const int n_take = min(full, n_sel);
    const int n_l = lane < full ? (full - lane + 31) / 32 : 0;
    for (int i = 1; i < n_l; ++i) {  // insertion sort, descending
        const uint64_t x = key[lane + 32 * i];
        int j = i - 1;
        while (j >= 0 && key[lane + 32 * j] < x) {
            key[lane + 32 * (j + 1)] = key[lane + 32 * j];
            --j;
        }
        key[lane + 32 * (j + 1)] = x;
    }
    int ptr = 0;
    uint64_t cand = n_l > 0 ? key[lane] : 0ull;
    int mine0 = -1, mine1 = -1;  // this lane's picks: rounds lane and lane + 32
    for (int r = 0; r < n_take; ++r) {
        const uint32_t hi = static_cast<uint32_t>(cand >> 32), lo = static_cast<uint32_t>(cand);
        const uint32_t mhi = __reduce_max_sync(0xffffffffu, hi);
        const uint32_t mlo = __reduce_max_sync(0xffffffffu, hi == mhi ? lo : 0u);
        const int page = static_cast<int>(0xffffffffu - mlo);
        if (lane == (r & 31)) {
            if (r < 32) mine0 = page; else mine1 = page;
        }
        if (cand != 0ull && hi == mhi && lo == mlo) {
            ++ptr;
            cand = ptr < n_l ? key[lane + 32 * ptr] : 0ull;
        }
    }
    // ascending order: each pick goes to its rank among the picks
    int rank0 = 0, rank1 = 0;
    for (int r = 0; r < n_take; ++r) {
        const int other = __shfl_sync(0xffffffffu, r < 32 ? mine0 : mine1, r & 31);
        rank0 += other < mine0;
        rank1 += other < mine1;
    }
    if (lane < n_take) out[rank0] = mine0;
    if (lane + 32 < n_take) out[rank1] = mine1;
    for (int r = n_take + lane; r < n_sel; r += 32) out[r] = -1;
}

// choose_pages for a head of at most 32 * kRegKeys full pages, with every key in registers:
// lane i holds the keys of pages i, i + 32, ... read straight from the bound row, sorts them
// by a bitonic network (no shared-memory round trip per step; the insertion sort above took
// ~4.3 us of the attention launch on the Llama-3 shapes, measured), then the rounds pick
// from the lanes' heads as above. Same pages, same order.
constexpr int kRegKeys = 16;
__device__ __forceinline__ void choose_pages_reg(const float* src, int full, int n_sel,
                                                 int32_t* out) {
    const int lane = threadIdx.x % 32;
    const int n_take = min(full, n_sel);
    uint64_t k[kRegKeys];
    {
        float v[kRegKeys];
#pragma unroll
        for (int j = 0; j < kRegKeys; ++j) {
            const int m = lane + 32 * j;
            v[j] = m < full ? __ldcg(src + m) : 0.f;
        }
#pragma unroll
        for (int j = 0; j < kRegKeys; ++j) {
            const int m = lane + 32 * j;
            k[j] = m < full ? bound_key(v[j], m) : 0ull;
        }
    }
    // bitonic sort, descending (0 keys, "no page", last)
#pragma unroll
    for (int size = 2; size <= kRegKeys; size <<= 1)
#pragma unroll
        for (int stride = size / 2; stride > 0; stride >>= 1)
#pragma unroll
            for (int i = 0; i < kRegKeys; ++i) {
                const int j = i ^ stride;
                if (j > i) {
                    const uint64_t a = k[i], c = k[j];
                    const bool swap = (i & size) == 0 ? a < c : a > c;
                    k[i] = swap ? c : a;
                    k[j] = swap ? a : c;
                }
            }
    int ptr = 0;
    uint64_t cand = k[0];
    int mine0 = -1, mine1 = -1;  // this lane's picks: rounds lane and lane + 32
    for (int r = 0; r < n_take; ++r) {
        const uint32_t hi = static_cast<uint32_t>(cand >> 32), lo = static_cast<uint32_t>(cand);
        const uint32_t mhi = __reduce_max_sync(0xffffffffu, hi);
        const uint32_t mlo = __reduce_max_sync(0xffffffffu, hi == mhi ? lo : 0u);
        const int page = static_cast<int>(0xffffffffu - mlo);
        if (lane == (r & 31)) {
            if (r < 32) mine0 = page; else mine1 = page;
        }
        if (cand != 0ull && hi == mhi && lo == mlo) {
            ++ptr;
            uint64_t nx = 0ull;
#pragma unroll
            for (int j = 1; j < kRegKeys; ++j) nx = j == ptr ? k[j] : nx;
            cand = nx;
        }
    }
    int rank0 = 0, rank1 = 0;
    for (int r = 0; r < n_take; ++r) {
        const int other = __shfl_sync(0xffffffffu, r < 32 ? mine0 : mine1, r & 31);
        rank0 += other < mine0;
        rank1 += other < mine1;
    }
    if (lane < n_take) out[rank0] = mine0;
    if (lane + 32 < n_take) out[rank1] = mine1;
    for (int r = n_take + lane; r < n_sel; r += 32) out[r] = -1;
}

__global__ void __launch_bounds__(kChooseWarps * 32) quest_choose_kernel(const QuestParams p) {
    extern __shared__ uint64_t ubs[];  // [kChooseWarps][max_pages] sort keys
    griddep_wait();
    const int warp = threadIdx.x / 32;
    const int bh = blockIdx.x * kChooseWarps + warp;
    if (bh >= p.B * p.Hq) return;
    const int b = bh / p.Hq;
    const int L = load_len(p.seq_lens, b, p.max_len, p.err);
    const int full = L / p.page_size;
    uint64_t* u = ubs + static_cast<size_t>(warp) * p.max_pages;
    load_bound_keys(p.ub_out + static_cast<size_t>(bh) * p.max_pages, full, u);
    __syncwarp();
    choose_pages(u, full, p.n_sel, p.sel + static_cast<size_t>(bh) * p.n_sel);
}

// ---------------------------------------------------------------------------- attention
// CHOOSE: warp 0 first picks the head's pages from its bounds (p.ub_out), writes them to
// p.sel for the caller, and the CTA attends over them (no separate choice launch).
template <int VEC, bool BF16, bool CHOOSE>
__global__ void __launch_bounds__(kAttnWarps * 32, kAttnCtasPerSm)
    quest_attn_kernel(const QuestParams p) {
    constexpr int D = VEC * 32;
    __shared__ float m_s[kAttnWarps], l_s[kAttnWarps];
    __shared__ float o_s[kAttnWarps][D];
    __shared__ int32_t sel_s[64];
    extern __shared__ uint64_t ubrow[];  // CHOOSE: the head's bound keys [max_pages]
    griddep_wait();
    const int b = blockIdx.x / p.Hq, h = blockIdx.x % p.Hq;
    const int g = h / (p.Hq / p.Hkv);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int L = load_len(p.seq_lens, b, p.max_len, p.err);
    const int full = L / p.page_size;
    const int n_take = min(full, p.n_sel);
    const int tail = L - full * p.page_size;
    const int32_t* sel = p.sel + (static_cast<size_t>(b) * p.Hq + h) * p.n_sel;
    if constexpr (CHOOSE) {
        if (warp == 0) {
            const float* ubh = p.ub_out + (static_cast<size_t>(b) * p.Hq + h) * p.max_pages;
            if (full <= 32 * kRegKeys) {
                choose_pages_reg(ubh, full, p.n_sel, sel_s);
            } else {
                load_bound_keys(ubh, full, ubrow);
                __syncwarp();
                choose_pages(ubrow, full, p.n_sel, sel_s);
            }
            __syncwarp();
            int32_t* dst = p.sel + (static_cast<size_t>(b) * p.Hq + h) * p.n_sel;
            for (int r = lane; r < p.n_sel; r += 32) dst[r] = sel_s[r];
        }
        __syncthreads();
        sel = sel_s;
    }

    float q[VEC];
    load_vec<VEC, BF16>(p.q, (static_cast<size_t>(b) * p.Hq + h) * D + lane * VEC, q);
#pragma unroll
    for (int i = 0; i < VEC; ++i) q[i] *= p.scale * kQLog2e;
    float m = -INFINITY, l = 0.f, o[VEC];
#pragma unroll
    for (int i = 0; i < VEC; ++i) o[i] = 0.f;

    // units of work: the chosen pages, then the tail as one more (partial) page; their
    // physical pages are resolved up front, all lanes at once (at most 65 units)
    __shared__ int unit_pg[65];
    const int n_units = n_take + (tail > 0 ? 1 : 0);
    for (int u = threadIdx.x; u < n_units; u += blockDim.x) {
        int lp = u < n_take ? sel[u] : full;
        if (lp < 0 || lp >= full + (u < n_take ? 0 : 1)) {
            record_error(p.err, KVD_ERR_DEVICE_OOB);
            unit_pg[u] = -1;
            continue;
        }
        unit_pg[u] = load_page(p.block_table, p.max_pages, p.num_pages, b, lp, p.err);
    }
    __syncthreads();
    for (int u = warp; u < n_units; u += kAttnWarps) {
        const int pg = unit_pg[u];
        if (pg < 0) continue;
        const int rows = u < n_take ? p.page_size : tail;
        const size_t row0 = (static_cast<size_t>(pg) * p.Hkv + g) * p.page_size;
        for (int t0 = 0; t0 < rows; t0 += kRowsInFlight) {
            // the K and V rows of the batch all in flight together
            Raw<VEC, BF16> k[kRowsInFlight], v[kRowsInFlight];
            float s[kRowsInFlight];
#pragma unroll
            for (int r = 0; r < kRowsInFlight; ++r)
                if (t0 + r < rows) {
                    k[r].load(p.k_pool, (row0 + t0 + r) * D + lane * VEC);
                    v[r].load(p.v_pool, (row0 + t0 + r) * D + lane * VEC);
                }
#pragma unroll
            for (int r = 0; r < kRowsInFlight; ++r) {
                float acc = 0.f;
                if (t0 + r < rows)
#pragma unroll
                    for (int i = 0; i < VEC; ++i) acc = fmaf(q[i], k[r].at(i), acc);
                s[r] = acc;
            }
#pragma unroll
            for (int off = 16; off; off >>= 1)
#pragma unroll
                for (int r = 0; r < kRowsInFlight; ++r)
                    s[r] += __shfl_xor_sync(0xffffffffu, s[r], off);
            float mx = m;
#pragma unroll
            for (int r = 0; r < kRowsInFlight; ++r)
                if (t0 + r < rows) mx = fmaxf(mx, s[r]);
            const float corr = exp2f(m - mx);
            l *= corr;
#pragma unroll
            for (int i = 0; i < VEC; ++i) o[i] *= corr;
            m = mx;
#pragma unroll
            for (int r = 0; r < kRowsInFlight; ++r) {
                if (t0 + r >= rows) break;
                const float e = exp2f(s[r] - m);
                l += e;
#pragma unroll
                for (int i = 0; i < VEC; ++i) o[i] = fmaf(e, v[r].at(i), o[i]);
            }
        }
    }
    // merge the warps
    if (lane == 0) m_s[warp] = m, l_s[warp] = l;
#pragma unroll
    for (int i = 0; i < VEC; ++i) o_s[warp][lane * VEC + i] = o[i];
    __syncthreads();
    if (warp == 0) {
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kAttnWarps; ++w) M = fmaxf(M, m_s[w]);
        float Lsum = 0.f, acc[VEC];
#pragma unroll
        for (int i = 0; i < VEC; ++i) acc[i] = 0.f;
#pragma unroll
        for (int w = 0; w < kAttnWarps; ++w) {
            const float f = m_s[w] == -INFINITY ? 0.f : exp2f(m_s[w] - M);
            Lsum += f * l_s[w];
#pragma unroll
            for (int i = 0; i < VEC; ++i) acc[i] += f * o_s[w][lane * VEC + i];
        }
        const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
        const size_t oo = (static_cast<size_t>(b) * p.Hq + h) * D + lane * VEC;
#pragma unroll
        for (int i = 0; i < VEC; ++i) {
            if constexpr (BF16)
                static_cast<__nv_bfloat16*>(p.out)[oo + i] = __float2bfloat16(acc[i] * inv);
            else
                static_cast<float*>(p.out)[oo + i] = acc[i] * inv;
        }
        if (p.lse_out && lane == 0)
            p.lse_out[static_cast<size_t>(b) * p.Hq + h] = (M + log2f(Lsum)) / kQLog2e;
    }
}

}  // namespace

#define KVD_QUEST_DISPATCH(KERNEL, GRID, BLOCK, SMEM)                                          \
    do {                                                                                       \
        cudaError_t e_ = cudaErrorInvalidValue;                                                \
        if (p.dtype == KVD_BF16 && p.D == 64)                                                  \
            e_ = launch_kernel(KERNEL<2, true>, GRID, BLOCK, SMEM, stream, p);                 \
        else if (p.dtype == KVD_BF16 && p.D == 128)                                            \
            e_ = launch_kernel(KERNEL<4, true>, GRID, BLOCK, SMEM, stream, p);                 \
        else if (p.dtype == KVD_F32 && p.D == 64)                                              \
            e_ = launch_kernel(KERNEL<2, false>, GRID, BLOCK, SMEM, stream, p);                \
        else if (p.dtype == KVD_F32 && p.D == 128)                                             \
            e_ = launch_kernel(KERNEL<4, false>, GRID, BLOCK, SMEM, stream, p);                \
        else                                                                                   \
            return KVD_ERR_UNSUPPORTED;                                                        \
        if (e_ != cudaSuccess) return KVD_ERR_CUDA;                                            \
    } while (0)

int quest_minmax_launch(const QuestParams& p, cudaStream_t stream) {
    const long long warps = static_cast<long long>(p.n_list) * p.Hkv;
    const dim3 grid(static_cast<unsigned>((warps + 7) / 8)), block(256);
    KVD_QUEST_DISPATCH(quest_minmax_kernel, grid, block, 0);
    return cudaGetLastError() == cudaSuccess ? KVD_OK : KVD_ERR_CUDA;
}

size_t quest_select_smem(int Hq, int Hkv, int max_pages) {
    (void)Hq;
    (void)Hkv;
    return sizeof(uint64_t) * static_cast<size_t>(kChooseWarps) * max_pages;
}

template <int VEC, bool BF16, int KG>
static cudaError_t bounds_launch_kg(const QuestParams& p, dim3 grid, cudaStream_t stream) {
    constexpr int kSmem = bound_smem_bytes<VEC, BF16>();
    static bool configured = false;
    if (!configured) {
        const cudaError_t e = cudaFuncSetAttribute(quest_bounds_kernel<VEC, BF16, KG>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   kSmem);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    return launch_kernel(quest_bounds_kernel<VEC, BF16, KG>, grid, dim3(kBoundWarps * 32), kSmem,
                         stream, p);
}

template <int VEC, bool BF16>
static cudaError_t bounds_launch(const QuestParams& p, dim3 grid, cudaStream_t stream) {
    const int G = p.Hq / p.Hkv;
    if (G <= 1) return bounds_launch_kg<VEC, BF16, 1>(p, grid, stream);
    if (G <= 2) return bounds_launch_kg<VEC, BF16, 2>(p, grid, stream);
    if (G <= 4) return bounds_launch_kg<VEC, BF16, 4>(p, grid, stream);
    if (G <= 8) return bounds_launch_kg<VEC, BF16, 8>(p, grid, stream);
    return bounds_launch_kg<VEC, BF16, 16>(p, grid, stream);
}

int quest_bounds_launch(const QuestParams& p, cudaStream_t stream) {
    const int per_cta = 32 * kBoundWarps;
    const dim3 grid(static_cast<unsigned>(p.B * p.Hkv),
                    static_cast<unsigned>((p.max_pages + per_cta - 1) / per_cta));
    cudaError_t e = cudaErrorInvalidValue;
    if (p.dtype == KVD_BF16 && p.D == 64) e = bounds_launch<2, true>(p, grid, stream);
    else if (p.dtype == KVD_BF16 && p.D == 128) e = bounds_launch<4, true>(p, grid, stream);
    else if (p.dtype == KVD_F32 && p.D == 64) e = bounds_launch<2, false>(p, grid, stream);
    else if (p.dtype == KVD_F32 && p.D == 128) e = bounds_launch<4, false>(p, grid, stream);
    else return KVD_ERR_UNSUPPORTED;
    if (e != cudaSuccess) return KVD_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? KVD_OK : KVD_ERR_CUDA;
}

int quest_select_launch(const QuestParams& p, cudaStream_t stream) {
    const int st = quest_bounds_launch(p, stream);
    if (st != KVD_OK) return st;
    const size_t smem = quest_select_smem(p.Hq, p.Hkv, p.max_pages);
    static size_t configured = 0;
    if (smem > 48 * 1024 && configured < smem) {
        if (cudaFuncSetAttribute(quest_choose_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem)) != cudaSuccess)
            return KVD_ERR_CUDA;
        configured = smem;
    }
    const unsigned blocks = static_cast<unsigned>((p.B * p.Hq + kChooseWarps - 1) / kChooseWarps);
    if (launch_kernel(quest_choose_kernel, dim3(blocks), dim3(kChooseWarps * 32), smem, stream,
                      p) != cudaSuccess)
        return KVD_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? KVD_OK : KVD_ERR_CUDA;
}

template <bool CHOOSE>
static int attn_launch(const QuestParams& p, cudaStream_t stream) {
    const dim3 grid(static_cast<unsigned>(p.B * p.Hq)), block(kAttnWarps * 32);
    const size_t smem = CHOOSE ? sizeof(uint64_t) * static_cast<size_t>(p.max_pages) : 0;
    if constexpr (CHOOSE) {
        if (smem > 48 * 1024) {
            static size_t configured = 0;
            if (configured < smem) {
                const int bytes = static_cast<int>(smem);
                constexpr auto attr = cudaFuncAttributeMaxDynamicSharedMemorySize;
                cudaError_t e = cudaSuccess;
                if (p.dtype == KVD_BF16 && p.D == 64)
                    e = cudaFuncSetAttribute(quest_attn_kernel<2, true, CHOOSE>, attr, bytes);
                if (p.dtype == KVD_BF16 && p.D == 128)
                    e = cudaFuncSetAttribute(quest_attn_kernel<4, true, CHOOSE>, attr, bytes);
                if (p.dtype == KVD_F32 && p.D == 64)
                    e = cudaFuncSetAttribute(quest_attn_kernel<2, false, CHOOSE>, attr, bytes);
                if (p.dtype == KVD_F32 && p.D == 128)
                    e = cudaFuncSetAttribute(quest_attn_kernel<4, false, CHOOSE>, attr, bytes);
                if (e != cudaSuccess) return KVD_ERR_CUDA;
                configured = smem;
            }
        }
    }
    cudaError_t e;
    if (p.dtype == KVD_BF16 && p.D == 64)
        e = launch_kernel(quest_attn_kernel<2, true, CHOOSE>, grid, block, smem, stream, p);
    else if (p.dtype == KVD_BF16 && p.D == 128)
        e = launch_kernel(quest_attn_kernel<4, true, CHOOSE>, grid, block, smem, stream, p);
    else if (p.dtype == KVD_F32 && p.D == 64)
        e = launch_kernel(quest_attn_kernel<2, false, CHOOSE>, grid, block, smem, stream, p);
    else if (p.dtype == KVD_F32 && p.D == 128)
        e = launch_kernel(quest_attn_kernel<4, false, CHOOSE>, grid, block, smem, stream, p);
    else
        return KVD_ERR_UNSUPPORTED;
    if (e != cudaSuccess) return KVD_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? KVD_OK : KVD_ERR_CUDA;
}

int quest_attn_launch(const QuestParams& p, bool choose, cudaStream_t stream) {
    return choose ? attn_launch<true>(p, stream) : attn_launch<false>(p, stream);
}

}  // namespace kvd
