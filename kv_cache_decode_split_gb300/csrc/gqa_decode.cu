// gqa_decode.cu -- split-KV decode attention for GQA / MHA / MQA over a paged cache,
// with an optional sliding window, sink tokens and a learned sink logit.
//
// What is computed ("Overview of Attention Mechanism", GQA / Code; "All the
// attentions", sections 1, 4 and 8; "Attention Optimizations", Attention sinks):
//   o_h = sum_{t in V} e^{s_t} v_{g(h),t} / (sum_{t in V} e^{s_t} + [sink] e^{sigma_h}),
//   s_t = scale * q_h . k_{g(h),t},  g(h) = h / (Hq / Hkv),
// with V the visible set of the query at position L-1 (all tokens, or the window of W
// tokens ending at the query plus the first n_sink tokens). On a rolling cache ("All the
// attentions", section 4: the window's cache is a buffer of W entries, the newest replacing
// the oldest; sinks in their own first slots) every filled slot is visible: the first
// min(L, n_sink + W) slots, in whatever order the ring holds them.
//
// How (GB300), bf16: one CTA per (sequence, group of HPT KV heads, block of <= 16 query
// heads per KV head, chunk of the visible range), two CTAs per SM. A producer warp streams
// 64-token tiles of K and V through a 3-stage mbarrier ring with one 3-D TMA instruction
// per page piece: all 64-dim column blocks at once and, for D = 64, two KV heads at once,
// so that every instruction moves 16 KB (a single issuing thread needs transfers that
// large to keep its share of HBM busy). Four consumer warps each take 16 tokens of every
// tile and run the running-max / running-sum softmax ("All the attentions", section 1) on
// warp-level tensor cores:
//   S^T[16 tok x 8 heads] = K[16 x D] q^T        (mma.sync m16n8k16, tokens as M)
//   O^T[D x 8 heads]     += V^T[D x 16 tok] P^T  (P^T via movmatrix, V^T via ldmatrix.trans)
// The warps are merged in shared memory into one (o, log2-sum-exp) partial per chunk and
// KV head. When groups are few, the chunks of a group form a thread-block cluster and push
// their partials into the combining CTAs' shared memory; otherwise the CTA that finishes
// last (a completion counter per group) combines them through the workspace. Either way
// the partials are weighted by log-sum-exp, the learned sink enters once, and one launch
// serves the call (on a rolling cache it can also write the newest token's rows first).
// Start and end of a call overlap its neighbours on the stream: before the dependency wait
// the producer has the first tiles prefetched into L2 (and issues their copies right after
// it when the values it read are unchanged), and once a CTA's copies are all issued it lets
// the next grid be scheduled.
//
// The float32 variant (tiny shapes, exact fp32 arithmetic) walks the block table with
// plain loads on CUDA cores and shares the merge and combine code.

#include "kvd_device.cuh"
#include "kvd_host.h"

namespace kvd {

namespace {

constexpr int kTile = 64;        // tokens per K/V tile
constexpr int kConsumers = 4;    // consumer warps, 16 tokens of each tile each
constexpr int kMaxHP = 16;       // query heads per KV head handled by one CTA
constexpr int kRowCache = 512;   // block-table entries the producer loads at once (one row)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Tokens the query sees through the cache: L (paged cache; checked against its capacity) or,
// on a rolling cache of p.ring slots, the filled slots min(L, ring) (L itself unbounded).
__device__ __forceinline__ int visible_len(const GqaParams& p, int b) {
    if (p.ring <= 0) return load_len(p.seq_lens, b, p.max_len, p.err);
    int L = p.seq_lens[b];
    if (L < 1) {
        record_error(p.err, KVD_ERR_DEVICE_OOB);
        L = 1;
    }
    return min(L, p.ring);
}

__device__ __forceinline__ float neg_inf() { return -__int_as_float(0x7f800000); }

// Per-warp partials of one KV head, merged into the chunk partial.
template <int D, int HP>
struct MergeSmem {
    float m[kConsumers][HP];
    float l[kConsumers][HP];
    float o[kConsumers][HP][D];
};

// Scratch of the final combine: one row per (KV head of the group, query head).
template <int ROWS>
struct CombineSmem {
    float wgt[ROWS][kGqaMaxChunks];
    float inv_denom[ROWS];
    float lse_nat[ROWS];
};

__device__ __forceinline__ size_t unit_of(const GqaParams& p, int b, int kvh, int hg) {
    return (static_cast<size_t>(b) * p.Hkv + kvh) * p.NHG + hg;
}

// Merge the four warps' partials of NKV KV heads into chunk c's (o, log2-sum-exp)
// partials: one thread per head turns the warps' (m, l) into weights 2^{m_w - M} / L
// (stored over m), then every thread sums float4 slices of the weighted warp outputs.
template <int D, int HP>
__device__ void merge_chunks(const GqaParams& p, MergeSmem<D, HP>* ms, int b, int kv0, int nkv,
                             int hg, int c, int G_cta) {
    const int rows = nkv * G_cta;
    for (int r = threadIdx.x; r < rows; r += blockDim.x) {
        MergeSmem<D, HP>& m = ms[r / G_cta];
        const int h = r % G_cta;
        float M = neg_inf();
#pragma unroll
        for (int w = 0; w < kConsumers; ++w) M = fmaxf(M, m.m[w][h]);
        float f[kConsumers], L = 0.f;
#pragma unroll
        for (int w = 0; w < kConsumers; ++w) {
            f[w] = fast_exp2(m.m[w][h] - M);
            L += m.l[w][h] * f[w];
        }
        const float inv = 1.f / L;
#pragma unroll
        for (int w = 0; w < kConsumers; ++w) m.m[w][h] = f[w] * inv;
        const size_t unit = unit_of(p, b, kv0 + r / G_cta, hg);
        __stcg(p.part_lse + (unit * p.max_chunks + c) * kMaxHP + h, M + log2f(L));
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < rows * (D / 4); idx += blockDim.x) {
        const int r = idx / (D / 4), d = (idx % (D / 4)) * 4;
        const MergeSmem<D, HP>& m = ms[r / G_cta];
        const int h = r % G_cta;
        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w = 0; w < kConsumers; ++w) {
            const float f = m.m[w][h];
            const float4 v = *reinterpret_cast<const float4*>(&m.o[w][h][d]);
            o.x += f * v.x;
            o.y += f * v.y;
            o.z += f * v.z;
            o.w += f * v.w;
        }
        const size_t unit = unit_of(p, b, kv0 + r / G_cta, hg);
        __stcg(reinterpret_cast<float4*>(p.part_o + ((unit * p.max_chunks + c) * kMaxHP + h) * D + d),
               o);
    }
}

// Combine every chunk partial of NKV KV heads of one (sequence, head block) and write the
// output rows, the learned sink added once to each denominator:
//   o = sum_c 2^{lse_c - M} o_c / (sum_c 2^{lse_c - M} + 2^{sigma - M}).
// All chunk log-sum-exps are fetched in one parallel pass, then one warp per row turns them
// into weights, then every thread sums float4 slices of the chunk outputs.
template <int D, int ROWS>
__device__ void combine_units(const GqaParams& p, CombineSmem<ROWS>& cs, int b, int kv0, int nkv,
                              int hg, int n_chunks, int G_cta) {
    constexpr int kBuf = 16;  // chunks of one output slice held in registers at once
    const int rows = nkv * G_cta;
    const int n_out = rows * (D / 4);
    const bool in_regs = n_chunks <= kBuf;
    auto slice = [&](int idx) -> const float* {
        const int r = idx / (D / 4), d = (idx % (D / 4)) * 4;
        const size_t unit = unit_of(p, b, kv0 + r / G_cta, hg);
        return p.part_o + (unit * p.max_chunks * kMaxHP + r % G_cta) * D + d;
    };
    auto fetch = [&](int idx, float4 (&v)[kBuf]) {
        const float* uo = slice(idx);
#pragma unroll
        for (int cc = 0; cc < kBuf; ++cc)
            if (cc < n_chunks)
                v[cc] = __ldcg(reinterpret_cast<const float4*>(uo + static_cast<size_t>(cc) * kMaxHP * D));
    };
    // the chunk log-sum-exps, with the first output slice's partials in flight alongside
    for (int idx = threadIdx.x; idx < rows * n_chunks; idx += blockDim.x) {
        const int r = idx / n_chunks, cc = idx % n_chunks;
        const size_t unit = unit_of(p, b, kv0 + r / G_cta, hg);
        cs.wgt[r][cc] = __ldcg(p.part_lse + (unit * p.max_chunks + cc) * kMaxHP + r % G_cta);
    }
    float4 v[kBuf];
    if (in_regs && static_cast<int>(threadIdx.x) < n_out) fetch(threadIdx.x, v);
    __syncthreads();
    // weights: one thread per row when there are few chunks (short serial loops over
    // shared memory, all rows at once), one warp per row otherwise
    if (n_chunks <= 32) {
        for (int r = threadIdx.x; r < rows; r += blockDim.x) {
            const int hq = (kv0 + r / G_cta) * p.G + hg * kMaxHP + r % G_cta;
            float M = p.sink_logit ? p.sink_logit[hq] * kLog2e : neg_inf();
            const float sig = M;
            for (int cc = 0; cc < n_chunks; ++cc) M = fmaxf(M, cs.wgt[r][cc]);
            float den = p.sink_logit ? fast_exp2(sig - M) : 0.f;
            for (int cc = 0; cc < n_chunks; ++cc) {
                const float wv = fast_exp2(cs.wgt[r][cc] - M);
                cs.wgt[r][cc] = wv;
                den += wv;
            }
            cs.inv_denom[r] = 1.f / den;
            cs.lse_nat[r] = (M + log2f(den)) * kLn2;
        }
    }
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32, nwarps = blockDim.x / 32;
    for (int r = warp; r < rows && n_chunks > 32; r += nwarps) {
        const int hq = (kv0 + r / G_cta) * p.G + hg * kMaxHP + r % G_cta;
        float M = neg_inf();
        for (int cc = lane; cc < n_chunks; cc += 32) M = fmaxf(M, cs.wgt[r][cc]);
        for (int off = 16; off; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
        const float sig = p.sink_logit ? p.sink_logit[hq] * kLog2e : neg_inf();
        M = fmaxf(M, sig);
        float den = 0.f;
        for (int cc = lane; cc < n_chunks; cc += 32) {
            const float wv = fast_exp2(cs.wgt[r][cc] - M);
            cs.wgt[r][cc] = wv;
            den += wv;
        }
        for (int off = 16; off; off >>= 1) den += __shfl_xor_sync(0xffffffffu, den, off);
        if (p.sink_logit) den += fast_exp2(sig - M);
        if (lane == 0) {
            cs.inv_denom[r] = 1.f / den;
            cs.lse_nat[r] = (M + log2f(den)) * kLn2;
        }
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < n_out; idx += blockDim.x) {
        const int r = idx / (D / 4), d = (idx % (D / 4)) * 4;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (in_regs) {
            if (idx != static_cast<int>(threadIdx.x)) fetch(idx, v);
#pragma unroll
            for (int cc = 0; cc < kBuf; ++cc) {
                if (cc < n_chunks) {
                    const float w = cs.wgt[r][cc];
                    acc.x += w * v[cc].x;
                    acc.y += w * v[cc].y;
                    acc.z += w * v[cc].z;
                    acc.w += w * v[cc].w;
                }
            }
        } else {
            const float* uo = slice(idx);
#pragma unroll 8
            for (int cc = 0; cc < n_chunks; ++cc) {
                const float w = cs.wgt[r][cc];
                const float4 x = __ldcg(reinterpret_cast<const float4*>(uo + static_cast<size_t>(cc) * kMaxHP * D));
                acc.x += w * x.x;
                acc.y += w * x.y;
                acc.z += w * x.z;
                acc.w += w * x.w;
            }
        }
        const float inv = cs.inv_denom[r];
        const int hq = (kv0 + r / G_cta) * p.G + hg * kMaxHP + r % G_cta;
        const size_t o = (static_cast<size_t>(b) * p.Hq + hq) * D + d;
        if (p.dtype == KVD_BF16) {
            __nv_bfloat162 lo2 = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
            __nv_bfloat162 hi2 = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
            *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(p.out) + o) =
                make_uint2(*reinterpret_cast<uint32_t*>(&lo2), *reinterpret_cast<uint32_t*>(&hi2));
        } else {
            *reinterpret_cast<float4*>(reinterpret_cast<float*>(p.out) + o) =
                make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
        }
        if (d == 0 && p.lse_out) p.lse_out[static_cast<size_t>(b) * p.Hq + hq] = cs.lse_nat[r];
    }
}

// After this CTA's chunk partials are written: count the chunk in, and if it was the last
// one of group `grp`, combine the NKV KV heads kv0 .. kv0+NKV-1 of that group.
template <int D, int ROWS>
__device__ void finish_group(const GqaParams& p, CombineSmem<ROWS>& cs, int b, int kv0, int nkv,
                             int hg, int grp, int n_chunks, int G_cta) {
    __shared__ int s_last;
    __threadfence();  // partials visible device-wide before the count
    __syncthreads();
    if (threadIdx.x == 0) {
        const int prev = atomicAdd(p.counters + grp, 1);
        s_last = prev == n_chunks - 1;
        if (s_last) p.counters[grp] = 0;  // ready for the next call on this workspace
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    combine_units<D, ROWS>(p, cs, b, kv0, nkv, hg, n_chunks, G_cta);
}

// ---------------------------------------------------------------------------------------
// Cluster combine: when the CTAs of one group (its chunks) form a thread-block cluster, the
// chunk partials never leave the cluster. Row r of the group is combined by CTA r mod CS:
// every CTA merges its four warps and stores each row's partial straight into the shared
// memory of that row's CTA (distributed shared memory); after one cluster barrier each
// CTA combines its rows from its own shared memory and writes them. No workspace counters,
// no global round trip, no remote load.
// ---------------------------------------------------------------------------------------
template <int D, int ROWS>
struct ClusterRx {
    // slot c * stride + i: chunk c's partial of this CTA's i-th row (stride = ceil(rows / CS))
    float lse[ROWS + 8];     // log2-sum-exp; -inf when the chunk saw nothing
    float o[ROWS + 8][D];    // the chunk's output, normalised by its own sum
};

// Both steps run once per CTA at the end of the call, while the SM's other CTA may still be
// streaming: every dependent step there costs ~0.4-0.6 us (measured), so each thread takes
// whole output pieces and derives the row's weights itself (a few redundant exponentials)
// instead of weights first, a barrier, then the outputs.
template <int D, int HP, int ROWS>
__device__ void merge_push(const MergeSmem<D, HP>* ms, ClusterRx<D, ROWS>& rx, int nkv,
                           int G_cta, int CS, int rank) {
    const int rows = nkv * G_cta;
    const int stride = (rows + CS - 1) / CS;
    const uint32_t lse0 = smem_u32(&rx.lse[0]), o0 = smem_u32(&rx.o[0][0]);
    const int n_items = rows * (D / 4);
    for (int idx = threadIdx.x; idx < n_items; idx += blockDim.x) {
        const int r = idx / (D / 4), d = (idx % (D / 4)) * 4;
        const MergeSmem<D, HP>& m = ms[r / G_cta];
        const int h = r % G_cta;
        float mw[kConsumers], lw[kConsumers];
#pragma unroll
        for (int w = 0; w < kConsumers; ++w) mw[w] = m.m[w][h], lw[w] = m.l[w][h];
        float M = neg_inf();
#pragma unroll
        for (int w = 0; w < kConsumers; ++w) M = fmaxf(M, mw[w]);
        const int slot = rank * stride + r / CS;
        const uint32_t peer = static_cast<uint32_t>(r % CS);
        if (M == neg_inf()) {  // an empty chunk (its outputs are zeros)
            if (d == 0) st_cluster_f32(map_peer(lse0 + slot * 4, peer), neg_inf());
            st_cluster_v4(map_peer(o0 + static_cast<uint32_t>((slot * D + d) * 4), peer), 0.f,
                          0.f, 0.f, 0.f);
            continue;
        }
        float f[kConsumers], L = 0.f;
#pragma unroll
        for (int w = 0; w < kConsumers; ++w) {
            f[w] = fast_exp2(mw[w] - M);
            L += lw[w] * f[w];
        }
        const float inv = 1.f / L;
        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w = 0; w < kConsumers; ++w) {
            const float g = f[w] * inv;
            const float4 v = *reinterpret_cast<const float4*>(&m.o[w][h][d]);
            o.x += g * v.x;
            o.y += g * v.y;
            o.z += g * v.z;
            o.w += g * v.w;
        }
        if (d == 0) st_cluster_f32(map_peer(lse0 + slot * 4, peer), M + log2f(L));
        st_cluster_v4(map_peer(o0 + static_cast<uint32_t>((slot * D + d) * 4), peer), o.x, o.y,
                      o.z, o.w);
    }
}

template <int D, int ROWS>
__device__ void combine_rx(const GqaParams& p, const ClusterRx<D, ROWS>& rx, int b, int kv0,
                           int nkv, int hg, int G_cta, int CS, int rank) {
    constexpr int kMaxCS = 8;  // portable cluster size
    const int rows = nkv * G_cta;
    const int stride = (rows + CS - 1) / CS;
    const int mine = rank < rows ? (rows - rank + CS - 1) / CS : 0;  // rows rank + CS i
    for (int idx = threadIdx.x; idx < mine * (D / 4); idx += blockDim.x) {
        const int i = idx / (D / 4), d = (idx % (D / 4)) * 4;
        const int r = rank + i * CS;
        const int hq = (kv0 + r / G_cta) * p.G + hg * kMaxHP + r % G_cta;
        float lc[kMaxCS];
        float M = p.sink_logit ? p.sink_logit[hq] * kLog2e : neg_inf();
        const float sig = M;
#pragma unroll
        for (int c = 0; c < kMaxCS; ++c) {
            lc[c] = c < CS ? rx.lse[c * stride + i] : neg_inf();
            M = fmaxf(M, lc[c]);
        }
        float den = p.sink_logit ? fast_exp2(sig - M) : 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int c = 0; c < kMaxCS; ++c) {
            if (c >= CS) break;
            const float w = fast_exp2(lc[c] - M);
            den += w;
            const float4 v = *reinterpret_cast<const float4*>(&rx.o[c * stride + i][d]);
            acc.x += w * v.x;
            acc.y += w * v.y;
            acc.z += w * v.z;
            acc.w += w * v.w;
        }
        const float inv = 1.f / den;
        const size_t o = (static_cast<size_t>(b) * p.Hq + hq) * D + d;
        __nv_bfloat162 lo2 = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
        __nv_bfloat162 hi2 = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
        *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(p.out) + o) =
            make_uint2(*reinterpret_cast<uint32_t*>(&lo2), *reinterpret_cast<uint32_t*>(&hi2));
        if (d == 0 && p.lse_out)
            p.lse_out[static_cast<size_t>(b) * p.Hq + hq] = (M + log2f(den)) * kLn2;
    }
}

// ---------------------------------------------------------------------------------------
// bf16 kernel: TMA ring + mma.sync, HPT KV heads per tile
// ---------------------------------------------------------------------------------------
template <int D, int NT, int HPT, bool kClu>
struct GqaBf16Cfg {
    static constexpr int kStages = 3;
    static constexpr int kTileBytes = HPT * kTile * D * 2;  // one K (or V) tile
    static constexpr int kRingBytes = 2 * kStages * kTileBytes;
    static constexpr int kMergeBytes = HPT * static_cast<int>(sizeof(MergeSmem<D, NT * 8>));
    static constexpr int kCombBytes = static_cast<int>(sizeof(CombineSmem<HPT * NT * 8>));
    static constexpr int kAfterRing = kMergeBytes + kCombBytes;
    static constexpr int kOverlay = kRingBytes > kAfterRing ? kRingBytes : kAfterRing;
    // cluster combine: the partials other CTAs push, outside the ring (they may arrive while
    // this CTA still streams)
    static constexpr int kRxBytes = kClu ? static_cast<int>(sizeof(ClusterRx<D, HPT * NT * 8>)) : 0;
    static constexpr int kSmem =
        1024 + kOverlay + kRxBytes + (2 * kStages + 1) * 8 + kRowCache * 4;
    static constexpr int kThreads = (kConsumers + 1) * 32;
};

// kClu: the grid's x blocks (the chunks of one group) form a cluster and combine through
// distributed shared memory; otherwise the last CTA of each group combines through the
// workspace.
template <int D, int NT, int HPT, bool kClu>
__global__ void __launch_bounds__(GqaBf16Cfg<D, NT, HPT, kClu>::kThreads, 2)
    gqa_decode_bf16_kernel(const __grid_constant__ CUtensorMap tmK,
                           const __grid_constant__ CUtensorMap tmV, const GqaParams p) {
    using Cfg = GqaBf16Cfg<D, NT, HPT, kClu>;
    using MS = MergeSmem<D, NT * 8>;
    using CS = CombineSmem<HPT * NT * 8>;
    using RX = ClusterRx<D, HPT * NT * 8>;
    constexpr int S = Cfg::kStages;
    constexpr int KT = D / 16;  // k-steps of QK, m-tiles of PV
    constexpr int NB = D / 64;  // 64-dim column blocks
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* sK = smem;
    uint8_t* sV = smem + S * Cfg::kTileBytes;
    RX& rx = *reinterpret_cast<RX*>(smem + Cfg::kOverlay);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + Cfg::kOverlay + Cfg::kRxBytes);
    uint64_t* empty = full + S;
    uint64_t* stall = empty + S;  // completed by nothing (give-up test only)
    int* bt_row = reinterpret_cast<int*>(stall + 1);  // the sequence's block-table row
    // once the ring is drained: per-KV-head merge areas, then the combine scratch
    MS* ms = reinterpret_cast<MS*>(smem);
    CS& cs = *reinterpret_cast<CS*>(smem + Cfg::kMergeBytes);

    const int c = blockIdx.x;
    const int n_kvg = p.Hkv / HPT;
    const int kvg = blockIdx.y % n_kvg;
    const int hg = blockIdx.y / n_kvg;
    const int b = blockIdx.z;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int bp = min(p.page_size, kTile);  // tokens per page piece (power of two)
    const int lbp = 31 - __clz(bp);

    // Before the dependency wait, while the previous grid drains: the producer warp reads the
    // length and the block-table entries of the chunk's first S tiles with L2-only loads and
    // has TMA prefetch those tiles into L2. The values may still be changing (the previous
    // grid's writes are not yet visible): they only choose what to prefetch, and a prefetch
    // cannot leave stale data (L2 is the point of coherence). The lane of piece k keeps the
    // page it read (spg) and the length (sLp): when both are read again unchanged after the
    // wait, the first copies are issued from them at once (nothing is copied before the wait).
    int sLp = -1, spg = -1, s_idx = 0, s_n = 0;
    if (warp == kConsumers) {
        if (lane == 0) {
            prefetch_tensormap(&tmK);
            prefetch_tensormap(&tmV);
        }
        int Lp = __ldcg(p.seq_lens + b);
        Lp = min(Lp, p.ring > 0 ? p.ring : p.max_len);
        int plo = 0, phi = 0;
        if (Lp >= 1 &&
            chunk_bounds(visible_ranges(Lp, p.window, p.n_sink), p.chunk, c, plo, phi)) {
            const int pt0 = plo & ~(kTile - 1);
            sLp = Lp;
            s_n = min(S, (phi - pt0 + kTile - 1) / kTile) * (kTile / bp);  // <= 32 pieces
            if (lane < s_n) {
                const int t = pt0 + lane * bp;
                s_idx = min(t, Lp - 1) / p.page_size;  // as the copy loop picks it
                spg = __ldcg(p.block_table + static_cast<size_t>(b) * p.max_pages + s_idx);
                if (spg < 0 || spg >= p.num_pages) spg = -1;
                if (spg >= 0 && t < Lp) {
                    const int y =
                        (spg * p.Hkv + kvg * HPT) * p.page_size + (t & (p.page_size - 1));
                    tma_prefetch_3d(&tmK, 0, y, 0);
                    tma_prefetch_3d(&tmV, 0, y, 0);
                }
            }
        }
    }
    if (threadIdx.x == 0) {  // shared memory only: published by the barrier after the wait
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumers);
        }
        mbar_init(stall, 1);
        fence_mbar_init();
    }
    griddep_wait();
    // The producer loads the sequence's whole block-table row (up to kRowCache entries) while
    // the sequence length is on its way, instead of the entries the length points to after
    // it: one memory round trip less before the first copy. Entries are checked when used.
    constexpr int kRowRegs = kRowCache / 32;
    const bool row_cached = p.max_pages <= kRowCache;
    int row[kRowRegs];
    int vpg = -1;  // the entry behind spg, read again
    if (warp == kConsumers) {
        const int32_t* btr = p.block_table + static_cast<size_t>(b) * p.max_pages;
        if (lane < s_n) vpg = btr[s_idx];
        if (row_cached) {
#pragma unroll
            for (int j = 0; j < kRowRegs; ++j)
                row[j] = lane + 32 * j < p.max_pages ? btr[lane + 32 * j] : 0;
        }
    }
    const int L = visible_len(p, b);
    const Ranges R = visible_ranges(L, p.window, p.n_sink);
    int lo = 0, hi = 0;
    // an empty chunk exits, except in a cluster, where it joins the combine with nothing
    const bool has = chunk_bounds(R, p.chunk, c, lo, hi);
    if (!kClu && !has) return;
    if (!has) lo = hi = 0;
    const int n_chunks = total_chunks(R, p.chunk);
    const int t0 = lo & ~(kTile - 1);
    const int n_tiles = (hi - t0 + kTile - 1) / kTile;
    const int G_cta = min(kMaxHP, p.G - hg * kMaxHP);
    __syncthreads();
    // cluster combine: no CTA stores into another's shared memory before every CTA of the
    // cluster has started (this arrival; the matching wait comes before the first store)
    if constexpr (kClu) cluster_arrive_relaxed();
    // Every wait of the ring is bounded; one that runs out records KVD_ERR_TIMEOUT and its
    // warp leaves the loop. The call's limit is normally kWaitCycles.
    const long long wait_limit = p.wait_cycles > 0 ? p.wait_cycles : kWaitCycles;

    if (warp == kConsumers) {
        // ------------------------------------------------------------------ producer
        // The warp resolves the page ids of the CTA's page pieces 32 at a time (lane k: piece
        // 32 m + k), the next batch in flight while the current one is used, so that filling
        // the ring costs one lookup round trip rather than one per tile; lane 0 issues.
        const int per_tile = kTile / bp;
        const int n_pieces = n_tiles * per_tile;
        const uint64_t pol = l2_evict_first_policy();  // K and V are read once
        // The newest token's ring slot, when this call appends it (below).
        int slot = -1;
        if (p.k_new != nullptr && has) {
            const int Lt = p.seq_lens[b];  // its validity is recorded by visible_len
            if (Lt >= 1) {
                const long long t = Lt - 1;
                const int win = p.ring - p.ring_sink;
                slot = t < p.ring_sink ? static_cast<int>(t)
                                       : p.ring_sink + static_cast<int>((t - p.ring_sink) % win);
                if (slot < lo || slot >= hi) slot = -1;
            }
        }
        // First copies from the values read before the wait, when the length and every entry
        // they used are unchanged now (a chunk that appends the newest token's rows first
        // writes them, so it takes the ordinary path).
        int n_fast = 0;
        if (slot < 0 && has && sLp == L && s_n == min(S, n_tiles) * per_tile &&
            __all_sync(0xffffffffu, lane >= s_n || (spg >= 0 && vpg == spg))) {
            n_fast = min(S, n_tiles);
            for (int i = 0; i < n_fast; ++i) {
                if (lane == 0) mbar_arrive_expect_tx(&full[i], 2 * Cfg::kTileBytes);
                for (int sub = 0; sub < per_tile; ++sub) {
                    const int pc = i * per_tile + sub;
                    const int pg = __shfl_sync(0xffffffffu, spg, pc);
                    if (lane == 0) {
                        const int t = t0 + pc * bp;
                        const int y =
                            (pg * p.Hkv + kvg * HPT) * p.page_size + (t & (p.page_size - 1));
                        const uint32_t off = static_cast<uint32_t>(sub * NB * HPT) << (lbp + 7);
                        tma_load_3d(sK + i * Cfg::kTileBytes + off, &tmK, &full[i], 0, y, 0, pol);
                        tma_load_3d(sV + i * Cfg::kTileBytes + off, &tmV, &full[i], 0, y, 0, pol);
                    }
                }
            }
        }
        if (row_cached) {
#pragma unroll
            for (int j = 0; j < kRowRegs; ++j)
                if (lane + 32 * j < p.max_pages) bt_row[lane + 32 * j] = row[j];
            __syncwarp();
        }
        auto piece_page = [&](int pc) -> int {
            if (pc >= n_pieces) return 0;
            const int t = t0 + pc * bp;
            const int tc = t < L ? t : L - 1;  // pieces past the end: any valid page
            if (!row_cached)
                return load_page(p.block_table, p.max_pages, p.num_pages, b, tc / p.page_size,
                                 p.err);
            int pg = bt_row[tc / p.page_size];
            if (pg < 0 || pg >= p.num_pages) {
                record_error(p.err, KVD_ERR_DEVICE_OOB);
                pg = 0;
            }
            return pg;
        };
        // Ring with the newest token's rows in the call (append + attention in one launch):
        // the CTA whose chunk holds the token's ring slot writes its KV heads' K and V rows
        // there before any copy of its own (every query-head block of the group writes the
        // same bytes), ordered before the copies' reads by the proxy fence; no other chunk
        // reads that slot, and the previous kernel has finished with it (dependency wait).
        if (slot >= 0) {
            const int pg = row_cached ? bt_row[slot / p.page_size]
                                      : p.block_table[static_cast<size_t>(b) * p.max_pages +
                                                      slot / p.page_size];
            if (pg < 0 || pg >= p.num_pages) {
                if (lane == 0) record_error(p.err, KVD_ERR_DEVICE_OOB);
            } else {
                constexpr int kPieces = D * 2 / 16;  // 16-byte pieces of a bf16 row
                for (int e = lane; e < HPT * 2 * kPieces; e += 32) {
                    const int hh = e / (2 * kPieces), isv = (e / kPieces) & 1;
                    const int pc = e % kPieces;
                    const int kvh = kvg * HPT + hh;
                    const size_t src = (static_cast<size_t>(b) * p.Hkv + kvh) * D * 2 + pc * 16;
                    const size_t dst =
                        ((static_cast<size_t>(pg) * p.Hkv + kvh) * p.page_size +
                         slot % p.page_size) * D * 2 + pc * 16;
                    const uint4 v = *reinterpret_cast<const uint4*>(
                        static_cast<const uint8_t*>(isv ? p.v_new : p.k_new) + src);
                    *reinterpret_cast<uint4*>(
                        const_cast<uint8_t*>(static_cast<const uint8_t*>(
                            isv ? p.v_pool : p.k_pool)) + dst) = v;
                }
                asm volatile("fence.proxy.async.global;" ::: "memory");
            }
            __syncwarp();
        }
        int cur = piece_page(lane), nxt = piece_page(32 + lane);
        int issued = n_fast;  // tiles whose copies are in flight or landed
        for (int i = n_fast; i < n_tiles; ++i) {  // (pieces of fast tiles are < 32)
            const int s = i % S;
            bool ok = true;
            if (lane == 0) {
                ok = mbar_wait(&empty[s], ((i / S) & 1) ^ 1, p.err, wait_limit);
                if (ok) mbar_arrive_expect_tx(&full[s], 2 * Cfg::kTileBytes);
            }
            if (!__shfl_sync(0xffffffffu, ok, 0)) break;
            for (int sub = 0; sub < per_tile; ++sub) {
                const int pc = i * per_tile + sub;
                if (pc > 0 && (pc & 31) == 0) {
                    cur = nxt;
                    nxt = piece_page(pc + 32 + lane);
                }
                const int pg = __shfl_sync(0xffffffffu, cur, pc & 31);
                if (lane == 0) {
                    const int t = t0 + pc * bp;
                    // rows of KV heads kvg*HPT .. +HPT-1 of this piece (HPT > 1 only when a
                    // piece is a whole page, so the heads' rows are adjacent), all blocks
                    const int y =
                        (pg * p.Hkv + kvg * HPT) * p.page_size + (t & (p.page_size - 1));
                    const uint32_t off = static_cast<uint32_t>(sub * NB * HPT) << (lbp + 7);
                    tma_load_3d(sK + s * Cfg::kTileBytes + off, &tmK, &full[s], 0, y, 0, pol);
                    tma_load_3d(sV + s * Cfg::kTileBytes + off, &tmV, &full[s], 0, y, 0, pol);
                }
            }
            issued = i + 1;
        }
        // Every copy of this CTA is issued: the next grid on the stream may be scheduled
        // (its prefetches then overlap this grid's last tiles, merge and combine).
        griddep_launch_dependents();
        // The merge below overwrites the ring, and consumers that gave up on a wait leave
        // tiles unread: every issued copy must have landed first. (After a normal loop these
        // are the last tiles, which the consumers wait for as well.) The tile issued last in
        // each stage completes that stage's latest phase; earlier ones completed before it
        // was issued.
        if (lane == 0)
            for (int i = issued > S ? issued - S : 0; i < issued; ++i)
                mbar_wait(&full[i % S], (i / S) & 1, p.err);
        __syncwarp();
        asm volatile("bar.sync 1, %0;" ::"r"((kConsumers + 1) * 32) : "memory");
    } else {
        // ------------------------------------------------------------------ consumers
        // tile layout [piece][block][head][slot][64]: 128-byte rows, 16-byte chunks XOR-ed
        // with (slot % 8) by the 128-byte swizzle
        auto addr = [&](int hh, int row, int col) -> uint32_t {
            const int piece = row >> lbp, slot = row & (bp - 1);
            return (static_cast<uint32_t>((piece * NB + (col >> 6)) * HPT + hh) << (lbp + 7)) +
                   (static_cast<uint32_t>(slot) << 7) +
                   static_cast<uint32_t>((((col & 63) >> 3) ^ (slot & 7)) << 4);
        };
        // q^T fragments (B operand of the score mma): lane holds head lane/4 of each 8-head
        // tile, dims 16kk + 2(lane%4) + {0,1} and the same +8
        uint32_t qf[HPT][NT][KT][2];
        const __nv_bfloat16* qb = reinterpret_cast<const __nv_bfloat16*>(p.q);
#pragma unroll
        for (int hh = 0; hh < HPT; ++hh)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int hl = nt * 8 + lane / 4;
                const bool ok = hl < G_cta;
                const int hq = (kvg * HPT + hh) * p.G + hg * kMaxHP + hl;
                const __nv_bfloat16* qr =
                    qb + (static_cast<size_t>(b) * p.Hq + (ok ? hq : 0)) * D;
#pragma unroll
                for (int kk = 0; kk < KT; ++kk) {
                    const int d0 = kk * 16 + 2 * (lane % 4);
                    qf[hh][nt][kk][0] = ok ? *reinterpret_cast<const uint32_t*>(qr + d0) : 0u;
                    qf[hh][nt][kk][1] = ok ? *reinterpret_cast<const uint32_t*>(qr + d0 + 8) : 0u;
                }
            }
        float oacc[HPT][KT][NT][4];
        float m_run[HPT][NT][2], l_run[HPT][NT][2];
#pragma unroll
        for (int hh = 0; hh < HPT; ++hh)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
                for (int mt = 0; mt < KT; ++mt)
#pragma unroll
                    for (int r = 0; r < 4; ++r) oacc[hh][mt][nt][r] = 0.f;
                m_run[hh][nt][0] = m_run[hh][nt][1] = neg_inf();
                l_run[hh][nt][0] = l_run[hh][nt][1] = 0.f;
            }
        const int r0 = warp * 16;
        const float sl2 = p.scale_log2;
        // give-up test: this wait runs out, so the consumers read no tile (the producer's
        // wait for a free stage then runs out as well)
        const int n_read = (p.stall_test && !mbar_wait(stall, 0, p.err, wait_limit)) ? 0 : n_tiles;

        for (int i = 0; i < n_read; ++i) {
            const int s = i % S;
            if (!mbar_wait(&full[s], (i / S) & 1, p.err, wait_limit)) break;
            const int T = t0 + i * kTile;
            uint8_t* kt = sK + s * Cfg::kTileBytes;
            uint8_t* vt = sV + s * Cfg::kTileBytes;
            const bool ragged = T < lo || T + kTile > hi;
            if (ragged) {
                // zero this warp's V rows outside [lo, hi): masked tokens then add 0 * 0
                // (their rows may hold anything, including NaN bit patterns)
                for (int idx = lane; idx < HPT * 16 * (D / 8); idx += 32) {
                    const int hh = idx / (16 * (D / 8));
                    const int rem = idx % (16 * (D / 8));
                    const int row = r0 + rem / (D / 8);
                    const int tok = T + row;
                    if (tok < lo || tok >= hi)
                        *reinterpret_cast<uint4*>(vt + addr(hh, row, (rem % (D / 8)) * 8)) =
                            make_uint4(0, 0, 0, 0);
                }
                __syncwarp();
            }
            const int tokA = T + r0 + lane / 4, tokB = tokA + 8;
            const bool inA = tokA >= lo && tokA < hi, inB = tokB >= lo && tokB < hi;
            const uint32_t kbase = smem_u32(kt), vbase = smem_u32(vt);
#pragma unroll
            for (int hh = 0; hh < HPT; ++hh) {
                // ---- scores S^T[16 tok x 8 heads], two independent accumulation chains
                float sacc[NT][4], sacc2[NT][4];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int r = 0; r < 4; ++r) sacc[nt][r] = sacc2[nt][r] = 0.f;
#pragma unroll
                for (int kk = 0; kk < KT; ++kk) {
                    uint32_t a[4];
                    ldsm_x4(kbase + addr(hh, r0 + (lane % 16), kk * 16 + (lane / 16) * 8), a);
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        if (kk & 1)
                            mma_bf16_16816(sacc2[nt], a, qf[hh][nt][kk][0], qf[hh][nt][kk][1]);
                        else
                            mma_bf16_16816(sacc[nt], a, qf[hh][nt][kk][0], qf[hh][nt][kk][1]);
                    }
                }
                // ---- online softmax over this warp's 16 tokens, per head column
                uint32_t pb[NT][2];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const float x0 = inA ? (sacc[nt][0] + sacc2[nt][0]) * sl2 : neg_inf();
                    const float x1 = inA ? (sacc[nt][1] + sacc2[nt][1]) * sl2 : neg_inf();
                    const float x2 = inB ? (sacc[nt][2] + sacc2[nt][2]) * sl2 : neg_inf();
                    const float x3 = inB ? (sacc[nt][3] + sacc2[nt][3]) * sl2 : neg_inf();
                    float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
                    for (int off = 4; off < 32; off <<= 1) {
                        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
                        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
                    }
                    const float mn0 = fmaxf(m_run[hh][nt][0], mx0);
                    const float mn1 = fmaxf(m_run[hh][nt][1], mx1);
                    // a column with nothing visible yet keeps a finite reference of 0
                    const float mu0 = mn0 == neg_inf() ? 0.f : mn0;
                    const float mu1 = mn1 == neg_inf() ? 0.f : mn1;
                    const float al0 = fast_exp2(m_run[hh][nt][0] - mu0);
                    const float al1 = fast_exp2(m_run[hh][nt][1] - mu1);
                    m_run[hh][nt][0] = mn0;
                    m_run[hh][nt][1] = mn1;
                    const float p0 = fast_exp2(x0 - mu0), p1 = fast_exp2(x1 - mu1);
                    const float p2 = fast_exp2(x2 - mu0), p3 = fast_exp2(x3 - mu1);
                    l_run[hh][nt][0] = l_run[hh][nt][0] * al0 + p0 + p2;
                    l_run[hh][nt][1] = l_run[hh][nt][1] * al1 + p1 + p3;
#pragma unroll
                    for (int mt = 0; mt < KT; ++mt) {
                        oacc[hh][mt][nt][0] *= al0;
                        oacc[hh][mt][nt][1] *= al1;
                        oacc[hh][mt][nt][2] *= al0;
                        oacc[hh][mt][nt][3] *= al1;
                    }
                    // P^T as the B operand: transpose the two 8x8 (token x head) blocks
                    pb[nt][0] = movmatrix_t(pack_bf16(p0, p1));
                    pb[nt][1] = movmatrix_t(pack_bf16(p2, p3));
                }
                // ---- O^T[D x 8] += V^T[D x 16 tok] P^T
#pragma unroll
                for (int mt = 0; mt < KT; ++mt) {
                    uint32_t a[4];
                    ldsm_x4_t(vbase + addr(hh, r0 + (lane % 8) + (lane / 16) * 8,
                                           mt * 16 + ((lane / 8) % 2) * 8),
                              a);
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
                        mma_bf16_16816(oacc[hh][mt][nt], a, pb[nt][0], pb[nt][1]);
                }
            }
            // the zeroing (generic proxy) ordered before the next TMA write into the stage
            if (ragged) fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
        }
        griddep_launch_dependents();  // (as the producer: every thread of the CTA has it)
        // row sums: reduce over the 8 lanes that share a head column
#pragma unroll
        for (int hh = 0; hh < HPT; ++hh)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int j = 0; j < 2; ++j)
#pragma unroll
                    for (int off = 4; off < 32; off <<= 1)
                        l_run[hh][nt][j] += __shfl_xor_sync(0xffffffffu, l_run[hh][nt][j], off);
        // every consumer warp is done with the ring, and every copy into it has landed,
        // before the merge area overwrites it
        asm volatile("bar.sync 1, %0;" ::"r"((kConsumers + 1) * 32) : "memory");
#pragma unroll
        for (int hh = 0; hh < HPT; ++hh)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int h0 = nt * 8 + 2 * (lane % 4);
                if (lane < 4) {
                    ms[hh].m[warp][h0] = m_run[hh][nt][0];
                    ms[hh].m[warp][h0 + 1] = m_run[hh][nt][1];
                    ms[hh].l[warp][h0] = l_run[hh][nt][0];
                    ms[hh].l[warp][h0 + 1] = l_run[hh][nt][1];
                }
#pragma unroll
                for (int mt = 0; mt < KT; ++mt) {
                    const int d0 = mt * 16 + lane / 4;
                    ms[hh].o[warp][h0][d0] = oacc[hh][mt][nt][0];
                    ms[hh].o[warp][h0 + 1][d0] = oacc[hh][mt][nt][1];
                    ms[hh].o[warp][h0][d0 + 8] = oacc[hh][mt][nt][2];
                    ms[hh].o[warp][h0 + 1][d0 + 8] = oacc[hh][mt][nt][3];
                }
            }
    }
    __syncthreads();
    if constexpr (kClu) {
        const int rank = static_cast<int>(cluster_rank());
        cluster_wait();  // every CTA of the cluster has started
        merge_push<D, NT * 8, HPT * NT * 8>(ms, rx, HPT, G_cta, gridDim.x, rank);
        cluster_sync();  // every chunk's partial is in its combining CTA
        combine_rx<D, HPT * NT * 8>(p, rx, b, kvg * HPT, HPT, hg, G_cta, gridDim.x, rank);
    } else {
        merge_chunks<D, NT * 8>(p, ms, b, kvg * HPT, HPT, hg, c, G_cta);
        const int grp = (b * n_kvg + kvg) * p.NHG + hg;
        finish_group<D, HPT * NT * 8>(p, cs, b, kvg * HPT, HPT, hg, grp, n_chunks, G_cta);
    }
}

// ---------------------------------------------------------------------------------------
// float32 kernel: one CTA per chunk, plain loads, one token per warp step, exact fp32 FMA
// ---------------------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(kConsumers * 32) gqa_decode_f32_kernel(const GqaParams p) {
    griddep_wait();
    constexpr int J = D / 32;  // dims per lane
    extern __shared__ uint8_t smem_raw[];
    MergeSmem<D, kMaxHP>& ms = *reinterpret_cast<MergeSmem<D, kMaxHP>*>(smem_raw);
    CombineSmem<kMaxHP>& cs =
        *reinterpret_cast<CombineSmem<kMaxHP>*>(smem_raw + sizeof(MergeSmem<D, kMaxHP>));
    const int c = blockIdx.x;
    const int kvh = blockIdx.y % p.Hkv;
    const int hg = blockIdx.y / p.Hkv;
    const int b = blockIdx.z;
    const int L = visible_len(p, b);
    const Ranges R = visible_ranges(L, p.window, p.n_sink);
    int lo, hi;
    if (!chunk_bounds(R, p.chunk, c, lo, hi)) return;
    const int n_chunks = total_chunks(R, p.chunk);
    const int G_cta = min(kMaxHP, p.G - hg * kMaxHP);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    const float* q = reinterpret_cast<const float*>(p.q);
    const float* kp = reinterpret_cast<const float*>(p.k_pool);
    const float* vp = reinterpret_cast<const float*>(p.v_pool);
    float qr[kMaxHP][J], o[kMaxHP][J], m[kMaxHP], l[kMaxHP];
#pragma unroll
    for (int h = 0; h < kMaxHP; ++h) {
        const int hq = kvh * p.G + hg * kMaxHP + min(h, G_cta - 1);
#pragma unroll
        for (int j = 0; j < J; ++j) {
            qr[h][j] = q[(static_cast<size_t>(b) * p.Hq + hq) * D + lane + 32 * j];
            o[h][j] = 0.f;
        }
        m[h] = neg_inf();
        l[h] = 0.f;
    }
    for (int t = lo + warp; t < hi; t += kConsumers) {
        const int pg = load_page(p.block_table, p.max_pages, p.num_pages, b, t / p.page_size, p.err);
        const size_t row = (static_cast<size_t>(pg) * p.Hkv + kvh) * p.page_size + t % p.page_size;
        float kr[J], vr[J];
#pragma unroll
        for (int j = 0; j < J; ++j) {
            kr[j] = kp[row * D + lane + 32 * j];
            vr[j] = vp[row * D + lane + 32 * j];
        }
#pragma unroll
        for (int h = 0; h < kMaxHP; ++h) {
            if (h >= G_cta) break;
            float dot = 0.f;
#pragma unroll
            for (int j = 0; j < J; ++j) dot = fmaf(qr[h][j], kr[j], dot);
            for (int off = 16; off; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
            const float x = dot * p.scale_log2;
            const float mn = fmaxf(m[h], x);
            const float al = exp2f(m[h] - mn);
            const float pr = exp2f(x - mn);
            m[h] = mn;
            l[h] = l[h] * al + pr;
#pragma unroll
            for (int j = 0; j < J; ++j) o[h][j] = o[h][j] * al + pr * vr[j];
        }
    }
#pragma unroll
    for (int h = 0; h < kMaxHP; ++h) {
        if (h >= G_cta) break;
        if (lane == 0) {
            ms.m[warp][h] = m[h];
            ms.l[warp][h] = l[h];
        }
#pragma unroll
        for (int j = 0; j < J; ++j) ms.o[warp][h][lane + 32 * j] = o[h][j];
    }
    __syncthreads();
    const size_t unit = unit_of(p, b, kvh, hg);
    merge_chunks<D, kMaxHP>(p, &ms, b, kvh, 1, hg, c, G_cta);
    finish_group<D, kMaxHP>(p, cs, b, kvh, 1, hg, static_cast<int>(unit), n_chunks, G_cta);
}

template <typename K>
int set_smem(K kernel, int bytes) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) ==
                   cudaSuccess
               ? KVD_OK
               : KVD_ERR_CUDA;
}

template <int D, int NT, int HPT>
int launch_bf16(const GqaPlan& plan, const GqaParams& p, const CUtensorMap& tk,
                const CUtensorMap& tv, cudaStream_t stream) {
    using Cfg = GqaBf16Cfg<D, NT, HPT, false>;
    using CfgC = GqaBf16Cfg<D, NT, HPT, true>;
    auto kern = gqa_decode_bf16_kernel<D, NT, HPT, false>;
    auto kern_clu = gqa_decode_bf16_kernel<D, NT, HPT, true>;
    // per cluster size: 0 not yet checked, 1 a cluster of that size fits on the GPU, -1 not
    static int configured = 0, clu_ok[9] = {};
    if (!configured) {
        if (set_smem(kern, Cfg::kSmem) != KVD_OK || set_smem(kern_clu, CfgC::kSmem) != KVD_OK)
            return KVD_ERR_CUDA;
        configured = 1;
    }
    const dim3 grid(plan.max_chunks, (p.Hkv / HPT) * p.NHG, p.B);
    const int cs = plan.cluster;
    if (cs >= 1 && cs <= 8 && cs == plan.max_chunks) {
        if (clu_ok[cs] == 0) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = grid;
            cfg.blockDim = dim3(CfgC::kThreads);
            cfg.dynamicSmemBytes = CfgC::kSmem;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = static_cast<unsigned>(cs);
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            int n = 0;
            clu_ok[cs] = (cudaOccupancyMaxActiveClusters(&n, kern_clu, &cfg) == cudaSuccess && n >= 1)
                             ? 1 : -1;
            cudaGetLastError();
        }
        if (clu_ok[cs] == 1) {
            if (launch_kernel_cluster(kern_clu, grid, dim3(CfgC::kThreads), CfgC::kSmem, cs,
                                      stream, tk, tv, p) != cudaSuccess)
                return KVD_ERR_CUDA;
            return cudaGetLastError() == cudaSuccess ? KVD_OK : KVD_ERR_CUDA;
        }
    }
    if (launch_kernel(kern, grid, dim3(Cfg::kThreads), Cfg::kSmem, stream, tk, tv, p) !=
        cudaSuccess)
        return KVD_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? KVD_OK : KVD_ERR_CUDA;
}

template <int D>
int launch_f32(const GqaPlan& plan, const GqaParams& p, cudaStream_t stream) {
    auto kern = gqa_decode_f32_kernel<D>;
    const int bytes =
        static_cast<int>(sizeof(MergeSmem<D, kMaxHP>) + sizeof(CombineSmem<kMaxHP>));
    static int configured = 0;
    if (!configured) {
        if (set_smem(kern, bytes) != KVD_OK) return KVD_ERR_CUDA;
        configured = 1;
    }
    const dim3 grid(plan.max_chunks, p.Hkv * p.NHG, p.B);
    if (launch_kernel(kern, grid, dim3(kConsumers * 32), bytes, stream, p) != cudaSuccess)
        return KVD_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? KVD_OK : KVD_ERR_CUDA;
}

}  // namespace

int gqa_launch(const GqaPlan& plan, const GqaParams& p, const CUtensorMap* tk,
               const CUtensorMap* tv, cudaStream_t stream) {
    if (p.dtype == KVD_F32) {
        return p.D == 128 ? launch_f32<128>(plan, p, stream) : launch_f32<64>(plan, p, stream);
    }
    const int hp = p.G < kMaxHP ? p.G : kMaxHP;
    if (p.D == 128) {
        return hp <= 8 ? launch_bf16<128, 1, 1>(plan, p, *tk, *tv, stream)
                       : launch_bf16<128, 2, 1>(plan, p, *tk, *tv, stream);
    }
    if (plan.hpt == 2) return launch_bf16<64, 1, 2>(plan, p, *tk, *tv, stream);
    return hp <= 8 ? launch_bf16<64, 1, 1>(plan, p, *tk, *tv, stream)
                   : launch_bf16<64, 2, 1>(plan, p, *tk, *tv, stream);
}

}  // namespace kvd
