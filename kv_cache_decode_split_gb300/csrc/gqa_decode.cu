// gqa_decode.cu -- split-KV decode attention for GQA / MHA / MQA over a paged cache,
// with an optional sliding window, sink tokens and a learned sink logit.
//
// What is computed ("Overview of Attention Mechanism", GQA / Code; "All the
// attentions", sections 1, 4 and 8; "Attention Optimizations", Attention sinks):
//   o_h = sum_{t in V} e^{s_t} v_{g(h),t} / (sum_{t in V} e^{s_t} + [sink] e^{sigma_h}),
//   s_t = scale * q_h . k_{g(h),t},  g(h) = h / (Hq / Hkv),
// with V the visible set of the query at position L-1 (all tokens, or the window of W
// tokens ending at the query plus the first n_sink tokens).
//
// How (GB300), bf16: a persistent kernel, one CTA per SM. Work items are (sequence, KV
// head, block of <= 16 query heads, chunk of the visible range); a producer warp takes
// them from a global queue and streams their 64-token K and V page tiles with TMA
// (128-byte swizzle) through a multi-stage mbarrier ring, together with the item's query
// rows (one bulk copy into the first tile's stage). The ring never drains between items.
// Four consumer warps each take 16 tokens of every tile and run the running-max /
// running-sum softmax ("All the attentions", section 1) on warp-level tensor cores:
//   S^T[16 tok x 8 heads] = K[16 x D] q^T        (mma.sync m16n8k16, tokens as M)
//   O^T[D x 8 heads]     += V^T[D x 16 tok] P^T  (P^T via movmatrix, V^T via ldmatrix.trans)
// At the end of an item the four warps are merged in shared memory into one (o,
// log2-sum-exp) partial; the CTA that finishes the last chunk of a (sequence, KV head,
// head block) combines all its chunk partials with log-sum-exp weights (plus the learned
// sink, once) and writes the output. One launch per call.
//
// The float32 variant (tiny shapes, exact fp32 arithmetic) walks the block table with
// plain loads on CUDA cores, one CTA per item, and shares the merge and combine code.

#include <cstdlib>

#include "kvd_device.cuh"
#include "kvd_host.h"

namespace kvd {

namespace {

constexpr int kTile = 64;        // tokens per K/V tile
constexpr int kConsumers = 4;    // consumer warps, 16 tokens of each tile each
constexpr int kMaxHP = 16;       // query heads handled per work item
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ float neg_inf() { return -__int_as_float(0x7f800000); }

__device__ __forceinline__ void consumer_sync() {
    asm volatile("bar.sync 1, %0;" ::"r"(kConsumers * 32) : "memory");
}

// Shared memory of the merge / combine phase for HP query heads per item.
template <int D, int HP>
struct MergeSmem {
    float m[kConsumers][HP];
    float l[kConsumers][HP];
    float o[kConsumers][HP][D];
};

struct Item {
    int b, kvh, hg, c, unit;
};

__device__ __forceinline__ Item decode_item(const GqaParams& p, int item) {
    Item it;
    it.unit = item / p.max_chunks;
    it.c = item % p.max_chunks;
    it.hg = it.unit % p.NHG;
    const int bk = it.unit / p.NHG;
    it.kvh = bk % p.Hkv;
    it.b = bk / p.Hkv;
    return it;
}

// Merge the per-warp partials in `ms` (written by the 128 consumer threads) into this
// chunk's (o, log2-sum-exp) partial in the workspace. `sync` is the consumers' barrier.
template <int D, int HP, typename Sync>
__device__ void merge_chunk(const GqaParams& p, MergeSmem<D, HP>& ms, const Item& it, int G_cta,
                            int tid, Sync sync) {
    constexpr int kThr = kConsumers * 32;
    const size_t unit = it.unit;
    float* part_o = p.part_o + (unit * p.max_chunks + it.c) * kMaxHP * D;
    float* part_lse = p.part_lse + (unit * p.max_chunks + it.c) * kMaxHP;
    for (int idx = tid; idx < G_cta * D; idx += kThr) {
        const int h = idx / D, d = idx % D;
        float M = neg_inf();
#pragma unroll
        for (int w = 0; w < kConsumers; ++w) M = fmaxf(M, ms.m[w][h]);
        float lsum = 0.f, osum = 0.f;
#pragma unroll
        for (int w = 0; w < kConsumers; ++w) {
            const float f = fast_exp2(ms.m[w][h] - M);
            lsum += ms.l[w][h] * f;
            osum += ms.o[w][h][d] * f;
        }
        __stcg(part_o + h * D + d, osum / lsum);
        if (d == 0) __stcg(part_lse + h, M + log2f(lsum));
    }
    sync();  // the merge area is free again
}

// Combine the chunk partials of one (sequence, KV head, head block) with log-sum-exp
// weights, the learned sink added once to the denominator:
//   o = sum_c 2^{lse_c - M} o_c / (sum_c 2^{lse_c - M} + 2^{sigma - M}).
// One CTA per unit; each thread owns four dims of one query head and streams every chunk.
template <int D>
__global__ void __launch_bounds__(256) gqa_combine_kernel(const GqaParams p) {
    const int unit = blockIdx.x;
    if (unit == 0 && threadIdx.x == 0) p.counters[p.units] = 0;  // work queue, next call
    const Item it = decode_item(p, unit * p.max_chunks);
    const int L = load_len(p.seq_lens, it.b, p.max_len, nullptr);
    const int n_chunks = total_chunks(visible_ranges(L, p.window, p.n_sink), p.chunk);
    const int G_cta = min(kMaxHP, p.G - it.hg * kMaxHP);
    const float* uo = p.part_o + static_cast<size_t>(unit) * p.max_chunks * kMaxHP * D;
    const float* ul = p.part_lse + static_cast<size_t>(unit) * p.max_chunks * kMaxHP;
    for (int idx = threadIdx.x; idx < G_cta * (D / 4); idx += blockDim.x) {
        const int h = idx / (D / 4), d = (idx % (D / 4)) * 4;
        const int hq = it.kvh * p.G + it.hg * kMaxHP + h;
        float M = neg_inf();
        for (int c = 0; c < n_chunks; ++c) M = fmaxf(M, ul[c * kMaxHP + h]);
        const float sig = p.sink_logit ? p.sink_logit[hq] * kLog2e : neg_inf();
        M = fmaxf(M, sig);
        float den = p.sink_logit ? fast_exp2(sig - M) : 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
        for (int c = 0; c < n_chunks; ++c) {
            const float w = fast_exp2(ul[c * kMaxHP + h] - M);
            den += w;
            const float4 v = __ldcg(reinterpret_cast<const float4*>(
                uo + (static_cast<size_t>(c) * kMaxHP + h) * D + d));
            acc.x += w * v.x;
            acc.y += w * v.y;
            acc.z += w * v.z;
            acc.w += w * v.w;
        }
        const float inv = 1.f / den;
        const size_t o = (static_cast<size_t>(it.b) * p.Hq + hq) * D + d;
        if (p.dtype == KVD_BF16) {
            __nv_bfloat162 lo2 = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
            __nv_bfloat162 hi2 = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
            *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(p.out) + o) =
                make_uint2(*reinterpret_cast<uint32_t*>(&lo2), *reinterpret_cast<uint32_t*>(&hi2));
        } else {
            *reinterpret_cast<float4*>(reinterpret_cast<float*>(p.out) + o) =
                make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
        }
        if (d == 0 && p.lse_out)
            p.lse_out[static_cast<size_t>(it.b) * p.Hq + hq] = (M + log2f(den)) * kLn2;
    }
}

// ---------------------------------------------------------------------------------------
// bf16 kernel: persistent, TMA ring + mma.sync
// ---------------------------------------------------------------------------------------
struct StageMeta {
    int item;     // < 0: no more work
    int tile;     // tile index within the item
    int n_tiles;
    int T;        // first token of the tile
    int lo, hi;   // visible token range of the item
    int n_chunks;
    int pad;
};

// A resolved work item: its visible token range and the physical page of every TMA box.
struct ItemDesc {
    int item;  // < 0: no more work
    int lo, hi, t0, n_tiles, n_chunks, pad0, pad1;
    int pages[kGqaMaxBoxesPerItem];
};

constexpr int kDesc = 8;  // descriptor ring: how far the resolver runs ahead

template <int D, int NT>
struct GqaBf16Cfg {
    static constexpr int kTileBytes = kTile * D * 2;   // one K (or V) tile
    static constexpr int kQBytes = NT * 8 * D * 2;     // the item's query rows
    static constexpr int kStageBytes = (2 * kTileBytes + kQBytes + 64 + 1023) / 1024 * 1024;
    static constexpr int kMergeBytes = static_cast<int>(sizeof(MergeSmem<D, NT * 8>));
    // one CTA per SM; the TMA ring takes all the shared memory the merge area leaves, so
    // that as many K/V bytes as possible are in flight per SM
    static constexpr int kSmemBudget = 227 * 1024;
    static constexpr int kBarBytes = 512;
    static constexpr int kDescBytes = kDesc * static_cast<int>(sizeof(ItemDesc));
    static constexpr int kStages =
        (kSmemBudget - 1024 - kBarBytes - kDescBytes - kMergeBytes) / kStageBytes;
    static_assert(kStages >= 2, "ring too small");
    static_assert((2 * kStages + 2 * kDesc) * 8 <= kBarBytes, "mbarriers must fit their slot");
    static constexpr int kSmem = 1024 + kStages * kStageBytes + kBarBytes + kDescBytes + kMergeBytes;
    // warps 0-3 consume tiles, warp 4 issues TMA, warp 5 resolves work items
    static constexpr int kThreads = (kConsumers + 2) * 32;
};

template <int D, int NT>
__global__ void __launch_bounds__(GqaBf16Cfg<D, NT>::kThreads, 1)
    gqa_decode_bf16_kernel(const __grid_constant__ CUtensorMap tmK,
                           const __grid_constant__ CUtensorMap tmV, const GqaParams p) {
    using Cfg = GqaBf16Cfg<D, NT>;
    using MS = MergeSmem<D, NT * 8>;
    constexpr int S = Cfg::kStages;
    constexpr int KT = D / 16;  // k-steps of QK, m-tiles of PV
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    // stage s: [K tile][V tile][q rows][meta]
    auto stageK = [&](int s) { return smem + s * Cfg::kStageBytes; };
    auto stageV = [&](int s) { return smem + s * Cfg::kStageBytes + Cfg::kTileBytes; };
    auto stageQ = [&](int s) { return smem + s * Cfg::kStageBytes + 2 * Cfg::kTileBytes; };
    auto stageM = [&](int s) {
        return reinterpret_cast<StageMeta*>(smem + s * Cfg::kStageBytes + 2 * Cfg::kTileBytes +
                                            Cfg::kQBytes);
    };
    // after the ring (1024-aligned): mbarriers, item descriptors, the merge area
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + S * Cfg::kStageBytes);
    uint64_t* empty = full + S;
    uint64_t* dfull = empty + S;
    uint64_t* dempty = dfull + kDesc;
    ItemDesc* desc = reinterpret_cast<ItemDesc*>(smem + S * Cfg::kStageBytes + Cfg::kBarBytes);
    MS& ms = *reinterpret_cast<MS*>(smem + S * Cfg::kStageBytes + Cfg::kBarBytes + Cfg::kDescBytes);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int total_items = p.units * p.max_chunks;
    int* work = p.counters + p.units;  // work queue head (reset by the combine kernel)

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumers);
        }
        for (int d = 0; d < kDesc; ++d) {
            mbar_init(&dfull[d], 1);
            mbar_init(&dempty[d], 1);
        }
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == kConsumers + 1) {
        // ------------------------------------------------------------------ resolver
        // Takes work items from the queue, resolves their visible range and the physical
        // page of every TMA box (the dependent loads of seq_lens and the block table), and
        // publishes them as descriptors up to kDesc items ahead of the TMA issuer. The next
        // item's length and the item after it are requested before this item's page loads.
        const int bp = min(p.page_size, kTile);
        const int subs = kTile / bp;
        uint32_t d = 0;
        bool ok = true;
        int it_a = 0, it_c = 0;
        if (lane == 0) {
            it_a = atomicAdd(work, 1);
            it_c = atomicAdd(work, 1);
        }
        it_a = __shfl_sync(0xffffffffu, it_a, 0);
        int it_b = __shfl_sync(0xffffffffu, it_c, 0);
        int L_a = it_a < total_items ? load_len(p.seq_lens, decode_item(p, it_a).b, p.max_len, p.err) : 1;
        while (it_a < total_items && ok) {
            const int L_b =
                it_b < total_items ? load_len(p.seq_lens, decode_item(p, it_b).b, p.max_len, p.err) : 1;
            if (lane == 0 && it_b < total_items) it_c = atomicAdd(work, 1);
            const Item it = decode_item(p, it_a);
            const Ranges R = visible_ranges(L_a, p.window, p.n_sink);
            int lo, hi;
            if (chunk_bounds(R, p.chunk, it.c, lo, hi)) {
                const int slot = d % kDesc;
                if (lane == 0) ok = mbar_wait(&dempty[slot], ((d / kDesc) & 1) ^ 1, p.err);
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (ok) {
                    ItemDesc& dd = desc[slot];
                    const int t0 = lo & ~(kTile - 1);
                    const int n_tiles = (hi - t0 + kTile - 1) / kTile;
                    for (int j = lane; j < n_tiles * subs; j += 32) {
                        const int t = t0 + j * bp;
                        const int tc = t < L_a ? t : L_a - 1;  // rows past the end: a valid page
                        dd.pages[j] = load_page(p.block_table, p.max_pages, p.num_pages, it.b,
                                                tc / p.page_size, p.err);
                    }
                    if (lane == 0) {
                        dd.item = it_a;
                        dd.lo = lo;
                        dd.hi = hi;
                        dd.t0 = t0;
                        dd.n_tiles = n_tiles;
                        dd.n_chunks = total_chunks(R, p.chunk);
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&dfull[slot]);
                    ++d;
                }
            }
            it_a = it_b;
            L_a = L_b;
            it_b = __shfl_sync(0xffffffffu, it_c, 0);
        }
        if (ok && lane == 0) {  // no more work
            const int slot = d % kDesc;
            if (mbar_wait(&dempty[slot], ((d / kDesc) & 1) ^ 1, p.err)) {
                desc[slot].item = -1;
                mbar_arrive(&dfull[slot]);
            }
        }
    } else if (warp == kConsumers) {
        // ------------------------------------------------------------------ TMA issuer
        if (lane == 0) {
            prefetch_tensormap(&tmK);
            prefetch_tensormap(&tmV);
            const int bp = min(p.page_size, kTile);  // rows per TMA box
            const int subs = kTile / bp;
            uint32_t d = 0, g = 0;
            while (true) {
                const int slot = d % kDesc;
                if (!mbar_wait(&dfull[slot], (d / kDesc) & 1, p.err)) break;
                const ItemDesc& dd = desc[slot];
                const int item = dd.item;
                if (item < 0) {  // tell the consumers there is no more work
                    const int s = g % S;
                    if (mbar_wait(&empty[s], ((g / S) & 1) ^ 1, p.err)) {
                        stageM(s)->item = -1;
                        mbar_arrive(&full[s]);
                    }
                    break;
                }
                const Item it = decode_item(p, item);
                const int G_cta = min(kMaxHP, p.G - it.hg * kMaxHP);
                const int n_tiles = dd.n_tiles, t0 = dd.t0;
                bool ok = true;
                for (int tile = 0; tile < n_tiles; ++tile) {
                    const int s = g % S;
                    if (!mbar_wait(&empty[s], ((g / S) & 1) ^ 1, p.err)) {
                        ok = false;
                        break;
                    }
                    StageMeta* mt = stageM(s);
                    mt->item = item;
                    mt->tile = tile;
                    mt->n_tiles = n_tiles;
                    mt->T = t0 + tile * kTile;
                    mt->lo = dd.lo;
                    mt->hi = dd.hi;
                    mt->n_chunks = dd.n_chunks;
                    const int qbytes = tile == 0 ? G_cta * D * 2 : 0;
                    mbar_arrive_expect_tx(&full[s], 2 * Cfg::kTileBytes + qbytes);
                    if (tile == 0) {
                        const __nv_bfloat16* qsrc = reinterpret_cast<const __nv_bfloat16*>(p.q) +
                                                    (static_cast<size_t>(it.b) * p.Hq +
                                                     it.kvh * p.G + it.hg * kMaxHP) * D;
                        bulk_load(stageQ(s), qsrc, qbytes, &full[s]);
                    }
                    for (int sub = 0; sub < subs; ++sub) {
                        // one instruction per piece for K and for V, all D/64 column blocks:
                        // shared layout [piece][block][row][64]
                        const int j = tile * subs + sub;
                        const int t = t0 + j * bp;
                        const int y = (dd.pages[j] * p.Hkv + it.kvh) * p.page_size + (t % p.page_size);
                        const uint32_t off = sub * (D / 64) * bp * 128;
                        tma_load_3d(stageK(s) + off, &tmK, &full[s], 0, y, 0);
                        tma_load_3d(stageV(s) + off, &tmV, &full[s], 0, y, 0);
                    }
                    ++g;
                }
                mbar_arrive(&dempty[slot]);
                ++d;
                if (!ok) break;
            }
        }
    } else {
        // ------------------------------------------------------------------ consumers
        const int tid = threadIdx.x;
        uint32_t qf[NT][KT][2];
        float oacc[KT][NT][4];
        float m_run[NT][2], l_run[NT][2];
        const int r0 = warp * 16;
        const float sl2 = p.scale_log2;
        // tile layout [piece][block][row][64] with pieces of bp rows (the page, at most 64)
        const int lbp = 31 - __clz(min(p.page_size, kTile));
        auto addr = [&](int row, int col) -> uint32_t {
            return static_cast<uint32_t>(((row >> lbp) * (D / 64) + (col >> 6)) << (lbp + 7)) +
                   (static_cast<uint32_t>(row & ((1 << lbp) - 1)) << 7) +
                   ((((col & 63) >> 3) ^ (row & 7)) << 4);
        };
        uint32_t g = 0;
        while (true) {
            const int s = g % S;
            if (!mbar_wait(&full[s], (g / S) & 1, p.err)) break;
            const StageMeta mt = *stageM(s);
            if (mt.item < 0) break;
            const Item it = decode_item(p, mt.item);
            const int G_cta = min(kMaxHP, p.G - it.hg * kMaxHP);
            if (mt.tile == 0) {
                // q^T fragments (B operand of the score mma): lane holds head lane/4 of
                // each 8-head tile, dims 16kk + 2(lane%4) + {0,1} and +8.
                const uint8_t* qs = stageQ(s);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const int hl = nt * 8 + lane / 4;
                    const bool okh = hl < G_cta;
#pragma unroll
                    for (int kk = 0; kk < KT; ++kk) {
                        const int d0 = kk * 16 + 2 * (lane % 4);
                        qf[nt][kk][0] =
                            okh ? *reinterpret_cast<const uint32_t*>(qs + (hl * D + d0) * 2) : 0u;
                        qf[nt][kk][1] =
                            okh ? *reinterpret_cast<const uint32_t*>(qs + (hl * D + d0 + 8) * 2)
                                : 0u;
                    }
                }
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
                    for (int mtl = 0; mtl < KT; ++mtl)
#pragma unroll
                        for (int r = 0; r < 4; ++r) oacc[mtl][nt][r] = 0.f;
                    m_run[nt][0] = m_run[nt][1] = neg_inf();
                    l_run[nt][0] = l_run[nt][1] = 0.f;
                }
            }
            const int T = mt.T, lo = mt.lo, hi = mt.hi;
            uint8_t* kt = stageK(s);
            uint8_t* vt = stageV(s);
            const bool partial = (T < lo) || (T + kTile > hi);
            if (partial) {
                // zero this warp's V rows outside [lo, hi) so that masked tokens add 0 * 0
                for (int idx = lane; idx < 16 * (D / 8); idx += 32) {
                    const int row = r0 + idx / (D / 8);
                    const int tok = T + row;
                    if (tok < lo || tok >= hi)
                        *reinterpret_cast<uint4*>(vt + addr(row, (idx % (D / 8)) * 8)) =
                            make_uint4(0, 0, 0, 0);
                }
                fence_proxy_async_smem();  // order these stores before later TMA writes
                __syncwarp();
            }
            // ---- scores: S^T[16 tok x 8 heads] per head tile
            // two independent accumulation chains (even / odd k-steps), summed at the end
            float sacc[NT][4], sacc2[NT][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int r = 0; r < 4; ++r) sacc[nt][r] = sacc2[nt][r] = 0.f;
            const uint32_t kbase = smem_u32(kt);
#pragma unroll
            for (int kk = 0; kk < KT; ++kk) {
                uint32_t a[4];
                ldsm_x4(kbase + addr(r0 + (lane % 16), kk * 16 + (lane / 16) * 8), a);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    if (kk & 1)
                        mma_bf16_16816(sacc2[nt], a, qf[nt][kk][0], qf[nt][kk][1]);
                    else
                        mma_bf16_16816(sacc[nt], a, qf[nt][kk][0], qf[nt][kk][1]);
                }
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int r = 0; r < 4; ++r) sacc[nt][r] += sacc2[nt][r];
            // ---- online softmax over this warp's 16 tokens, per head column
            const int tokA = T + r0 + lane / 4, tokB = tokA + 8;
            const bool inA = tokA >= lo && tokA < hi, inB = tokB >= lo && tokB < hi;
            uint32_t pb[NT][2];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const float x0 = inA ? sacc[nt][0] * sl2 : neg_inf();
                const float x1 = inA ? sacc[nt][1] * sl2 : neg_inf();
                const float x2 = inB ? sacc[nt][2] * sl2 : neg_inf();
                const float x3 = inB ? sacc[nt][3] * sl2 : neg_inf();
                float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
                for (int off = 4; off < 32; off <<= 1) {
                    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
                    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
                }
                const float mn0 = fmaxf(m_run[nt][0], mx0), mn1 = fmaxf(m_run[nt][1], mx1);
                const float mu0 = mn0 == neg_inf() ? 0.f : mn0;
                const float mu1 = mn1 == neg_inf() ? 0.f : mn1;
                const float al0 = fast_exp2(m_run[nt][0] - mu0);
                const float al1 = fast_exp2(m_run[nt][1] - mu1);
                m_run[nt][0] = mn0;
                m_run[nt][1] = mn1;
                const float p0 = fast_exp2(x0 - mu0), p1 = fast_exp2(x1 - mu1);
                const float p2 = fast_exp2(x2 - mu0), p3 = fast_exp2(x3 - mu1);
                l_run[nt][0] = l_run[nt][0] * al0 + p0 + p2;
                l_run[nt][1] = l_run[nt][1] * al1 + p1 + p3;
#pragma unroll
                for (int mtl = 0; mtl < KT; ++mtl) {
                    oacc[mtl][nt][0] *= al0;
                    oacc[mtl][nt][1] *= al1;
                    oacc[mtl][nt][2] *= al0;
                    oacc[mtl][nt][3] *= al1;
                }
                // P^T as the B operand: transpose the two 8x8 (token x head) blocks
                pb[nt][0] = movmatrix_t(pack_bf16(p0, p1));
                pb[nt][1] = movmatrix_t(pack_bf16(p2, p3));
            }
            // ---- O^T[D x 8] += V^T[D x 16 tok] P^T
            const uint32_t vbase = smem_u32(vt);
#pragma unroll
            for (int mtl = 0; mtl < KT; ++mtl) {
                uint32_t a[4];
                ldsm_x4_t(vbase + addr(r0 + (lane % 8) + (lane / 16) * 8,
                                       mtl * 16 + ((lane / 8) % 2) * 8),
                          a);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
                    mma_bf16_16816(oacc[mtl][nt], a, pb[nt][0], pb[nt][1]);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
            ++g;
            if (mt.tile != mt.n_tiles - 1) continue;

            // ---- end of the item: merge the four warps, write the chunk partial
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int j = 0; j < 2; ++j)
#pragma unroll
                    for (int off = 4; off < 32; off <<= 1)
                        l_run[nt][j] += __shfl_xor_sync(0xffffffffu, l_run[nt][j], off);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int h0 = nt * 8 + 2 * (lane % 4);
                if (lane < 4) {
                    ms.m[warp][h0] = m_run[nt][0];
                    ms.m[warp][h0 + 1] = m_run[nt][1];
                    ms.l[warp][h0] = l_run[nt][0];
                    ms.l[warp][h0 + 1] = l_run[nt][1];
                }
#pragma unroll
                for (int mtl = 0; mtl < KT; ++mtl) {
                    const int d0 = mtl * 16 + lane / 4;
                    ms.o[warp][h0][d0] = oacc[mtl][nt][0];
                    ms.o[warp][h0 + 1][d0] = oacc[mtl][nt][1];
                    ms.o[warp][h0][d0 + 8] = oacc[mtl][nt][2];
                    ms.o[warp][h0 + 1][d0 + 8] = oacc[mtl][nt][3];
                }
            }
            consumer_sync();
            merge_chunk<D, NT * 8>(p, ms, it, G_cta, tid, consumer_sync);
        }
    }
}

// ---------------------------------------------------------------------------------------
// float32 kernel: one CTA per item, plain loads, one token per warp step, exact fp32 FMA
// ---------------------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(kConsumers * 32) gqa_decode_f32_kernel(const GqaParams p) {
    constexpr int J = D / 32;  // dims per lane
    extern __shared__ uint8_t smem_raw[];
    MergeSmem<D, kMaxHP>& ms = *reinterpret_cast<MergeSmem<D, kMaxHP>*>(smem_raw);
    const Item it = decode_item(p, blockIdx.x);
    const int L = load_len(p.seq_lens, it.b, p.max_len, p.err);
    const Ranges R = visible_ranges(L, p.window, p.n_sink);
    int lo, hi;
    if (!chunk_bounds(R, p.chunk, it.c, lo, hi)) return;
    const int G_cta = min(kMaxHP, p.G - it.hg * kMaxHP);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    const float* q = reinterpret_cast<const float*>(p.q);
    const float* kp = reinterpret_cast<const float*>(p.k_pool);
    const float* vp = reinterpret_cast<const float*>(p.v_pool);
    float qr[kMaxHP][J], o[kMaxHP][J], m[kMaxHP], l[kMaxHP];
#pragma unroll
    for (int h = 0; h < kMaxHP; ++h) {
        const int hq = it.kvh * p.G + it.hg * kMaxHP + min(h, G_cta - 1);
#pragma unroll
        for (int j = 0; j < J; ++j) {
            qr[h][j] = q[(static_cast<size_t>(it.b) * p.Hq + hq) * D + lane + 32 * j];
            o[h][j] = 0.f;
        }
        m[h] = neg_inf();
        l[h] = 0.f;
    }
    for (int t = lo + warp; t < hi; t += kConsumers) {
        const int pg =
            load_page(p.block_table, p.max_pages, p.num_pages, it.b, t / p.page_size, p.err);
        const size_t row =
            (static_cast<size_t>(pg) * p.Hkv + it.kvh) * p.page_size + t % p.page_size;
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
    merge_chunk<D, kMaxHP>(p, ms, it, G_cta, threadIdx.x, [] { __syncthreads(); });
}

template <typename K>
int set_smem(K kernel, int bytes) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) ==
                   cudaSuccess
               ? KVD_OK
               : KVD_ERR_CUDA;
}

template <int D, int NT>
int launch_bf16(const GqaPlan& plan, const GqaParams& p, const CUtensorMap& tk,
                const CUtensorMap& tv, cudaStream_t stream) {
    using Cfg = GqaBf16Cfg<D, NT>;
    auto kern = gqa_decode_bf16_kernel<D, NT>;
    static int configured = 0;
    if (!configured) {
        if (set_smem(kern, Cfg::kSmem) != KVD_OK) return KVD_ERR_CUDA;
        configured = 1;
    }
    const int items = plan.units * plan.max_chunks;
    const int ctas = num_sms();
    const int grid = items < ctas ? items : ctas;
    kern<<<grid, Cfg::kThreads, Cfg::kSmem, stream>>>(tk, tv, p);
    gqa_combine_kernel<D><<<plan.units, 256, 0, stream>>>(p);
    return cudaGetLastError() == cudaSuccess ? KVD_OK : KVD_ERR_CUDA;
}

template <int D>
int launch_f32(const GqaPlan& plan, const GqaParams& p, cudaStream_t stream) {
    auto kern = gqa_decode_f32_kernel<D>;
    const int bytes = static_cast<int>(sizeof(MergeSmem<D, kMaxHP>));
    static int configured = 0;
    if (!configured) {
        if (set_smem(kern, bytes) != KVD_OK) return KVD_ERR_CUDA;
        configured = 1;
    }
    kern<<<plan.units * plan.max_chunks, kConsumers * 32, bytes, stream>>>(p);
    gqa_combine_kernel<D><<<plan.units, 256, 0, stream>>>(p);
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
        return hp <= 8 ? launch_bf16<128, 1>(plan, p, *tk, *tv, stream)
                       : launch_bf16<128, 2>(plan, p, *tk, *tv, stream);
    }
    return hp <= 8 ? launch_bf16<64, 1>(plan, p, *tk, *tv, stream)
                   : launch_bf16<64, 2>(plan, p, *tk, *tv, stream);
}

}  // namespace kvd
