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
// How (GB300): one CTA per (sequence, KV head, head block of <= 16 query heads, chunk of
// the visible range). A producer warp streams 64-token K and V page tiles with TMA
// (128-byte swizzle) through a multi-stage mbarrier ring; four consumer warps each take
// 16 tokens of every tile and run the running-max / running-sum softmax ("All the
// attentions", section 1, online softmax) on warp-level tensor cores:
//   S^T[16 tok x 8 heads] = K[16 x D] q^T        (mma.sync m16n8k16, tokens as M)
//   O^T[D x 8 heads]     += V^T[D x 16 tok] P^T  (P^T via movmatrix, V^T via ldmatrix.trans)
// Warps are merged in shared memory into one (o, log2-sum-exp) partial per chunk; the last
// CTA of a (sequence, KV head, head block) combines all chunk partials (log-sum-exp
// weights plus the learned sink, once) and writes the output. No second launch.
//
// The float32 variant (tiny shapes, exact fp32 arithmetic) walks the block table with
// plain loads on CUDA cores and shares the merge and combine code.

#include "kvd_device.cuh"
#include "kvd_host.h"

namespace kvd {

namespace {

constexpr int kTile = 64;        // tokens per K/V tile
constexpr int kConsumers = 4;    // consumer warps, 16 tokens of each tile each
constexpr int kMaxHP = 16;       // query heads handled per CTA
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ float neg_inf() { return -__int_as_float(0x7f800000); }

// Shared memory of the merge / combine phase (overlays the K/V ring).
template <int D>
struct MergeSmem {
    float m[kConsumers][kMaxHP];
    float l[kConsumers][kMaxHP];
    float o[kConsumers][kMaxHP][D];
    float wgt[kMaxHP][kGqaMaxChunks];
    float inv_denom[kMaxHP];
    float lse_nat[kMaxHP];
    int is_last;
};

// Combine the per-warp partials in `ms` into this chunk's partial, then, if this CTA is
// the last of its (b, kvh, hg) unit, combine every chunk partial and write the output.
template <int D>
__device__ void merge_and_combine(const GqaParams& p, MergeSmem<D>& ms, int b, int kvh,
                                  int hg, int c, int n_chunks, int G_cta) {
    const int tid = threadIdx.x;
    const int nthr = blockDim.x;
    const size_t unit = (static_cast<size_t>(b) * p.Hkv + kvh) * p.NHG + hg;
    float* part_o = p.part_o + (unit * p.max_chunks + c) * kMaxHP * D;
    float* part_lse = p.part_lse + (unit * p.max_chunks + c) * kMaxHP;

    for (int idx = tid; idx < G_cta * D; idx += nthr) {
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
        part_o[h * D + d] = osum / lsum;
        if (d == 0) part_lse[h] = M + log2f(lsum);
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        const int prev = atomicAdd(p.counters + unit, 1);
        ms.is_last = (prev == n_chunks - 1);
    }
    __syncthreads();
    if (!ms.is_last) return;
    __threadfence();

    const float* uo = p.part_o + unit * p.max_chunks * kMaxHP * D;
    const float* ul = p.part_lse + unit * p.max_chunks * kMaxHP;
    const int warp = tid / 32, lane = tid % 32, nwarps = nthr / 32;
    for (int h = warp; h < G_cta; h += nwarps) {
        const int hq = kvh * p.G + hg * kMaxHP + h;
        float M = neg_inf();
        for (int cc = lane; cc < n_chunks; cc += 32) M = fmaxf(M, __ldcg(ul + cc * kMaxHP + h));
        for (int off = 16; off; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
        const float sig = p.sink_logit ? p.sink_logit[hq] * kLog2e : neg_inf();
        M = fmaxf(M, sig);
        float den = 0.f;
        for (int cc = lane; cc < n_chunks; cc += 32) {
            const float wv = fast_exp2(__ldcg(ul + cc * kMaxHP + h) - M);
            ms.wgt[h][cc] = wv;
            den += wv;
        }
        for (int off = 16; off; off >>= 1) den += __shfl_xor_sync(0xffffffffu, den, off);
        if (p.sink_logit) den += fast_exp2(sig - M);
        if (lane == 0) {
            ms.inv_denom[h] = 1.f / den;
            ms.lse_nat[h] = (M + log2f(den)) * kLn2;
        }
    }
    __syncthreads();
    for (int idx = tid; idx < G_cta * D; idx += nthr) {
        const int h = idx / D, d = idx % D;
        float acc = 0.f;
        for (int cc = 0; cc < n_chunks; ++cc)
            acc += ms.wgt[h][cc] * __ldcg(uo + (static_cast<size_t>(cc) * kMaxHP + h) * D + d);
        acc *= ms.inv_denom[h];
        const int hq = kvh * p.G + hg * kMaxHP + h;
        const size_t o_idx = (static_cast<size_t>(b) * p.Hq + hq) * D + d;
        if (p.dtype == KVD_BF16)
            reinterpret_cast<__nv_bfloat16*>(p.out)[o_idx] = __float2bfloat16_rn(acc);
        else
            reinterpret_cast<float*>(p.out)[o_idx] = acc;
        if (d == 0 && p.lse_out) p.lse_out[static_cast<size_t>(b) * p.Hq + hq] = ms.lse_nat[h];
    }
    if (tid == 0) p.counters[unit] = 0;  // ready for the next call
}

// ---------------------------------------------------------------------------------------
// bf16 kernel: TMA ring + mma.sync
// ---------------------------------------------------------------------------------------
template <int D>
struct GqaBf16Cfg {
    static constexpr int kStages = (D == 128) ? 3 : 4;
    static constexpr int kTileBytes = kTile * D * 2;  // one K (or V) tile
    static constexpr int kRingBytes = 2 * kStages * kTileBytes;
    static constexpr int kSmem =
        1024 + (kRingBytes > static_cast<int>(sizeof(MergeSmem<D>)) ? kRingBytes
                                                                    : static_cast<int>(sizeof(MergeSmem<D>))) +
        2 * kStages * 8 + 16;
    static constexpr int kThreads = (kConsumers + 1) * 32;
};

template <int D, int NT>
__global__ void __launch_bounds__(GqaBf16Cfg<D>::kThreads)
    gqa_decode_bf16_kernel(const __grid_constant__ CUtensorMap tmK,
                           const __grid_constant__ CUtensorMap tmV, const GqaParams p) {
    using Cfg = GqaBf16Cfg<D>;
    constexpr int S = Cfg::kStages;
    constexpr int KT = D / 16;  // k-steps of QK, m-tiles of PV
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int ring_or_merge =
        Cfg::kRingBytes > static_cast<int>(sizeof(MergeSmem<D>)) ? Cfg::kRingBytes
                                                                 : static_cast<int>(sizeof(MergeSmem<D>));
    uint8_t* sK = smem;
    uint8_t* sV = smem + S * Cfg::kTileBytes;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + ring_or_merge);
    uint64_t* empty = full + S;
    MergeSmem<D>& ms = *reinterpret_cast<MergeSmem<D>*>(smem);

    const int c = blockIdx.x;
    const int kvh = blockIdx.y % p.Hkv;
    const int hg = blockIdx.y / p.Hkv;
    const int b = blockIdx.z;
    const int L = load_len(p.seq_lens, b, p.max_len, p.err);
    const Ranges R = visible_ranges(L, p.window, p.n_sink);
    int lo, hi;
    if (!chunk_bounds(R, p.chunk, c, lo, hi)) return;
    const int n_chunks = total_chunks(R, p.chunk);
    const int t0 = lo & ~(kTile - 1);
    const int n_tiles = (hi - t0 + kTile - 1) / kTile;
    const int G_cta = min(kMaxHP, p.G - hg * kMaxHP);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumers);
        }
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == kConsumers) {
        // ------------------------------------------------------------------ producer
        if (lane == 0) {
            prefetch_tensormap(&tmK);
            prefetch_tensormap(&tmV);
            const int bp = min(p.page_size, kTile);  // rows per TMA box
            for (int i = 0; i < n_tiles; ++i) {
                const int s = i % S;
                const uint32_t ph = (i / S) & 1;
                if (!mbar_wait(&empty[s], ph ^ 1, p.err)) break;
                mbar_arrive_expect_tx(&full[s], 2 * Cfg::kTileBytes);
                const int T = t0 + i * kTile;
                for (int sub = 0; sub < kTile / bp; ++sub) {
                    const int t = T + sub * bp;
                    const int tc = t < L ? t : L - 1;  // rows past the end: any valid page
                    const int pg = load_page(p.block_table, p.max_pages, p.num_pages, b,
                                             tc / p.page_size, p.err);
                    const int y = (pg * p.Hkv + kvh) * p.page_size + (t % p.page_size);
#pragma unroll
                    for (int box = 0; box < D / 64; ++box) {
                        const uint32_t off = box * kTile * 128 + sub * bp * 128;
                        tma_load_2d(sK + s * Cfg::kTileBytes + off, &tmK, &full[s], box * 64, y);
                        tma_load_2d(sV + s * Cfg::kTileBytes + off, &tmV, &full[s], box * 64, y);
                    }
                }
            }
        }
    } else {
        // ------------------------------------------------------------------ consumers
        // q^T fragments (B operand of the score mma): lane holds head n = lane/4 of each
        // 8-head tile, dims 16kk + 2(lane%4) + {0,1} and +8.
        uint32_t qf[NT][KT][2];
        const __nv_bfloat16* qb = reinterpret_cast<const __nv_bfloat16*>(p.q);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int hl = nt * 8 + lane / 4;
            const bool ok = hl < G_cta;
            const int hq = kvh * p.G + hg * kMaxHP + hl;
            const __nv_bfloat16* qr = qb + (static_cast<size_t>(b) * p.Hq + (ok ? hq : 0)) * D;
#pragma unroll
            for (int kk = 0; kk < KT; ++kk) {
                const int d0 = kk * 16 + 2 * (lane % 4);
                uint32_t lo2 = ok ? *reinterpret_cast<const uint32_t*>(qr + d0) : 0u;
                uint32_t hi2 = ok ? *reinterpret_cast<const uint32_t*>(qr + d0 + 8) : 0u;
                qf[nt][kk][0] = lo2;
                qf[nt][kk][1] = hi2;
            }
        }
        float oacc[KT][NT][4];
#pragma unroll
        for (int mt = 0; mt < KT; ++mt)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int r = 0; r < 4; ++r) oacc[mt][nt][r] = 0.f;
        float m_run[NT][2], l_run[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            m_run[nt][0] = m_run[nt][1] = neg_inf();
            l_run[nt][0] = l_run[nt][1] = 0.f;
        }
        const int r0 = warp * 16;
        const float sl2 = p.scale_log2;

        for (int i = 0; i < n_tiles; ++i) {
            const int s = i % S;
            const uint32_t ph = (i / S) & 1;
            if (!mbar_wait(&full[s], ph, p.err)) break;
            const int T = t0 + i * kTile;
            uint8_t* kt = sK + s * Cfg::kTileBytes;
            uint8_t* vt = sV + s * Cfg::kTileBytes;
            const bool partial = (T < lo) || (T + kTile > hi);
            if (partial) {
                // zero this warp's V rows outside [lo, hi) so that masked tokens add 0 * 0
                for (int idx = lane; idx < 16 * (D / 8); idx += 32) {
                    const int row = r0 + idx / (D / 8);
                    const int tok = T + row;
                    if (tok < lo || tok >= hi)
                        *reinterpret_cast<uint4*>(vt + swz128(row, (idx % (D / 8)) * 8, kTile)) =
                            make_uint4(0, 0, 0, 0);
                }
                __syncwarp();
            }
            // ---- scores: S^T[16 tok x 8 heads] per head tile
            float sacc[NT][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int r = 0; r < 4; ++r) sacc[nt][r] = 0.f;
            const uint32_t kbase = smem_u32(kt);
#pragma unroll
            for (int kk = 0; kk < KT; ++kk) {
                uint32_t a[4];
                ldsm_x4(kbase + swz128(r0 + (lane % 16), kk * 16 + (lane / 16) * 8, kTile), a);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) mma_bf16_16816(sacc[nt], a, qf[nt][kk][0], qf[nt][kk][1]);
            }
            // ---- online softmax over this warp's 16 tokens, per head column
            const int tokA = T + r0 + lane / 4, tokB = tokA + 8;
            const bool inA = tokA >= lo && tokA < hi, inB = tokB >= lo && tokB < hi;
            uint32_t pb[NT][2];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                float x0 = inA ? sacc[nt][0] * sl2 : neg_inf();
                float x1 = inA ? sacc[nt][1] * sl2 : neg_inf();
                float x2 = inB ? sacc[nt][2] * sl2 : neg_inf();
                float x3 = inB ? sacc[nt][3] * sl2 : neg_inf();
                float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
                for (int off = 4; off < 32; off <<= 1) {
                    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
                    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
                }
                const float mn0 = fmaxf(m_run[nt][0], mx0), mn1 = fmaxf(m_run[nt][1], mx1);
                const float mu0 = mn0 == neg_inf() ? 0.f : mn0;
                const float mu1 = mn1 == neg_inf() ? 0.f : mn1;
                const float al0 = fast_exp2(m_run[nt][0] - mu0), al1 = fast_exp2(m_run[nt][1] - mu1);
                m_run[nt][0] = mn0;
                m_run[nt][1] = mn1;
                const float p0 = fast_exp2(x0 - mu0), p1 = fast_exp2(x1 - mu1);
                const float p2 = fast_exp2(x2 - mu0), p3 = fast_exp2(x3 - mu1);
                l_run[nt][0] = l_run[nt][0] * al0 + p0 + p2;
                l_run[nt][1] = l_run[nt][1] * al1 + p1 + p3;
#pragma unroll
                for (int mt = 0; mt < KT; ++mt) {
                    oacc[mt][nt][0] *= al0;
                    oacc[mt][nt][1] *= al1;
                    oacc[mt][nt][2] *= al0;
                    oacc[mt][nt][3] *= al1;
                }
                // P^T as the B operand: transpose the two 8x8 (token x head) blocks
                pb[nt][0] = movmatrix_t(pack_bf16(p0, p1));
                pb[nt][1] = movmatrix_t(pack_bf16(p2, p3));
            }
            // ---- O^T[D x 8] += V^T[D x 16 tok] P^T
            const uint32_t vbase = smem_u32(vt);
#pragma unroll
            for (int mt = 0; mt < KT; ++mt) {
                uint32_t a[4];
                ldsm_x4_t(vbase + swz128(r0 + (lane % 8) + (lane / 16) * 8,
                                         mt * 16 + ((lane / 8) % 2) * 8, kTile),
                          a);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) mma_bf16_16816(oacc[mt][nt], a, pb[nt][0], pb[nt][1]);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
        }
        // row sums: reduce over the 8 lanes that share a head column
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int j = 0; j < 2; ++j)
#pragma unroll
                for (int off = 4; off < 32; off <<= 1)
                    l_run[nt][j] += __shfl_xor_sync(0xffffffffu, l_run[nt][j], off);
        // stash this warp's partial (after every warp is done with the ring)
        __syncwarp();
        asm volatile("bar.sync 1, %0;" ::"r"(kConsumers * 32));
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
            for (int mt = 0; mt < KT; ++mt) {
                const int d0 = mt * 16 + lane / 4;
                ms.o[warp][h0][d0] = oacc[mt][nt][0];
                ms.o[warp][h0 + 1][d0] = oacc[mt][nt][1];
                ms.o[warp][h0][d0 + 8] = oacc[mt][nt][2];
                ms.o[warp][h0 + 1][d0 + 8] = oacc[mt][nt][3];
            }
        }
    }
    __syncthreads();
    merge_and_combine<D>(p, ms, b, kvh, hg, c, n_chunks, G_cta);
}

// ---------------------------------------------------------------------------------------
// float32 kernel: plain loads, one token per warp step, exact fp32 FMA
// ---------------------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(kConsumers * 32)
    gqa_decode_f32_kernel(const GqaParams p) {
    constexpr int J = D / 32;  // dims per lane
    extern __shared__ uint8_t smem_raw[];
    MergeSmem<D>& ms = *reinterpret_cast<MergeSmem<D>*>(smem_raw);
    const int c = blockIdx.x;
    const int kvh = blockIdx.y % p.Hkv;
    const int hg = blockIdx.y / p.Hkv;
    const int b = blockIdx.z;
    const int L = load_len(p.seq_lens, b, p.max_len, p.err);
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
    merge_and_combine<D>(p, ms, b, kvh, hg, c, n_chunks, G_cta);
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
    using Cfg = GqaBf16Cfg<D>;
    auto kern = gqa_decode_bf16_kernel<D, NT>;
    static int configured = 0;
    if (!configured) {
        if (set_smem(kern, Cfg::kSmem) != KVD_OK) return KVD_ERR_CUDA;
        configured = 1;
    }
    dim3 grid(plan.max_chunks, p.Hkv * p.NHG, p.B);
    kern<<<grid, Cfg::kThreads, Cfg::kSmem, stream>>>(tk, tv, p);
    return cudaGetLastError() == cudaSuccess ? KVD_OK : KVD_ERR_CUDA;
}

template <int D>
int launch_f32(const GqaPlan& plan, const GqaParams& p, cudaStream_t stream) {
    auto kern = gqa_decode_f32_kernel<D>;
    const int bytes = static_cast<int>(sizeof(MergeSmem<D>));
    static int configured = 0;
    if (!configured) {
        if (set_smem(kern, bytes) != KVD_OK) return KVD_ERR_CUDA;
        configured = 1;
    }
    dim3 grid(plan.max_chunks, p.Hkv * p.NHG, p.B);
    kern<<<grid, kConsumers * 32, bytes, stream>>>(p);
    return cudaGetLastError() == cudaSuccess ? KVD_OK : KVD_ERR_CUDA;
}

}  // namespace

int gqa_stage_bytes(int D) { return D == 128 ? GqaBf16Cfg<128>::kSmem : GqaBf16Cfg<64>::kSmem; }

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
