// mla_decode.cu -- absorbed-latent MLA decode (DeepSeek-V3 shapes: 128 heads, one 576-wide
// row per cached token, value = its first 512 entries), over all cached tokens or over the
// tokens a DSA selection kept.
//
// What is computed ("Attention Optimizations", DSA / Computation Path; "Overview of
// Attention Mechanism", MLA: W^UK folded into the query, W^UV into the output):
//   s_{h,t} = scale * q_h . c_t   (576 dims),   o_h = sum_t softmax_t(s_{h,.}) c_t[0:512].
//
// How (GB300): a cluster of two CTAs per work unit (one sequence, one split of its tokens).
// The 128 x 512 fp32 output accumulator alone fills a CTA's tensor memory, so the pair
// splits the work without repeating any of it:
//   * CTA 0 holds q[:, 0:256] and loads dims 0-255 of every latent row; CTA 1 holds
//     q[:, 256:576] and loads dims 256-575. Each row is read from memory once.
//   * Each CTA computes a partial score tile S_r = q_r C_r^T (tcgen05, M = 128 heads,
//     N = 64 tokens, fp32 in TMEM), and the two exchange their partials through
//     distributed shared memory. Float addition is commutative, so both CTAs hold the
//     bit-identical full tile and run the same online softmax.
//   * Each CTA accumulates its half of the value dims, O_r += P V_r (tcgen05, M = 128,
//     N = 256, K = 64 tokens; P in shared memory, V read MN-major from the same tile).
// The running max is only raised (and O rescaled in TMEM) when it grows by more than 2^8,
// so the common tile touches O only through the MMA. Splits are merged by log-sum-exp in
// a small combine kernel.

#include <algorithm>

#include "kvd_device.cuh"
#include "kvd_host.h"

namespace kvd {

namespace {

constexpr int kH = 128;               // heads (MMA M)
constexpr int kDqk = 576;
constexpr int kDv = 512;
constexpr int kTok = 64;              // tokens per tile
constexpr int kNBox = 5;              // 64-dim boxes held per CTA (rank 0 uses 4)
constexpr int kStages = 4;
constexpr int kTileBox = kTok * 128;  // 8 KB: 64 tokens x 64 dims
constexpr int kStageBytes = kNBox * kTileBox;
constexpr int kThreads = 6 * 32;      // warps 0-3 softmax, 4 loads, 5 MMA
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr float kLn2 = 0.6931471805599453f;

struct MlaSmem {
    uint8_t stage[kStages][kStageBytes];   // offset 0, 1024-aligned
    float x[2][kH][kTok];                  // the partner's partial scores (float4-swizzled)
    uint64_t full[kStages], empty[kStages], qready, sfull, sempty, xfull[2], peer_free[2], pfull,
        pvdone, ofinal;
    uint32_t tmem_base;
};

// Tensor-memory columns (all 512): this CTA's query slice (bf16 pairs, up to 320 dims), one
// score tile, one P tile (bf16 pairs) and the 256-wide output accumulator.
constexpr uint32_t kColQ = 0, kColS = 160, kColP = 224, kColO = 256;
constexpr int kMlaSmem = static_cast<int>(sizeof(MlaSmem)) + 1024;
static_assert(kMlaSmem <= 227 * 1024, "MLA shared memory");

__device__ __forceinline__ float neg_inf() { return -__int_as_float(0x7f800000); }

template <bool kSparse>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    mla_decode_kernel(const __grid_constant__ CUtensorMap tmC0,
                      const __grid_constant__ CUtensorMap tmC1,
                      const __grid_constant__ CUtensorMap tmC2, const MlaParams p) {
    extern __shared__ uint8_t smem_raw[];
    MlaSmem& sm = *reinterpret_cast<MlaSmem*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t rank = cluster_rank();
    const uint32_t peer = rank ^ 1u;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int unit = blockIdx.x >> 1;
    const int b = unit / p.n_splits, split = unit % p.n_splits;
    const int L = load_len(p.seq_lens, b, p.max_len, rank == 0 ? p.err : nullptr);
    int n_items = L;
    if (kSparse) n_items = min(max(p.idx_count[b], 0), p.idx_stride);
    const int lo = split * p.chunk;
    const int hi = min(n_items, lo + p.chunk);
    if (lo >= hi) return;  // both CTAs of the pair take this exit together
    const int n_tiles = (hi - lo + kTok - 1) / kTok;
    const int nbox = rank == 0 ? 4 : 5;   // 64-dim boxes this CTA loads
    const int dim0 = rank == 0 ? 0 : 256;
    const CUtensorMap& tmC = rank == 0 ? tmC0 : tmC1;  // 3-D maps with 4 / 5 blocks per box

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&sm.full[s], kSparse ? 32 : 1);
            mbar_init(&sm.empty[s], 1);
        }
        mbar_init(&sm.qready, 4);
        mbar_init(&sm.sfull, 1);
        mbar_init(&sm.sempty, 4);
        mbar_init(&sm.pfull, 4);
        mbar_init(&sm.pvdone, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sm.xfull[i], 1);      // armed with the exchanged byte count each tile
            mbar_init(&sm.peer_free[i], 4);  // one arrive per softmax warp of the partner
        }
        mbar_init(&sm.ofinal, 1);
        fence_mbar_init();
    }
    if (warp == 5) tmem_alloc(&sm.tmem_base, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    cluster_sync();  // the partner's barriers exist before anyone signals them
    const uint32_t tmem = sm.tmem_base;

    if (warp == 4) {
        // ------------------------------------------------------------------ loads
        if (!kSparse) {
            if (lane == 0) {
                prefetch_tensormap(&tmC);
                prefetch_tensormap(&tmC2);
                const int bp = min(p.page_size, kTok);
                for (int i = 0; i < n_tiles; ++i) {
                    const int s = i % kStages;
                    if (!mbar_wait(&sm.empty[s], ((i / kStages) & 1) ^ 1, p.err)) break;
                    mbar_arrive_expect_tx(&sm.full[s], nbox * kTileBox);
                    const int T = lo + i * kTok;
                    for (int sub = 0; sub < kTok / bp; ++sub) {
                        const int t = T + sub * bp;
                        const int tc = t < L ? t : L - 1;
                        const int pg = load_page(p.block_table, p.max_pages, p.num_pages, b,
                                                 tc / p.page_size, p.err);
                        const int y = pg * p.page_size + (t % p.page_size);
                        if (bp == kTok) {
                            // all of this CTA's 64-dim blocks in one instruction
                            tma_load_3d(sm.stage[s], &tmC, &sm.full[s], 0, y, dim0 / 64);
                        } else {
                            for (int bx = 0; bx < nbox; ++bx)
                                tma_load_2d(sm.stage[s] + bx * kTileBox + sub * bp * 128, &tmC2,
                                            &sm.full[s], dim0 + 64 * bx, y);
                        }
                    }
                }
                const int first = n_tiles > kStages ? n_tiles - kStages : 0;
                for (int i = first; i < n_tiles; ++i)
                    mbar_wait(&sm.full[i % kStages], (i / kStages) & 1, p.err);
            }
        } else {
            // gather the selected rows: each lane copies rows lane and lane + 32 of the tile
            const __nv_bfloat16* cpool = reinterpret_cast<const __nv_bfloat16*>(p.c_pool);
            const int32_t* idx = p.idx + static_cast<size_t>(b) * p.idx_stride;
            bool ok = true;
            for (int i = 0; i < n_tiles; ++i) {
                const int s = i % kStages;
                if (lane == 0) ok = mbar_wait(&sm.empty[s], ((i / kStages) & 1) ^ 1, p.err);
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
                const uint32_t base = smem_u32(sm.stage[s]);
                for (int rr = 0; rr < 2; ++rr) {
                    const int r = lane + 32 * rr;
                    const int j = lo + i * kTok + r;
                    int t = j < hi ? idx[j] : -1;
                    bool valid = t >= 0 && t < L;
                    if (j < hi && !valid) record_error(p.err, KVD_ERR_DEVICE_OOB);
                    const __nv_bfloat16* src = cpool;
                    if (valid) {
                        const int pg = load_page(p.block_table, p.max_pages, p.num_pages, b,
                                                 t / p.page_size, p.err);
                        src = cpool + (static_cast<size_t>(pg) * p.page_size + t % p.page_size) *
                                          kDqk + dim0;
                    }
                    for (int c = 0; c < nbox * 8; ++c) {
                        const int bx = c >> 3, cc = c & 7;
                        const uint32_t dst = base + bx * kTileBox + r * 128 + ((cc ^ (r & 7)) << 4);
                        cp_async_16(dst, valid ? src + c * 8 : cpool, valid ? 16u : 0u);
                    }
                }
                cp_async_commit();
                if (i >= 1) {
                    cp_async_wait<1>();
                    fence_proxy_async_smem();
                    mbar_arrive(&sm.full[(i - 1) % kStages]);
                }
            }
            if (ok) {
                cp_async_wait<0>();
                fence_proxy_async_smem();
                mbar_arrive(&sm.full[(n_tiles - 1) % kStages]);
            } else {
                cp_async_wait<0>();
            }
        }
    } else if (warp == 5) {
        // ------------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_qk = idesc_bf16_f32(kH, kTok, 0, 0);
            constexpr uint32_t idesc_pv = idesc_bf16_f32(kH, 256, 0, 1);
            const int nk = nbox * 4;  // 16-dim k-steps of the score product
            bool ok = mbar_wait(&sm.qready, 0, p.err);
            auto qk = [&](int i) {
                const int s = i % kStages;
                ok = ok && mbar_wait(&sm.full[s], (i / kStages) & 1, p.err);
                ok = ok && mbar_wait(&sm.sempty, (i & 1) ^ 1, p.err);
                if (!ok) return;
                tc_fence_after();
                const uint32_t ca = smem_u32(sm.stage[s]);
                for (int ks = 0; ks < nk; ++ks) {
                    const uint64_t bd =
                        sw128_kmajor_desc(ca + (ks >> 2) * kTileBox + (ks & 3) * 32);
                    tc_mma_bf16_ts(tmem + kColS, tmem + kColQ + ks * 8, bd, idesc_qk,
                                   ks > 0 ? 1u : 0u);
                }
                tc_commit(&sm.sfull);
            };
            auto pv = [&](int i) {
                const int s = i % kStages;
                ok = ok && mbar_wait(&sm.pfull, i & 1, p.err);
                if (!ok) return;
                tc_fence_after();
                const uint32_t va = smem_u32(sm.stage[s]);
                for (int ks = 0; ks < kTok / 16; ++ks) {
                    const uint64_t bd = sw128_mnmajor_desc(va + ks * 16 * 128, kTileBox);
                    tc_mma_bf16_ts(tmem + kColO, tmem + kColP + ks * 8, bd, idesc_pv,
                                   (i > 0 || ks > 0) ? 1u : 0u);
                }
                tc_commit(&sm.pvdone);
                tc_commit(&sm.empty[s]);
            };
            // The softmax warps read score tile j + 1 (and send it to the partner) before
            // they finish tile j, so the score product runs two tiles ahead of the value
            // product: tile j + 2's scores are issued as soon as tile j + 1's have been read,
            // and overlap the exchange and softmax of tile j.
            qk(0);
            if (n_tiles > 1) qk(1);
            for (int j = 0; j < n_tiles; ++j) {
                if (j + 2 < n_tiles) qk(j + 2);
                pv(j);
            }
            tc_commit(&sm.ofinal);
            mbar_wait(&sm.ofinal, 0, p.err);  // every MMA of this CTA has completed
        }
    } else {
        // ------------------------------------------------------------------ softmax
        const int h = threadIdx.x;  // head = TMEM lane
        const uint32_t trow = tmem + (static_cast<uint32_t>(warp * 32) << 16);
        {
            // this CTA's query slice into TMEM (the A operand of the score product)
            const uint4* qrow = reinterpret_cast<const uint4*>(
                reinterpret_cast<const __nv_bfloat16*>(p.q) + (static_cast<size_t>(b) * kH + h) * kDqk +
                dim0);
            // 64 dims (32 columns) per box; the loads of up to three boxes are in flight at once
            for (int c0 = 0; c0 < nbox; c0 += 3) {
                uint4 v[3][8];
#pragma unroll
                for (int bx = 0; bx < 3; ++bx)
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        if (c0 + bx < nbox) v[bx][j] = __ldg(qrow + (c0 + bx) * 8 + j);
#pragma unroll
                for (int bx = 0; bx < 3; ++bx) {
                    if (c0 + bx >= nbox) break;
                    uint32_t r[32];
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        r[4 * j] = v[bx][j].x;
                        r[4 * j + 1] = v[bx][j].y;
                        r[4 * j + 2] = v[bx][j].z;
                        r[4 * j + 3] = v[bx][j].w;
                    }
                    tmem_st_32x32b_x32(trow + kColQ + (c0 + bx) * 32, r);
                }
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.qready);
        }
        // Tile j's partial score row is read (freeing the score tile for the next product)
        // and sent to the partner one tile ahead of combining tile j - 1, so the exchange
        // latency overlaps the previous tile's softmax.
        const uint32_t peer_x0 = map_peer(smem_u32(&sm.x[0][h][0]), peer);
        const uint32_t peer_x1 = map_peer(smem_u32(&sm.x[1][h][0]), peer);
        const uint32_t peer_xfull0 = map_peer(smem_u32(&sm.xfull[0]), peer);
        const uint32_t peer_xfull1 = map_peer(smem_u32(&sm.xfull[1]), peer);
        const uint32_t peer_free0 = map_peer(smem_u32(&sm.peer_free[0]), peer);
        const uint32_t peer_free1 = map_peer(smem_u32(&sm.peer_free[1]), peer);
        const float sl2 = p.scale_log2;
        float m_ref = neg_inf(), l = 0.f;
        bool ok = true;
        auto send = [&](int j, float (&s)[kTok]) -> bool {
            const int xb = j & 1;
            if (!mbar_wait(&sm.sfull, j & 1, p.err)) return false;
            tc_fence_after();
            {
                uint32_t r[32];
                tmem_ld_32x32b_x32(trow + kColS, r);
                tmem_ld_wait(r);
#pragma unroll
                for (int c = 0; c < 32; ++c) s[c] = __uint_as_float(r[c]);
                tmem_ld_32x32b_x32(trow + kColS + 32, r);
                tmem_ld_wait(r);
#pragma unroll
                for (int c = 0; c < 32; ++c) s[32 + c] = __uint_as_float(r[c]);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.sempty);  // the score tile may be overwritten
            if (h == 0) mbar_arrive_expect_tx(&sm.xfull[xb], kH * kTok * 4);
            if (!mbar_wait_cluster(&sm.peer_free[xb], ((j >> 1) & 1) ^ 1, p.err)) return false;
            const uint32_t px = xb ? peer_x1 : peer_x0;
            const uint32_t pf = xb ? peer_xfull1 : peer_xfull0;
#pragma unroll
            for (int c4 = 0; c4 < kTok / 4; ++c4)
                st_async_v4(px + ((c4 ^ (h & 15)) << 4), s[4 * c4], s[4 * c4 + 1], s[4 * c4 + 2],
                            s[4 * c4 + 3], pf);
            return true;
        };
        float s[kTok];
        ok = send(0, s);
        for (int i = 0; i < n_tiles && ok; ++i) {
            float sn[kTok];
            if (i + 1 < n_tiles && !(ok = send(i + 1, sn))) break;
            const int xb = i & 1;
            if (!(ok = mbar_wait_cluster(&sm.xfull[xb], (i >> 1) & 1, p.err))) break;
#pragma unroll
            for (int c4 = 0; c4 < kTok / 4; ++c4) {
                const float4 v = *reinterpret_cast<const float4*>(&sm.x[xb][h][(c4 ^ (h & 15)) * 4]);
                s[4 * c4] += v.x;
                s[4 * c4 + 1] += v.y;
                s[4 * c4 + 2] += v.z;
                s[4 * c4 + 3] += v.w;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive_remote(xb ? peer_free1 : peer_free0);  // slot read
            // online softmax in log2 units, lazily rescaled
            const int T0 = lo + i * kTok;
            float mt = neg_inf();
#pragma unroll
            for (int j = 0; j < kTok; ++j) {
                s[j] = (T0 + j < hi) ? s[j] * sl2 : neg_inf();
                mt = fmaxf(mt, s[j]);
            }
            bool resc = false;
            float alpha = 1.f;
            if (mt > m_ref) {
                if (m_ref == neg_inf()) {
                    m_ref = mt;
                } else if (mt > m_ref + kRescaleThreshold) {
                    alpha = fast_exp2(m_ref - mt);
                    m_ref = mt;
                    l *= alpha;
                    resc = true;
                }
            }
            const float mu = m_ref == neg_inf() ? 0.f : m_ref;
            uint32_t pk[kTok / 2];
            float psum = 0.f;
#pragma unroll
            for (int j = 0; j < kTok / 2; ++j) {
                const __nv_bfloat162 v =
                    __floats2bfloat162_rn(fast_exp2(s[2 * j] - mu), fast_exp2(s[2 * j + 1] - mu));
                const float2 f = __bfloat1622float2(v);
                psum += f.x + f.y;
                pk[j] = *reinterpret_cast<const uint32_t*>(&v);
            }
            l += psum;
            // the P tile (and O) are free once tile i - 1's value product has completed
            if (i >= 1 && !(ok = mbar_wait(&sm.pvdone, (i - 1) & 1, p.err))) break;
            tc_fence_after();
            if (__any_sync(0xffffffffu, resc)) {
                for (int c = 0; c < 8; ++c) {
                    uint32_t r[32];
                    tmem_ld_32x32b_x32(trow + kColO + c * 32, r);
                    tmem_ld_wait(r);
#pragma unroll
                    for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * alpha);
                    tmem_st_32x32b_x32(trow + kColO + c * 32, r);
                }
            }
            tmem_st_32x32b_x32(trow + kColP, pk);  // P row: 64 bf16
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.pfull);
#pragma unroll
            for (int j = 0; j < kTok; ++j) s[j] = sn[j];
        }
        // the split's partial: O / l for this CTA's 256 value dims, and log2-sum-exp
        if (ok && mbar_wait(&sm.ofinal, 0, p.err)) {
            tc_fence_after();
            const float inv = l > 0.f ? 1.f / l : 0.f;
            float* po = p.part_o + (static_cast<size_t>(unit) * kH + h) * kDv + rank * 256;
            for (int c = 0; c < 8; ++c) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(trow + kColO + c * 32, r);
                tmem_ld_wait(r);
#pragma unroll
                for (int j = 0; j < 32; j += 4)
                    __stcg(reinterpret_cast<float4*>(po + c * 32 + j),
                           make_float4(__uint_as_float(r[j]) * inv, __uint_as_float(r[j + 1]) * inv,
                                       __uint_as_float(r[j + 2]) * inv,
                                       __uint_as_float(r[j + 3]) * inv));
            }
            if (rank == 0)
                p.part_lse[static_cast<size_t>(unit) * kH + h] = l > 0.f ? m_ref + log2f(l) : neg_inf();
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    cluster_sync();  // the partner is done with this CTA's shared memory
    if (warp == 5) tmem_dealloc(tmem, 512);
}

// Merge the splits of each (sequence, head): o = sum_s 2^{lse_s - M} o_s / sum_s 2^{lse_s - M}.
// Two heads per block; each thread owns four value dims and streams every split.
__global__ void __launch_bounds__(256) mla_combine_kernel(const MlaParams p, __nv_bfloat16* out,
                                                          float* lse_out) {
    const int b = blockIdx.x / (kH / 2);
    const int h = (blockIdx.x % (kH / 2)) * 2 + threadIdx.x / 128;
    const int d = (threadIdx.x % 128) * 4;
    const int L = load_len(p.seq_lens, b, p.max_len, nullptr);
    const int n_items = p.sparse ? min(max(p.idx_count[b], 0), p.idx_stride) : L;
    const int ns = min(p.n_splits, (n_items + p.chunk - 1) / p.chunk);
    const size_t u0 = static_cast<size_t>(b) * p.n_splits;
    const float* lse = p.part_lse + u0 * kH + h;
    float M = neg_inf();
    for (int s = 0; s < ns; ++s) M = fmaxf(M, lse[s * kH]);
    float den = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
    for (int s = 0; s < ns; ++s) {
        const float w = (M == neg_inf()) ? 0.f : fast_exp2(lse[s * kH] - M);
        den += w;
        const float4 v = __ldcg(reinterpret_cast<const float4*>(p.part_o + ((u0 + s) * kH + h) * kDv + d));
        acc.x += w * v.x;
        acc.y += w * v.y;
        acc.z += w * v.z;
        acc.w += w * v.w;
    }
    const float inv = den > 0.f ? 1.f / den : 0.f;
    __nv_bfloat162 lo2 = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
    __nv_bfloat162 hi2 = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
    uint2 pk = make_uint2(*reinterpret_cast<uint32_t*>(&lo2), *reinterpret_cast<uint32_t*>(&hi2));
    *reinterpret_cast<uint2*>(out + (static_cast<size_t>(b) * kH + h) * kDv + d) = pk;
    if (d == 0 && lse_out)
        lse_out[static_cast<size_t>(b) * kH + h] = den > 0.f ? (M + log2f(den)) * kLn2 : neg_inf();
}

}  // namespace

int mla_launch(const MlaParams& p, const CUtensorMap& tc0, const CUtensorMap& tc1,
               const CUtensorMap& tc2, void* out, float* lse_out, cudaStream_t stream) {
    static int configured[2] = {0, 0};
    const int which = p.sparse ? 1 : 0;
    if (!configured[which]) {
        const cudaError_t e =
            p.sparse ? cudaFuncSetAttribute(mla_decode_kernel<true>,
                                            cudaFuncAttributeMaxDynamicSharedMemorySize, kMlaSmem)
                     : cudaFuncSetAttribute(mla_decode_kernel<false>,
                                            cudaFuncAttributeMaxDynamicSharedMemorySize, kMlaSmem);
        if (e != cudaSuccess) return KVD_ERR_CUDA;
        configured[which] = 1;
    }
    const int grid = 2 * p.B * p.n_splits;
    if (p.sparse)
        mla_decode_kernel<true><<<grid, kThreads, kMlaSmem, stream>>>(tc0, tc1, tc2, p);
    else
        mla_decode_kernel<false><<<grid, kThreads, kMlaSmem, stream>>>(tc0, tc1, tc2, p);
    mla_combine_kernel<<<p.B * (kH / 2), 256, 0, stream>>>(p, static_cast<__nv_bfloat16*>(out),
                                                            lse_out);
    return cudaGetLastError() == cudaSuccess ? KVD_OK : KVD_ERR_CUDA;
}

}  // namespace kvd
