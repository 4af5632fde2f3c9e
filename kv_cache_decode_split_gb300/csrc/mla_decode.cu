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
//     N = 256, K = 64 tokens; P in tensor memory, V read MN-major from the same tile).
// The exchange (32 KB per tile each way) is the slowest step, so two groups of four softmax
// warps take alternate tiles: while one group's partial scores drain to the partner, the
// other group runs its softmax. The running max passes from group to group through shared
// memory; it is only raised (and O rescaled in TMEM) when it grows by more than 2^8, so the
// common tile touches O only through the MMA. Score and value products are issued by two
// threads, so that a score product never waits behind a value product that waits for a
// softmax. Splits are merged by log-sum-exp in a small combine kernel.

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
constexpr int kStages = 3;
constexpr int kTileBox = kTok * 128;  // 8 KB: 64 tokens x 64 dims
constexpr int kStageBytes = kNBox * kTileBox;
// warps 0-7: softmax (group = warp / 4 takes tiles of that parity, TMEM lane quarter =
// warp % 4); warp 8: loads; warp 9: score products (and TMEM allocation); warp 10: value
// products; warp 11: score exchange
constexpr int kThreads = 12 * 32;
constexpr int kWarpLoad = 8, kWarpQK = 9, kWarpPV = 10, kWarpX = 11;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr float kLn2 = 0.6931471805599453f;

struct MlaSmem {
    uint8_t stage[kStages][kStageBytes];   // offset 0, 1024-aligned
    float x[2][kH][kTok];                  // the partner's partial scores, one slot per group
                                           // (16-byte chunks XOR-ed with row % 16)
    float y[kH][kTok];                     // this CTA's partial scores on their way out
    float mref[2][kH];                     // running max after each group's latest tile
    // Barriers waited by one group only exist once per group (tile parity), so that each
    // waiter goes through its barrier's phases in order.
    uint64_t full[kStages], empty[kStages], qready, sfull[2], sempty, pfull, pvdone[2], ofinal;
    uint64_t xfull[2];       // the partner's partial of a tile has arrived in x[parity]
    uint64_t xused[2];       // x[parity] has been read (four warps of that group)
    uint64_t peer_free[2];   // the partner has read our previous partial in its x[parity]
    uint64_t yfull, yfree[2];  // y written (four warps) / y read by the copy of a tile
    uint64_t hand[2];        // group published its running max
    uint32_t tmem_base;
};

// Tensor-memory columns (all 512): this CTA's query slice (bf16 pairs, up to 320 dims), one
// score tile, one P tile (bf16 pairs) and the 256-wide output accumulator.
constexpr uint32_t kColQ = 0, kColS = 160, kColP = 224, kColO = 256;
constexpr int kMlaSmem = static_cast<int>(sizeof(MlaSmem)) + 1024;
static_assert(kMlaSmem <= 227 * 1024, "MLA shared memory");

__device__ __forceinline__ float neg_inf() { return -__int_as_float(0x7f800000); }

// Score product of one tile: S (TMEM) = q_r (TMEM, NK 16-dim k-steps) x this CTA's
// 64-dim boxes of the tile (shared memory, K-major). Fully unrolled with the descriptors
// advanced by constants, so that one thread keeps the tensor pipe fed.
template <int NK>
__device__ __forceinline__ void issue_qk(uint32_t tmem, uint32_t tile_addr) {
    constexpr uint32_t idesc = idesc_bf16_f32(kH, kTok, 0, 0);
    const uint64_t bd = sw128_kmajor_desc(tile_addr);
#pragma unroll
    for (int ks = 0; ks < NK; ++ks)
        tc_mma_bf16_ts(tmem + kColS, tmem + kColQ + ks * 8,
                       bd + static_cast<uint64_t>(((ks >> 2) * kTileBox + (ks & 3) * 32) >> 4),
                       idesc, ks > 0 ? 1u : 0u);
}

// Value product of one tile: O_r (TMEM, 256 columns) += P (TMEM) x V_r, V_r being this
// CTA's first four boxes of the tile read MN-major (16 tokens x 256 dims per k-step).
__device__ __forceinline__ void issue_pv(uint32_t tmem, uint32_t tile_addr, bool accumulate) {
    constexpr uint32_t idesc = idesc_bf16_f32(kH, 256, 0, 1);
    const uint64_t bd = sw128_mnmajor_desc(tile_addr, kTileBox);
#pragma unroll
    for (int ks = 0; ks < kTok / 16; ++ks)
        tc_mma_bf16_ts(tmem + kColO, tmem + kColP + ks * 8,
                       bd + static_cast<uint64_t>((ks * 16 * 128) >> 4), idesc,
                       (accumulate || ks > 0) ? 1u : 0u);
}

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
    constexpr uint32_t kXBytes = kH * kTok * 4;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&sm.full[s], kSparse ? 32 : 1);
            mbar_init(&sm.empty[s], 1);
        }
        mbar_init(&sm.qready, 8);
        mbar_init(&sm.sempty, 4);  // the four warps of the group that owns the tile
        mbar_init(&sm.pfull, 4);
        mbar_init(&sm.yfull, 4);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sm.sfull[i], 1);
            mbar_init(&sm.pvdone[i], 1);
            mbar_init(&sm.xfull[i], 1);      // armed with the exchanged byte count each tile
            mbar_init(&sm.xused[i], 4);
            mbar_init(&sm.peer_free[i], 1);  // remote arrive by the partner's exchange thread
            mbar_init(&sm.yfree[i], 1);
            mbar_init(&sm.hand[i], 4);
        }
        mbar_init(&sm.ofinal, 1);
        fence_mbar_init();
        // the partner's partial scores of tiles 0 and 1 (later tiles: armed by the group
        // once the slot's previous phase has completed)
        for (int i = 0; i < 2 && i < n_tiles; ++i) mbar_arrive_expect_tx(&sm.xfull[i], kXBytes);
    }
    if (warp == kWarpQK) tmem_alloc(&sm.tmem_base, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    cluster_sync();  // the partner's barriers exist before anyone signals them
    const uint32_t tmem = sm.tmem_base;

    if (warp == kWarpLoad) {
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
    } else if (warp == kWarpQK) {
        // ------------------------------------------------------------------ score products
        // Tile j's product starts as soon as its data is in and tile j - 1's scores have been
        // read, independently of the value products.
        if (lane == 0) {
            bool ok = mbar_wait(&sm.qready, 0, p.err);
            for (int j = 0; j < n_tiles && ok; ++j) {
                const int s = j % kStages;
                ok = mbar_wait(&sm.full[s], (j / kStages) & 1, p.err) &&
                     mbar_wait(&sm.sempty, (j & 1) ^ 1, p.err);
                if (!ok) break;
                tc_fence_after();
                if (nbox == 4)
                    issue_qk<16>(tmem, smem_u32(sm.stage[s]));
                else
                    issue_qk<20>(tmem, smem_u32(sm.stage[s]));
                tc_commit(&sm.sfull[j & 1]);
            }
        }
    } else if (warp == kWarpPV) {
        // ------------------------------------------------------------------ value products
        if (lane == 0) {
            bool ok = true;
            for (int j = 0; j < n_tiles && ok; ++j) {
                const int s = j % kStages;
                if (!(ok = mbar_wait(&sm.pfull, j & 1, p.err))) break;
                tc_fence_after();
                issue_pv(tmem, smem_u32(sm.stage[s]), j > 0);
                tc_commit(&sm.pvdone[j & 1]);
                tc_commit(&sm.empty[s]);  // the tile's score product completed before its P
            }
            tc_commit(&sm.ofinal);
            mbar_wait(&sm.ofinal, 0, p.err);  // every value product of this CTA has completed
        }
    } else if (warp == kWarpX) {
        // ------------------------------------------------------------------ score exchange
        // One bulk copy per tile moves this CTA's partial scores (staged in y by the tile's
        // group) into the partner's slot for that tile's parity. The copies drain over
        // distributed shared memory at its own rate, off the softmax warps' instruction path.
        if (lane == 0) {
            uint32_t peer_x[2], peer_xfull[2], peer_free[2];
            for (int i = 0; i < 2; ++i) {
                peer_x[i] = map_peer(smem_u32(&sm.x[i][0][0]), peer);
                peer_xfull[i] = map_peer(smem_u32(&sm.xfull[i]), peer);
                peer_free[i] = map_peer(smem_u32(&sm.peer_free[i]), peer);
            }
            for (int j = 0; j < n_tiles; ++j) {
                const int xb = j & 1;
                // our x[xb] has been read for tile j - 2: the partner may send tile j into it
                if (j >= 2) {
                    if (!mbar_wait(&sm.xused[xb], ((j - 2) >> 1) & 1, p.err)) break;
                    mbar_arrive_remote_relaxed(peer_free[xb]);
                }
                if (!mbar_wait(&sm.yfull, j & 1, p.err)) break;
                if (!mbar_wait_cluster(&sm.peer_free[xb], ((j >> 1) & 1) ^ 1, p.err)) break;
                bulk_copy_to_peer(peer_x[xb], &sm.y[0][0], kXBytes, peer_xfull[xb]);
                bulk_wait_read_all();
                mbar_arrive(&sm.yfree[xb]);
            }
        }
    } else {
        // ------------------------------------------------------------------ softmax
        const int grp = warp >> 2;                 // takes tiles j with j % 2 == grp
        const int h = (warp & 3) * 32 + lane;      // head = TMEM lane
        const uint32_t trow = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
        {
            // this CTA's query slice into TMEM (the A operand of the score product): group 0
            // boxes 0-2, group 1 the rest
            const uint4* qrow = reinterpret_cast<const uint4*>(
                reinterpret_cast<const __nv_bfloat16*>(p.q) + (static_cast<size_t>(b) * kH + h) * kDqk +
                dim0);
            const int bx0 = grp == 0 ? 0 : 3, bx1 = grp == 0 ? 3 : nbox;
            uint4 v[3][8];
#pragma unroll
            for (int k = 0; k < 3; ++k)
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    if (bx0 + k < bx1) v[k][j] = __ldg(qrow + (bx0 + k) * 8 + j);
#pragma unroll
            for (int k = 0; k < 3; ++k) {
                if (bx0 + k >= bx1) break;
                uint32_t r[32];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    r[4 * j] = v[k][j].x;
                    r[4 * j + 1] = v[k][j].y;
                    r[4 * j + 2] = v[k][j].z;
                    r[4 * j + 3] = v[k][j].w;
                }
                tmem_st_32x32b_x32(trow + kColQ + (bx0 + k) * 32, r);
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.qready);
        }
        const float sl2 = p.scale_log2;
        float l = 0.f, m_l = neg_inf();  // this group's sum of P, relative to 2^m_l
        float m_last = neg_inf();        // running max after this group's latest tile
        bool ok = true;
        for (int j = grp; j < n_tiles && ok; j += 2) {
            const int it = j >> 1;  // this group's iteration
            // 1. this CTA's partial scores; reading them frees S for tile j + 1's product
            if (!(ok = mbar_wait(&sm.sfull[grp], it & 1, p.err))) break;
            tc_fence_after();
            float s[kTok];
            {
                uint32_t r0[32], r1[32];
                tmem_ld_32x32b_x32(trow + kColS, r0);
                tmem_ld_32x32b_x32(trow + kColS + 32, r1);
                tmem_ld_wait(r0);
                tmem_ld_wait(r1);
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    s[c] = __uint_as_float(r0[c]);
                    s[32 + c] = __uint_as_float(r1[c]);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.sempty);
            // 2. stage them for the exchange thread once tile j - 1's copy has read y
            if (j >= 1 && !(ok = mbar_wait(&sm.yfree[grp ^ 1], ((j - 1) >> 1) & 1, p.err))) break;
#pragma unroll
            for (int c4 = 0; c4 < kTok / 4; ++c4)
                *reinterpret_cast<float4*>(&sm.y[h][(c4 ^ (h & 15)) * 4]) =
                    make_float4(s[4 * c4], s[4 * c4 + 1], s[4 * c4 + 2], s[4 * c4 + 3]);
            fence_proxy_async_smem();  // generic stores before the bulk copy reads them
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.yfull);
            // 3. the partner's partial
            if (!(ok = mbar_wait_cluster(&sm.xfull[grp], it & 1, p.err))) break;
#pragma unroll
            for (int c4 = 0; c4 < kTok / 4; ++c4) {
                const float4 v = *reinterpret_cast<const float4*>(&sm.x[grp][h][(c4 ^ (h & 15)) * 4]);
                s[4 * c4] += v.x;
                s[4 * c4 + 1] += v.y;
                s[4 * c4 + 2] += v.z;
                s[4 * c4 + 3] += v.w;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.xused[grp]);
            // the slot's phase is complete: arm it for this group's next tile
            if (warp == 4 * grp && lane == 0 && j + 2 < n_tiles)
                mbar_arrive_expect_tx(&sm.xfull[grp], kXBytes);
            // 4. tile max, then the running max handed over from tile j - 1
            const int T0 = lo + j * kTok;
            float mt = neg_inf();
#pragma unroll
            for (int c = 0; c < kTok; ++c) {
                s[c] = (T0 + c < hi) ? s[c] * sl2 : neg_inf();
                mt = fmaxf(mt, s[c]);
            }
            float m_prev = neg_inf();
            if (j >= 1) {
                if (!(ok = mbar_wait(&sm.hand[grp ^ 1], ((j - 1) >> 1) & 1, p.err))) break;
                m_prev = sm.mref[grp ^ 1][h];
            }
            // raise the reference only on the first tile or when the max grows by > 2^8
            float m_new = m_prev;
            bool resc = false;
            if (mt > m_prev) {
                if (m_prev == neg_inf()) {
                    m_new = mt;
                } else if (mt > m_prev + kRescaleThreshold) {
                    m_new = mt;
                    resc = true;
                }
            }
            sm.mref[grp][h] = m_new;
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.hand[grp]);
            m_last = m_new;
            // 5. P relative to 2^m_new, and this group's running sum moved to that reference
            if (m_new != m_l) {
                if (l > 0.f) l *= fast_exp2(m_l - m_new);
                m_l = m_new;
            }
            const float mu = m_new == neg_inf() ? 0.f : m_new;
            uint32_t pk[kTok / 2];
            float psum = 0.f;
#pragma unroll
            for (int c = 0; c < kTok / 2; ++c) {
                const __nv_bfloat162 v =
                    __floats2bfloat162_rn(fast_exp2(s[2 * c] - mu), fast_exp2(s[2 * c + 1] - mu));
                const float2 f = __bfloat1622float2(v);
                psum += f.x + f.y;
                pk[c] = *reinterpret_cast<const uint32_t*>(&v);
            }
            l += psum;
            // 6. P (and O) are free once tile j - 1's value product has completed
            if (j >= 1 && !(ok = mbar_wait(&sm.pvdone[grp ^ 1], ((j - 1) >> 1) & 1, p.err))) break;
            tc_fence_after();
            if (__any_sync(0xffffffffu, resc)) {
                // rare: O was accumulated relative to 2^m_prev
                const float alpha = resc ? fast_exp2(m_prev - m_new) : 1.f;
#pragma unroll 1
                for (int c = 0; c < 8; ++c) {
                    uint32_t r[32];
                    tmem_ld_32x32b_x32(trow + kColO + c * 32, r);
                    tmem_ld_wait(r);
#pragma unroll
                    for (int k = 0; k < 32; ++k) r[k] = __float_as_uint(__uint_as_float(r[k]) * alpha);
                    tmem_st_32x32b_x32(trow + kColO + c * 32, r);
                }
            }
            tmem_st_32x32b_x32(trow + kColP, pk);  // P row: 64 bf16
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.pfull);
        }
        // the split's partial: O / l for this CTA's 256 value dims, and log2-sum-exp. The
        // final reference is the running max after the last tile.
        const int jl = n_tiles - 1;
        if (ok && (jl & 1) != grp) {
            ok = mbar_wait(&sm.hand[grp ^ 1], (jl >> 1) & 1, p.err);
            if (ok) m_last = sm.mref[grp ^ 1][h];
        }
        // both groups' sums relative to 2^m_last, added through shared memory (the exchange
        // slots are no longer written by the partner once its last partial has arrived)
        float* lsum = &sm.x[0][0][0];
        lsum[grp * kH + h] = (l > 0.f) ? l * fast_exp2(m_l - m_last) : 0.f;
        asm volatile("bar.sync 1, %0;" ::"r"(8 * 32) : "memory");
        const float l_tot = lsum[h] + lsum[kH + h];
        if (ok && mbar_wait(&sm.ofinal, 0, p.err)) {
            tc_fence_after();
            const float inv = l_tot > 0.f ? 1.f / l_tot : 0.f;
            float* po = p.part_o + (static_cast<size_t>(unit) * kH + h) * kDv + rank * 256;
            // group g writes value dims 128 g .. 128 g + 127 of this CTA's half
            for (int c = 4 * grp; c < 4 * grp + 4; ++c) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(trow + kColO + c * 32, r);
                tmem_ld_wait(r);
#pragma unroll
                for (int k = 0; k < 32; k += 4)
                    __stcg(reinterpret_cast<float4*>(po + c * 32 + k),
                           make_float4(__uint_as_float(r[k]) * inv, __uint_as_float(r[k + 1]) * inv,
                                       __uint_as_float(r[k + 2]) * inv,
                                       __uint_as_float(r[k + 3]) * inv));
            }
            if (rank == 0 && grp == 0)
                p.part_lse[static_cast<size_t>(unit) * kH + h] =
                    l_tot > 0.f ? m_last + log2f(l_tot) : neg_inf();
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    cluster_sync();  // the partner is done with this CTA's shared memory
    if (warp == kWarpQK) tmem_dealloc(tmem, 512);
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
