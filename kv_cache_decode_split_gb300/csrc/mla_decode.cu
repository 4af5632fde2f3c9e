// mla_decode.cu -- absorbed-latent MLA decode (DeepSeek-V3 shapes: 128 heads, one 576-wide
// row per cached token, value = its first 512 entries), over all cached tokens or over the
// tokens a DSA selection kept.
//
// What is computed ("Attention Optimizations", DSA / Computation Path; "Overview of
// Attention Mechanism", MLA: W^UK folded into the query, W^UV into the output):
//   s_{h,t} = scale * q_h . c_t   (576 dims),   o_h = sum_t softmax_t(s_{h,.}) c_t[0:512].
//
// How (GB300): a persistent grid of two-CTA clusters. All sequences' 64-token tiles form
// one list, cut into equal contiguous ranges, one per cluster; a range that spans several
// sequences is processed as one piece per sequence, each writing its own partial.
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
// softmax. Pieces are merged by log-sum-exp in a small combine kernel.

#include <algorithm>

#include "mla_common.cuh"

namespace kvd {

namespace {

using namespace mla;

constexpr int kTok = 64;              // tokens per tile
constexpr int kNBox = 5;              // 64-dim boxes held per CTA (rank 0 uses 4)
constexpr int kStages = 4;
constexpr int kTileBox = kTok * 128;  // 8 KB: 64 tokens x 64 dims
constexpr int kStageBytes = kNBox * kTileBox;
// warps 0-7: softmax (group = warp / 4 takes tiles of that parity, TMEM lane quarter =
// warp % 4); warp 8: loads; warp 9: score products (and TMEM allocation); warp 10: value
// products; warp 11: score exchange
constexpr int kGroups = 3;  // softmax warp groups, taking tiles j with j % kGroups == group
constexpr int kSoftWarps = 4 * kGroups;
constexpr int kThreads = (kSoftWarps + 4) * 32;
constexpr int kWarpLoad = kSoftWarps, kWarpQK = kSoftWarps + 1, kWarpPV = kSoftWarps + 2,
              kWarpX = kSoftWarps + 3;

struct MlaSmem {
    uint8_t stage[kStages][kStageBytes];   // offset 0, 1024-aligned
    // Partial scores cross in two halves of 32 columns (16 KB each), so that the next
    // tile's first half can follow the current tile's second half without a gap.
    float x[2][kH][kTok / 2];              // the partner's halves, one slot per half (16-byte
                                           // chunks XOR-ed with row % 8)
    float y[2][kH][kTok / 2];              // this CTA's halves on their way out
    float mref[kGroups][kH];               // running max after each group's latest tile; at
                                           // the end of a piece: each group's row sum
    // Barriers waited by one group only exist once per group (tile parity), so that each
    // waiter goes through its barrier's phases in order.
    uint64_t full[kStages], empty[kStages], qready, sfull[kGroups], sempty, pfull,
        pvdone[kGroups], ofinal;
    uint64_t xfull[2][kGroups];  // [half][tile group]: the partner's half has arrived
    uint64_t peer_free[2];   // the partner has read our previous half in its x[half] (remote
                             // arrives by the four warps of the partner's group)
    uint64_t yfull[2];       // y[half] written (four warps of the tile's group)
    uint64_t yfree[2][kGroups];  // [half][tile group]: the copy of y[half] has read it
    uint64_t hand[kGroups];  // group published its running max
    uint64_t ofree;          // O of the current piece has been read (eight softmax warps)
    uint64_t qfull;          // the first piece's queries have landed in stages 2-3
    uint64_t qkend, pvend;   // every product the score / value issuer started has completed
    uint32_t tmem_base;
    Sched sched;             // the cluster's tile range and pieces, built once
};

// Tensor-memory columns (all 512): this CTA's query slice (bf16 pairs, up to 320 dims), one
// score tile, one P tile (bf16 pairs) and the 256-wide output accumulator.
constexpr uint32_t kColQ = 0, kColS = 160, kColP = 224, kColO = 256;
// No alignment slack fits: the dynamic shared memory window starts 1024-byte aligned when
// the kernel declares no static shared memory (checked at run time).
constexpr int kMlaSmem = static_cast<int>(sizeof(MlaSmem));
static_assert(kMlaSmem <= 227 * 1024, "MLA shared memory");

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
                      const __grid_constant__ CUtensorMap tmC2,
                      const __grid_constant__ CUtensorMap tmQ, const MlaParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    MlaSmem& sm = *reinterpret_cast<MlaSmem*>(smem_raw);
    const uint32_t rank = cluster_rank();
    const uint32_t peer = rank ^ 1u;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int cl = blockIdx.x >> 1, n_cl = gridDim.x >> 1;
    if (smem_u32(smem_raw) & 1023u) {  // the layout needs a 1024-byte aligned window
        griddep_wait();
        if (threadIdx.x == 0) record_error(p.err, KVD_ERR_CUDA);
        return;
    }
    const int nbox = rank == 0 ? 4 : 5;   // 64-dim boxes this CTA loads
    const int dim0 = rank == 0 ? 0 : 256;
    const CUtensorMap& tmC = rank == 0 ? tmC0 : tmC1;  // 3-D maps with 4 / 5 blocks per box
    constexpr uint32_t kXBytes = kH * kTok * 4;

    // Set-up that touches no global memory runs while the previous kernel on the stream
    // may still be finishing (programmatic launch).
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&sm.full[s], kSparse ? 32 : 1);
            mbar_init(&sm.empty[s], 1);
        }
        mbar_init(&sm.qready, kSoftWarps);
        mbar_init(&sm.sempty, 4);  // the four warps of the group that owns the tile
        mbar_init(&sm.pfull, 4);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sm.peer_free[i], 4);
            mbar_init(&sm.yfull[i], 4);
        }
        for (int g = 0; g < kGroups; ++g) {
            mbar_init(&sm.sfull[g], 1);
            mbar_init(&sm.pvdone[g], 1);
            mbar_init(&sm.xfull[0][g], 1);   // armed with the exchanged byte count each tile
            mbar_init(&sm.xfull[1][g], 1);
            mbar_init(&sm.yfree[0][g], 1);
            mbar_init(&sm.yfree[1][g], 1);
            mbar_init(&sm.hand[g], 4);
        }
        mbar_init(&sm.ofinal, 1);
        mbar_init(&sm.ofree, kSoftWarps);
        mbar_init(&sm.qfull, 1);
        mbar_init(&sm.qkend, 1);
        mbar_init(&sm.pvend, 1);
        fence_mbar_init();
    }
    if (warp == kWarpQK) tmem_alloc(&sm.tmem_base, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    cluster_sync();  // the partner's barriers exist before anyone signals them
    const uint32_t tmem = sm.tmem_base;

    griddep_wait();  // lengths, selected indices and the workspace are read from here on
    if (warp == 0)
        build_schedule<kSparse, kTok>(p, cl, n_cl, sm.sched, lane, rank == 0 ? p.err : nullptr);
    __syncthreads();
    const int n_tiles = sm.sched.n_tiles;
    if (n_tiles == 0) {  // both CTAs of the pair take this exit together, with no remote access
        if (warp == kWarpQK) tmem_dealloc(tmem, 512);
        return;
    }
    // With the piece table: the first piece's query slice comes by TMA into ring stages 2-3
    // (16 KB per 64-dim box), issued ahead of the first tiles, which take stages 0-1; the
    // producer reuses stages 2-3 once the queries are in tensor memory.
    const bool tma_q = sm.sched.n_pieces > 0;
    constexpr int kQBox = kH * 128;
    // the partner's partial scores of the first tile of each group (later tiles: armed by
    // the group once the slot's previous phase has completed). A copy that lands before
    // its arming leaves the transaction count below zero until then.
    if (threadIdx.x == 0)
        for (int i = 0; i < kGroups && i < n_tiles; ++i)
            for (int hf = 0; hf < 2; ++hf) mbar_arrive_expect_tx(&sm.xfull[hf][i], kXBytes / 2);

    if (warp == kWarpLoad) {
        // ------------------------------------------------------------------ loads
        if (lane == 0) {
            prefetch_tensormap(&tmC);
            prefetch_tensormap(&tmC2);
            if (tma_q) {
                mbar_arrive_expect_tx(&sm.qfull, nbox * kQBox);
                for (int bx = 0; bx < nbox; ++bx)
                    tma_load_2d(sm.stage[2] + bx * kQBox, &tmQ, &sm.qfull, dim0 + 64 * bx,
                                sm.sched.piece[0].b * kH);
            }
        }
        int g = 0;  // tile index within this CTA's range
        bool ok = true;
        const uint64_t pol = l2_evict_first_policy();  // latent rows are read once
        // Dense: no tile is of use before the first piece's queries are in tensor memory, so
        // their loads go out first instead of queueing behind every SM's first tiles (page
        // ids of the first tiles are resolved meanwhile).
        auto wait_queries = [&]() {
            if (lane == 0) ok = mbar_wait(&sm.qready, 0, p.err);
            ok = __shfl_sync(0xffffffffu, ok, 0);
        };
        for_each_piece<kSparse, kTok>(p, sm.sched, [&](int b, int items, int lo, int hi, int) {
            if (!ok) return;
            const int nt = (hi - lo + kTok - 1) / kTok;
            if (!kSparse) {
                // page ids of the piece, 32 at a time (lane k holds piece 32 m + k), the
                // next batch in flight while the current one is used
                const int L = items;
                const int bp = min(p.page_size, kTok);
                const int per_tile = kTok / bp;
                const int n_pieces = nt * per_tile;
                auto piece_page = [&](int pc) -> int {
                    if (pc >= n_pieces) return 0;
                    const int t = min(lo + pc * bp, L - 1);  // past the end: any valid page
                    return load_page(p.block_table, p.max_pages, p.num_pages, b,
                                     t / p.page_size, p.err);
                };
                int cur = piece_page(lane), nxt = piece_page(32 + lane);
                for (int i = 0; i < nt && ok; ++i, ++g) {
                    const int s = g % kStages;
                    if (g == (tma_q ? 2 : 0)) wait_queries();
                    if (lane == 0 && ok)
                        ok = mbar_wait(&sm.empty[s], ((g / kStages) & 1) ^ 1, p.err);
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                    if (!ok) break;
                    if (lane == 0) mbar_arrive_expect_tx(&sm.full[s], nbox * kTileBox);
                    for (int sub = 0; sub < per_tile; ++sub) {
                        const int pc = i * per_tile + sub;
                        if (pc > 0 && (pc & 31) == 0) {
                            cur = nxt;
                            nxt = piece_page(pc + 32 + lane);
                        }
                        const int pg = __shfl_sync(0xffffffffu, cur, pc & 31);
                        if (lane == 0) {
                            const int t = lo + pc * bp;
                            const int y = pg * p.page_size + (t % p.page_size);
                            if (bp == kTok) {
                                // all of this CTA's 64-dim blocks in one instruction
                                tma_load_3d(sm.stage[s], &tmC, &sm.full[s], 0, y, dim0 / 64,
                                            pol);
                            } else {
                                for (int bx = 0; bx < nbox; ++bx)
                                    tma_load_2d(sm.stage[s] + bx * kTileBox + sub * bp * 128,
                                                &tmC2, &sm.full[s], dim0 + 64 * bx, y, pol);
                            }
                        }
                    }
                }
            } else {
                // gather the selected rows: each lane copies rows lane and lane + 32 of the
                // tile (one row per lane and instruction issues faster than one row per
                // instruction); each lane's copies arrive on the tile's barrier when they land,
                // without the lane waiting. Row sources are resolved a tile ahead (token
                // indices two tiles ahead), so that neither dependent load waits in front of
                // the copies.
                const int L = load_len(p.seq_lens, b, p.max_len, nullptr);
                const __nv_bfloat16* cpool = reinterpret_cast<const __nv_bfloat16*>(p.c_pool);
                const int32_t* idx = p.idx + static_cast<size_t>(b) * p.idx_stride;
                auto has_row = [&](int i, int rr) {
                    return i < nt && lo + i * kTok + lane + 32 * rr < hi;
                };
                auto tok_of = [&](int i, int rr) -> int {
                    return has_row(i, rr) ? idx[lo + i * kTok + lane + 32 * rr] : -1;
                };
                // the block-table entry of t's page, read without waiting for the length
                // (checked once both have arrived)
                auto page_of = [&](int t) -> int {
                    if (t < 0) return 0;
                    const int pg = p.block_table[static_cast<size_t>(b) * p.max_pages +
                                                 min(t / p.page_size, p.max_pages - 1)];
                    if (t >= L) return 0;
                    if (pg < 0 || pg >= p.num_pages) {
                        record_error(p.err, KVD_ERR_DEVICE_OOB);
                        return 0;
                    }
                    return pg;
                };
                // the row's first element of this CTA's dims, or null for a zero row
                auto src_of = [&](bool has, int t, int pg) -> const __nv_bfloat16* {
                    if (!has) return nullptr;
                    if (t < 0 || t >= L) {
                        record_error(p.err, KVD_ERR_DEVICE_OOB);
                        return nullptr;
                    }
                    return cpool +
                           (static_cast<size_t>(pg) * p.page_size + t % p.page_size) * kDqk + dim0;
                };
                const __nv_bfloat16* src_cur[2];
                int t_nxt[2];
                {
                    const int t0a = tok_of(0, 0), t0b = tok_of(0, 1);
                    t_nxt[0] = tok_of(1, 0);
                    t_nxt[1] = tok_of(1, 1);
                    const int pa = page_of(t0a), pb = page_of(t0b);
                    src_cur[0] = src_of(has_row(0, 0), t0a, pa);
                    src_cur[1] = src_of(has_row(0, 1), t0b, pb);
                }
                for (int i = 0; i < nt && ok; ++i, ++g) {
                    const int s = g % kStages;
                    if (tma_q && g == 2) wait_queries();  // stages 2-3 held the queries
                    if (lane == 0 && ok)
                        ok = mbar_wait(&sm.empty[s], ((g / kStages) & 1) ^ 1, p.err);
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                    if (!ok) break;
                    const int t_nn0 = tok_of(i + 2, 0), t_nn1 = tok_of(i + 2, 1);
                    const int pg_n0 = page_of(t_nxt[0]), pg_n1 = page_of(t_nxt[1]);
                    const uint32_t base = smem_u32(sm.stage[s]);
#pragma unroll
                    for (int rr = 0; rr < 2; ++rr) {
                        const int r = lane + 32 * rr;
                        const __nv_bfloat16* src = src_cur[rr];
                        for (int c = 0; c < nbox * 8; ++c) {
                            const int bx = c >> 3, cc = c & 7;
                            const uint32_t dst =
                                base + bx * kTileBox + r * 128 + ((cc ^ (r & 7)) << 4);
                            cp_async_16(dst, src ? src + c * 8 : cpool, src ? 16u : 0u, pol);
                        }
                    }
                    // the tile's arrival: each lane's share once its copies have landed (the
                    // product issuers order these generic-proxy writes before their reads)
                    cp_async_arrive_noinc(&sm.full[s]);
                    src_cur[0] = src_of(has_row(i + 1, 0), t_nxt[0], pg_n0);
                    src_cur[1] = src_of(has_row(i + 1, 1), t_nxt[1], pg_n1);
                    t_nxt[0] = t_nn0;
                    t_nxt[1] = t_nn1;
                }
            }
        });
        if (kSparse) {
            cp_async_wait<0>();  // every issued copy lands before the CTA goes on
        } else if (lane == 0) {
            // every issued copy lands before the CTA goes on (also after a wait gave up: the
            // ring's shared memory must not be written once the CTA has exited)
            const int first = g > kStages ? g - kStages : 0;
            for (int i = first; i < g; ++i)
                mbar_wait(&sm.full[i % kStages], (i / kStages) & 1, p.err);
        }
    } else if (warp == kWarpQK) {
        // ------------------------------------------------------------------ score products
        // Tile g's product starts as soon as its data is in and tile g - 1's scores have been
        // read, independently of the value products. A piece's first product also waits for
        // that piece's query in TMEM.
        if (lane == 0) {
            int g = 0;
            bool ok = true;
            for_each_piece<kSparse, kTok>(p, sm.sched, [&](int, int, int lo, int hi, int k) {
                if (!ok || !(ok = mbar_wait(&sm.qready, k & 1, p.err))) return;
                const int nt = (hi - lo + kTok - 1) / kTok;
                for (int i = 0; i < nt; ++i, ++g) {
                    const int s = g % kStages;
                    ok = mbar_wait(&sm.full[s], (g / kStages) & 1, p.err) &&
                         mbar_wait(&sm.sempty, (g & 1) ^ 1, p.err);
                    if (!ok) return;
                    // gathered rows were written by cp.async (generic proxy): ordered before
                    // the tensor core's reads here
                    if (kSparse) fence_proxy_async_smem();
                    tc_fence_after();
                    if (nbox == 4)
                        issue_qk<16>(tmem, smem_u32(sm.stage[s]));
                    else
                        issue_qk<20>(tmem, smem_u32(sm.stage[s]));
                    tc_commit(&sm.sfull[g % kGroups]);
                }
            });
            // every product issued here completes before TMEM can be released (also after a
            // wait gave up)
            tc_commit(&sm.qkend);
            mbar_wait(&sm.qkend, 0, p.err);
        }
    } else if (warp == kWarpPV) {
        // ------------------------------------------------------------------ value products
        if (lane == 0) {
            int g = 0;
            bool ok = true;
            for_each_piece<kSparse, kTok>(p, sm.sched, [&](int, int, int lo, int hi, int k) {
                if (!ok) return;
                const int nt = (hi - lo + kTok - 1) / kTok;
                for (int i = 0; i < nt; ++i, ++g) {
                    const int s = g % kStages;
                    // a piece's first product overwrites O: the previous piece's O is read
                    if (i == 0 && k > 0 && !(ok = mbar_wait(&sm.ofree, (k - 1) & 1, p.err))) return;
                    if (!(ok = mbar_wait(&sm.pfull, g & 1, p.err))) return;
                    if (kSparse) fence_proxy_async_smem();
                    tc_fence_after();
                    issue_pv(tmem, smem_u32(sm.stage[s]), i > 0);
                    tc_commit(&sm.pvdone[g % kGroups]);
                    tc_commit(&sm.empty[s]);  // the tile's score product completed before its P
                }
                tc_commit(&sm.ofinal);  // every product of the piece (and before) completed
            });
            tc_commit(&sm.pvend);
            mbar_wait(&sm.pvend, 0, p.err);
        }
    } else if (warp == kWarpX) {
        // ------------------------------------------------------------------ score exchange
        // One bulk copy per half tile moves this CTA's partial scores (staged in y by the
        // tile's group) into the partner's slot for that half. The copies drain over
        // distributed shared memory at its own rate, off the softmax warps' instruction path;
        // each half of y is released as soon as its own copy has read it.
        if (lane == 0) {
            uint32_t peer_x[2], peer_xfull[2][kGroups];
            for (int hf = 0; hf < 2; ++hf) {
                peer_x[hf] = map_peer(smem_u32(&sm.x[hf][0][0]), peer);
                for (int g = 0; g < kGroups; ++g)
                    peer_xfull[hf][g] = map_peer(smem_u32(&sm.xfull[hf][g]), peer);
            }
            bool ok = true;
            for (int j = 0; j < n_tiles && ok; ++j) {
                for (int hf = 0; hf < 2; ++hf) {
                    if (!(ok = mbar_wait(&sm.yfull[hf], j & 1, p.err))) break;
                    if (!(ok = mbar_wait_cluster(&sm.peer_free[hf], (j & 1) ^ 1, p.err))) break;
                    bulk_copy_to_peer(peer_x[hf], &sm.y[hf][0][0], kXBytes / 2,
                                      peer_xfull[hf][j % kGroups]);
                    // the previous copy (the other half) has been read: release it
                    asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
                    if (hf == 1)
                        mbar_arrive(&sm.yfree[0][j % kGroups]);
                    else if (j >= 1)
                        mbar_arrive(&sm.yfree[1][(j - 1) % kGroups]);
                }
            }
            bulk_wait_read_all();
            if (ok) mbar_arrive(&sm.yfree[1][(n_tiles - 1) % kGroups]);
            // the copies have landed in the partner before the pair's final barrier lets it exit
            bulk_wait_all();
        }
    } else {
        // ------------------------------------------------------------------ softmax
        const int grp = warp >> 2;                 // takes tiles j with j % kGroups == grp
        const int h = (warp & 3) * 32 + lane;      // head = TMEM lane
        const uint32_t trow = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
        const float sl2 = p.scale_log2;
        const uint32_t peer_free_hf[2] = {map_peer(smem_u32(&sm.peer_free[0]), peer),
                                          map_peer(smem_u32(&sm.peer_free[1]), peer)};
        int g0 = 0;  // first tile of the current piece within this CTA's range
        bool ok = true;
        constexpr int kQBoxes = (kNBox + kGroups - 1) / kGroups;
        const int bx0 = grp * kQBoxes, bx1 = min(nbox, bx0 + kQBoxes);
        auto q_rows = [&](int b) {  // this lane's head row of sequence b's queries, our dims
            return reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(p.q) +
                                                  (static_cast<size_t>(b) * kH + h) * kDqk +
                                                  dim0);
        };
        auto prefetch_q = [&](int b) {
#pragma unroll
            for (int bi = 0; bi < kQBoxes; ++bi)
                if (bx0 + bi < bx1) prefetch_l2(q_rows(b) + (bx0 + bi) * 8);
        };
        // Sequence b's query slice into TMEM (the A operand of the score product), the group's
        // 64-dim boxes one at a time (few registers), then the group's share of qready.
        auto load_q = [&](int b) {
            const uint4* qrow = q_rows(b);
#pragma unroll 1
            for (int bx = bx0; bx < bx1; ++bx) {
                uint4 v[8];
#pragma unroll
                for (int jj = 0; jj < 8; ++jj) v[jj] = __ldg(qrow + bx * 8 + jj);
                uint32_t r[32];
#pragma unroll
                for (int jj = 0; jj < 8; ++jj) {
                    r[4 * jj] = v[jj].x;
                    r[4 * jj + 1] = v[jj].y;
                    r[4 * jj + 2] = v[jj].z;
                    r[4 * jj + 3] = v[jj].w;
                }
                tmem_st_32x32b_x32(trow + kColQ + bx * 32, r);
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.qready);
        };
        // The first piece's queries from the TMA copy in stages 2-3 (128-byte swizzled rows).
        auto load_q_staged = [&]() {
            if (!(ok = mbar_wait(&sm.qfull, 0, p.err))) return;
#pragma unroll 1
            for (int bx = bx0; bx < bx1; ++bx) {
                const uint8_t* row = sm.stage[2] + bx * kQBox + h * 128;
                uint32_t r[32];
#pragma unroll
                for (int jj = 0; jj < 8; ++jj) {
                    const uint4 v = *reinterpret_cast<const uint4*>(row + ((jj ^ (h & 7)) << 4));
                    r[4 * jj] = v.x;
                    r[4 * jj + 1] = v.y;
                    r[4 * jj + 2] = v.z;
                    r[4 * jj + 3] = v.w;
                }
                tmem_st_32x32b_x32(trow + kColQ + bx * 32, r);
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.qready);
        };
        // With the piece table, the next piece's queries are loaded as soon as the current
        // piece's score products have all completed (before its output is written), so that
        // the next products overlap that write; otherwise each piece loads its own.
        const int n_pieces = sm.sched.n_pieces;
        // Every piece ends in two named barriers of all eight warps, reached even after a
        // failed wait, so that no warp is left waiting there.
        for_each_piece<kSparse, kTok>(p, sm.sched, [&](int b, int, int lo, int hi, int k) {
            const int nt = (hi - lo + kTok - 1) / kTok;
            const int next_b = (n_pieces >= 0 && k + 1 < n_pieces) ? sm.sched.piece[k + 1].b : -1;
            if (ok && k == 0 && tma_q) {
                load_q_staged();
            } else if (ok && (k == 0 || n_pieces < 0)) {
                prefetch_q(b);
                load_q(b);
            }
            bool next_prefetched = false;
            float l = 0.f, m_l = neg_inf();  // this group's sum of P, relative to 2^m_l
            float m_last = neg_inf();        // running max after this group's latest tile
            for (int i = 0; i < nt && ok; ++i) {
                const int j = g0 + i;  // tile index within the range (barrier phases)
                if (j % kGroups != grp) continue;
                if (next_b >= 0 && !next_prefetched && i + 2 * kGroups >= nt) {
                    prefetch_q(next_b);  // a few tiles before it is needed
                    next_prefetched = true;
                }
                const int it = j / kGroups;  // this group's iteration
                const int pg = (j + kGroups - 1) % kGroups;  // group of tile j - 1
                const int pit = ((j - 1) / kGroups) & 1;     // its barrier parity
                // 1. this CTA's partial scores; reading them frees S for the next product
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
                const int T0 = lo + i * kTok;
                // Dense, the sequence's last tile: the slots past its end (the rest of the last
                // page, or another page of the sequence when pages are shorter than a tile) may
                // hold anything, NaN and Inf included, and a zero probability times NaN is NaN.
                // The score product has read the stage, so the group clears those rows of this
                // CTA's four value boxes before the value product reads them (pfull below).
                if (!kSparse && T0 + kTok > hi) {
                    const int r0 = hi - T0;
                    const int n16 = (kTok - r0) * 8;  // 16-byte chunks to clear per box
                    uint8_t* st = sm.stage[j % kStages];
                    for (int e = (warp & 3) * 32 + lane; e < 4 * n16; e += 128) {
                        const int bx = e / n16, rem = e % n16;
                        *reinterpret_cast<uint4*>(st + bx * kTileBox + (r0 + rem / 8) * 128 +
                                                  (rem % 8) * 16) = make_uint4(0u, 0u, 0u, 0u);
                    }
                    fence_proxy_async_smem();  // before the tensor core reads the stage
                }
                // 2. stage them for the exchange thread, each half once tile j - 1's copy of
                //    that half has read y
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    if (j >= 1 &&
                        !(ok = mbar_wait(&sm.yfree[hf][pg], pit, p.err)))
                        break;
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        *reinterpret_cast<float4*>(&sm.y[hf][h][(c ^ (h & 7)) * 4]) =
                            make_float4(s[32 * hf + 4 * c], s[32 * hf + 4 * c + 1],
                                        s[32 * hf + 4 * c + 2], s[32 * hf + 4 * c + 3]);
                    fence_proxy_async_smem();  // generic stores before the bulk copy reads them
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&sm.yfull[hf]);
                }
                if (!ok) break;
                // 3. the partner's partial, half by half
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    if (!(ok = mbar_wait_cluster(&sm.xfull[hf][grp], it & 1, p.err))) break;
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const float4 v =
                            *reinterpret_cast<const float4*>(&sm.x[hf][h][(c ^ (h & 7)) * 4]);
                        s[32 * hf + 4 * c] += v.x;
                        s[32 * hf + 4 * c + 1] += v.y;
                        s[32 * hf + 4 * c + 2] += v.z;
                        s[32 * hf + 4 * c + 3] += v.w;
                    }
                    __syncwarp();
                    // x[hf] has been read: the partner may send its next half into it (the
                    // values are in registers, so a relaxed arrive suffices)
                    if (lane == 0) mbar_arrive_remote_relaxed(peer_free_hf[hf]);
                    // the slot's phase is complete: arm it for this group's next tile
                    if (warp == 4 * grp && lane == 0 && j + kGroups < n_tiles)
                        mbar_arrive_expect_tx(&sm.xfull[hf][grp], kXBytes / 2);
                }
                if (!ok) break;
                // 4. tile max, then the running max handed over from tile j - 1 (within the
                //    piece; the hand-over barrier is passed at every tile to keep its phases)
                float mt = neg_inf();
#pragma unroll
                for (int c = 0; c < kTok; ++c) {
                    s[c] = (T0 + c < hi) ? s[c] * sl2 : neg_inf();
                    mt = fmaxf(mt, s[c]);
                }
                float m_prev = neg_inf();
                if (j >= 1) {
                    if (!(ok = mbar_wait(&sm.hand[pg], pit, p.err))) break;
                    if (i > 0) m_prev = sm.mref[pg][h];
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
                    const __nv_bfloat162 v = __floats2bfloat162_rn(fast_exp2(s[2 * c] - mu),
                                                                   fast_exp2(s[2 * c + 1] - mu));
                    const float2 f = __bfloat1622float2(v);
                    psum += f.x + f.y;
                    pk[c] = *reinterpret_cast<const uint32_t*>(&v);
                }
                l += psum;
                // 6. P (and O) are free once tile j - 1's value product has completed
                if (j >= 1 &&
                    !(ok = mbar_wait(&sm.pvdone[pg], pit, p.err)))
                    break;
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
                        for (int kk = 0; kk < 32; ++kk)
                            r[kk] = __float_as_uint(__uint_as_float(r[kk]) * alpha);
                        tmem_st_32x32b_x32(trow + kColO + c * 32, r);
                    }
                }
                tmem_st_32x32b_x32(trow + kColP, pk);  // P row: 64 bf16
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&sm.pfull);
            }
            // The piece's partial: O / l for this CTA's 256 value dims, and log2-sum-exp.
            // The final reference is the running max after the piece's last tile.
            const int jl = g0 + nt - 1;
            const int lg = jl % kGroups;  // group of the piece's last tile
            if (ok && lg != grp) {
                ok = mbar_wait(&sm.hand[lg], (jl / kGroups) & 1, p.err);
                if (ok) m_last = sm.mref[lg][h];
            }
            // every score product of the piece has completed (the last tile's scores have
            // been read): the query slice may now take the next piece's queries
            if (ok && next_b >= 0) {
                if (!next_prefetched) prefetch_q(next_b);
                load_q(next_b);
            }
            // every group's sum relative to 2^m_last, added through shared memory (over the
            // running-max array, once every group has read the final max)
            asm volatile("bar.sync 1, %0;" ::"r"(kSoftWarps * 32) : "memory");
            sm.mref[grp][h] = (l > 0.f) ? l * fast_exp2(m_l - m_last) : 0.f;
            asm volatile("bar.sync 1, %0;" ::"r"(kSoftWarps * 32) : "memory");
            float l_tot = 0.f;
#pragma unroll
            for (int g = 0; g < kGroups; ++g) l_tot += sm.mref[g][h];
            asm volatile("bar.sync 1, %0;" ::"r"(kSoftWarps * 32) : "memory");  // sums read
            if (ok && (ok = mbar_wait(&sm.ofinal, k & 1, p.err))) {
                tc_fence_after();
                const size_t slot = static_cast<size_t>(cl) + b;
                const float inv = l_tot > 0.f ? 1.f / l_tot : 0.f;
                // rows of the eight heads of this lane's group of eight lanes; after the
                // transpose below, lane i of the group holds 16-byte chunk i of each of them
                float* po = p.part_o +
                            (slot * kH + (h & ~7)) * kDv + rank * 256 + (lane & 7) * 4;
                // the groups split this CTA's 256 value dims in 32-column slices
                constexpr int kOSlices = (8 + kGroups - 1) / kGroups;
                for (int c = grp * kOSlices; c < min(8, (grp + 1) * kOSlices); ++c) {
                    uint32_t r[32];
                    tmem_ld_32x32b_x32(trow + kColO + c * 32, r);
                    tmem_ld_wait(r);
                    float4 ch[8];
#pragma unroll
                    for (int jj = 0; jj < 8; ++jj)
                        ch[jj] = make_float4(__uint_as_float(r[4 * jj]) * inv,
                                             __uint_as_float(r[4 * jj + 1]) * inv,
                                             __uint_as_float(r[4 * jj + 2]) * inv,
                                             __uint_as_float(r[4 * jj + 3]) * inv);
                    transpose8_chunks(ch, lane);
                    // each store writes four whole 128-byte rows (one per group of lanes)
#pragma unroll
                    for (int jj = 0; jj < 8; ++jj)
                        __stcg(reinterpret_cast<float4*>(po + jj * kDv + c * 32), ch[jj]);
                }
                if (rank == 0 && grp == 0)
                    p.part_lse[slot * kH + h] = l_tot > 0.f ? m_last + log2f(l_tot) : neg_inf();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&sm.ofree);
            }
            g0 += nt;
        });
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    cluster_sync();  // the partner is done with this CTA's shared memory
    if (warp == kWarpQK) tmem_dealloc(tmem, 512);
}

// Merge the pieces of each (sequence, head): o = sum_i 2^{lse_i - M} o_i / sum_i 2^{lse_i - M}.
// Two heads per block; each thread owns four value dims and streams every piece. Sequence
// b's pieces come from the clusters whose tile ranges meet b's tiles (slot = cluster + b).
// kBuf partials of each thread in flight at once: 16 for the sparse decode (its sequences
// meet about 16 pieces each), 8 for the dense one (about 5, four blocks per SM).
template <int kBuf>
__global__ void __launch_bounds__(256, kBuf > 8 ? 2 : 4) mla_combine_kernel(const MlaParams p,
                                                             __nv_bfloat16* out,
                                                             float* lse_out) {
    griddep_wait();
    const int b = blockIdx.x / (kH / 2);
    const int h = (blockIdx.x % (kH / 2)) * 2 + threadIdx.x / 128;
    const int d = (threadIdx.x % 128) * 4;
    // Tile counts of all sequences, their total T and sequence b's first tile Sb and count nb:
    // the first warp loads 32 sequences' lengths at a time and scans them.
    // Clusters whose ranges [V c / C, V (c + 1) / C) of the virtual tile list (V = T plus a
    // gap of X positions before every later sequence) meet b's tiles: the one holding
    // position v is floor((v C + C - 1) / V). When every range holds tiles (a gap, or at
    // least as many tiles as clusters), the clusters holding b's first and last tiles bound
    // a contiguous run; otherwise (no gap, fewer tiles than clusters) each tile names its
    // cluster. Block-wide, once.
    constexpr int kMaxRun = 256;
    __shared__ int s_slot[kMaxRun];
    __shared__ int s_n;
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        long long T = 0, Sb = 0;
        int nb = 0;
        for (int base = 0; base < p.B; base += 32) {
            const int bb = base + lane;
            int items = 0;
            if (bb < p.B)
                items = p.sparse ? min(max(p.idx_count[bb], 0), p.idx_stride)
                                 : load_len(p.seq_lens, bb, p.max_len, nullptr);
            const int n = (items + p.tile - 1) / p.tile;
            int incl = n;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += v;
            }
            if (bb == b) {
                Sb = T + incl - n;
                nb = n;
            }
            T += __shfl_sync(0xffffffffu, incl, 31);
        }
        Sb = __shfl_sync(0xffffffffu, Sb, b & 31);
        nb = __shfl_sync(0xffffffffu, nb, b & 31);
        if (lane == 0) {
            const long long C = p.n_clusters;
            // the decode kernel's virtual tile list (a gap before every later sequence)
            const long long X = piece_gap(T, p.B, p.n_clusters, p.gap);
            const long long V = T + X * (p.B - 1), Vb = Sb + X * b;
            int n = 0;
            if (nb > 0 && (X > 0 || T >= C)) {
                const int c0 = static_cast<int>((Vb * C + C - 1) / V);
                const int c1 = static_cast<int>(((Vb + nb - 1) * C + C - 1) / V);
                for (int c = c0; c <= c1 && n < kMaxRun; ++c) s_slot[n++] = c + b;
            } else {
                int last = -1;
                for (int t = 0; t < nb && n < kMaxRun; ++t) {
                    const int c = static_cast<int>(((Sb + t) * C + C - 1) / T);
                    if (c != last) s_slot[n++] = c + b;
                    last = c;
                }
            }
            s_n = n;
        }
    }
    __shared__ float s_lse[2][kMaxRun];
    __syncthreads();
    const int n_slots = s_n;
    // both heads' log-sum-exps of every slot, fetched in parallel with the first kBuf
    // partials of this thread's dims
    for (int i = threadIdx.x; i < 2 * n_slots; i += blockDim.x)
        s_lse[i / n_slots][i % n_slots] =
            __ldcg(p.part_lse + static_cast<size_t>(s_slot[i % n_slots]) * kH +
                   (blockIdx.x % (kH / 2)) * 2 + i / n_slots);
    auto part = [&](int i) {
        return __ldcg(reinterpret_cast<const float4*>(
            p.part_o + (static_cast<size_t>(s_slot[i]) * kH + h) * kDv + d));
    };
    float4 vb[kBuf];
#pragma unroll
    for (int i = 0; i < kBuf; ++i)
        if (i < n_slots) vb[i] = part(i);
    __syncthreads();
    const float* lse = s_lse[threadIdx.x / 128];
    float M = neg_inf();
    for (int i = 0; i < n_slots; ++i) M = fmaxf(M, lse[i]);
    float den = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    auto add = [&](int i, const float4& v) {
        const float w = (M == neg_inf()) ? 0.f : fast_exp2(lse[i] - M);
        den += w;
        acc.x += w * v.x;
        acc.y += w * v.y;
        acc.z += w * v.z;
        acc.w += w * v.w;
    };
#pragma unroll
    for (int i = 0; i < kBuf; ++i)
        if (i < n_slots) add(i, vb[i]);
#pragma unroll 8
    for (int i = kBuf; i < n_slots; ++i) add(i, part(i));
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
               const CUtensorMap& tc2, const CUtensorMap& tq, void* out, float* lse_out,
               cudaStream_t stream) {
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
    const int grid = 2 * p.n_clusters;
    const cudaError_t e1 =
        p.sparse ? launch_kernel(mla_decode_kernel<true>, dim3(grid), dim3(kThreads), kMlaSmem,
                                 stream, tc0, tc1, tc2, tq, p)
                 : launch_kernel(mla_decode_kernel<false>, dim3(grid), dim3(kThreads), kMlaSmem,
                                 stream, tc0, tc1, tc2, tq, p);
    if (e1 != cudaSuccess) return KVD_ERR_CUDA;
    const cudaError_t e2 =
        p.sparse ? launch_kernel(mla_combine_kernel<16>, dim3(p.B * (kH / 2)), dim3(256), 0,
                                 stream, p, static_cast<__nv_bfloat16*>(out), lse_out)
                 : launch_kernel(mla_combine_kernel<8>, dim3(p.B * (kH / 2)), dim3(256), 0,
                                 stream, p, static_cast<__nv_bfloat16*>(out), lse_out);
    if (e2 != cudaSuccess) return KVD_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? KVD_OK : KVD_ERR_CUDA;
}

}  // namespace kvd
