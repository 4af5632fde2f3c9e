// dsa_indexer_fp8.cu -- the lightning indexer over an FP8 (e4m3) key cache, and the e4m3
// row quantizer that fills such a cache and quantizes the indexer queries.
//
// What is computed ("Long context, KV eviction and sparse attention", exact selection with a
// fast scorer: the lightning indexer scores every past token with few heads in FP8): codes
// are e4m3 with one float32 scale per key row (token) and per query row (head), so for every
// cached token t of sequence b
//   I_t = sk_t * sum_h (w_h sq_h) * ReLU(q8_h . k8_t)
// (a scale is never negative, so it leaves the ReLU), followed by the same top-k selection
// as the bf16 indexer. Quantization: scale = amax / 448 (1 for a row of zeros), code = the
// nearest e4m3 value to x / scale in float32, ties to even, saturating at 448.
//
// GB300: the bf16 indexer's structure with 16 KB tiles (128 tokens x 128 one-byte dims: one
// 128-byte swizzled box), tcgen05.mma kind::f8f6f4 (e4m3 x e4m3 -> f32, K = 32 a step), an
// 8-stage ring, and a ring of per-token scales (512 bytes per tile, 1-D bulk copies issued
// with the tile's TMA) that the epilogue releases once it has read them.

#include <algorithm>

#include <cuda_fp8.h>

#include "kvd_device.cuh"
#include "kvd_host.h"

namespace kvd {

namespace {

constexpr int kFTile = 128;                       // tokens per tile (MMA M)
constexpr int kFHi = 64;                          // indexer heads (MMA N)
constexpr int kFDi = 128;                         // head dim = bytes per key row (MMA K)
constexpr int kFTileBytes = kFTile * kFDi;        // 16 KB
constexpr int kFQBytes = kFHi * kFDi;             // 8 KB
constexpr int kFStages = 4;
constexpr int kFScaleSlots = 4;
constexpr int kFCtasPerSm = 2;                    // two independent pipelines per SM
constexpr int kFThreads = 6 * 32;                 // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
constexpr int kFHistBins = 2048;                  // top 11 key bits
constexpr int kFRowCap = 512;                     // page pieces resolved ahead (a chunk)

struct IdxF8Smem {
    uint8_t stage[kFStages][kFTileBytes];         // 1024-aligned (offset 0)
    uint8_t qbuf[2][kFQBytes];
    float ks[kFScaleSlots][kFTile];               // per-token scales of a tile
    alignas(16) uint32_t hist[kFHistBins];  // read as uint4 by the flush
    float wv[2][kFHi];                            // w_h * sq_h of the current sequence
    uint64_t full[kFStages], empty[kFStages], sfull[kFScaleSlots], sempty[kFScaleSlots];
    uint64_t qfull[2], qempty[2], tfull[2], tempty[2], done;
    uint32_t tmem_base;
    int prow[kFRowCap];                           // first physical row of each piece
};
constexpr int kFSmem = static_cast<int>(sizeof(IdxF8Smem)) + 1024;

struct F8Range {
    int begin, end;
};
__device__ __forceinline__ F8Range f8_tiles(int total) {
    const long long G = gridDim.x, i = blockIdx.x;
    return F8Range{static_cast<int>(i * total / G), static_cast<int>((i + 1) * total / G)};
}

// (sequence, tile within it) of flat tile f, advanced without a division per tile
struct TileCursor {
    int b, j, per_b;
    __device__ TileCursor(int f, int tiles_per_b)
        : b(f / tiles_per_b), j(f % tiles_per_b), per_b(tiles_per_b) {}
    __device__ void next() {
        if (++j == per_b) {
            j = 0;
            ++b;
        }
    }
};

__global__ void __launch_bounds__(kFThreads, kFCtasPerSm)
    dsa_indexer_fp8_kernel(const __grid_constant__ CUtensorMap tmK,
                           const __grid_constant__ CUtensorMap tmK128,
                           const __grid_constant__ CUtensorMap tmQ, const IdxParams p) {
    extern __shared__ uint8_t smem_raw[];
    IdxF8Smem& sm = *reinterpret_cast<IdxF8Smem*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int total = p.B * p.tiles_per_b;
    const F8Range tr = f8_tiles(total);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kFStages; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], 1);
        }
        for (int s = 0; s < kFScaleSlots; ++s) {
            mbar_init(&sm.sfull[s], 1);
            mbar_init(&sm.sempty[s], 4);  // the four epilogue warps
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sm.qfull[i], 1);
            mbar_init(&sm.qempty[i], 1);
            mbar_init(&sm.tfull[i], 1);
            mbar_init(&sm.tempty[i], 4);
        }
        mbar_init(&sm.done, 1);
        fence_mbar_init();
    }
    for (int i = threadIdx.x; i < kFHistBins; i += blockDim.x) sm.hist[i] = 0;
    if (warp == 1) tmem_alloc(&sm.tmem_base, 128);  // two 64-column fp32 accumulators
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;
    // the set-up above touches no global memory: it runs while the previous kernel on the
    // stream may still be finishing (programmatic launch)
    griddep_wait();
    // the selection's counters start from zero whatever an earlier call left in them
    if (blockIdx.x == 0)
        for (int i = threadIdx.x; i < 4 * p.B; i += blockDim.x) p.counts[i] = 0;

    if (warp == 0) {
        // ------------------------------------------------------------------ TMA producer
        // The warp resolves the physical rows of the range's page pieces a chunk at a time
        // into shared memory; lane 0 then issues the key copies and the copies of the
        // matching per-token scales.
        if (lane == 0) {
            prefetch_tensormap(&tmK);
            prefetch_tensormap(&tmK128);
            prefetch_tensormap(&tmQ);
        }
        const int bp = min(p.page_size, kFTile);
        const int per_tile = kFTile / bp;  // 1, 2, 4 or 8 pieces a tile
        const int chunk = kFRowCap / per_tile;
        uint32_t g = 0, nq = 0;
        int cur_b = -1;
        bool ok = true;
        const uint64_t pol = l2_evict_first_policy();  // codes and scales are read once
        for (int c0 = tr.begin; c0 < tr.end && ok; c0 += chunk) {
            const int c1 = min(tr.end, c0 + chunk);
            // the warp resolves the chunk's piece rows (first physical row of each piece, or
            // -1 for a tile past its sequence's end), lane k taking pieces k, k + 32, ...
            for (int q = lane; q < (c1 - c0) * per_tile; q += 32) {
                const int f = c0 + q / per_tile, sub = q % per_tile;
                const int b = f / p.tiles_per_b, j = f % p.tiles_per_b;
                sm.prow[q] = piece_row(p.seq_lens, p.block_table, p.max_len, p.max_pages,
                                       p.num_pages, p.page_size, b, j * kFTile,
                                       j * kFTile + sub * bp, p.err);
            }
            __syncwarp();
            // lane 0 alone issues the chunk's copies: no warp-wide step per tile
            if (lane == 0) {
                TileCursor tc(c0, p.tiles_per_b);
                for (int f = c0; f < c1 && ok; ++f, tc.next()) {
                    const int* ys = sm.prow + (f - c0) * per_tile;
                    if (ys[0] < 0) continue;  // the tile lies past its sequence's end
                    const int b = tc.b;
                    if (b != cur_b) {
                        const int qs = nq & 1;
                        ok = mbar_wait(&sm.qempty[qs], ((nq >> 1) & 1) ^ 1, p.err);
                        if (!ok) break;
                        mbar_arrive_expect_tx(&sm.qfull[qs], kFQBytes);
                        tma_load_2d(sm.qbuf[qs], &tmQ, &sm.qfull[qs], 0, b * kFHi);
                        ++nq;
                        cur_b = b;
                    }
                    const int s = g % kFStages, ss = g % kFScaleSlots;
                    ok = mbar_wait(&sm.empty[s], ((g / kFStages) & 1) ^ 1, p.err) &&
                         mbar_wait(&sm.sempty[ss], ((g / kFScaleSlots) & 1) ^ 1, p.err);
                    if (!ok) break;
                    mbar_arrive_expect_tx(&sm.full[s], kFTileBytes);
                    mbar_arrive_expect_tx(&sm.sfull[ss], kFTile * 4);
                    // one 16 KB instruction when the pieces are contiguous (adjacent pages, or
                    // pages of >= 128 tokens)
                    bool contiguous = true;
                    for (int sub = 1; sub < per_tile; ++sub)
                        if (ys[sub] != ys[0] + sub * bp) contiguous = false;
                    if (contiguous && ys[0] + kFTile <= p.num_pages * p.page_size) {
                        tma_load_2d(sm.stage[s], &tmK128, &sm.full[s], 0, ys[0], pol);
                        bulk_load(sm.ks[ss], p.k_scale + ys[0], kFTile * 4, &sm.sfull[ss], pol);
                    } else {
                        for (int sub = 0; sub < per_tile; ++sub) {
                            tma_load_2d(sm.stage[s] + sub * bp * kFDi, &tmK, &sm.full[s], 0,
                                        ys[sub], pol);
                            bulk_load(sm.ks[ss] + sub * bp, p.k_scale + ys[sub], bp * 4,
                                      &sm.sfull[ss], pol);
                        }
                    }
                    ++g;
                }
            }
            // the rows of this chunk stay until lane 0 has issued them
            ok = __shfl_sync(0xffffffffu, ok, 0);
        }
        // copies still in flight complete before the CTA may exit
        if (lane == 0) {
            const uint32_t first = g > kFStages ? g - kFStages : 0;
            for (uint32_t i = first; i < g; ++i)
                mbar_wait(&sm.full[i % kFStages], (i / kFStages) & 1, p.err);
            const uint32_t sfirst = g > kFScaleSlots ? g - kFScaleSlots : 0;
            for (uint32_t i = sfirst; i < g; ++i)
                mbar_wait(&sm.sfull[i % kFScaleSlots], (i / kFScaleSlots) & 1, p.err);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_e4m3_f32(kFTile, kFHi);
            int cur_b = -1, L = 0;
            uint32_t g = 0, nq = 0, nt = 0;
            int qs = 0;
            bool ok = true;
            TileCursor tc(tr.begin, p.tiles_per_b);
            for (int f = tr.begin; f < tr.end && ok; ++f, tc.next()) {
                const int b = tc.b, j = tc.j;
                if (b != cur_b) L = load_len(p.seq_lens, b, p.max_len, nullptr);
                if (j * kFTile >= L) continue;
                if (b != cur_b) {
                    if (cur_b >= 0) tc_commit(&sm.qempty[qs]);  // previous q free after its MMAs
                    qs = nq & 1;
                    if (!(ok = mbar_wait(&sm.qfull[qs], (nq >> 1) & 1, p.err))) break;
                    ++nq;
                    cur_b = b;
                }
                const int s = g % kFStages;
                if (!(ok = mbar_wait(&sm.full[s], (g / kFStages) & 1, p.err))) break;
                const int acc = nt & 1;
                if (!(ok = mbar_wait(&sm.tempty[acc], ((nt >> 1) & 1) ^ 1, p.err))) break;
                tc_fence_after();
                const uint32_t a0 = smem_u32(sm.stage[s]);
                const uint32_t b0 = smem_u32(sm.qbuf[qs]);
#pragma unroll
                for (int k = 0; k < kFDi / 32; ++k) {  // 32 one-byte elements per k-step
                    const uint64_t ad = sw128_kmajor_desc(a0 + k * 32);
                    const uint64_t bd = sw128_kmajor_desc(b0 + k * 32);
                    tc_mma_e4m3(tmem + acc * kFHi, ad, bd, idesc, k > 0 ? 1u : 0u);
                }
                tc_commit(&sm.empty[s]);     // the smem stage is free once these MMAs are done
                tc_commit(&sm.tfull[acc]);   // the accumulator is ready
                ++g;
                ++nt;
            }
            tc_commit(&sm.done);  // every MMA of this CTA has completed
            mbar_wait(&sm.done, 0, p.err);
        }
    } else {
        // ------------------------------------------------------------------ epilogue
        const int quad = warp & 3;  // TMEM lane quadrant this warp may access
        const int row = quad * 32 + lane;
        const int etid = threadIdx.x - 64;  // 0..127
        int cur_b = -1, L = 0;
        uint32_t nt = 0, nb = 0;
        float wr[kFHi];  // w_h * sq_h of the current sequence
        // The sequence's counts into the global histogram (16-byte reads, all in flight at
        // once), the shared one left zeroed for the next sequence (`last`: no next one, no
        // barrier after).
        auto flush_hist = [&](int b, bool last) {
            asm volatile("bar.sync 2, 128;" ::: "memory");
            uint32_t* gh = p.hist + static_cast<size_t>(b) * kFHistBins;
            uint4 v[kFHistBins / 4 / 128];
#pragma unroll
            for (int k = 0; k < kFHistBins / 4 / 128; ++k)
                v[k] = reinterpret_cast<const uint4*>(sm.hist)[etid + 128 * k];
#pragma unroll
            for (int k = 0; k < kFHistBins / 4 / 128; ++k) {
                const int i = 4 * (etid + 128 * k);
                if (v[k].x) atomicAdd(gh + i, v[k].x);
                if (v[k].y) atomicAdd(gh + i + 1, v[k].y);
                if (v[k].z) atomicAdd(gh + i + 2, v[k].z);
                if (v[k].w) atomicAdd(gh + i + 3, v[k].w);
                if (!last && (v[k].x | v[k].y | v[k].z | v[k].w))
                    reinterpret_cast<uint4*>(sm.hist)[etid + 128 * k] = make_uint4(0u, 0u, 0u, 0u);
            }
            if (!last) asm volatile("bar.sync 2, 128;" ::: "memory");
        };
        TileCursor tc(tr.begin, p.tiles_per_b);
        for (int f = tr.begin; f < tr.end; ++f, tc.next()) {
            const int b = tc.b, j = tc.j;
            if (b != cur_b) L = load_len(p.seq_lens, b, p.max_len, nullptr);
            if (j * kFTile >= L) continue;
            if (b != cur_b) {
                if (cur_b >= 0) flush_hist(cur_b, false);
                if (etid < kFHi) {
                    const size_t i = static_cast<size_t>(b) * kFHi + etid;
                    sm.wv[nb & 1][etid] = p.w[i] * p.q_scale[i];
                }
                asm volatile("bar.sync 2, 128;" ::: "memory");
#pragma unroll
                for (int h = 0; h < kFHi; ++h) wr[h] = sm.wv[nb & 1][h];
                ++nb;
                cur_b = b;
            }
            const int acc = nt & 1, ss = nt % kFScaleSlots;
            if (!mbar_wait(&sm.tfull[acc], (nt >> 1) & 1, p.err)) break;
            if (!mbar_wait(&sm.sfull[ss], (nt / kFScaleSlots) & 1, p.err)) break;
            const float sk = sm.ks[ss][row];
            tc_fence_after();
            const uint32_t taddr = tmem + (static_cast<uint32_t>(quad * 32) << 16) + acc * kFHi;
            // both 32-column halves of the row in flight at once; four independent sums
            uint32_t r0[32], r1[32];
            tmem_ld_32x32b_x32(taddr, r0);
            tmem_ld_32x32b_x32(taddr + 32, r1);
            tmem_ld_wait(r0);
            tmem_ld_wait(r1);
            float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
            for (int c = 0; c < 32; c += 2) {
                a0 = fmaf(wr[c], fmaxf(__uint_as_float(r0[c]), 0.f), a0);
                a1 = fmaf(wr[c + 1], fmaxf(__uint_as_float(r0[c + 1]), 0.f), a1);
                a2 = fmaf(wr[32 + c], fmaxf(__uint_as_float(r1[c]), 0.f), a2);
                a3 = fmaf(wr[33 + c], fmaxf(__uint_as_float(r1[c + 1]), 0.f), a3);
            }
            const float score = ((a0 + a1) + (a2 + a3)) * sk;
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&sm.tempty[acc]);
                mbar_arrive(&sm.sempty[ss]);
            }
            const int t = j * kFTile + row;
            if (t < L) {
                p.scores[static_cast<size_t>(b) * p.score_stride + t] = score;
                atomicAdd(&sm.hist[float_key(score) >> 21], 1u);
            }
            ++nt;
        }
        if (cur_b >= 0) flush_hist(cur_b, true);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, 128);
}

// Row quantization to e4m3: one warp per row. dst_rows: null -> row r goes to row r of
// codes / scales; else the row's destination is computed from the block table (the cache
// append: sequence r's newest token, position seq_lens[r] - 1).
__global__ void __launch_bounds__(256) quantize_e4m3_kernel(const QuantParams p) {
    griddep_wait();
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) / 32, lane = threadIdx.x % 32;
    if (warp >= p.rows) return;
    const __nv_bfloat16* x = reinterpret_cast<const __nv_bfloat16*>(p.x) +
                             static_cast<size_t>(warp) * p.cols;
    long long dst = warp;
    if (p.block_table) {
        const int L = load_len(p.seq_lens, warp, p.max_len, p.err);
        const int t = L - 1;
        const int pg = load_page(p.block_table, p.max_pages, p.num_pages, warp, t / p.page_size,
                                 p.err);
        dst = static_cast<long long>(pg) * p.page_size + (t % p.page_size);
    }
    float amax = 0.f;
    for (int c = lane; c < p.cols; c += 32) amax = fmaxf(amax, fabsf(__bfloat162float(x[c])));
#pragma unroll
    for (int off = 16; off; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    const float s = amax > 0.f ? amax / 448.0f : 1.0f;
    uint8_t* out = static_cast<uint8_t*>(p.codes) + dst * p.cols;
    for (int c = lane; c < p.cols; c += 32)
        out[c] = static_cast<uint8_t>(
            __nv_cvt_float_to_fp8(__bfloat162float(x[c]) / s, __NV_SATFINITE, __NV_E4M3));
    if (lane == 0) p.scales[dst] = s;
}

}  // namespace

int dsa_indexer_fp8_launch(const IdxParams& p, const CUtensorMap& tk, const CUtensorMap& tk128,
                           const CUtensorMap& tq, cudaStream_t stream) {
    static int configured = 0;
    if (!configured) {
        if (cudaFuncSetAttribute(dsa_indexer_fp8_kernel,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kFSmem) != cudaSuccess)
            return KVD_ERR_CUDA;
        configured = 1;
    }
    const int total = p.B * p.tiles_per_b;
    const int grid = std::min(total, kFCtasPerSm * num_sms());
    if (launch_kernel(dsa_indexer_fp8_kernel, dim3(grid), dim3(kFThreads), kFSmem, stream, tk,
                      tk128, tq, p) != cudaSuccess)
        return KVD_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? KVD_OK : KVD_ERR_CUDA;
}

int quantize_e4m3_launch(const QuantParams& p, cudaStream_t stream) {
    const int blocks = (p.rows + 7) / 8;  // eight warps a block
    if (launch_kernel(quantize_e4m3_kernel, dim3(blocks), dim3(256), 0, stream, p) !=
        cudaSuccess)
        return KVD_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? KVD_OK : KVD_ERR_CUDA;
}

}  // namespace kvd
