// dsa_indexer.cu -- the DSA lightning indexer and the top-k selection over its scores.
//
// What is computed ("Attention Optimizations", DSA / Computation Path; "All the
// attentions", section 5): for every cached token t of sequence b,
//   I_t = sum_h w_h * ReLU(q_h . k_t)        (64 heads x 128 dims, one 128-wide key per token)
// then the indices of the k largest I_t (ties to the lower position), in ascending order.
//
// Indexer (GB300): a persistent kernel, one CTA per SM, each CTA owning a contiguous range
// of 128-token tiles. One warp resolves the tiles' page rows ahead of time and one of its
// threads streams key tiles with TMA (128-byte swizzle) through a shared-memory ring; one thread issues tcgen05.mma with the tokens as M and the heads as
// N: D[128 tok x 64 heads] (TMEM, fp32) = K[128 x 128] * Q^T, double-buffered in tensor
// memory; four epilogue warps read one token row each (tcgen05.ld), apply ReLU and the head
// weights, write the fp32 score and count its top 11 key bits into a shared-memory
// histogram, the first pass of the radix selection.
//
// Selection: one kernel. Its blocks split each sequence's scores, find from that histogram
// the bucket holding the k-th largest score, and sort tokens into selected (above it) and
// candidates (inside it). The last block of a sequence to finish narrows the candidates with
// further radix passes over a 64-bit key (score key, then position reversed, so the order is
// total and ties go to the lower position) and writes the k chosen positions ascending.

#include <algorithm>

#include "kvd_device.cuh"
#include "kvd_host.h"

namespace kvd {

namespace {

constexpr int kItile = 128;             // tokens per indexer tile (MMA M)
constexpr int kHi = 64;                 // indexer heads (MMA N)
constexpr int kDi = 128;                // indexer head dim (MMA K)
constexpr int kIdxTileBytes = kItile * kDi * 2;   // 32 KB: two 64-dim boxes of 16 KB
constexpr int kIdxQBytes = kHi * kDi * 2;         // 16 KB: two 64-dim boxes of 8 KB
constexpr int kIdxStages = 2;
constexpr int kIdxCtasPerSm = 2;        // two independent pipelines per SM
constexpr int kIdxThreads = 6 * 32;     // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
constexpr int kHistBins = 2048;         // top 11 key bits
constexpr int kIdxRowCap = 512;         // page pieces resolved ahead (a chunk)

struct IdxSmem {
    uint8_t stage[kIdxStages][kIdxTileBytes];   // 1024-aligned (offset 0)
    uint8_t qbuf[2][kIdxQBytes];
    alignas(16) uint32_t hist[kHistBins];  // read as uint4 by the flush
    float wv[2][kHi];
    uint64_t full[kIdxStages], empty[kIdxStages];
    uint64_t qfull[2], qempty[2], tfull[2], tempty[2], done;
    uint32_t tmem_base;
    int prow[kIdxRowCap];                       // first physical row of each piece
};
constexpr int kIdxSmem = static_cast<int>(sizeof(IdxSmem)) + 1024;

// The tiles a CTA owns: a contiguous slice of the flattened (sequence, tile) list.
struct TileRange {
    int begin, end;
};

// (sequence, tile within it) of flat tile f, advanced without a division per tile
struct IdxCursor {
    int b, j, per_b;
    __device__ IdxCursor(int f, int tiles_per_b)
        : b(f / tiles_per_b), j(f % tiles_per_b), per_b(tiles_per_b) {}
    __device__ void next() {
        if (++j == per_b) {
            j = 0;
            ++b;
        }
    }
};
__device__ __forceinline__ TileRange my_tiles(int total) {
    const long long G = gridDim.x, i = blockIdx.x;
    return TileRange{static_cast<int>(i * total / G), static_cast<int>((i + 1) * total / G)};
}

__global__ void __launch_bounds__(kIdxThreads, kIdxCtasPerSm)
    dsa_indexer_kernel(const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmK128,
                       const __grid_constant__ CUtensorMap tmQ, const IdxParams p) {
    extern __shared__ uint8_t smem_raw[];
    IdxSmem& sm = *reinterpret_cast<IdxSmem*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int total = p.B * p.tiles_per_b;
    const TileRange tr = my_tiles(total);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kIdxStages; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], 1);
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
    for (int i = threadIdx.x; i < kHistBins; i += blockDim.x) sm.hist[i] = 0;
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
        // into shared memory; lane 0 then issues the copies.
        if (lane == 0) {
            prefetch_tensormap(&tmK);
            prefetch_tensormap(&tmK128);
            prefetch_tensormap(&tmQ);
        }
        const int bp = min(p.page_size, kItile);
        const int per_tile = kItile / bp;  // 1, 2, 4 or 8 pieces a tile
        const int chunk = kIdxRowCap / per_tile;
        uint32_t g = 0, nq = 0;
        int cur_b = -1;
        bool ok = true;
        const uint64_t pol = l2_evict_first_policy();  // keys are read once
        for (int c0 = tr.begin; c0 < tr.end && ok; c0 += chunk) {
            const int c1 = min(tr.end, c0 + chunk);
            // the warp resolves the chunk's piece rows (first physical row of each piece, or
            // -1 for a tile past its sequence's end), lane k taking pieces k, k + 32, ...
            for (int q = lane; q < (c1 - c0) * per_tile; q += 32) {
                const int f = c0 + q / per_tile, sub = q % per_tile;
                const int b = f / p.tiles_per_b, j = f % p.tiles_per_b;
                sm.prow[q] = piece_row(p.seq_lens, p.block_table, p.max_len, p.max_pages,
                                       p.num_pages, p.page_size, b, j * kItile,
                                       j * kItile + sub * bp, p.err);
            }
            __syncwarp();
            // lane 0 alone issues the chunk's copies: no warp-wide step per tile
            if (lane == 0) {
                IdxCursor tc(c0, p.tiles_per_b);
                for (int f = c0; f < c1 && ok; ++f, tc.next()) {
                    const int* ys = sm.prow + (f - c0) * per_tile;
                    if (ys[0] < 0) continue;  // the tile lies past its sequence's end
                    const int b = tc.b;
                    if (b != cur_b) {
                        const int qs = nq & 1;
                        ok = mbar_wait(&sm.qempty[qs], ((nq >> 1) & 1) ^ 1, p.err);
                        if (!ok) break;
                        mbar_arrive_expect_tx(&sm.qfull[qs], kIdxQBytes);
                        tma_load_2d(sm.qbuf[qs], &tmQ, &sm.qfull[qs], 0, b * kHi);
                        tma_load_2d(sm.qbuf[qs] + kIdxQBytes / 2, &tmQ, &sm.qfull[qs], 64,
                                    b * kHi);
                        ++nq;
                        cur_b = b;
                    }
                    const int s = g % kIdxStages;
                    ok = mbar_wait(&sm.empty[s], ((g / kIdxStages) & 1) ^ 1, p.err);
                    if (!ok) break;
                    mbar_arrive_expect_tx(&sm.full[s], kIdxTileBytes);
                    // one 32 KB instruction when the pieces are contiguous (adjacent pages, or
                    // pages of >= 128 tokens)
                    bool contiguous = true;
                    for (int sub = 1; sub < per_tile; ++sub)
                        if (ys[sub] != ys[0] + sub * bp) contiguous = false;
                    if (contiguous && ys[0] + kItile <= p.num_pages * p.page_size) {
                        tma_load_3d(sm.stage[s], &tmK128, &sm.full[s], 0, ys[0], 0, pol);
                    } else {
                        for (int sub = 0; sub < per_tile; ++sub)
                            for (int half = 0; half < 2; ++half)
                                tma_load_2d(sm.stage[s] + half * (kIdxTileBytes / 2) +
                                                sub * bp * 128,
                                            &tmK, &sm.full[s], half * 64, ys[sub], pol);
                    }
                    ++g;
                }
            }
            // the rows of this chunk stay until lane 0 has issued them
            ok = __shfl_sync(0xffffffffu, ok, 0);
        }
        // copies still in flight complete before the CTA may exit
        if (lane == 0) {
            const uint32_t first = g > kIdxStages ? g - kIdxStages : 0;
            for (uint32_t i = first; i < g; ++i)
                mbar_wait(&sm.full[i % kIdxStages], (i / kIdxStages) & 1, p.err);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(kItile, kHi);
            int cur_b = -1, L = 0;
            uint32_t g = 0, nq = 0, nt = 0;
            int qs = 0;
            bool ok = true;
            IdxCursor tc(tr.begin, p.tiles_per_b);
            for (int f = tr.begin; f < tr.end && ok; ++f, tc.next()) {
                const int b = tc.b, j = tc.j;
                if (b != cur_b) L = load_len(p.seq_lens, b, p.max_len, nullptr);
                if (j * kItile >= L) continue;
                if (b != cur_b) {
                    if (cur_b >= 0) tc_commit(&sm.qempty[qs]);  // previous q free after its MMAs
                    qs = nq & 1;
                    if (!(ok = mbar_wait(&sm.qfull[qs], (nq >> 1) & 1, p.err))) break;
                    ++nq;
                    cur_b = b;
                }
                const int s = g % kIdxStages;
                if (!(ok = mbar_wait(&sm.full[s], (g / kIdxStages) & 1, p.err))) break;
                const int acc = nt & 1;
                if (!(ok = mbar_wait(&sm.tempty[acc], ((nt >> 1) & 1) ^ 1, p.err))) break;
                tc_fence_after();
                const uint32_t a0 = smem_u32(sm.stage[s]);
                const uint32_t b0 = smem_u32(sm.qbuf[qs]);
#pragma unroll
                for (int k = 0; k < kDi / 16; ++k) {
                    const uint32_t koff = (k & 3) * 32;  // 16 bf16 = 32 bytes per k-step
                    const uint64_t ad =
                        sw128_kmajor_desc(a0 + (k >> 2) * (kIdxTileBytes / 2) + koff);
                    const uint64_t bd = sw128_kmajor_desc(b0 + (k >> 2) * (kIdxQBytes / 2) + koff);
                    tc_mma_bf16(tmem + acc * kHi, ad, bd, idesc, k > 0 ? 1u : 0u);
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
        float wr[kHi];  // the head weights of the current sequence
        // The sequence's counts into the global histogram (16-byte reads, all in flight at
        // once), the shared one left zeroed for the next sequence (`last`: no next one, no
        // barrier after).
        auto flush_hist = [&](int b, bool last) {
            asm volatile("bar.sync 2, 128;" ::: "memory");
            uint32_t* gh = p.hist + static_cast<size_t>(b) * kHistBins;
            uint4 v[kHistBins / 4 / 128];
#pragma unroll
            for (int k = 0; k < kHistBins / 4 / 128; ++k)
                v[k] = reinterpret_cast<const uint4*>(sm.hist)[etid + 128 * k];
#pragma unroll
            for (int k = 0; k < kHistBins / 4 / 128; ++k) {
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
        IdxCursor tc(tr.begin, p.tiles_per_b);
        for (int f = tr.begin; f < tr.end; ++f, tc.next()) {
            const int b = tc.b, j = tc.j;
            if (b != cur_b) L = load_len(p.seq_lens, b, p.max_len, nullptr);
            if (j * kItile >= L) continue;
            if (b != cur_b) {
                if (cur_b >= 0) flush_hist(cur_b, false);
                if (etid < kHi) sm.wv[nb & 1][etid] = p.w[static_cast<size_t>(b) * kHi + etid];
                asm volatile("bar.sync 2, 128;" ::: "memory");
#pragma unroll
                for (int h = 0; h < kHi; ++h) wr[h] = sm.wv[nb & 1][h];
                ++nb;
                cur_b = b;
            }
            const int acc = nt & 1;
            if (!mbar_wait(&sm.tfull[acc], (nt >> 1) & 1, p.err)) break;
            tc_fence_after();
            const uint32_t taddr = tmem + (static_cast<uint32_t>(quad * 32) << 16) + acc * kHi;
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
            const float score = (a0 + a1) + (a2 + a3);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.tempty[acc]);
            const int t = j * kItile + row;
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

// ---------------------------------------------------------------------------------------
// Selection kernels
// ---------------------------------------------------------------------------------------

// Histogram of the top 11 key bits of caller-provided scores (dsa_topk only).
__global__ void __launch_bounds__(256) topk_hist_kernel(const TopkParams p) {
    griddep_wait();
    __shared__ __align__(16) uint32_t h[kHistBins];
    const int b = blockIdx.y;
    // the selection's counters start from zero whatever an earlier call left in them
    if (blockIdx.x == 0 && threadIdx.x < 4) p.counts[4 * b + threadIdx.x] = 0;
    for (int i = threadIdx.x; i < kHistBins; i += blockDim.x) h[i] = 0;
    __syncthreads();
    const int L = load_len(p.lens, b, p.max_len, p.err);
    const float* sc = p.scores + static_cast<size_t>(b) * p.score_stride;
    for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < L; t += gridDim.x * blockDim.x)
        atomicAdd(&h[float_key(sc[t]) >> 21], 1u);
    __syncthreads();
    for (int i = threadIdx.x; i < kHistBins; i += blockDim.x)
        if (h[i]) atomicAdd(p.hist + static_cast<size_t>(b) * kHistBins + i, h[i]);
}

// Block-wide inclusive scan of one int per thread (warp shuffles, then the warp totals).
template <int NT>
__device__ __forceinline__ int block_incl_scan(int v, int* s_warp) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= off) v += n;
    }
    if (lane == 31) s_warp[warp] = v;
    __syncthreads();
    if (warp == 0) {
        int t = lane < NT / 32 ? s_warp[lane] : 0;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, t, off);
            if (lane >= off) t += n;
        }
        if (lane < NT / 32) s_warp[lane] = t;
    }
    __syncthreads();
    const int r = v + (warp > 0 ? s_warp[warp - 1] : 0);
    __syncthreads();
    return r;
}

// Find the bucket holding the k-th largest key, scanning buckets from the top. Returns the
// bucket, the number of keys in higher buckets, the bucket's own count and (if asked) the
// total over all buckets. All threads of the block take part; s_tmp holds NT/32 + 4 ints.
template <int NT>
__device__ void find_bucket(const uint32_t* bins, int nbins, int k, int& bucket, int& above,
                            int& in_bucket, int* s_tmp, int* total = nullptr) {
    const int per = (nbins + NT - 1) / NT;  // each thread owns `per` bins counted from the top
    const int tid = threadIdx.x;
    int local = 0;
    for (int i = 0; i < per; ++i) {
        const int r = tid * per + i;
        if (r < nbins) local += bins[nbins - 1 - r];
    }
    const int incl = block_incl_scan<NT>(local, s_tmp);
    const int excl = incl - local;
    if (tid == NT - 1) s_tmp[NT / 32 + 3] = incl;
    if (excl < k && incl >= k) {
        int cum = excl;
        for (int i = 0; i < per; ++i) {
            const int r = tid * per + i;
            if (r >= nbins) break;
            const int c = bins[nbins - 1 - r];
            if (cum + c >= k) {
                s_tmp[NT / 32] = nbins - 1 - r;
                s_tmp[NT / 32 + 1] = cum;
                s_tmp[NT / 32 + 2] = c;
                break;
            }
            cum += c;
        }
    }
    __syncthreads();
    bucket = s_tmp[NT / 32];
    above = s_tmp[NT / 32 + 1];
    in_bucket = s_tmp[NT / 32 + 2];
    if (total) *total = s_tmp[NT / 32 + 3];
    __syncthreads();
}

// The 2048-bin histogram of one sequence into shared memory, all loads in flight at once.
template <int NT>
__device__ __forceinline__ void load_hist(uint32_t* h, const uint32_t* src) {
    constexpr int kVec = kHistBins / 4;  // uint4 loads
    constexpr int kPer = (kVec + NT - 1) / NT;
    uint4 v[kPer];
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
        const int i = threadIdx.x + k * NT;
        if (i < kVec) v[k] = __ldcg(reinterpret_cast<const uint4*>(src) + i);
    }
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
        const int i = threadIdx.x + k * NT;
        if (i < kVec) reinterpret_cast<uint4*>(h)[i] = v[k];
    }
}

constexpr int kSelThreads = 512;
static_assert(kSelThreads >= 256, "a thread per second-level bin");
constexpr int kSelPerThread = 8;
constexpr int kRankMax = 256;  // a threshold bucket this small is finished by ranking its keys
constexpr int kRadixBits = 8;  // digit of the passes after the histogram's top 11 bits

__device__ __forceinline__ uint64_t composite_key(float score, int t) {
    return (static_cast<uint64_t>(float_key(score)) << 32) |
           static_cast<uint64_t>(0xFFFFFFFFu - static_cast<uint32_t>(t));
}

// Shared-memory copies for the final step when they fit: the candidates' keys (reused by
// every radix pass) and the bitmap of chosen positions (no global atomics, fence or
// read-back); larger cases use the global copies.
constexpr int kFinCandSmem = 4096;
constexpr int kFinWordsSmem = 8192;
constexpr int kSelDynSmem = kFinCandSmem * 8 + kFinWordsSmem * 4 + kTopkMaxK * 4;

// Reserve consecutive slots of a shared counter for the lanes of a warp whose `pred` holds
// (one atomic per warp); returns the lane's slot, or -1. Every lane of the warp calls it.
__device__ __forceinline__ int warp_append(bool pred, int* counter) {
    const unsigned mask = __ballot_sync(0xffffffffu, pred);
    if (mask == 0u) return -1;
    const int lane = threadIdx.x & 31;
    const int leader = __ffs(mask) - 1;
    int base = 0;
    if (lane == leader) base = atomicAdd(counter, __popc(mask));
    base = __shfl_sync(0xffffffffu, base, leader);
    return pred ? base + __popc(mask & ((1u << lane) - 1u)) : -1;
}

// The top-k selection of each sequence, given its scores and the histogram of their top 11
// key bits. All blocks of a sequence split its scores: tokens whose bucket is above the
// k-th's are selected (positions), tokens inside it are candidates (64-bit keys: score key,
// then reversed position, so that ties go to the lower position). Each block classifies its
// scores in registers, counts both lists with one block scan and reserves its space with
// one atomic per list. The block that finishes last (a counter per sequence) narrows the
// candidates with radix passes until the bucket holding the threshold either holds exactly
// the keys still needed or at most kRankMax keys (then ranked against each other), marks all
// chosen positions in a bitmap, and writes each one at its rank in ascending order (chosen
// positions before its bitmap word, from per-word prefix counts, plus those below it in the
// word), then leaves histogram and counters zeroed for the next call.
__global__ void __launch_bounds__(kSelThreads) topk_select_kernel(const TopkParams p) {
    griddep_wait();
    __shared__ __align__(16) uint32_t h[kHistBins];
    __shared__ int tmp[kSelThreads / 32 + 4];
    __shared__ int s_nlist, s_nchosen;
    __shared__ int s_base[2];
    __shared__ int s_last;
    __shared__ uint32_t h2[256];  // this block's candidates by their next 8 key bits
    extern __shared__ uint64_t sel_dyn[];
    const int b = blockIdx.y;
    const int tid = threadIdx.x;
    const int L = load_len(p.lens, b, p.max_len, nullptr);
    int* cnt = p.counts + 4 * b;
    uint32_t* hist = p.hist + static_cast<size_t>(b) * kHistBins;
    int32_t* idx_out = p.topk_idx + static_cast<size_t>(b) * p.k;
    if (L <= p.k) {
        // every token is selected: block 0 writes the identity and clears the histogram
        if (blockIdx.x == 0) {
            for (int i = tid; i < p.k; i += kSelThreads) idx_out[i] = i < L ? i : -1;
            for (int i = tid; i < kHistBins; i += kSelThreads) hist[i] = 0;
            for (int i = tid; i < 256; i += kSelThreads)
                p.hist2[static_cast<size_t>(b) * 256 + i] = 0u;
            if (tid == 0) p.topk_count[b] = L;
        }
        return;
    }
    const float* sc = p.scores + static_cast<size_t>(b) * p.score_stride;
    int* sel = p.sel + static_cast<size_t>(b) * p.k;
    uint64_t* cand = p.cand + static_cast<size_t>(b) * p.max_len;
    constexpr int kSpan = kSelThreads * kSelPerThread;
    // all of this thread's scores of a span in flight at once (the first span's while the
    // histogram is read)
    float v[kSelPerThread];
    auto load_span = [&](int base) {
#pragma unroll
        for (int k = 0; k < kSelPerThread; ++k) {
            const int t = base + k * kSelThreads + tid;
            v[k] = t < L ? __ldcg(sc + t) : 0.f;
        }
    };
    load_span(blockIdx.x * kSpan);
    load_hist<kSelThreads>(h, hist);
    for (int i = tid; i < 256; i += kSelThreads) h2[i] = 0u;
    __syncthreads();
    int b1, above, in_b1, total;
    find_bucket<kSelThreads>(h, kHistBins, p.k, b1, above, in_b1, tmp, &total);
    // a histogram left by anything but this call's scores does not count L tokens
    if (tid == 0 && total != L) record_error(p.err, KVD_ERR_DEVICE_STATE);
    for (int base = blockIdx.x * kSpan; base < L; base += gridDim.x * kSpan) {
        if (base != blockIdx.x * kSpan) load_span(base);
        uint32_t cls = 0;  // 2 bits per element: 1 = selected, 2 = candidate
        int n_sel = 0, n_cand = 0;
#pragma unroll
        for (int k = 0; k < kSelPerThread; ++k) {
            const int t = base + k * kSelThreads + tid;
            const int bk = static_cast<int>(float_key(v[k]) >> 21);
            if (t < L && bk > b1) {
                cls |= 1u << (2 * k);
                ++n_sel;
            } else if (t < L && bk == b1) {
                cls |= 2u << (2 * k);
                ++n_cand;
            }
        }
        // both counts in one scan (each at most 4096 per block)
        const int packed = n_sel | (n_cand << 16);
        const int incl = block_incl_scan<kSelThreads>(packed, tmp);
        const int excl = incl - packed;
        if (tid == kSelThreads - 1) {
            // both lists' slots in one 64-bit atomic (selected count low, candidates high)
            const unsigned long long inc =
                (static_cast<unsigned long long>(incl >> 16) << 32) | static_cast<unsigned>(incl & 0xFFFF);
            const unsigned long long old =
                atomicAdd(reinterpret_cast<unsigned long long*>(cnt), inc);
            s_base[0] = static_cast<int>(static_cast<uint32_t>(old));
            s_base[1] = static_cast<int>(static_cast<uint32_t>(old >> 32));
        }
        __syncthreads();
        int si = s_base[0] + (excl & 0xFFFF), ci = s_base[1] + (excl >> 16);
        __syncthreads();  // s_base read before the next span overwrites it
#pragma unroll
        for (int k = 0; k < kSelPerThread; ++k) {
            const int t = base + k * kSelThreads + tid;
            const uint32_t c = (cls >> (2 * k)) & 3u;
            // a zeroed workspace keeps both lists inside their buffers (fewer than k tokens
            // lie above the k-th's bucket); counters left non-zero by other kernels must not
            // write outside them
            if (c == 1u) {
                if (si >= 0 && si < p.k) sel[si] = t;
                else record_error(p.err, KVD_ERR_DEVICE_STATE);
                ++si;
            } else if (c == 2u) {
                atomicAdd(&h2[(float_key(v[k]) >> 13) & 255u], 1u);
                if (ci >= 0 && ci < p.max_len) cand[ci] = composite_key(v[k], t);
                else record_error(p.err, KVD_ERR_DEVICE_STATE);
                ++ci;
            }
        }
    }
    // the candidates' next-digit counts go to the sequence's second-level histogram, so that
    // the finishing block starts its radix search one digit further
    __syncthreads();
    for (int i = tid; i < 256; i += kSelThreads)
        if (h2[i]) atomicAdd(p.hist2 + static_cast<size_t>(b) * 256 + i, h2[i]);
    // the last block of the sequence finishes it
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = atomicAdd(cnt + 2, 1) == static_cast<int>(gridDim.x) - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    uint64_t* keys = sel_dyn;
    uint32_t* sbits = reinterpret_cast<uint32_t*>(sel_dyn + kFinCandSmem);
    int* chosen = reinterpret_cast<int*>(sbits + kFinWordsSmem);  // chosen candidates' positions
    const int n_words = (L + 31) / 32;
    const bool bits_in_smem = n_words <= kFinWordsSmem;
    uint32_t* bits =
        bits_in_smem ? sbits : p.bitmap + static_cast<size_t>(b) * ((p.max_len + 31) / 32);
    // the candidate keys (as many as shared memory holds) and the selected positions, all in
    // flight together with the candidate count
    constexpr int kKeyPer = kFinCandSmem / kSelThreads;
    constexpr int kPosPer = kTopkMaxK / kSelThreads;
    static_assert(kKeyPer * kSelThreads == kFinCandSmem && kPosPer * kSelThreads == kTopkMaxK, "");
    const int n_pre = min(kFinCandSmem, p.max_len);
    const int above_c = min(max(above, 0), p.k - 1);
    uint64_t kv[kKeyPer];
    int tv[kPosPer];
#pragma unroll
    for (int r = 0; r < kKeyPer; ++r) {
        const int i = r * kSelThreads + tid;
        kv[r] = i < n_pre ? __ldcg(cand + i) : 0ull;
    }
#pragma unroll
    for (int r = 0; r < kPosPer; ++r) {
        const int i = r * kSelThreads + tid;
        tv[r] = i < above_c ? __ldcg(sel + i) : -1;
    }
    int nc = __ldcg(cnt + 1);
    // the second-level histogram, in flight with the lists
    const uint32_t h2v = tid < 256 ? __ldcg(p.hist2 + static_cast<size_t>(b) * 256 + tid) : 0u;
    if (nc < 0 || nc > L || above != above_c) {  // not a zeroed workspace
        if (tid == 0) record_error(p.err, KVD_ERR_DEVICE_STATE);
        nc = min(max(nc, 0), L);
        above = above_c;
    }
    const bool keys_in_smem = nc <= kFinCandSmem;
    if (keys_in_smem) {
#pragma unroll
        for (int r = 0; r < kKeyPer; ++r) {
            const int i = r * kSelThreads + tid;
            if (i < nc) keys[i] = kv[r];
        }
    }
    if (bits_in_smem)
        for (int i = tid; i < n_words; i += kSelThreads) sbits[i] = 0;
    __syncthreads();
    auto cand_key = [&](int i) -> uint64_t { return keys_in_smem ? keys[i] : __ldcg(cand + i); };
    auto key_pos = [](uint64_t ck) { return static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(ck)); };
    const int need0 = p.k - above;  // to take from the candidates (>= 1)
#pragma unroll
    for (int r = 0; r < kPosPer; ++r)
        if (tv[r] >= 0 && tv[r] < L) atomicOr(bits + (tv[r] >> 5), 1u << (tv[r] & 31));
    // radix passes (8-bit digits, a bin per thread) over the 64-bit key below its top 11
    // bits, until the bucket that holds the threshold either holds exactly the keys still
    // needed or is small enough to rank
    int need = need0;
    uint64_t prefix = static_cast<uint64_t>(b1);
    int done_bits = 11;
    int in_b = in_b1;
    // the first digit below the top 11 bits from the second-level histogram (when it counts
    // exactly the candidates: else the radix passes start from the top 11 bits)
    if (in_b != need && in_b > kRankMax) {
        if (tid < 256) h[tid] = h2v;
        __syncthreads();
        int bb, ab, ib, tot2;
        find_bucket<kSelThreads>(h, 256, need, bb, ab, ib, tmp, &tot2);
        if (tot2 == nc && nc == in_b1) {
            prefix = (prefix << 8) | static_cast<uint64_t>(bb);
            need -= ab;
            in_b = ib;
            done_bits = 19;
        } else if (tid == 0) {
            record_error(p.err, KVD_ERR_DEVICE_STATE);
        }
    }
    while (done_bits < 64 && in_b != need && in_b > kRankMax) {
        const int wdt = min(kRadixBits, 64 - done_bits);
        const int shift = 64 - done_bits - wdt;
        const int nb = 1 << wdt;
        for (int i = tid; i < nb; i += kSelThreads) h[i] = 0;
        __syncthreads();
        for (int i = tid; i < nc; i += kSelThreads) {
            const uint64_t ck = cand_key(i);
            if ((ck >> (64 - done_bits)) == prefix)
                atomicAdd(&h[static_cast<int>((ck >> shift) & (nb - 1))], 1u);
        }
        __syncthreads();
        int bb, ab;
        find_bucket<kSelThreads>(h, nb, need, bb, ab, in_b, tmp);
        prefix = (prefix << wdt) | static_cast<uint64_t>(bb);
        need -= ab;
        done_bits += wdt;
    }
    // keys above the bucket are chosen; the bucket's keys all are when it holds exactly the
    // ones needed, else they go to a short list and are chosen by rank (keys are distinct:
    // the position is part of the key). Chosen positions are marked in the bitmap and listed.
    const bool rank_bucket = in_b != need;
    uint64_t* lst = reinterpret_cast<uint64_t*>(h);  // kRankMax keys
    if (tid == 0) {
        s_nlist = 0;
        s_nchosen = 0;
    }
    __syncthreads();
    auto choose = [&](bool pick, int t) {  // all lanes of the warp take part
        const bool ok = pick && t >= 0 && t < L;
        const int slot = warp_append(ok, &s_nchosen);
        if (ok) {
            atomicOr(bits + (t >> 5), 1u << (t & 31));
            if (slot < kTopkMaxK) chosen[slot] = t;
        }
    };
    for (int i0 = 0; i0 < nc; i0 += kSelThreads) {
        const int i = i0 + tid;
        const uint64_t ck = i < nc ? cand_key(i) : 0ull;
        const uint64_t top = done_bits < 64 ? ck >> (64 - done_bits) : ck;
        const bool above_b = i < nc && (top > prefix || (top == prefix && !rank_bucket));
        choose(above_b, key_pos(ck));
        const int slot = warp_append(i < nc && top == prefix && rank_bucket, &s_nlist);
        if (slot >= 0 && slot < kRankMax) lst[slot] = ck;
    }
    __syncthreads();
    if (rank_bucket) {
        const int nl = min(s_nlist, kRankMax);
        if (tid == 0 && s_nlist != in_b) record_error(p.err, KVD_ERR_DEVICE_STATE);
        static_assert(kRankMax <= kSelThreads, "one list key per thread");
        const uint64_t ck = tid < nl ? lst[tid] : 0ull;
        int rank = 0;
        if (tid < nl)
            for (int jj = 0; jj < nl; ++jj) rank += lst[jj] > ck ? 1 : 0;
        choose(tid < nl && rank < need, key_pos(ck));
    }
    if (!bits_in_smem) __threadfence();  // global bit updates land in L2 first
    __syncthreads();
    if (tid == 0 && above + s_nchosen != p.k) record_error(p.err, KVD_ERR_DEVICE_STATE);
    if (bits_in_smem) {
        // every chosen position goes straight to its rank: the chosen positions before its
        // bitmap word (a prefix count per word, in the key buffer that is no longer read)
        // plus those below it in its own word
        int* wpre = reinterpret_cast<int*>(keys);
        static_assert(kFinCandSmem * 2 >= kFinWordsSmem, "");
        const int per = ((n_words + kSelThreads - 1) / kSelThreads + 3) & ~3;
        const int w0 = min(n_words, tid * per), w1 = min(n_words, w0 + per);
        int c = 0;
        for (int wi = w0; wi < w1; wi += 4) {
            if (wi + 4 <= w1) {
                const uint4 x = *reinterpret_cast<const uint4*>(sbits + wi);
                c += __popc(x.x) + __popc(x.y) + __popc(x.z) + __popc(x.w);
            } else {
                for (int r = wi; r < w1; ++r) c += __popc(sbits[r]);
            }
        }
        int run = block_incl_scan<kSelThreads>(c, tmp) - c;
        for (int wi = w0; wi < w1; wi += 4) {
            if (wi + 4 <= w1) {
                const uint4 x = *reinterpret_cast<const uint4*>(sbits + wi);
                int4 o;
                o.x = run;
                o.y = o.x + __popc(x.x);
                o.z = o.y + __popc(x.y);
                o.w = o.z + __popc(x.z);
                run = o.w + __popc(x.w);
                *reinterpret_cast<int4*>(wpre + wi) = o;
            } else {
                for (int r = wi; r < w1; ++r) {
                    wpre[r] = run;
                    run += __popc(sbits[r]);
                }
            }
        }
        __syncthreads();
        auto place = [&](int t) {
            const int wi = t >> 5;
            const int rk = wpre[wi] + __popc(sbits[wi] & ((1u << (t & 31)) - 1u));
            if (rk >= 0 && rk < p.k) idx_out[rk] = t;
        };
#pragma unroll
        for (int r = 0; r < kPosPer; ++r)
            if (tv[r] >= 0 && tv[r] < L) place(tv[r]);
        const int n_ch = min(s_nchosen, kTopkMaxK);
        for (int i = tid; i < n_ch; i += kSelThreads) place(chosen[i]);
    } else {
        // a bitmap in global memory: each warp owns a contiguous run of words, each lane 16
        // consecutive words a round; warp totals first, then one warp scan a round, after
        // which every lane writes its own positions and clears its words
        constexpr int kWarps = kSelThreads / 32;
        constexpr int kLaneWords = 16;
        const int warp = tid / 32, lane = tid % 32;
        const int wrun = ((n_words + kWarps - 1) / kWarps + kLaneWords - 1) & ~(kLaneWords - 1);
        const int wbeg = min(n_words, warp * wrun), wend = min(n_words, wbeg + wrun);
        int cnt_w = 0;
        for (int i = wbeg + kLaneWords * lane; i < wend; i += 32 * kLaneWords)
            for (int r = 0; r < kLaneWords && i + r < wend; ++r) cnt_w += __popc(__ldcg(bits + i + r));
        for (int off = 16; off; off >>= 1) cnt_w += __shfl_xor_sync(0xffffffffu, cnt_w, off);
        if (lane == 0) tmp[warp] = cnt_w;
        __syncthreads();
        int pos = 0;
        for (int w2 = 0; w2 < warp; ++w2) pos += tmp[w2];
        __syncthreads();
        for (int i0 = wbeg; i0 < wend; i0 += 32 * kLaneWords) {
            const int i = i0 + kLaneWords * lane;
            int c = 0;
            for (int r = 0; r < kLaneWords && i + r < wend; ++r) c += __popc(__ldcg(bits + i + r));
            int incl = c;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int n = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += n;
            }
            int q = pos + incl - c;
            for (int r = 0; r < kLaneWords && i + r < wend; ++r) {
                uint32_t m = __ldcg(bits + i + r);
                bits[i + r] = 0;  // leave the bitmap clear
                while (m) {
                    const int bit = __ffs(m) - 1;
                    if (q < p.k) idx_out[q] = (i + r) * 32 + bit;
                    ++q;
                    m &= m - 1;
                }
            }
            pos += __shfl_sync(0xffffffffu, incl, 31);
        }
    }
    if (tid == 0) p.topk_count[b] = p.k;
    // leave the histogram and counters zeroed for the next call
    for (int i = tid; i < kHistBins; i += kSelThreads) hist[i] = 0;
    for (int i = tid; i < 256; i += kSelThreads) p.hist2[static_cast<size_t>(b) * 256 + i] = 0u;
    if (tid < 3) cnt[tid] = 0;
}

}  // namespace

int idx_smem_bytes() { return kIdxSmem; }

int dsa_indexer_launch(const IdxParams& p, const CUtensorMap& tk, const CUtensorMap& tk128,
                       const CUtensorMap& tq, cudaStream_t stream) {
    static int configured = 0;
    if (!configured) {
        if (cudaFuncSetAttribute(dsa_indexer_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kIdxSmem) != cudaSuccess)
            return KVD_ERR_CUDA;
        configured = 1;
    }
    const int total = p.B * p.tiles_per_b;
    const int grid = std::min(total, kIdxCtasPerSm * num_sms());
    if (launch_kernel(dsa_indexer_kernel, dim3(grid), dim3(kIdxThreads), kIdxSmem, stream, tk,
                      tk128, tq, p) != cudaSuccess)
        return KVD_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? KVD_OK : KVD_ERR_CUDA;
}

int topk_launch(const TopkParams& p, bool need_hist, cudaStream_t stream) {
    const int blocks_per_b = std::max(1, std::min(64, (p.max_len + 4095) / 4096));
    if (need_hist && launch_kernel(topk_hist_kernel, dim3(blocks_per_b, p.B), dim3(256), 0,
                                   stream, p) != cudaSuccess)
        return KVD_ERR_CUDA;
    static int configured = 0;
    if (!configured) {
        if (cudaFuncSetAttribute(topk_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kSelDynSmem) != cudaSuccess)
            return KVD_ERR_CUDA;
        configured = 1;
    }
    const int sel_per_b =
        std::max(1, std::min(64, (p.max_len + kSelThreads * kSelPerThread - 1) /
                                     (kSelThreads * kSelPerThread)));
    if (launch_kernel(topk_select_kernel, dim3(sel_per_b, p.B), dim3(kSelThreads), kSelDynSmem,
                      stream, p) != cudaSuccess)
        return KVD_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? KVD_OK : KVD_ERR_CUDA;
}

}  // namespace kvd
