// dsa_indexer.cu -- the DSA lightning indexer and the top-k selection over its scores.
//
// What is computed ("Attention Optimizations", DSA / Computation Path; "All the
// attentions", section 5): for every cached token t of sequence b,
//   I_t = sum_h w_h * ReLU(q_h . k_t)        (64 heads x 128 dims, one 128-wide key per token)
// then the indices of the k largest I_t (ties to the lower position), in ascending order.
//
// Indexer (GB300): a persistent kernel, one CTA per SM, each CTA owning a contiguous range
// of 128-token tiles. One thread streams key tiles with TMA (128-byte swizzle) through a
// shared-memory ring; one thread issues tcgen05.mma with the tokens as M and the heads as
// N: D[128 tok x 64 heads] (TMEM, fp32) = K[128 x 128] * Q^T, double-buffered in tensor
// memory; four epilogue warps read one token row each (tcgen05.ld), apply ReLU and the head
// weights, write the fp32 score and count its top 11 key bits into a shared-memory
// histogram, the first pass of the radix selection.
//
// Selection: a filter kernel finds, from that histogram, the bucket holding the k-th
// largest score; tokens above it are selected and tokens inside it become candidates. A
// finalize kernel (one CTA per sequence) narrows the candidates with further radix passes
// over a 64-bit key (score key, then position reversed, so the order is total and ties go
// to the lower position), then sorts the k chosen positions ascending.

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
constexpr int kIdxStages = 5;
constexpr int kIdxThreads = 6 * 32;     // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
constexpr int kHistBins = 2048;         // top 11 key bits

struct IdxSmem {
    uint8_t stage[kIdxStages][kIdxTileBytes];   // 1024-aligned (offset 0)
    uint8_t qbuf[2][kIdxQBytes];
    uint32_t hist[kHistBins];
    float wv[2][kHi];
    uint64_t full[kIdxStages], empty[kIdxStages];
    uint64_t qfull[2], qempty[2], tfull[2], tempty[2], done;
    uint32_t tmem_base;
};
constexpr int kIdxSmem = static_cast<int>(sizeof(IdxSmem)) + 1024;

// The tiles a CTA owns: a contiguous slice of the flattened (sequence, tile) list.
struct TileRange {
    int begin, end;
};
__device__ __forceinline__ TileRange my_tiles(int total) {
    const long long G = gridDim.x, i = blockIdx.x;
    return TileRange{static_cast<int>(i * total / G), static_cast<int>((i + 1) * total / G)};
}

__global__ void __launch_bounds__(kIdxThreads, 1)
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

    if (warp == 0) {
        // ------------------------------------------------------------------ TMA producer
        if (lane == 0) {
            prefetch_tensormap(&tmK);
            prefetch_tensormap(&tmK128);
            prefetch_tensormap(&tmQ);
            const int bp = min(p.page_size, kItile);
            int cur_b = -1, L = 0;
            uint32_t g = 0, nq = 0;
            bool ok = true;
            for (int f = tr.begin; f < tr.end && ok; ++f) {
                const int b = f / p.tiles_per_b, j = f % p.tiles_per_b;
                if (b != cur_b) {
                    L = load_len(p.seq_lens, b, p.max_len, p.err);
                }
                if (j * kItile >= L) continue;
                if (b != cur_b) {
                    const int qs = nq & 1;
                    if (!(ok = mbar_wait(&sm.qempty[qs], ((nq >> 1) & 1) ^ 1, p.err))) break;
                    mbar_arrive_expect_tx(&sm.qfull[qs], kIdxQBytes);
                    tma_load_2d(sm.qbuf[qs], &tmQ, &sm.qfull[qs], 0, b * kHi);
                    tma_load_2d(sm.qbuf[qs] + kIdxQBytes / 2, &tmQ, &sm.qfull[qs], 64, b * kHi);
                    ++nq;
                    cur_b = b;
                }
                const int s = g % kIdxStages;
                if (!(ok = mbar_wait(&sm.empty[s], ((g / kIdxStages) & 1) ^ 1, p.err))) break;
                mbar_arrive_expect_tx(&sm.full[s], kIdxTileBytes);
                // physical rows of the tile's page pieces; one 32 KB instruction when they
                // are contiguous (adjacent pages, or pages of >= 128 tokens)
                int ys[kItile / 16];
                bool contiguous = true;
                for (int sub = 0; sub < kItile / bp; ++sub) {
                    const int t = j * kItile + sub * bp;
                    const int tc = t < L ? t : L - 1;  // rows past the end: a valid page
                    const int pg = load_page(p.block_table, p.max_pages, p.num_pages, b,
                                             tc / p.page_size, p.err);
                    ys[sub] = pg * p.page_size + (t % p.page_size);
                    if (sub > 0 && ys[sub] != ys[0] + sub * bp) contiguous = false;
                }
                if (contiguous && ys[0] + kItile <= p.num_pages * p.page_size) {
                    tma_load_3d(sm.stage[s], &tmK128, &sm.full[s], 0, ys[0], 0);
                } else {
                    for (int sub = 0; sub < kItile / bp; ++sub)
                        for (int half = 0; half < 2; ++half)
                            tma_load_2d(sm.stage[s] + half * (kIdxTileBytes / 2) + sub * bp * 128,
                                        &tmK, &sm.full[s], half * 64, ys[sub]);
                }
                ++g;
            }
            // copies still in flight complete before the CTA may exit
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
            for (int f = tr.begin; f < tr.end && ok; ++f) {
                const int b = f / p.tiles_per_b, j = f % p.tiles_per_b;
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
        auto flush_hist = [&](int b) {
            asm volatile("bar.sync 2, 128;" ::: "memory");
            for (int i = etid; i < kHistBins; i += 128) {
                const uint32_t c = sm.hist[i];
                if (c) {
                    atomicAdd(p.hist + static_cast<size_t>(b) * kHistBins + i, c);
                    sm.hist[i] = 0;
                }
            }
            asm volatile("bar.sync 2, 128;" ::: "memory");
        };
        for (int f = tr.begin; f < tr.end; ++f) {
            const int b = f / p.tiles_per_b, j = f % p.tiles_per_b;
            if (b != cur_b) L = load_len(p.seq_lens, b, p.max_len, nullptr);
            if (j * kItile >= L) continue;
            if (b != cur_b) {
                if (cur_b >= 0) flush_hist(cur_b);
                if (etid < kHi) sm.wv[nb & 1][etid] = p.w[static_cast<size_t>(b) * kHi + etid];
                asm volatile("bar.sync 2, 128;" ::: "memory");
                ++nb;
                cur_b = b;
            }
            const float* wv = sm.wv[(nb - 1) & 1];
            const int acc = nt & 1;
            if (!mbar_wait(&sm.tfull[acc], (nt >> 1) & 1, p.err)) break;
            tc_fence_after();
            const uint32_t taddr = tmem + (static_cast<uint32_t>(quad * 32) << 16) + acc * kHi;
            float score = 0.f;
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(taddr + half * 32, r);
                tmem_ld_wait(r);
#pragma unroll
                for (int c = 0; c < 32; ++c)
                    score = fmaf(wv[half * 32 + c], fmaxf(__uint_as_float(r[c]), 0.f), score);
            }
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
        if (cur_b >= 0) flush_hist(cur_b);
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
    __shared__ __align__(16) uint32_t h[kHistBins];
    const int b = blockIdx.y;
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
// bucket, the number of keys in higher buckets and the bucket's own count. All threads of
// the block take part; s_tmp holds at least NT/32 + 3 ints.
template <int NT>
__device__ void find_bucket(const uint32_t* bins, int nbins, int k, int& bucket, int& above,
                            int& in_bucket, int* s_tmp) {
    const int per = (nbins + NT - 1) / NT;  // each thread owns `per` bins counted from the top
    const int tid = threadIdx.x;
    int local = 0;
    for (int i = 0; i < per; ++i) {
        const int r = tid * per + i;
        if (r < nbins) local += bins[nbins - 1 - r];
    }
    const int incl = block_incl_scan<NT>(local, s_tmp);
    const int excl = incl - local;
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

// Tokens whose bucket is above the k-th's are selected; tokens inside it are candidates.
// Each block classifies its share of the scores in registers, counts both lists with one
// block scan and reserves its space with one atomic per list, so the two per-sequence
// counters see a few dozen atomics instead of one per warp and 32 scores.
constexpr int kFiltThreads = 256;
constexpr int kFiltPerThread = 16;
__global__ void __launch_bounds__(kFiltThreads) topk_filter_kernel(const TopkParams p) {
    __shared__ __align__(16) uint32_t h[kHistBins];
    __shared__ int tmp[kFiltThreads / 32 + 3];
    __shared__ int s_base[2];
    const int b = blockIdx.y;
    const int L = load_len(p.lens, b, p.max_len, nullptr);
    if (L <= p.k) return;  // everything is selected; the finalize kernel writes it
    load_hist<kFiltThreads>(h, p.hist + static_cast<size_t>(b) * kHistBins);
    __syncthreads();
    int b1, above, in_b1;
    find_bucket<kFiltThreads>(h, kHistBins, p.k, b1, above, in_b1, tmp);
    const float* sc = p.scores + static_cast<size_t>(b) * p.score_stride;
    int* sel = p.sel + static_cast<size_t>(b) * p.k;
    int* cand = p.cand + static_cast<size_t>(b) * p.max_len;
    constexpr int kSpan = kFiltThreads * kFiltPerThread;
    for (int base = blockIdx.x * kSpan; base < L; base += gridDim.x * kSpan) {
        // 2 bits per element: 1 = selected, 2 = candidate
        uint32_t cls = 0;
        int n_sel = 0, n_cand = 0;
#pragma unroll
        for (int k = 0; k < kFiltPerThread; ++k) {
            const int t = base + k * kFiltThreads + threadIdx.x;
            if (t < L) {
                const int bk = static_cast<int>(float_key(sc[t]) >> 21);
                if (bk > b1) {
                    cls |= 1u << (2 * k);
                    ++n_sel;
                } else if (bk == b1) {
                    cls |= 2u << (2 * k);
                    ++n_cand;
                }
            }
        }
        // both counts in one scan (each at most 4096 per block)
        const int packed = n_sel | (n_cand << 16);
        const int incl = block_incl_scan<kFiltThreads>(packed, tmp);
        const int excl = incl - packed;
        if (threadIdx.x == kFiltThreads - 1) {
            s_base[0] = (incl & 0xFFFF) ? atomicAdd(p.counts + 2 * b, incl & 0xFFFF) : 0;
            s_base[1] = (incl >> 16) ? atomicAdd(p.counts + 2 * b + 1, incl >> 16) : 0;
        }
        __syncthreads();
        int si = s_base[0] + (excl & 0xFFFF), ci = s_base[1] + (excl >> 16);
        __syncthreads();  // s_base read before the next span overwrites it
#pragma unroll
        for (int k = 0; k < kFiltPerThread; ++k) {
            const int t = base + k * kFiltThreads + threadIdx.x;
            const uint32_t c = (cls >> (2 * k)) & 3u;
            // a zeroed workspace keeps both lists inside their buffers (fewer than k tokens
            // lie above the k-th's bucket); counters left non-zero by other kernels must not
            // write outside them
            if (c == 1u) {
                if (si >= 0 && si < p.k) sel[si] = t;
                else record_error(p.err, KVD_ERR_DEVICE_STATE);
                ++si;
            } else if (c == 2u) {
                if (ci >= 0 && ci < p.max_len) cand[ci] = t;
                else record_error(p.err, KVD_ERR_DEVICE_STATE);
                ++ci;
            }
        }
    }
}

constexpr int kFinThreads = 1024;

__device__ __forceinline__ uint64_t composite_key(float score, int t) {
    return (static_cast<uint64_t>(float_key(score)) << 32) |
           static_cast<uint64_t>(0xFFFFFFFFu - static_cast<uint32_t>(t));
}

// Shared-memory copies of the finalize step when they fit: the candidates' composite keys
// (read once from global memory, then reused by every radix pass) and the bitmap of chosen
// positions (no global atomics, fence or read-back).
constexpr int kFinCandSmem = 4096;
constexpr int kFinWordsSmem = 8192;
constexpr int kFinDynSmem = kFinCandSmem * 8 + kFinWordsSmem * 4;

// One CTA per sequence: exact threshold among the candidates, then the output in
// ascending position order from a bitmap of the chosen positions and a prefix scan.
__global__ void __launch_bounds__(kFinThreads) topk_finalize_kernel(const TopkParams p) {
    __shared__ __align__(16) uint32_t h[kHistBins];
    __shared__ int tmp[kFinThreads / 32 + 3];
    extern __shared__ uint64_t fin_dyn[];
    uint64_t* keys = fin_dyn;
    uint32_t* sbits = reinterpret_cast<uint32_t*>(fin_dyn + kFinCandSmem);
    const int b = blockIdx.x;
    const int tid = threadIdx.x;
    const int L = load_len(p.lens, b, p.max_len, nullptr);
    int32_t* idx_out = p.topk_idx + static_cast<size_t>(b) * p.k;
    const int count = min(p.k, L);
    if (tid == 0) p.topk_count[b] = count;
    if (L <= p.k) {
        for (int i = tid; i < p.k; i += kFinThreads) idx_out[i] = i < L ? i : -1;
    } else {
        const float* sc = p.scores + static_cast<size_t>(b) * p.score_stride;
        const int* cand = p.cand + static_cast<size_t>(b) * p.max_len;
        const int* sel = p.sel + static_cast<size_t>(b) * p.k;
        const int n_words = (L + 31) / 32;
        const bool bits_in_smem = n_words <= kFinWordsSmem;
        uint32_t* bits = bits_in_smem
                             ? sbits
                             : p.bitmap + static_cast<size_t>(b) * ((p.max_len + 31) / 32);
        load_hist<kFinThreads>(h, p.hist + static_cast<size_t>(b) * kHistBins);
        if (bits_in_smem)
            for (int i = tid; i < n_words; i += kFinThreads) sbits[i] = 0;
        __syncthreads();
        int b1, above, in_b;
        find_bucket<kFinThreads>(h, kHistBins, p.k, b1, above, in_b, tmp);
        int nc = p.counts[2 * b + 1];
        if (nc < 0 || nc > L || above < 0 || above >= p.k) {  // not a zeroed workspace
            if (tid == 0) record_error(p.err, KVD_ERR_DEVICE_STATE);
            nc = min(max(nc, 0), L);
            above = min(max(above, 0), p.k - 1);
        }
        // the candidates' keys (a position outside [0, L) only follows a non-zeroed
        // workspace; its key is 0 and it is never chosen below)
        const bool keys_in_smem = nc <= kFinCandSmem;
        auto cand_key = [&](int i) -> uint64_t {
            if (keys_in_smem) return keys[i];
            const int t = cand[i];
            return (t >= 0 && t < L) ? composite_key(sc[t], t) : 0ull;
        };
        if (keys_in_smem) {
            for (int i = tid; i < nc; i += kFinThreads) {
                const int t = cand[i];
                keys[i] = (t >= 0 && t < L) ? composite_key(sc[t], t) : 0ull;
            }
            __syncthreads();
        }
        int need = p.k - above;  // to take from the candidates (>= 1)
        // radix passes over the 64-bit composite key below its top 11 bits, until the
        // bucket that holds the threshold holds exactly the keys still needed
        uint64_t prefix = static_cast<uint64_t>(b1);
        int done_bits = 11;
        while (done_bits < 64 && in_b != need) {
            const int wdt = min(11, 64 - done_bits);
            const int shift = 64 - done_bits - wdt;
            const int nb = 1 << wdt;
            for (int i = tid; i < nb; i += kFinThreads) h[i] = 0;
            __syncthreads();
            for (int i = tid; i < nc; i += kFinThreads) {
                const uint64_t ck = cand_key(i);
                if (ck != 0ull && (ck >> (64 - done_bits)) == prefix)
                    atomicAdd(&h[static_cast<int>((ck >> shift) & (nb - 1))], 1u);
            }
            __syncthreads();
            int bb, ab;
            find_bucket<kFinThreads>(h, nb, need, bb, ab, in_b, tmp);
            prefix = (prefix << wdt) | static_cast<uint64_t>(bb);
            need -= ab;
            done_bits += wdt;
        }
        // every key at or above T is chosen (T: the threshold prefix, low bits zero)
        const uint64_t T = done_bits < 64 ? prefix << (64 - done_bits) : prefix;
        for (int i = tid; i < above; i += kFinThreads) {
            const int t = sel[i];
            if (t >= 0 && t < L) atomicOr(bits + (t >> 5), 1u << (t & 31));
        }
        for (int i = tid; i < nc; i += kFinThreads) {
            const uint64_t ck = cand_key(i);
            if (ck != 0ull && ck >= T) {
                const int t = static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(ck));
                atomicOr(bits + (t >> 5), 1u << (t & 31));
            }
        }
        if (!bits_in_smem) __threadfence();  // global bit updates land in L2 first
        __syncthreads();
        // positions in ascending order: popcount prefix scan over the bitmap words
        const int per = (n_words + kFinThreads - 1) / kFinThreads;
        const int w0 = tid * per;
        int local = 0;
        for (int i = 0; i < per; ++i)
            if (w0 + i < n_words)
                local += __popc(bits_in_smem ? sbits[w0 + i] : __ldcg(bits + w0 + i));
        int pos = block_incl_scan<kFinThreads>(local, tmp) - local;
        for (int i = 0; i < per; ++i) {
            if (w0 + i >= n_words) break;
            uint32_t w = bits_in_smem ? sbits[w0 + i] : __ldcg(bits + w0 + i);
            if (!bits_in_smem) bits[w0 + i] = 0;  // leave the global bitmap clear
            while (w) {
                const int bit = __ffs(w) - 1;
                if (pos < p.k) idx_out[pos] = (w0 + i) * 32 + bit;
                ++pos;
                w &= w - 1;
            }
        }
    }
    // leave the histogram and counters zeroed for the next call
    __syncthreads();
    for (int i = tid; i < kHistBins; i += kFinThreads)
        p.hist[static_cast<size_t>(b) * kHistBins + i] = 0;
    if (tid < 2) p.counts[2 * b + tid] = 0;
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
    const int grid = total < num_sms() ? total : num_sms();
    dsa_indexer_kernel<<<grid, kIdxThreads, kIdxSmem, stream>>>(tk, tk128, tq, p);
    return cudaGetLastError() == cudaSuccess ? KVD_OK : KVD_ERR_CUDA;
}

int topk_launch(const TopkParams& p, bool need_hist, cudaStream_t stream) {
    const int blocks_per_b = std::max(1, std::min(64, (p.max_len + 4095) / 4096));
    if (need_hist) topk_hist_kernel<<<dim3(blocks_per_b, p.B), 256, 0, stream>>>(p);
    const int filt_per_b =
        std::max(1, std::min(64, (p.max_len + kFiltThreads * kFiltPerThread - 1) /
                                     (kFiltThreads * kFiltPerThread)));
    topk_filter_kernel<<<dim3(filt_per_b, p.B), kFiltThreads, 0, stream>>>(p);
    static int fin_configured = 0;
    if (!fin_configured) {
        if (cudaFuncSetAttribute(topk_finalize_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kFinDynSmem) != cudaSuccess)
            return KVD_ERR_CUDA;
        fin_configured = 1;
    }
    topk_finalize_kernel<<<p.B, kFinThreads, kFinDynSmem, stream>>>(p);
    return cudaGetLastError() == cudaSuccess ? KVD_OK : KVD_ERR_CUDA;
}

}  // namespace kvd
