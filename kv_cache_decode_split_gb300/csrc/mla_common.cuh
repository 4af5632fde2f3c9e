// mla_common.cuh -- what the MLA decode kernels share: the DeepSeek-V3 shapes, the
// persistent schedule (every sequence's tiles in one list, cut into one contiguous range per
// cluster, each range met as one piece per sequence) and small warp helpers.
#pragma once

#include "kvd_device.cuh"
#include "kvd_host.h"

namespace kvd {
namespace mla {

constexpr int kH = 128;    // heads
constexpr int kDqk = 576;  // latent row: 512 value dims + 64 RoPE dims
constexpr int kDv = 512;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: O is rescaled only past 2^8

__device__ __forceinline__ float neg_inf() { return -__int_as_float(0x7f800000); }

// Part of a cluster's tile range inside one sequence: tokens [lo, hi) of sequence b, which
// holds `items` tokens (or selected tokens).
struct Piece {
    int b, items, lo, hi;
};
constexpr int kMaxPieces = 32;

// A cluster's schedule, built once into shared memory: its virtual tile range, the gap
// before each later sequence, the number of real tiles and the pieces (n_pieces < 0: more
// pieces than the table holds, walked from the sequence lengths instead).
struct Sched {
    long long t0, t1, gap;
    int n_tiles;
    int n_pieces;
    Piece piece[kMaxPieces];
};

// A range that moves on to the next sequence pays for an output write and a query load,
// worth about `gap` tiles of streaming. Ranges are cut in a virtual tile list with `gap`
// empty positions before every sequence but the first, so that such a range holds fewer
// tiles; only when ranges span at least 2 gap positions, so that every range still holds
// tiles.
__device__ __forceinline__ long long piece_gap(long long T, int B, int n_clusters, int gap) {
    const long long V = T + static_cast<long long>(gap) * (B - 1);
    return V >= 2LL * gap * n_clusters ? gap : 0;
}

// Work of one sequence: its item count (tokens, or selected tokens).
template <bool kSparse>
__device__ __forceinline__ int seq_items(const MlaParams& p, int b, int* err) {
    if (kSparse) return min(max(p.idx_count[b], 0), p.idx_stride);
    return load_len(p.seq_lens, b, p.max_len, err);
}

// Cluster c's range [t0, t1) of the list of all sequences' kTok-token tiles and the pieces
// it meets. One warp: the lanes load 32 sequences' lengths at a time and a warp scan turns
// their tile counts into tile offsets, so that the walk costs one memory round trip per 32
// sequences.
template <bool kSparse, int kTok>
__device__ void build_schedule(const MlaParams& p, int c, int n_clusters, Sched& sc, int lane,
                               int* err) {
    long long T = 0;
    for (int base = 0; base < p.B; base += 32) {
        const int bb = base + lane;
        int n = bb < p.B ? (seq_items<kSparse>(p, bb, err) + kTok - 1) / kTok : 0;
#pragma unroll
        for (int off = 16; off; off >>= 1) n += __shfl_xor_sync(0xffffffffu, n, off);
        T += n;
    }
    const long long X = piece_gap(T, p.B, n_clusters, p.gap);
    const long long V = T + X * (p.B - 1);
    const long long t0 = V * c / n_clusters, t1 = V * (c + 1) / n_clusters;
    long long run = 0;  // tiles of the sequences before this batch
    int np = 0, n_real = 0;
    for (int base = 0; base < p.B && run + X * base < t1; base += 32) {
        const int bb = base + lane;
        const int items = bb < p.B ? seq_items<kSparse>(p, bb, nullptr) : 0;
        const int n = (items + kTok - 1) / kTok;
        int incl = n;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += v;
        }
        const long long sb = run + incl - n + X * bb;  // the lane's sequence's first position
        const long long lo_t = max(t0, sb) - sb, hi_t = min(t1, sb + n) - sb;
        const bool has = bb < p.B && hi_t > lo_t;
        const unsigned m = __ballot_sync(0xffffffffu, has);
        const int slot = np + __popc(m & ((1u << lane) - 1u));
        if (has && slot < kMaxPieces)
            sc.piece[slot] = Piece{bb, items, static_cast<int>(lo_t) * kTok,
                                   min(static_cast<int>(hi_t) * kTok, items)};
        int nr = has ? static_cast<int>(hi_t - lo_t) : 0;
#pragma unroll
        for (int off = 16; off; off >>= 1) nr += __shfl_xor_sync(0xffffffffu, nr, off);
        n_real += nr;
        np += __popc(m);
        run += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) {
        sc.t0 = t0;
        sc.t1 = t1;
        sc.gap = X;
        sc.n_tiles = n_real;
        sc.n_pieces = np <= kMaxPieces ? np : -1;
    }
}

// Calls f(b, items, lo, hi, k) for the k-th piece of the range: tokens [lo, hi) of
// sequence b (multiples of kTok except at the end of the sequence).
template <bool kSparse, int kTok, typename F>
__device__ __forceinline__ void for_each_piece(const MlaParams& p, const Sched& sc, F&& f) {
    const int np = sc.n_pieces;
    if (np >= 0) {
        for (int k = 0; k < np; ++k) {
            const Piece pc = sc.piece[k];
            f(pc.b, pc.items, pc.lo, pc.hi, k);
        }
        return;
    }
    const long long t0 = sc.t0, t1 = sc.t1, X = sc.gap;
    long long base = 0;  // virtual position of sequence b's first tile
    int k = 0;
    for (int b = 0; b < p.B && base < t1; ++b) {
        const int items = seq_items<kSparse>(p, b, nullptr);
        const int n = (items + kTok - 1) / kTok;
        const long long lo_t = max(t0, base) - base, hi_t = min(t1, base + n) - base;
        if (hi_t > lo_t) {
            f(b, items, static_cast<int>(lo_t) * kTok,
              min(static_cast<int>(hi_t) * kTok, items), k);
            ++k;
        }
        base += n + X;
    }
}

// Transpose an 8 x 8 array of 16-byte chunks held by each group of eight lanes: lane i of the
// group holds chunk j of row i in ch[j] on entry and chunk i of row j on exit (three
// butterfly stages of shuffles). All lanes of the warp take part.
__device__ __forceinline__ void transpose8_chunks(float4 (&ch)[8], int lane) {
#pragma unroll
    for (int m = 4; m >= 1; m >>= 1) {
        const bool upper = (lane & m) != 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if (j & m) continue;
            const int hi = j | m;
            float4 send = upper ? ch[j] : ch[hi];
            float4 recv;
            recv.x = __shfl_xor_sync(0xffffffffu, send.x, m);
            recv.y = __shfl_xor_sync(0xffffffffu, send.y, m);
            recv.z = __shfl_xor_sync(0xffffffffu, send.z, m);
            recv.w = __shfl_xor_sync(0xffffffffu, send.w, m);
            if (upper)
                ch[j] = recv;
            else
                ch[hi] = recv;
        }
    }
}

}  // namespace mla
}  // namespace kvd
