// delta_decode.cu -- one decode step of the gated delta rule (Gated DeltaNet / KDA) for
// many independent heads.
//
// What is computed ("All the attentions", sections 6 Gated DeltaNet and 7 KDA; "Attention
// Optimizations", KDA): each head keeps a fixed-size state S of dv rows by dk columns. One
// token's step fades S column by column (KDA: one decay a_j per key channel; Gated
// DeltaNet: one decay for the whole head), asks the faded memory what it returns for the
// key (S k), writes beta times the error v - S k along the key (outer product), and reads
// the output o = S q with the updated state.
//
// GB300: the step reads and writes the whole state once and does a few flops per element,
// so it is bound by HBM bandwidth. Rows are independent: a warp owns eight rows at a time
// (a lane holds dk/32 consecutive columns of each, read with 8- or 16-byte streaming
// loads), the two dot products per row are warp reductions, and the updated row is stored
// in place with streaming stores. A CTA covers 32 rows of one head, so even a few heads
// spread over every SM. There is no contraction here for the tensor cores.

#include "kvd_device.cuh"
#include "kvd_host.h"

namespace kvd {

namespace {

constexpr int kDeltaWarps = 4;
constexpr int kDeltaRows = 8;                            // rows a warp keeps in flight
constexpr int kDeltaRowsPerCta = kDeltaWarps * kDeltaRows;

// VEC consecutive floats of a lane (VEC = 2, 4 or 8), 8- or 16-byte aligned.
template <int VEC>
__device__ __forceinline__ void load_lane(const float* src, float (&x)[VEC]) {
    if constexpr (VEC == 2) {
        const float2 t = *reinterpret_cast<const float2*>(src);
        x[0] = t.x, x[1] = t.y;
    } else {
#pragma unroll
        for (int i = 0; i < VEC; i += 4) {
            const float4 t = *reinterpret_cast<const float4*>(src + i);
            x[i] = t.x, x[i + 1] = t.y, x[i + 2] = t.z, x[i + 3] = t.w;
        }
    }
}

// The state is touched once per step: evict-first loads and stores.
template <int VEC>
__device__ __forceinline__ void load_lane_stream(const float* src, float (&x)[VEC]) {
    if constexpr (VEC == 2) {
        const float2 t = __ldcs(reinterpret_cast<const float2*>(src));
        x[0] = t.x, x[1] = t.y;
    } else {
#pragma unroll
        for (int i = 0; i < VEC; i += 4) {
            const float4 t = __ldcs(reinterpret_cast<const float4*>(src + i));
            x[i] = t.x, x[i + 1] = t.y, x[i + 2] = t.z, x[i + 3] = t.w;
        }
    }
}

template <int VEC>
__device__ __forceinline__ void store_lane_stream(float* dst, const float (&x)[VEC]) {
    if constexpr (VEC == 2) {
        __stcs(reinterpret_cast<float2*>(dst), make_float2(x[0], x[1]));
    } else {
#pragma unroll
        for (int i = 0; i < VEC; i += 4)
            __stcs(reinterpret_cast<float4*>(dst + i),
                   make_float4(x[i], x[i + 1], x[i + 2], x[i + 3]));
    }
}

// Butterfly sums of kDeltaRows values across the warp (every lane gets every sum).
__device__ __forceinline__ void warp_sum_rows(float (&x)[kDeltaRows]) {
#pragma unroll
    for (int off = 16; off; off >>= 1)
#pragma unroll
        for (int r = 0; r < kDeltaRows; ++r) x[r] += __shfl_xor_sync(0xffffffffu, x[r], off);
}

template <int VEC>
__global__ void __launch_bounds__(kDeltaWarps * 32) delta_step_kernel(const DeltaParams p) {
    constexpr int dk = VEC * 32;
    griddep_wait();
    const int per_head = (p.dv + kDeltaRowsPerCta - 1) / kDeltaRowsPerCta;
    const int h = blockIdx.x / per_head;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int row0 = (blockIdx.x % per_head) * kDeltaRowsPerCta + warp * kDeltaRows;
    if (row0 >= p.dv) return;
    const int c0 = lane * VEC;  // this lane's first column

    float s[kDeltaRows][VEC];
    float* Sh = p.S + static_cast<size_t>(h) * p.dv * dk;
    // the rows first, so that their loads are in flight while the vectors arrive
#pragma unroll
    for (int r = 0; r < kDeltaRows; ++r) {
        if (row0 + r < p.dv) {
            load_lane_stream<VEC>(Sh + static_cast<size_t>(row0 + r) * dk + c0, s[r]);
        } else {
#pragma unroll
            for (int i = 0; i < VEC; ++i) s[r][i] = 0.f;
        }
    }
    float kk[VEC], qq[VEC], aa[VEC];
    load_lane<VEC>(p.k + static_cast<size_t>(h) * dk + c0, kk);
    load_lane<VEC>(p.q + static_cast<size_t>(h) * dk + c0, qq);
    if (p.a_per_channel) {
        load_lane<VEC>(p.a + static_cast<size_t>(h) * dk + c0, aa);
    } else {
        const float ah = p.a[h];
#pragma unroll
        for (int i = 0; i < VEC; ++i) aa[i] = ah;
    }
    const float beta = p.beta[h];
    float vr[kDeltaRows];
#pragma unroll
    for (int r = 0; r < kDeltaRows; ++r)
        vr[r] = row0 + r < p.dv ? p.v[static_cast<size_t>(h) * p.dv + row0 + r] : 0.f;

    // fade, then what the faded memory returns for k
    float pred[kDeltaRows];
#pragma unroll
    for (int r = 0; r < kDeltaRows; ++r) {
        float acc = 0.f;
#pragma unroll
        for (int i = 0; i < VEC; ++i) {
            s[r][i] *= aa[i];
            acc = fmaf(s[r][i], kk[i], acc);
        }
        pred[r] = acc;
    }
    warp_sum_rows(pred);
    // write the correction along k, then read with q
    float out[kDeltaRows];
#pragma unroll
    for (int r = 0; r < kDeltaRows; ++r) {
        const float w = beta * (vr[r] - pred[r]);
        float acc = 0.f;
#pragma unroll
        for (int i = 0; i < VEC; ++i) {
            s[r][i] = fmaf(w, kk[i], s[r][i]);
            acc = fmaf(s[r][i], qq[i], acc);
        }
        out[r] = acc;
    }
#pragma unroll
    for (int r = 0; r < kDeltaRows; ++r)
        if (row0 + r < p.dv)
            store_lane_stream<VEC>(Sh + static_cast<size_t>(row0 + r) * dk + c0, s[r]);
    warp_sum_rows(out);
    if (lane < kDeltaRows && row0 + lane < p.dv) {
        float mine = out[0];
#pragma unroll
        for (int r = 1; r < kDeltaRows; ++r)
            if (lane == r) mine = out[r];
        p.o[static_cast<size_t>(h) * p.dv + row0 + lane] = mine;
    }
}

}  // namespace

int delta_step_launch(const DeltaParams& p, cudaStream_t stream) {
    const long long per_head = (p.dv + kDeltaRowsPerCta - 1) / kDeltaRowsPerCta;
    const long long grid = per_head * p.n;
    if (grid > 0x7fffffffLL) return KVD_ERR_UNSUPPORTED;
    cudaError_t e;
    const dim3 g(static_cast<unsigned>(grid)), b(kDeltaWarps * 32);
    switch (p.dk) {
        case 64: e = launch_kernel(delta_step_kernel<2>, g, b, 0, stream, p); break;
        case 128: e = launch_kernel(delta_step_kernel<4>, g, b, 0, stream, p); break;
        case 256: e = launch_kernel(delta_step_kernel<8>, g, b, 0, stream, p); break;
        default: return KVD_ERR_UNSUPPORTED;
    }
    if (e != cudaSuccess) return KVD_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? KVD_OK : KVD_ERR_CUDA;
}

}  // namespace kvd
