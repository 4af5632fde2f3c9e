// cache_append.cu -- the newest token's rows written into the cache before attention.
//
// What is computed ("Attention Optimizations", DSA / Computation Path: the new token's
// latent row is written to the cache, then attention reads the cache; "All the attentions",
// section 4: a sliding window's cache is a rolling buffer of W entries, the newest entry
// replacing the oldest; "Attention Optimizations", Attention sinks: the first tokens stay):
// token t = L - 1 of sequence b goes to logical slot
//   r = t                                   (paged cache, every token kept), or
//   r = t for t < n_sink, else n_sink + (t - n_sink) mod W   (rolling cache of n_sink + W)
// whose physical row is page block_table[b][r / P], offset r % P. The rows are copied as
// bytes: the cache holds exactly what the caller computed.
//
// GB300: a few kilobytes per call; one thread per 16-byte piece of a row, K and V copied by
// the same thread. Indices read from device memory are checked before any store: a bad
// length or page id records an error and skips the write rather than clamping to a
// different page.

#include <algorithm>

#include "kvd_device.cuh"
#include "kvd_host.h"

namespace kvd {

namespace {

__global__ void __launch_bounds__(256) cache_append_kernel(const AppendParams p) {
    griddep_wait();
    const int chunks = p.row_bytes / 16;
    const long long total = static_cast<long long>(p.B) * p.H * chunks;
    const long long cap = p.window > 0 ? static_cast<long long>(p.n_sink) + p.window
                                       : static_cast<long long>(p.max_pages) * p.page_size;
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
         i < total; i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int c = static_cast<int>(i % chunks);
        const long long bh = i / chunks;
        const int h = static_cast<int>(bh % p.H), b = static_cast<int>(bh / p.H);
        const int L = p.seq_lens[b];
        if (L < 1 || (p.window <= 0 && L > cap)) {
            record_error(p.err, KVD_ERR_DEVICE_OOB);
            continue;
        }
        const int t = L - 1;
        const long long r = (p.window <= 0 || t < p.n_sink)
                                ? t
                                : p.n_sink + (static_cast<long long>(t) - p.n_sink) % p.window;
        const int pg = p.block_table[static_cast<size_t>(b) * p.max_pages + r / p.page_size];
        if (pg < 0 || pg >= p.num_pages) {
            record_error(p.err, KVD_ERR_DEVICE_OOB);
            continue;
        }
        const size_t dst =
            ((static_cast<size_t>(pg) * p.H + h) * p.page_size + r % p.page_size) * p.row_bytes +
            static_cast<size_t>(c) * 16;
        const size_t src = (static_cast<size_t>(b) * p.H + h) * p.row_bytes +
                           static_cast<size_t>(c) * 16;
        for (int k = 0; k < p.n_pools; ++k) {
            const uint4 v = *reinterpret_cast<const uint4*>(
                static_cast<const uint8_t*>(p.src[k]) + src);
            *reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.pool[k]) + dst) = v;
        }
    }
}

}  // namespace

int append_launch(const AppendParams& p, cudaStream_t stream) {
    const long long total = static_cast<long long>(p.B) * p.H * (p.row_bytes / 16);
    const long long blocks = std::min<long long>((total + 255) / 256, 8LL * num_sms());
    if (launch_kernel(cache_append_kernel, dim3(static_cast<unsigned>(std::max(1LL, blocks))),
                      dim3(256), 0, stream, p) != cudaSuccess)
        return KVD_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? KVD_OK : KVD_ERR_CUDA;
}

}  // namespace kvd
