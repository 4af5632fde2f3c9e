// gqa_static_ws.cu -- attn_decode_gqa_paged with a library-owned scratch buffer, for
// callers that cannot pass (or allocate) a workspace.
//
// Some callers hold only the input and output buffers and may not call cudaMalloc: a
// plugin inside a serving engine whose memory pool already owns all device memory and
// hands out nothing else, or a decode loop that must not take the implicit device-wide
// synchronisation that cudaMalloc / cudaFree bring. This entry point gives them the GQA
// decode without any allocation: the split-KV scratch (partial outputs, log-sum-exp
// values, completion counters) lives in a file-scope __device__ array of fixed size,
// which every GPU that loads this library holds until the process exits.

#include <mutex>

#include "kvd_host.h"

namespace {

// Maximum scratch of one call. Shapes whose split plan needs more are rejected with
// KVD_ERR_WORKSPACE_TOO_SMALL.
constexpr size_t kStaticWsBytes = 32u << 20;
constexpr int kMaxDevices = 64;

// The scratch itself. In host code this name is only a host-side stand-in for the device
// array, never a device address: the device address comes from cudaGetSymbolAddress.
__device__ __align__(256) unsigned char g_gqa_static_ws[kStaticWsBytes];

std::mutex g_mu;
void* g_ws_addr[kMaxDevices] = {};

// Device address of the scratch on the current device, looked up once per device.
int static_ws_addr(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return KVD_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return KVD_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_ws_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_gqa_static_ws) != cudaSuccess || !p) return KVD_ERR_CUDA;
        g_ws_addr[dev] = p;
    }
    *out = g_ws_addr[dev];
    return KVD_OK;
}

}  // namespace

extern "C" int attn_decode_gqa_paged_static_ws(const void* q, const void* k_pool,
                                               const void* v_pool, const int32_t* block_table,
                                               const int32_t* seq_lens, void* out,
                                               float* lse_out, int B, int Hq, int Hkv, int D,
                                               int page_size, int max_pages, int num_pages,
                                               float scale, int dtype, cudaStream_t stream) {
    // Every argument check runs before the shared array is touched: a rejected call leaves
    // it (and any call still running on it) alone.
    const int st = kvd::gqa_check(q, k_pool, v_pool, block_table, seq_lens, out, B, Hq, Hkv, D,
                                  page_size, max_pages, num_pages, scale, dtype, 0, 0, 0);
    if (st != KVD_OK) return st;
    kvd::GqaPlan plan;
    if (kvd::gqa_plan(B, Hq, Hkv, D, page_size, max_pages * page_size, 0, 0, dtype, &plan) !=
        KVD_OK)
        return KVD_ERR_UNSUPPORTED;
    if (plan.total > kStaticWsBytes) return KVD_ERR_WORKSPACE_TOO_SMALL;
    void* ws = nullptr;
    const int sa = static_ws_addr(&ws);
    if (sa != KVD_OK) return sa;
    // Every call shares the array and finds the previous call's contents in it: the error
    // flag and the completion counters must start at zero.
    if (cudaMemsetAsync(ws, 0, plan.off_lse, stream) != cudaSuccess) return KVD_ERR_CUDA;
    return kvd::gqa_run(q, k_pool, v_pool, block_table, seq_lens, out, lse_out, B, Hq, Hkv, D,
                        page_size, max_pages, num_pages, scale, dtype, 0, 0, nullptr, ws,
                        kStaticWsBytes, stream);
}
