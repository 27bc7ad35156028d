// kda_prefill_static_ws: kda_prefill with its workspace taken from a fixed
// device array that this library owns, so the caller passes inputs and
// outputs only and nothing is allocated on the call path.
//
// Some callers cannot allocate device memory themselves: a plugin that is
// handed only input and output pointers by its host application and has no
// allocator of its own, or a latency-critical serving loop that forbids
// cudaMalloc because it can synchronise the device.  This entry point serves
// them.  The source pages have no counterpart; the library adds it.
//
// The array is a file-scope __device__ array of KDA_STATIC_WORKSPACE_BYTES.
// Every GPU that loads the library holds it until the process exits.  Host
// code must not use the array's name as a device address: on the first call
// on a device (with that device current) the entry point resolves the address
// with cudaGetSymbolAddress and caches it per device.
#include <mutex>

#include "kda_common.h"

namespace kda {
namespace {

static __device__ __align__(256) unsigned char g_static_ws[KDA_STATIC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_ws_mutex;
void* g_ws_addr[kMaxDevices] = {};

// Device address of g_static_ws on the current device, resolved once.
kda_status static_ws_address(void** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        set_error("kda_prefill_static_ws: cudaGetDevice failed: %s", cudaGetErrorString(e));
        return KDA_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) {
        set_error("kda_prefill_static_ws: device %d out of range", dev);
        return KDA_ERR_UNSUPPORTED;
    }
    std::lock_guard<std::mutex> lock(g_ws_mutex);
    if (!g_ws_addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_static_ws);
        if (e != cudaSuccess || !p) {
            set_error("kda_prefill_static_ws: cudaGetSymbolAddress failed: %s",
                      cudaGetErrorString(e));
            return KDA_ERR_CUDA;
        }
        g_ws_addr[dev] = p;
    }
    *out = g_ws_addr[dev];
    return KDA_OK;
}

}  // namespace
}  // namespace kda

using namespace kda;

extern "C" kda_status kda_prefill_static_ws(float* state, const void* q, const void* k,
                                            const void* v, const void* g, const void* beta,
                                            float* o, int t, int t_pad, int chunk, float pad_fill,
                                            int heads, int head_dim, int in_dtype,
                                            int64_t qkv_row_stride, const int* cu_seqlens,
                                            int n_seqs, uint64_t stream) {
    // the same checks, and statuses, as kda_prefill before the size check
    const kda_status vs = validate_prefill("kda_prefill_static_ws", state, q, k, v, g, beta, o, t,
                                           t_pad, chunk, heads, head_dim, in_dtype,
                                           qkv_row_stride, cu_seqlens, n_seqs);
    if (vs != KDA_OK) return vs;
    const long long rows = cu_seqlens ? (long long)t : (long long)t_pad * n_seqs;
    const size_t need = kda_prefill_workspace_size(rows, n_seqs, chunk, heads, head_dim, in_dtype);
    KDA_REQUIRE(need <= (size_t)KDA_STATIC_WORKSPACE_BYTES, KDA_ERR_WORKSPACE,
                "kda_prefill_static_ws: this call needs %zu B of workspace; the static "
                "workspace holds %zu B (KDA_STATIC_WORKSPACE_BYTES)",
                need, (size_t)KDA_STATIC_WORKSPACE_BYTES);
    void* ws = nullptr;
    if (need > 0) {
        kda_status st = static_ws_address(&ws);
        if (st != KDA_OK) return st;
    }
    return kda_prefill(state, q, k, v, g, beta, o, t, t_pad, chunk, pad_fill, heads, head_dim,
                       in_dtype, qkv_row_stride, cu_seqlens, n_seqs, ws,
                       need > 0 ? (size_t)KDA_STATIC_WORKSPACE_BYTES : 0, stream);
}
