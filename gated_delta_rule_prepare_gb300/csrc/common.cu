// Error reporting, status words and the version string of libkda.
#include "kda_common.h"

namespace kda {

static thread_local char g_last_error[512] = "";

void set_error(const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
    va_end(ap);
}

bool fault_injected(const char* what) {
    const char* s = getenv("KDA_FAULT_INJECT");
    return s && strcmp(s, what) == 0;
}

}  // namespace kda

extern "C" const char* kda_last_error(void) { return kda::g_last_error; }

extern "C" const char* kda_version(void) { return "libkda 0.1 (sm_103a)"; }

extern "C" kda_status kda_sync_status(uint64_t stream) {
    cudaError_t e = cudaStreamSynchronize(kda::as_stream(stream));
    if (e != cudaSuccess) {
        kda::set_error("kda_sync_status: stream error: %s", cudaGetErrorString(e));
        return KDA_ERR_CUDA;
    }
    unsigned a = 0, b = 0, c = 0;
    e = kda::read_and_clear_status_prefill(&a);
    if (e == cudaSuccess) e = kda::read_and_clear_status_conv(&b);
    if (e == cudaSuccess) e = kda::read_and_clear_status_prefill_tc(&c);
    a |= c;
    if (e != cudaSuccess) {
        kda::set_error("kda_sync_status: reading the status word failed: %s",
                       cudaGetErrorString(e));
        return KDA_ERR_CUDA;
    }
    if (a | b) {
        kda::set_error("kda_sync_status: device-side check failed (prefill 0x%x, conv 0x%x): %s",
                       a, b,
                       ((a | b) & kda::STATUS_TIMEOUT)      ? "a bounded wait timed out"
                       : ((a | b) & kda::STATUS_SMEM_ALIGN) ? "shared memory misaligned"
                                                            : "malformed cu_seqlens");
        return KDA_ERR_DEVICE;
    }
    return KDA_OK;
}
