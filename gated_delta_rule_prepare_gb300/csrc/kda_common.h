// Internal helpers shared by the libkda translation units: error reporting,
// argument checks, the fault-injection hook and the device status words.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>

#include "kda.h"

namespace kda {

constexpr int D = KDA_HEAD_DIM;

// Thread-local last-error text (kda_last_error).
void set_error(const char* fmt, ...);

// Returns true when the environment variable KDA_FAULT_INJECT equals `what`
// (failure testing, read per call):
//   "launch"     -- the API reports a launch failure without enqueuing anything;
//   "ready_wait" -- the fused prefill grid's prepare CTAs release no ready
//                   flag and the chains' flag wait is cut to a few
//                   milliseconds, so the waits run out on the device, the
//                   kernel still returns, and kda_sync_status reports
//                   KDA_ERR_DEVICE (a bounded wait timed out).
bool fault_injected(const char* what = "launch");

// Values of the fused prefill grid's `fault` argument.
enum : uint32_t { FAULT_NONE = 0, FAULT_READY_WAIT = 1 };

inline cudaStream_t as_stream(uint64_t s) { return reinterpret_cast<cudaStream_t>(s); }

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Bits of the device status words (one per translation unit that checks).
enum : unsigned {
    STATUS_BAD_CU_SEQLENS = 1u << 0,
    STATUS_TIMEOUT = 1u << 1,  // a bounded wait on a copy or an MMA gave up
    STATUS_SMEM_ALIGN = 1u << 2,  // dynamic shared memory not 1024-byte aligned
};

// Each checking unit exposes a reader that returns and clears its word on the
// current device (synchronous; called from kda_sync_status only).
cudaError_t read_and_clear_status_prefill(unsigned* out);
cudaError_t read_and_clear_status_conv(unsigned* out);
cudaError_t read_and_clear_status_prefill_tc(unsigned* out);

// kda_prefill's argument checks, shared with kda_prefill_static_ws (prefill.cu).
kda_status validate_prefill(const char* fn, const float* state, const void* q, const void* k,
                            const void* v, const void* g, const void* beta, const float* o,
                            int t, int t_pad, int chunk, int heads, int head_dim, int in_dtype,
                            int64_t qkv_row_stride, const int* cu_seqlens, int n_seqs);

// Tensor-core prefill for BF16 inputs (prefill_tc.cu): its
// workspace size for `rows` token rows, and the launch (arguments validated by
// kda_prefill).
// Workspace of the tensor-core prefill; FP32 inputs add the FP16 copies of
// q, k and v the kernels read.
size_t prefill_tc_workspace_bytes(long long rows, int n_seqs, int heads, bool f32_in = false);
// Forget-gate inputs of kda_prefill_gated: g and beta are then the raw gate
// projection g_raw and the raw b_proj output, turned into the core's g and
// beta inside the prepare kernel.
struct PrefillGate {
    const float* dt_bias;  // [heads * 128]
    const float* a_log;    // [heads]
    float lb;              // gate_lower_bound
    long long g_stride;    // elements between token rows of g_raw
    long long b_stride;    // elements between token rows of b_raw
};
// The sigmoid-gated RMSNorm fused into the tensor-core prefill's epilogue
// (kda_prefill_o_norm): BF16 gate and output [rows][heads * 128] with their
// row pitches, the BF16 o_norm weight [128] and epsilon.
struct PrefillNorm {
    const uint16_t* gate;
    long long gate_stride;
    const uint16_t* w;
    float eps;
    uint16_t* out;
    long long out_stride;
};
kda_status launch_prefill_tc(float* state, const void* q, const void* k, const void* v,
                             const void* g, const void* beta, float* o, int t, int t_pad,
                             int heads, long long stride, const int* cu, int n_seqs,
                             void* workspace, cudaStream_t s, const PrefillGate* gate = nullptr,
                             const PrefillNorm* norm = nullptr, bool f32_in = false);

// decode_k's row walk (decode.cu) for kda_prefill's short FP32 sequences:
// n_seqs sequences of krows token rows, sequence n starting at row
// n * seq_rows of the [rows][heads][128] inputs and output.
kda_status launch_row_walk(float* state, const void* q, const void* k, const void* v,
                           const void* g, const void* beta, float* o, int n_seqs, int krows,
                           long long seq_rows, int heads, bool in_bf16, cudaStream_t s);

// Programmatic dependent launch.  Kernels launched with launch_pdl() may be
// scheduled while the previous kernel on the stream drains: pdl_wait() blocks
// until that kernel has finished and its writes are visible (call it before
// the first global access that may depend on it), pdl_release() lets the
// next such launch begin scheduling.  Without the attribute both are no-ops.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_release() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

#define KDA_REQUIRE(cond, code, ...)      \
    do {                                  \
        if (!(cond)) {                    \
            ::kda::set_error(__VA_ARGS__); \
            return (code);                \
        }                                 \
    } while (0)

// Check a launch; on failure record the CUDA error text.
inline kda_status launch_result(const char* what) {
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error("%s: launch failed: %s", what, cudaGetErrorString(e));
        return KDA_ERR_CUDA;
    }
    return KDA_OK;
}

}  // namespace kda
