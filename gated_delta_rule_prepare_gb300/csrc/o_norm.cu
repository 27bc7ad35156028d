// Sigmoid-gated RMSNorm of the KDA core output: the block pipeline's
// "sigmoid-gated RMSNorm(o_norm, g_b(g_a(h)))" step (glm5next_kda module
// index), from the workspace's FP32 pre-norm core [T, heads, head_dim] and the
// BF16 output gate [T, heads * head_dim] to the BF16 o_norm_out (Glm5NextKda
// Workspace), with the [head_dim] BF16 o_norm weight and rms_norm_eps
// (config.rs).  Per token and head:
//     out[j] = core[j] / sqrt(mean_j core[j]^2 + eps) * w[j] * sigmoid(gate[j])
// computed in FP32 and rounded once to BF16.
//
// One warp per 4 (token, head) units, their loads issued together: lane l
// holds channels 4l .. 4l + 3 of each, read as one 16-byte FP32 load and one
// 8-byte BF16 load and written as one 8-byte BF16 store; the sum of squares is
// a 5-step shuffle tree.  HBM-bound: 512 + 256 +
// 256 bytes per (token, head).
#include <cuda_bf16.h>

#include "kda_common.h"

namespace kda {
namespace {

constexpr int kWarps = 8;

__device__ __forceinline__ float2 bf2(uint32_t u) {
    return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
}

__device__ __forceinline__ uint32_t pack_bf2(float a, float b) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ float sigmoid(float x) { return 1.0f / (1.0f + __expf(-x)); }

constexpr int kUnits = 4;  // (token, head) units per warp, loads issued together

__global__ void __launch_bounds__(kWarps * 32)
o_norm_kernel(const float* __restrict__ core, const uint16_t* __restrict__ gate,
              const uint16_t* __restrict__ w, uint16_t* __restrict__ out, long long units,
              float eps) {
    pdl_wait();
    pdl_release();
    const int lane = threadIdx.x & 31;
    const long long u0 = ((long long)blockIdx.x * kWarps + (threadIdx.x >> 5)) * kUnits;
    if (u0 >= units) return;  // whole warps leave together
    const uint2 wv = __ldg(reinterpret_cast<const uint2*>(w + 4 * lane));
    const float2 w01 = bf2(wv.x), w23 = bf2(wv.y);
    float4 y[kUnits];
    uint2 gt[kUnits];
#pragma unroll
    for (int i = 0; i < kUnits; ++i) {
        const long long u = u0 + i;
        const size_t base = (size_t)(u < units ? u : u0) * D + 4 * lane;
        y[i] = __ldcs(reinterpret_cast<const float4*>(core + base));
        gt[i] = __ldcs(reinterpret_cast<const uint2*>(gate + base));
    }
#pragma unroll
    for (int i = 0; i < kUnits; ++i) {
        if (u0 + i >= units) break;  // uniform over the warp
        float ss = y[i].x * y[i].x;
        ss = __fmaf_rn(y[i].y, y[i].y, ss);
        ss = __fmaf_rn(y[i].z, y[i].z, ss);
        ss = __fmaf_rn(y[i].w, y[i].w, ss);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
        const float r = rsqrtf(ss * (1.0f / D) + eps);
        const float2 g01 = bf2(gt[i].x), g23 = bf2(gt[i].y);
        uint2 o;
        o.x = pack_bf2(y[i].x * r * w01.x * sigmoid(g01.x), y[i].y * r * w01.y * sigmoid(g01.y));
        o.y = pack_bf2(y[i].z * r * w23.x * sigmoid(g23.x), y[i].w * r * w23.y * sigmoid(g23.y));
        __stcs(reinterpret_cast<uint2*>(out + (size_t)(u0 + i) * D + 4 * lane), o);
    }
}

inline bool aligned8(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 7u) == 0; }

}  // namespace
}  // namespace kda

using namespace kda;

extern "C" kda_status kda_o_norm_gated(const float* core, const uint16_t* gate,
                                       const uint16_t* w, uint16_t* out, int64_t rows,
                                       int heads, int head_dim, float eps, uint64_t stream) {
    KDA_REQUIRE(head_dim == D, KDA_ERR_UNSUPPORTED,
                "kda_o_norm_gated: head_dim %d unsupported (only 128)", head_dim);
    KDA_REQUIRE(rows >= 0 && heads >= 1, KDA_ERR_INVALID_ARG,
                "kda_o_norm_gated: rows (%lld) must be >= 0 and heads (%d) >= 1",
                (long long)rows, heads);
    KDA_REQUIRE(eps >= 0.f, KDA_ERR_INVALID_ARG, "kda_o_norm_gated: eps must be >= 0");
    if (rows == 0) return KDA_OK;  // nothing to read or write
    KDA_REQUIRE(core && gate && w && out, KDA_ERR_INVALID_ARG,
                "kda_o_norm_gated: null pointer argument");
    KDA_REQUIRE(aligned16(core) && aligned8(gate) && aligned8(w) && aligned8(out),
                KDA_ERR_INVALID_ARG,
                "kda_o_norm_gated: core must be 16-byte aligned, gate, w and out 8-byte aligned");
    const long long units = (long long)rows * heads;
    const long long per_cta = (long long)kWarps * kUnits;
    KDA_REQUIRE(units / per_cta < 0x7fffffffLL, KDA_ERR_INVALID_ARG,
                "kda_o_norm_gated: problem too large");
    KDA_REQUIRE(!fault_injected(), KDA_ERR_CUDA, "kda_o_norm_gated: injected launch failure");
    launch_pdl(o_norm_kernel, dim3((unsigned)((units + per_cta - 1) / per_cta)), dim3(kWarps * 32),
               0, as_stream(stream), core, gate, w, out, units, eps);
    return launch_result("kda_o_norm_gated");
}
