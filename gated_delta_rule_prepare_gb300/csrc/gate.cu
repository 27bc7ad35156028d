// Forget gate and beta of the KDA core: the block pipeline's
// "kda_gate / sigmoid(b_proj)" step (glm5next_kda module index), from the
// forget-gate projection g_raw = f_b(f_a(h)) [T, heads * head_dim] BF16 and
// the b_proj output [T, heads] BF16 to the core's inputs of
// Glm5NextKdaWorkspace: gate [T, heads, head_dim], a log-decay bounded below,
// and beta [T, heads], the b_proj output after a sigmoid, with the
// Glm5NextKdaWeights parameters dt_bias [heads * head_dim] (one per channel)
// and a_log [heads] (one per head) and config.rs gate_lower_bound.  The pages
// give these inputs and the bound, not the formula; the reading taken:
//     g[r][c]    = lb * sigmoid(exp(a_log[h]) * (g_raw[r][c] + dt_bias[c]))
//     beta[r][h] = sigmoid(b[r][h])
// so that lb < g < 0 (lb <= g <= 0 once rounded).  FP32 arithmetic on channel
// pairs: sigmoid(z) = 1 / (1 + 2^(-z log2 e)) with the hardware 2^x and 1/x
// (a few ulp; the result's absolute error stays below 1e-5 |lb|), one
// rounding to the output type.
//
// A group is 8 channels of one head in one row.  The grid is one wave of
// resident CTAs whose thread count is a multiple of the groups in a row, so
// each thread keeps one column of groups (its channels, its head, their
// dt_bias and exp(a_log) in registers, no per-group index division) and walks
// its rows one grid apart, 4 rows per step, the step's four 16-byte BF16 loads
// issued before any of its arithmetic (each load instruction covers 512
// contiguous bytes of a warp); 16-byte stores; the thread holding a
// head's first group also writes that head's beta.  HBM-bound: 2 bytes in and
// 2 (BF16) or 4 (FP32) bytes out per channel.
#include <cuda_bf16.h>

#include <algorithm>

#include "f32x2.h"
#include "kda_common.h"
#include "tma_map.h"

namespace kda {
namespace {

constexpr int kGateThreads = 256;
constexpr int kGroupCh = 8;  // channels per group
constexpr int kUnits = 4;    // groups per thread

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&v);
}

// lb * sigmoid(c * (x + dt)) for a channel pair, given nc = -c log2 e.
__device__ __forceinline__ float2 gate2(float2 x, float2 dt, float nc, float lb) {
    const float2 t = mul2(add2(x, dt), make_float2(nc, nc));
    const float2 d = add2(make_float2(ex2_approx(t.x), ex2_approx(t.y)), make_float2(1.f, 1.f));
    return make_float2(lb * rcp_approx(d.x), lb * rcp_approx(d.y));
}
__device__ __forceinline__ float sigmoid_fast(float z) {
    return rcp_approx(1.0f + ex2_approx(z * -1.4426950408889634f));
}

__device__ __forceinline__ void gate_store(void* g_out, bool out_bf16, size_t o, const float* g) {
    if (out_bf16) {
        __stcs(reinterpret_cast<uint4*>(static_cast<uint16_t*>(g_out) + o),
               make_uint4(pack_bf16x2(g[0], g[1]), pack_bf16x2(g[2], g[3]),
                          pack_bf16x2(g[4], g[5]), pack_bf16x2(g[6], g[7])));
    } else {
        float* go = static_cast<float*>(g_out) + o;
        __stcs(reinterpret_cast<float4*>(go), make_float4(g[0], g[1], g[2], g[3]));
        __stcs(reinterpret_cast<float4*>(go + 4), make_float4(g[4], g[5], g[6], g[7]));
    }
}

// row_step = gridDim.x * kGateThreads / (heads * 16): the rows between two
// consecutive rows of one thread (the host makes the division exact).
__global__ void __launch_bounds__(kGateThreads)
gate_kernel(const uint16_t* __restrict__ g_raw, long long g_stride,
            const float* __restrict__ dt_bias, const float* __restrict__ a_log, float lb,
            const uint16_t* __restrict__ b_raw, long long b_stride, void* __restrict__ g_out,
            void* __restrict__ beta_out, bool out_bf16, long long rows, int heads,
            long long row_step) {
    pdl_wait();
    pdl_release();
    constexpr float kLog2e = 1.4426950408889634f;
    const unsigned per_row = (unsigned)heads * (D / kGroupCh);
    const unsigned g0 = blockIdx.x * kGateThreads + threadIdx.x;
    const unsigned r0 = g0 / per_row;
    if (r0 >= rows) return;
    const int c = (int)(g0 - r0 * per_row) * kGroupCh;
    const int h = c / D;
    const bool head_first = (c & (D - 1)) == 0;
    // -exp(a_log[h]) log2 e: the exponent's factor of this head
    const float nc = -ex2_approx(__ldg(a_log + h) * kLog2e) * kLog2e;
    const float4 b0 = __ldg(reinterpret_cast<const float4*>(dt_bias + c));
    const float4 b1 = __ldg(reinterpret_cast<const float4*>(dt_bias + c + 4));
    const float2 bias[4] = {make_float2(b0.x, b0.y), make_float2(b0.z, b0.w),
                            make_float2(b1.x, b1.y), make_float2(b1.z, b1.w)};
    const long long step = kUnits * row_step;

    for (long long r = r0; r < rows; r += step) {
        uint4 xs[kUnits];
#pragma unroll
        for (int u = 0; u < kUnits; ++u) {  // all of this step's loads first
            const long long rr = r + u * row_step;
            if (rr < rows) xs[u] = __ldcs(reinterpret_cast<const uint4*>(g_raw + rr * g_stride + c));
        }
#pragma unroll
        for (int u = 0; u < kUnits; ++u) {
            const long long rr = r + u * row_step;
            if (rr >= rows) break;
            const uint32_t xw[4] = {xs[u].x, xs[u].y, xs[u].z, xs[u].w};
            float g[8];
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                const float2 xv = make_float2(__uint_as_float(xw[p] << 16),
                                              __uint_as_float(xw[p] & 0xffff0000u));
                const float2 gv = gate2(xv, bias[p], nc, lb);
                g[2 * p] = gv.x;
                g[2 * p + 1] = gv.y;
            }
            gate_store(g_out, out_bf16, (size_t)rr * heads * D + c, g);
            if (head_first) {  // this head's beta
                const float bv = __uint_as_float((uint32_t)__ldg(b_raw + rr * b_stride + h) << 16);
                const float beta = sigmoid_fast(bv);
                const size_t bo = (size_t)rr * heads + h;
                if (out_bf16) {
                    const __nv_bfloat16 bb = __float2bfloat16_rn(beta);
                    static_cast<uint16_t*>(beta_out)[bo] = *reinterpret_cast<const uint16_t*>(&bb);
                } else {
                    static_cast<float*>(beta_out)[bo] = beta;
                }
            }
        }
    }
}

// Resident CTAs of gate_kernel per multiprocessor (queried once per process).
int gate_ctas_per_sm() {
    static int n = 0;
    if (!n) {
        int v = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, gate_kernel, kGateThreads, 0) !=
                cudaSuccess ||
            v < 1)
            v = 1;
        n = v;
    }
    return n;
}

}  // namespace
}  // namespace kda

using namespace kda;

extern "C" kda_status kda_gate(const uint16_t* g_raw, int64_t g_raw_stride, const float* dt_bias,
                               const float* a_log, float gate_lower_bound, const uint16_t* b_raw,
                               int64_t b_stride, void* g_out, void* beta_out, int out_dtype,
                               int64_t rows, int heads, int head_dim, uint64_t stream) {
    KDA_REQUIRE(head_dim == D, KDA_ERR_UNSUPPORTED, "kda_gate: head_dim %d unsupported (only 128)",
                head_dim);
    KDA_REQUIRE(rows >= 0 && heads >= 1, KDA_ERR_INVALID_ARG,
                "kda_gate: rows (%lld) must be >= 0 and heads (%d) >= 1", (long long)rows, heads);
    KDA_REQUIRE(out_dtype == KDA_F32 || out_dtype == KDA_BF16, KDA_ERR_INVALID_ARG,
                "kda_gate: out_dtype must be KDA_F32 or KDA_BF16");
    KDA_REQUIRE(gate_lower_bound < 0.f && gate_lower_bound > -INFINITY, KDA_ERR_INVALID_ARG,
                "kda_gate: gate_lower_bound must be finite and negative");
    KDA_REQUIRE(g_raw_stride >= (int64_t)heads * D && g_raw_stride % 8 == 0 && b_stride >= heads,
                KDA_ERR_INVALID_ARG,
                "kda_gate: g_raw_stride must be >= heads*128 and a multiple of 8, b_stride >= heads");
    if (rows == 0) return KDA_OK;  // nothing to read or write
    KDA_REQUIRE(g_raw && dt_bias && a_log && b_raw && g_out && beta_out, KDA_ERR_INVALID_ARG,
                "kda_gate: null pointer argument");
    KDA_REQUIRE(aligned16(g_raw) && aligned16(dt_bias) && aligned16(g_out), KDA_ERR_INVALID_ARG,
                "kda_gate: g_raw, dt_bias and g_out must be 16-byte aligned");
    // One wave of resident CTAs (fewer when the problem is small), rounded up
    // to a multiple of m so that the grid's threads cover whole rows of groups.
    const long long per_row = (long long)heads * (D / kGroupCh);
    long long a = per_row, b = kGateThreads;
    while (b) { const long long t = a % b; a = b; b = t; }
    const long long m = per_row / a;  // per_row / gcd(per_row, kGateThreads)
    const long long groups = rows * per_row;
    const int sms = sm_count();
    KDA_REQUIRE(sms > 0, KDA_ERR_CUDA, "kda_gate: no current CUDA device");
    long long ctas = (groups + (long long)kGateThreads * kUnits - 1) / ((long long)kGateThreads * kUnits);
    ctas = std::min(ctas, (long long)sms * gate_ctas_per_sm());
    ctas = (ctas + m - 1) / m * m;
    KDA_REQUIRE(ctas * kGateThreads <= 0xffffffffLL, KDA_ERR_INVALID_ARG,
                "kda_gate: heads (%d) too large", heads);
    KDA_REQUIRE(!fault_injected(), KDA_ERR_CUDA, "kda_gate: injected launch failure");
    launch_pdl(gate_kernel, dim3((unsigned)ctas), dim3(kGateThreads), 0, as_stream(stream), g_raw,
               (long long)g_raw_stride, dt_bias, a_log, gate_lower_bound, b_raw,
               (long long)b_stride, g_out, beta_out, out_dtype == KDA_BF16, (long long)rows, heads,
               ctas * kGateThreads / per_row);
    return launch_result("kda_gate");
}
