// Front end of the KDA block: depthwise causal conv1d + SiLU, then L2 over the
// q and k channels (block pipeline "conv1d + SiLU -> L2(q,k only)"; fused at
// decode as causal_conv1d_update_l2norm, split at prefill into conv_prefill
// and l2_norm_bf16; config.rs: conv state of conv_kernel slots, L2 applied as
// 1/sqrt(sum + eps)).
//
// Kernel 1 (conv_silu_l2_kernel): one CTA per (head-sized group of 128
// channels, block of 32 consecutive tokens); a thread owns one channel and
// slides a register window of the last conv_kernel - 1 inputs along the
// tokens.  History before a sequence's first token comes from the conv
// state, which this kernel only reads.  The L2 sum over a q/k head's 128
// channels is a warp shuffle reduction plus a 4-warp smem reduction per token.
// Kernel 2 (conv_state_kernel): after kernel 1, each thread rewrites one
// (sequence, channel) state row to hold that sequence's last conv_kernel
// inputs, reading the old row first; separating it from kernel 1 keeps any
// CTA from reading a state row another CTA has already replaced.
#include <cuda_bf16.h>

#include "kda_common.h"

namespace kda {
namespace {

__device__ unsigned g_conv_status = 0;

constexpr int kTok = 32;        // tokens per CTA
constexpr int kThreads = D;     // two heads of 128 channels, two channels per thread

__device__ __forceinline__ float bf16_to_f32(uint16_t b) {
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

__device__ __forceinline__ uint16_t f32_to_bf16(float f) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

__device__ __forceinline__ float2 bf16x2_to_f32(uint32_t u) {
    return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
}

__device__ __forceinline__ uint32_t f32x2_to_bf16x2(float a, float b) {
    return (uint32_t)f32_to_bf16(a) | ((uint32_t)f32_to_bf16(b) << 16);
}

// Sequence holding packed token tau: largest n with cu[n] <= tau.  Returns
// false when the offsets do not bracket tau (malformed cu_seqlens).
__device__ __forceinline__ bool find_seq(const int* __restrict__ cu, int n_seqs, int tau,
                                         int& n, int& start) {
    int lo = 0, hi = n_seqs - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(cu + mid) <= tau) lo = mid;
        else hi = mid - 1;
    }
    n = lo;
    start = __ldg(cu + lo);
    const int end = __ldg(cu + lo + 1);
    return start >= 0 && start <= tau && tau < end;
}

__device__ __forceinline__ float silu(float a) {
    return __fdividef(a, 1.0f + __expf(-a));  // rounded to BF16 by the caller
}

template <int K>
__global__ void __launch_bounds__(kThreads)
conv_silu_l2_kernel(const float* __restrict__ conv_state, const uint16_t* __restrict__ x,
                    const uint16_t* __restrict__ w, uint16_t* __restrict__ out, int total,
                    int t_per_seq, const int* __restrict__ cu, int n_seqs, int heads,
                    float l2_eps) {
    __shared__ float red[kThreads / 32][kTok];
    const int pair = blockIdx.x;  // head groups 2 pair and 2 pair + 1 of the 3H groups
    const int c = pair * 2 * D + 2 * threadIdx.x;  // first of this thread's two channels
    const size_t conv_dim = (size_t)3 * heads * D;
    // The first 2H groups (q and k) always pair up fully; with an odd head count the
    // last v pair has only one group, and its second half of threads stays idle.
    if ((size_t)c >= conv_dim) return;
    const bool normalise = pair < heads;
    float w0[K], w1[K];
#pragma unroll
    for (int j = 0; j < K; ++j) {
        w0[j] = bf16_to_f32(__ldg(w + (size_t)c * K + j));
        w1[j] = bf16_to_f32(__ldg(w + (size_t)(c + 1) * K + j));
    }

    const int tok0 = blockIdx.y * kTok;
    const int tok_end = min(total, tok0 + kTok);
    // The block's tokens are consecutive: find the first one's sequence once,
    // then step to the next sequence whenever a token reaches its end.
    int n, start, end;
    bool ok = true;
    if (cu) {
        ok = find_seq(cu, n_seqs, tok0, n, start);
        end = ok ? __ldg(cu + n + 1) : tok0;
    } else {
        n = tok0 / t_per_seq;
        start = n * t_per_seq;
        end = start + t_per_seq;
    }
    // All of the block's inputs first, as independent loads.
    const uint32_t* xp = reinterpret_cast<const uint32_t*>(x + (size_t)tok0 * conv_dim + c);
    const size_t step = conv_dim / 2;  // one token row, in channel pairs
    float2 xs[kTok];
#pragma unroll
    for (int m = 0; m < kTok; ++m)
        xs[m] = (tok0 + m < tok_end) ? bf16x2_to_f32(__ldg(xp + m * step)) : make_float2(0.f, 0.f);
    // h0[j], h1[j]: the two channels' inputs at token tau - (K - 1) + j.
    float h0[K > 1 ? K - 1 : 1], h1[K > 1 ? K - 1 : 1];
    auto state_history = [&]() {  // a sequence's first token: history from its state
        const float* st = conv_state + ((size_t)n * conv_dim + c) * K;
#pragma unroll
        for (int j = 0; j < K - 1; ++j) {
            h0[j] = __ldg(st + j + 1);
            h1[j] = __ldg(st + K + j + 1);
        }
    };
    if (ok) {
        const float* st = conv_state + ((size_t)n * conv_dim + c) * K;
#pragma unroll
        for (int j = 0; j < K - 1; ++j) {
            const int src = tok0 - (K - 1) + j;
            if (src >= start) {
                const float2 v = bf16x2_to_f32(__ldg(reinterpret_cast<const uint32_t*>(
                    x + (size_t)src * conv_dim + c)));
                h0[j] = v.x;
                h1[j] = v.y;
            } else {
                h0[j] = __ldg(st + K + (src - start));
                h1[j] = __ldg(st + K + K + (src - start));
            }
        }
    }
    float2 y[kTok];
#pragma unroll
    for (int m = 0; m < kTok; ++m) {
        const int tau = tok0 + m;
        y[m] = make_float2(0.f, 0.f);
        if (!ok || tau >= tok_end) continue;
        if (tau >= end) {  // a new sequence starts at tau (skipping empty ones)
            if (cu) {
                while (n + 1 < n_seqs && __ldg(cu + n + 1) <= tau) ++n;
                start = __ldg(cu + n);
                end = __ldg(cu + n + 1);
                if (!(start == tau && tau < end)) {
                    ok = false;
                    continue;
                }
            } else {
                ++n;
                start = n * t_per_seq;
                end = start + t_per_seq;
            }
            state_history();
        }
        float a0 = 0.f, a1 = 0.f;
#pragma unroll
        for (int j = 0; j < K - 1; ++j) {
            a0 = __fmaf_rn(w0[j], h0[j], a0);
            a1 = __fmaf_rn(w1[j], h1[j], a1);
        }
        a0 = __fmaf_rn(w0[K - 1], xs[m].x, a0);
        a1 = __fmaf_rn(w1[K - 1], xs[m].y, a1);
#pragma unroll
        for (int j = 0; j + 1 < K - 1; ++j) {
            h0[j] = h0[j + 1];
            h1[j] = h1[j + 1];
        }
        if constexpr (K > 1) {
            h0[K - 2] = xs[m].x;
            h1[K - 2] = xs[m].y;
        }
        y[m] = make_float2(silu(a0), silu(a1));
    }
    if (!ok && threadIdx.x == 0) atomicOr(&g_conv_status, STATUS_BAD_CU_SEQLENS);

    if (normalise) {  // uniform per CTA: both heads are q/k heads or neither is
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
        for (int m = 0; m < kTok; ++m) {
            float p = y[m].x * y[m].x + y[m].y * y[m].y;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) p += __shfl_xor_sync(0xffffffffu, p, off);
            if (lane == 0) red[warp][m] = p;
        }
        __syncthreads();
        const int hw = warp & ~1;  // the two warps of this thread's head
#pragma unroll
        for (int m = 0; m < kTok; ++m) {
            const float inv = rsqrtf(red[hw][m] + red[hw + 1][m] + l2_eps);
            y[m].x *= inv;
            y[m].y *= inv;
        }
    }
    uint32_t* op = reinterpret_cast<uint32_t*>(out + (size_t)tok0 * conv_dim + c);
#pragma unroll
    for (int m = 0; m < kTok; ++m)
        if (tok0 + m < tok_end) op[m * step] = f32x2_to_bf16x2(y[m].x, y[m].y);
}

template <int K>
__global__ void conv_state_kernel(float* __restrict__ conv_state, const uint16_t* __restrict__ x,
                                  int total, int t_per_seq, const int* __restrict__ cu,
                                  int n_seqs, int heads) {
    const size_t conv_dim = (size_t)3 * heads * D;
    const size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= (size_t)n_seqs * conv_dim) return;
    const int n = (int)(idx / conv_dim);
    const size_t c = idx % conv_dim;
    int start, end;
    if (cu) {
        start = __ldg(cu + n);
        end = __ldg(cu + n + 1);
        bool ok = start >= 0 && start <= end && end <= total;
        if (n == 0) ok = ok && start == 0;
        if (n == n_seqs - 1) ok = ok && end == total;
        if (!ok) {
            atomicOr(&g_conv_status, STATUS_BAD_CU_SEQLENS);
            return;
        }
    } else {
        start = n * t_per_seq;
        end = start + t_per_seq;
    }
    const int len = end - start;
    float* st = conv_state + idx * K;
    float old[K], nw[K];
#pragma unroll
    for (int j = 0; j < K; ++j) old[j] = st[j];
#pragma unroll
    for (int j = 0; j < K; ++j) {
        const int rel = len - K + j;  // position relative to the sequence start
        nw[j] = (rel >= 0) ? bf16_to_f32(__ldg(x + (size_t)(start + rel) * conv_dim + c))
                           : old[(j + len < K) ? j + len : K - 1];
    }
#pragma unroll
    for (int j = 0; j < K; ++j) st[j] = nw[j];
}

template <int K>
kda_status launch(float* conv_state, const uint16_t* x, const uint16_t* w, uint16_t* out,
                  int total, int t_per_seq, const int* cu, int n_seqs, int heads, float eps,
                  cudaStream_t s) {
    dim3 grid((3 * heads + 1) / 2, (total + kTok - 1) / kTok);
    conv_silu_l2_kernel<K><<<grid, kThreads, 0, s>>>(conv_state, x, w, out, total, t_per_seq,
                                                      cu, n_seqs, heads, eps);
    kda_status st = launch_result("kda_conv_silu_l2 (conv)");
    if (st != KDA_OK) return st;
    const size_t rows = (size_t)n_seqs * 3 * heads * D;
    conv_state_kernel<K><<<(unsigned)((rows + 255) / 256), 256, 0, s>>>(conv_state, x, total,
                                                                        t_per_seq, cu, n_seqs,
                                                                        heads);
    return launch_result("kda_conv_silu_l2 (state)");
}

}  // namespace

cudaError_t read_and_clear_status_conv(unsigned* out) {
    unsigned zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(out, g_conv_status, sizeof(unsigned));
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_conv_status, &zero, sizeof(unsigned));
    return e;
}

}  // namespace kda

using namespace kda;

extern "C" kda_status kda_conv_silu_l2(float* conv_state, const uint16_t* x, const uint16_t* w,
                                       uint16_t* out, int t, int n_seqs, const int* cu_seqlens,
                                       int conv_kernel, float l2_eps, int heads, int head_dim,
                                       uint64_t stream) {
    KDA_REQUIRE(conv_state && x && w && out, KDA_ERR_INVALID_ARG,
                "kda_conv_silu_l2: null pointer argument");
    KDA_REQUIRE(aligned16(conv_state) && aligned16(x) && aligned16(out), KDA_ERR_INVALID_ARG,
                "kda_conv_silu_l2: conv_state, x and out must be 16-byte aligned");
    KDA_REQUIRE(head_dim == D, KDA_ERR_UNSUPPORTED,
                "kda_conv_silu_l2: head_dim %d unsupported (only 128)", head_dim);
    KDA_REQUIRE(heads >= 1 && n_seqs >= 1 && t >= 1, KDA_ERR_INVALID_ARG,
                "kda_conv_silu_l2: heads (%d), n_seqs (%d) and t (%d) must be >= 1", heads,
                n_seqs, t);
    KDA_REQUIRE(conv_kernel >= 1 && conv_kernel <= KDA_MAX_CONV_KERNEL, KDA_ERR_UNSUPPORTED,
                "kda_conv_silu_l2: conv_kernel %d outside [1, %d]", conv_kernel,
                KDA_MAX_CONV_KERNEL);
    KDA_REQUIRE(l2_eps >= 0.f, KDA_ERR_INVALID_ARG, "kda_conv_silu_l2: l2_eps must be >= 0");
    const long long total = cu_seqlens ? (long long)t : (long long)t * n_seqs;
    KDA_REQUIRE(total <= 0x7fffffffLL && (long long)3 * heads * D * total < (1LL << 46),
                KDA_ERR_INVALID_ARG, "kda_conv_silu_l2: problem too large");
    KDA_REQUIRE((total + kTok - 1) / kTok <= 65535, KDA_ERR_INVALID_ARG,
                "kda_conv_silu_l2: more than %d tokens in one call", 65535 * kTok);
    KDA_REQUIRE(!fault_injected(), KDA_ERR_CUDA, "kda_conv_silu_l2: injected launch failure");
    cudaStream_t s = as_stream(stream);
    const int tps = cu_seqlens ? 0 : t;
    switch (conv_kernel) {
        case 1: return launch<1>(conv_state, x, w, out, (int)total, tps, cu_seqlens, n_seqs, heads, l2_eps, s);
        case 2: return launch<2>(conv_state, x, w, out, (int)total, tps, cu_seqlens, n_seqs, heads, l2_eps, s);
        case 3: return launch<3>(conv_state, x, w, out, (int)total, tps, cu_seqlens, n_seqs, heads, l2_eps, s);
        default: return launch<4>(conv_state, x, w, out, (int)total, tps, cu_seqlens, n_seqs, heads, l2_eps, s);
    }
}
