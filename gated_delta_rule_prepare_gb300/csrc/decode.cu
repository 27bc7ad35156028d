// Single-token decode and the decode_k row walk of the KDA core.
//
// Glm5NextKdaLayer::decode / decode_k and Glm5NextKdaKernels::recurrent_smem:
// the per-head gated delta-rule step, streaming the FP32 [128 x 128] state of
// each (sequence, head) once in and once out (1R + 1W).
//
// Mapping: one CTA of 512 threads per (sequence, head).  Warp w owns key rows
// [8w, 8w + 8); lane l owns value columns [4l, 4l + 4) as one float4, so each
// warp-wide load or store is one contiguous 512-byte state row.  A thread
// keeps its 8 x 4 block of the state in registers for the whole step (and, in
// decode_k, for all k rows).  The two reductions over the key index (S^T k
// and S^T q) sum 8 rows inside each thread, then the 16 warp partials through
// shared memory in a fixed order.
//
// Bit-identity of decode_k with k serial decodes: both run the very same
// token_step() with explicit round-to-nearest intrinsics (no contraction
// choices left to the compiler), the same thread mapping and the same
// reduction order; an FP32 state written to memory and read back is exact.
#include "kda_common.h"

namespace kda {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kRows = D / kWarps;  // key rows per warp

struct TokenSmem {
    float dec[D];  // exp(g_i)
    float kk[D];   // k_i
    float bk[D];   // beta * k_i
    float qs[D];   // KDA_Q_SCALE * q_i
    float v[D];
    float u[D];    // v - S^T k (decayed S)
    float red[kWarps][D];
    // decode_k (FP32 inputs): the next token's raw inputs, copied in by
    // cp.async while the current token's step runs; channel c's entries are
    // written and read by thread c alone
    float nq[D], nk[D], nv[D], ng[D], nb[D];
};

// 4-byte asynchronous global -> shared copy, and the wait for this thread's
// outstanding ones.
__device__ __forceinline__ void cp_async4(float* dst_smem, const float* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(
                     static_cast<uint32_t>(__cvta_generic_to_shared(dst_smem))),
                 "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_all;" ::: "memory");
}

// One input element widened to FP32: FP32 as is, BF16 (raw bits) exactly.
__device__ __forceinline__ float ld_in(const float* p) { return __ldg(p); }
__device__ __forceinline__ float ld_in(const uint16_t* p) {
    return __uint_as_float(static_cast<uint32_t>(__ldg(p)) << 16);
}

// Stage one token of one head: threads 0..127 take one channel each.
template <typename TIn>
__device__ __forceinline__ void stage_token(TokenSmem& sm, const TIn* __restrict__ q,
                                            const TIn* __restrict__ k,
                                            const TIn* __restrict__ v,
                                            const TIn* __restrict__ g, float beta) {
    const int c = threadIdx.x;
    if (c < D) {
        const float kc = ld_in(k + c);
        sm.dec[c] = expf(ld_in(g + c));
        sm.kk[c] = kc;
        sm.bk[c] = __fmul_rn(beta, kc);
        sm.qs[c] = __fmul_rn(KDA_Q_SCALE, ld_in(q + c));
        sm.v[c] = ld_in(v + c);
    }
}

__device__ __forceinline__ void scale4(float4& s, float a) {
    s.x = __fmul_rn(s.x, a);
    s.y = __fmul_rn(s.y, a);
    s.z = __fmul_rn(s.z, a);
    s.w = __fmul_rn(s.w, a);
}

__device__ __forceinline__ void fma4(float4& acc, const float4& s, float a) {
    acc.x = __fmaf_rn(s.x, a, acc.x);
    acc.y = __fmaf_rn(s.y, a, acc.y);
    acc.z = __fmaf_rn(s.z, a, acc.z);
    acc.w = __fmaf_rn(s.w, a, acc.w);
}

// Sum the kWarps (16) warp partials of column j in warp order.
__device__ __forceinline__ float reduce_col(const TokenSmem& sm, int j) {
    float t = sm.red[0][j];
#pragma unroll
    for (int w = 1; w < kWarps; ++w) t = __fadd_rn(t, sm.red[w][j]);
    return t;
}

// One token step on the register-resident state block `s` (inputs staged and
// visible).  Writes o[j] for j < 128.  Ends with every thread past its last
// read of the staged inputs, so the caller may stage the next token.
__device__ __forceinline__ void token_step(float4 (&s)[kRows], TokenSmem& sm,
                                           float* __restrict__ o) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int i0 = warp * kRows;

    // decay rows, then partial S^T k over this warp's rows
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
        scale4(s[r], sm.dec[i0 + r]);
        fma4(acc, s[r], sm.kk[i0 + r]);
    }
    reinterpret_cast<float4*>(sm.red[warp])[lane] = acc;
    __syncthreads();
    if (threadIdx.x < D) {
        const int j = threadIdx.x;
        sm.u[j] = __fsub_rn(sm.v[j], reduce_col(sm, j));
    }
    __syncthreads();

    // rank-1 update, then partial S^T (scale q) over this warp's rows
    const float4 u = reinterpret_cast<const float4*>(sm.u)[lane];
    acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
        const float b = sm.bk[i0 + r];
        s[r].x = __fmaf_rn(b, u.x, s[r].x);
        s[r].y = __fmaf_rn(b, u.y, s[r].y);
        s[r].z = __fmaf_rn(b, u.z, s[r].z);
        s[r].w = __fmaf_rn(b, u.w, s[r].w);
        fma4(acc, s[r], sm.qs[i0 + r]);
    }
    reinterpret_cast<float4*>(sm.red[warp])[lane] = acc;
    __syncthreads();
    if (threadIdx.x < D) {
        const int j = threadIdx.x;
        o[j] = reduce_col(sm, j);
    }
}

__device__ __forceinline__ void pdl_enter() {
    pdl_wait();
    pdl_release();
}

__device__ __forceinline__ void load_state(float4 (&s)[kRows], const float* __restrict__ S) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
    for (int r = 0; r < kRows; ++r)
        s[r] = __ldcs(reinterpret_cast<const float4*>(S + (size_t)(warp * kRows + r) * D) + lane);
}

__device__ __forceinline__ void store_state(const float4 (&s)[kRows], float* __restrict__ S) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
    for (int r = 0; r < kRows; ++r)
        __stcs(reinterpret_cast<float4*>(S + (size_t)(warp * kRows + r) * D) + lane, s[r]);
}

__global__ void __launch_bounds__(kThreads, 2)
decode_kernel(float* __restrict__ state, const float* __restrict__ q,
              const float* __restrict__ k, const float* __restrict__ v,
              const float* __restrict__ g, const float* __restrict__ beta,
              float* __restrict__ o) {
    __shared__ TokenSmem sm;
    pdl_enter();
    const size_t nh = blockIdx.x;  // n * heads + h
    float* S = state + nh * (size_t)(D * D);
    float4 s[kRows];
    load_state(s, S);
    stage_token(sm, q + nh * D, k + nh * D, v + nh * D, g + nh * D, __ldg(beta + nh));
    __syncthreads();
    token_step(s, sm, o + nh * D);
    store_state(s, S);
}

struct SnapList {
    float* p[KDA_MAX_K];
};

// TIn: float (kda_decode_k, and kda_prefill's short FP32 sequences) or the
// BF16 bits of kda_prefill's short BF16 sequences, widened exactly.
template <typename TIn>
__global__ void __launch_bounds__(kThreads, 2)
decode_k_kernel(float* __restrict__ state, const TIn* __restrict__ q,
                const TIn* __restrict__ k, const TIn* __restrict__ v,
                const TIn* __restrict__ g, const TIn* __restrict__ beta,
                float* __restrict__ o, int heads, int krows, long long seq_rows, SnapList snaps,
                int n_snap) {
    __shared__ TokenSmem sm;
    pdl_enter();
    const size_t nh = blockIdx.x;
    const size_t n = nh / heads, h = nh % heads;
    float* S = state + nh * (size_t)(D * D);
    const int c = threadIdx.x;
    auto row_of = [&](int t) { return (n * (size_t)seq_rows + t) * heads + h; };
    // FP32 inputs: token t + 1's inputs travel while token t's step runs (the
    // first token's with the state), so no step waits on a global load
    auto prefetch = [&](int t) {
        if constexpr (sizeof(TIn) == 4) {
            if (c < D) {
                const size_t row = row_of(t);
                cp_async4(sm.nq + c, q + row * D + c);
                cp_async4(sm.nk + c, k + row * D + c);
                cp_async4(sm.nv + c, v + row * D + c);
                cp_async4(sm.ng + c, g + row * D + c);
                cp_async4(sm.nb + c, beta + row);
            }
        }
    };
    prefetch(0);
    float4 s[kRows];
    load_state(s, S);
    for (int t = 0; t < krows; ++t) {
        const size_t row = row_of(t);
        if constexpr (sizeof(TIn) == 4) {
            if (c < D) {  // stage_token's arithmetic, from the copies
                cp_async_wait_all();
                const float kc = sm.nk[c];
                sm.dec[c] = expf(sm.ng[c]);
                sm.kk[c] = kc;
                sm.bk[c] = __fmul_rn(sm.nb[c], kc);
                sm.qs[c] = __fmul_rn(KDA_Q_SCALE, sm.nq[c]);
                sm.v[c] = sm.nv[c];
            }
            if (t + 1 < krows) prefetch(t + 1);  // after this thread's reads of its channel
        } else {
            stage_token(sm, q + row * D, k + row * D, v + row * D, g + row * D,
                        ld_in(beta + row));
        }
        __syncthreads();
        token_step(s, sm, o + row * D);
        if (t < n_snap) store_state(s, snaps.p[t] + nh * (size_t)(D * D));
    }
    store_state(s, S);
}

kda_status check_common(const char* fn, float* state, const float* q, const float* k,
                        const float* v, const float* g, const float* beta, float* o,
                        int n_seqs, int heads, int head_dim) {
    KDA_REQUIRE(state && q && k && v && g && beta && o, KDA_ERR_INVALID_ARG,
                "%s: null pointer argument", fn);
    KDA_REQUIRE(aligned16(state) && aligned16(q) && aligned16(k) && aligned16(v) &&
                    aligned16(g) && aligned16(o),
                KDA_ERR_INVALID_ARG, "%s: state, q, k, v, g and o must be 16-byte aligned", fn);
    KDA_REQUIRE(head_dim == D, KDA_ERR_UNSUPPORTED, "%s: head_dim %d unsupported (only 128)", fn,
                head_dim);
    KDA_REQUIRE(n_seqs >= 1 && heads >= 1, KDA_ERR_INVALID_ARG,
                "%s: n_seqs (%d) and heads (%d) must be >= 1", fn, n_seqs, heads);
    KDA_REQUIRE((long long)n_seqs * heads <= 0x7fffffffLL, KDA_ERR_INVALID_ARG,
                "%s: n_seqs * heads too large", fn);
    KDA_REQUIRE(!fault_injected(), KDA_ERR_CUDA, "%s: injected launch failure", fn);
    return KDA_OK;
}

}  // namespace
}  // namespace kda

namespace kda {

// The decode_k row walk over n_seqs sequences of krows consecutive token rows,
// sequences seq_rows rows apart (arguments checked by the caller), no
// snapshots: kda_prefill's route for short sequences, FP32 (in_bf16 false) or
// BF16 inputs.
kda_status launch_row_walk(float* state, const void* q, const void* k, const void* v,
                           const void* g, const void* beta, float* o, int n_seqs, int krows,
                           long long seq_rows, int heads, bool in_bf16, cudaStream_t s) {
    if (in_bf16)
        launch_pdl(decode_k_kernel<uint16_t>, dim3(n_seqs * heads), dim3(kThreads), 0, s, state,
                   (const uint16_t*)q, (const uint16_t*)k, (const uint16_t*)v,
                   (const uint16_t*)g, (const uint16_t*)beta, o, heads, krows, seq_rows,
                   SnapList{}, 0);
    else
        launch_pdl(decode_k_kernel<float>, dim3(n_seqs * heads), dim3(kThreads), 0, s, state,
                   (const float*)q, (const float*)k, (const float*)v, (const float*)g,
                   (const float*)beta, o, heads, krows, seq_rows, SnapList{}, 0);
    return launch_result("kda_prefill (row walk)");
}

}  // namespace kda

using namespace kda;

extern "C" kda_status kda_decode(float* state, const float* q, const float* k, const float* v,
                                 const float* g, const float* beta, float* o, int n_seqs,
                                 int heads, int head_dim, uint64_t stream) {
    kda_status st = check_common("kda_decode", state, q, k, v, g, beta, o, n_seqs, heads,
                                 head_dim);
    if (st != KDA_OK) return st;
    launch_pdl(decode_kernel, dim3(n_seqs * heads), dim3(kThreads), 0, as_stream(stream), state,
               q, k, v, g, beta, o);
    return launch_result("kda_decode");
}

extern "C" kda_status kda_decode_k(float* state, const float* q, const float* k, const float* v,
                                   const float* g, const float* beta, float* o, int n_seqs,
                                   int krows, int heads, int head_dim, float* const* snapshots,
                                   int n_snap, uint64_t stream) {
    kda_status st = check_common("kda_decode_k", state, q, k, v, g, beta, o, n_seqs, heads,
                                 head_dim);
    if (st != KDA_OK) return st;
    KDA_REQUIRE(krows >= 1 && krows <= KDA_MAX_K, KDA_ERR_INVALID_ARG,
                "kda_decode_k: k = %d outside [1, %d]", krows, KDA_MAX_K);
    KDA_REQUIRE(n_snap >= 0 && n_snap <= krows, KDA_ERR_INVALID_ARG,
                "kda_decode_k: n_snap = %d outside [0, k = %d]", n_snap, krows);
    KDA_REQUIRE(n_snap == 0 || snapshots, KDA_ERR_INVALID_ARG,
                "kda_decode_k: snapshots is NULL with n_snap = %d", n_snap);
    SnapList sl = {};
    for (int t = 0; t < n_snap; ++t) {
        KDA_REQUIRE(snapshots[t] && aligned16(snapshots[t]), KDA_ERR_INVALID_ARG,
                    "kda_decode_k: snapshot %d is NULL or not 16-byte aligned", t);
        KDA_REQUIRE(snapshots[t] != state, KDA_ERR_INVALID_ARG,
                    "kda_decode_k: snapshot %d aliases the state", t);
        sl.p[t] = snapshots[t];
    }
    launch_pdl(decode_k_kernel<float>, dim3(n_seqs * heads), dim3(kThreads), 0, as_stream(stream),
               state, q, k, v, g, beta, o, heads, krows, (long long)krows, sl, n_snap);
    return launch_result("kda_decode_k");
}
