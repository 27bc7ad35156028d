// Chunked prefill of the KDA core (Glm5NextKdaLayer::prefill_with_pad_fill;
// Glm5NextKdaKernels::chunk_prepare and chunk_scan; config.rs smem_prepare /
// smem_scan for the per-chunk working set).
//
// For a chunk of L <= C tokens of one head, starting from state S, with
// Gamma_r = sum_{s<=r} g_s (per key channel) and qh = KDA_Q_SCALE * q:
//   A_rs = beta_s sum_i k_ri k_si exp(Gamma_ri - Gamma_si)     (s < r)
//   P_rs = beta_s sum_i qh_ri k_si exp(Gamma_ri - Gamma_si)    (s <= r)
//   T    = (I + A)^-1                 (unit lower triangular)
//   Ktil = exp(Gamma) (.) k,  Qtil = exp(Gamma) (.) qh,
//   Khat_s = exp(Gamma_{L-1} - Gamma_s) (.) k_s
//   U    = T (V - Ktil S)             (the chunk's delta-rule residuals)
//   O    = Qtil S + P U
//   S   <- diag(exp(Gamma_{L-1})) S + Khat^T diag(beta) U
// The V-independent part (Gamma, A, P, T, Ktil, Qtil, Khat) is the "prepare"
// stage; the U / O / S recurrence over chunks is the "scan".
//
// This is the SIMT FP32 version: one CTA per (sequence, head, 32-column
// value slice); value columns of the state evolve independently, so the four
// slices of a head need no exchange.  Each CTA recomputes the prepare stage
// for its slice.  Rows at or past a sequence's end are never loaded.
#include <cuda_bf16.h>

#include <cmath>

#include "kda_common.h"

namespace kda {
namespace {

__device__ unsigned g_prefill_status = 0;

constexpr int kThreads = 256;
constexpr int kDV = 32;            // value columns per CTA
constexpr int kSlices = D / kDV;   // CTAs per head
constexpr int kCMax = 64;          // largest chunk this kernel holds on chip
constexpr int kKP = D + 1;         // padded row pitch of [C][128] tiles
constexpr int kLP = kCMax + 1;     // padded row pitch of [C][C] tiles
constexpr int kVP = kDV + 1;       // padded row pitch of [C][32] tiles

struct ChunkSmem {
    float kc[kCMax][kKP];   // k, then Ktil
    float qc[kCMax][kKP];   // qh, then Qtil
    float gc[kCMax][kKP];   // g, then Gamma, then Khat
    float am[kCMax][kLP];   // A
    float tm[kCMax][kLP];   // T
    float pm[kCMax][kLP];   // P
    float vc[kCMax][kVP];   // V slice
    float xm[kCMax][kVP];   // V - Ktil S
    float um[kCMax][kVP];   // U
    float sm[D][kVP];       // state slice, [key][value]
    float beta[kCMax];
    float glast[D];
    float dec[D];
};

__device__ __forceinline__ float ld_in(const float* p) { return __ldg(p); }
__device__ __forceinline__ float ld_in(const uint16_t* p) {
    return __uint_as_float(static_cast<uint32_t>(__ldg(p)) << 16);
}

// Token range [start, end) of sequence n; false when cu_seqlens is malformed.
__device__ __forceinline__ bool seq_range(const int* __restrict__ cu, int n, int n_seqs, int t,
                                          int t_pad, int& start, int& end) {
    if (!cu) {
        start = n * t_pad;
        end = start + t;
        return true;
    }
    start = __ldg(cu + n);
    end = __ldg(cu + n + 1);
    bool ok = start >= 0 && start <= end && end <= t;
    if (n == 0) ok = ok && start == 0;
    if (n == n_seqs - 1) ok = ok && end == t;
    return ok;
}

template <typename TIn>
__global__ void __launch_bounds__(kThreads, 1)
prefill_simt_kernel(float* __restrict__ state, const TIn* __restrict__ q,
                    const TIn* __restrict__ k, const TIn* __restrict__ v,
                    const TIn* __restrict__ g, const TIn* __restrict__ beta,
                    float* __restrict__ o, int t, int t_pad, int chunk, int heads,
                    long long qkv_stride, const int* __restrict__ cu, int n_seqs) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    ChunkSmem& sm = *reinterpret_cast<ChunkSmem*>(smem_raw);
    const int slice = blockIdx.x, h = blockIdx.y, n = blockIdx.z;
    const int tid = threadIdx.x;
    int start, end;
    if (!seq_range(cu, n, n_seqs, t, t_pad, start, end)) {
        if (tid == 0) atomicOr(&g_prefill_status, STATUS_BAD_CU_SEQLENS);
        return;
    }
    const int j0 = slice * kDV;
    float* Sg = state + ((size_t)n * heads + h) * D * D;
    const size_t hd = (size_t)heads * D;

    for (int e = tid; e < D * kDV; e += kThreads) {
        const int i = e / kDV, j = e % kDV;
        sm.sm[i][j] = Sg[(size_t)i * D + j0 + j];
    }

    for (int c0 = start; c0 < end; c0 += chunk) {
        const int L = min(chunk, end - c0);
        __syncthreads();  // previous chunk fully consumed
        // ---- load the chunk's rows (rows >= L are never touched)
        for (int e = tid; e < L * D; e += kThreads) {
            const int r = e / D, i = e % D;
            const size_t row = (size_t)(c0 + r);
            sm.kc[r][i] = ld_in(k + row * qkv_stride + (size_t)h * D + i);
            sm.qc[r][i] = __fmul_rn(KDA_Q_SCALE, ld_in(q + row * qkv_stride + (size_t)h * D + i));
            sm.gc[r][i] = ld_in(g + row * hd + (size_t)h * D + i);
        }
        for (int e = tid; e < L * kDV; e += kThreads) {
            const int r = e / kDV, j = e % kDV;
            sm.vc[r][j] = ld_in(v + (size_t)(c0 + r) * qkv_stride + (size_t)h * D + j0 + j);
        }
        if (tid < L) sm.beta[tid] = ld_in(beta + (size_t)(c0 + tid) * heads + h);
        __syncthreads();
        // ---- Gamma: running sum of g down the chunk, per key channel
        if (tid < D) {
            float acc = 0.f;
            for (int r = 0; r < L; ++r) {
                acc = __fadd_rn(acc, sm.gc[r][tid]);
                sm.gc[r][tid] = acc;
            }
        }
        __syncthreads();
        // ---- A (s < r) and P (s <= r) over the lower triangle
        const int npairs = L * (L + 1) / 2;
        for (int p = tid; p < npairs; p += kThreads) {
            int r = (int)((sqrtf(8.f * p + 1.f) - 1.f) * 0.5f);
            while ((r + 1) * (r + 2) / 2 <= p) ++r;
            while (r * (r + 1) / 2 > p) --r;
            const int s = p - r * (r + 1) / 2;
            float a = 0.f, pp = 0.f;
            for (int i = 0; i < D; ++i) {
                const float ex = expf(sm.gc[r][i] - sm.gc[s][i]);
                const float ke = sm.kc[s][i] * ex;
                a = __fmaf_rn(sm.kc[r][i], ke, a);
                pp = __fmaf_rn(sm.qc[r][i], ke, pp);
            }
            const float b = sm.beta[s];
            sm.am[r][s] = (s < r) ? b * a : 0.f;
            sm.pm[r][s] = b * pp;
        }
        if (tid < D) {
            sm.glast[tid] = sm.gc[L - 1][tid];
            sm.dec[tid] = expf(sm.gc[L - 1][tid]);
        }
        __syncthreads();
        // ---- T = (I + A)^-1, one column per thread
        if (tid < L) {
            const int c = tid;
            sm.tm[c][c] = 1.f;
            for (int r = c + 1; r < L; ++r) {
                float x = 0.f;
                for (int s = c; s < r; ++s) x = __fmaf_rn(sm.am[r][s], sm.tm[s][c], x);
                sm.tm[r][c] = -x;
            }
        }
        // ---- Ktil, Qtil, Khat in place
        for (int e = tid; e < L * D; e += kThreads) {
            const int r = e / D, i = e % D;
            const float gam = sm.gc[r][i];
            const float ex = expf(gam);
            const float kv = sm.kc[r][i];
            sm.gc[r][i] = expf(sm.glast[i] - gam) * kv;
            sm.kc[r][i] = ex * kv;
            sm.qc[r][i] = ex * sm.qc[r][i];
        }
        __syncthreads();
        // ---- X = V - Ktil S
        const int j = tid & 31, rw = tid >> 5;
        for (int r = rw; r < L; r += kThreads / 32) {
            float acc = 0.f;
            for (int i = 0; i < D; ++i) acc = __fmaf_rn(sm.kc[r][i], sm.sm[i][j], acc);
            sm.xm[r][j] = sm.vc[r][j] - acc;
        }
        __syncthreads();
        // ---- U = T X
        for (int r = rw; r < L; r += kThreads / 32) {
            float acc = 0.f;
            for (int s = 0; s <= r; ++s) acc = __fmaf_rn(sm.tm[r][s], sm.xm[s][j], acc);
            sm.um[r][j] = acc;
        }
        __syncthreads();
        // ---- O = Qtil S + P U
        for (int r = rw; r < L; r += kThreads / 32) {
            float acc = 0.f;
            for (int i = 0; i < D; ++i) acc = __fmaf_rn(sm.qc[r][i], sm.sm[i][j], acc);
            for (int s = 0; s <= r; ++s) acc = __fmaf_rn(sm.pm[r][s], sm.um[s][j], acc);
            o[((size_t)(c0 + r) * heads + h) * D + j0 + j] = acc;
        }
        __syncthreads();
        // ---- S <- diag(dec) S + Khat^T diag(beta) U
        for (int i = rw; i < D; i += kThreads / 32) {
            float acc = sm.dec[i] * sm.sm[i][j];
            for (int s = 0; s < L; ++s)
                acc = __fmaf_rn(sm.gc[s][i] * sm.beta[s], sm.um[s][j], acc);
            sm.sm[i][j] = acc;
        }
    }
    __syncthreads();
    for (int e = tid; e < D * kDV; e += kThreads) {
        const int i = e / kDV, jj = e % kDV;
        Sg[(size_t)i * D + j0 + jj] = sm.sm[i][jj];
    }
}

// True when the caller pins the SIMT chunk kernel (KDA_PREFILL_IMPL=simt,
// for comparisons).
bool simt_pinned() {
    const char* impl = getenv("KDA_PREFILL_IMPL");
    return impl && strcmp(impl, "simt") == 0;
}

// True when this call runs on the tensor-core kernels (which need a
// workspace): every call unless the SIMT kernel is pinned (FP32 inputs are
// rounded to FP16 copies in the workspace first).  Those kernels step through
// the sequence 64 tokens at a time whatever the chunk width: the chunked form
// gives the same result for any width (the recurrence it reorganises), up to
// rounding, so the width is the kernels' choice.
bool uses_tensor_cores(int chunk, int in_dtype) {
    (void)chunk;
    (void)in_dtype;
    return !simt_pinned();
}

template <typename TIn>
kda_status launch(float* state, const void* q, const void* k, const void* v, const void* g,
                  const void* beta, float* o, int t, int t_pad, int chunk, int heads,
                  long long stride, const int* cu, int n_seqs, void* workspace, cudaStream_t s) {
    // The SIMT kernel holds chunks of at most kCMax tokens on chip; a wider
    // chunk runs as consecutive kCMax-token chunks (the same result).
    chunk = chunk < kCMax ? chunk : kCMax;
    // Short sequences (uniform form, heads packed in each token row) take
    // decode_k's row walk, the pages' dispatch for pieces that do not take the
    // chunked arm: one state read, t token steps in registers, one state write
    // (BF16 inputs widened exactly, FP32 arithmetic).
    if (!cu && t <= KDA_MAX_K && stride == (long long)heads * D && !simt_pinned())
        return launch_row_walk(state, q, k, v, g, beta, o, n_seqs, t, t_pad, heads,
                               sizeof(TIn) == 2, s);
    // Everything else takes the tensor-core kernels unless the caller pins
    // the SIMT kernel (KDA_PREFILL_IMPL=simt, for comparisons).
    if (uses_tensor_cores(chunk, sizeof(TIn) == 2 ? KDA_BF16 : KDA_F32))
        return launch_prefill_tc(state, q, k, v, g, beta, o, t, t_pad, heads, stride, cu, n_seqs,
                                 workspace, s, nullptr, nullptr, sizeof(TIn) == 4);
    const size_t smem = sizeof(ChunkSmem);
    cudaError_t e = cudaFuncSetAttribute(prefill_simt_kernel<TIn>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) {
        set_error("kda_prefill: cannot reserve %zu B of shared memory: %s", smem,
                  cudaGetErrorString(e));
        return KDA_ERR_CUDA;
    }
    dim3 grid(kSlices, heads, n_seqs);
    prefill_simt_kernel<TIn><<<grid, kThreads, smem, s>>>(
        state, (const TIn*)q, (const TIn*)k, (const TIn*)v, (const TIn*)g, (const TIn*)beta, o,
        t, t_pad, chunk, heads, stride, cu, n_seqs);
    return launch_result("kda_prefill");
}

}  // namespace

cudaError_t read_and_clear_status_prefill(unsigned* out) {
    unsigned zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(out, g_prefill_status, sizeof(unsigned));
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_prefill_status, &zero, sizeof(unsigned));
    return e;
}

}  // namespace kda

using namespace kda;

extern "C" size_t kda_prefill_workspace_size(int64_t rows, int n_seqs, int chunk, int heads,
                                             int head_dim, int in_dtype) {
    if (rows < 0 || n_seqs < 1 || heads < 1 || head_dim != D) return 0;
    if (!uses_tensor_cores(chunk, in_dtype)) return 0;
    return prefill_tc_workspace_bytes(rows, n_seqs, heads, in_dtype == KDA_F32);
}

namespace kda {

// Argument checks of kda_prefill and kda_prefill_static_ws (everything but the
// workspace), so that both refuse the same call with the same status.
kda_status validate_prefill(const char* fn, const float* state, const void* q, const void* k,
                            const void* v, const void* g, const void* beta, const float* o,
                            int t, int t_pad, int chunk, int heads, int head_dim, int in_dtype,
                            int64_t qkv_row_stride, const int* cu_seqlens, int n_seqs) {
    KDA_REQUIRE(state && q && k && v && g && beta && o, KDA_ERR_INVALID_ARG,
                "%s: null pointer argument", fn);
    KDA_REQUIRE(aligned16(state) && aligned16(q) && aligned16(k) && aligned16(v) &&
                    aligned16(g) && aligned16(o),
                KDA_ERR_INVALID_ARG, "%s: state, q, k, v, g and o must be 16-byte aligned", fn);
    KDA_REQUIRE(head_dim == D, KDA_ERR_UNSUPPORTED, "%s: head_dim %d unsupported", fn, head_dim);
    KDA_REQUIRE(chunk == 16 || chunk == 32 || chunk == 64 || chunk == 128, KDA_ERR_UNSUPPORTED,
                "%s: chunk %d unsupported (16, 32, 64 or 128)", fn, chunk);
    KDA_REQUIRE(in_dtype == KDA_F32 || in_dtype == KDA_BF16, KDA_ERR_INVALID_ARG,
                "%s: in_dtype %d unknown", fn, in_dtype);
    KDA_REQUIRE(heads >= 1 && n_seqs >= 1 && heads <= 65535 && n_seqs <= 65535,
                KDA_ERR_INVALID_ARG, "%s: heads (%d) / n_seqs (%d) out of range", fn, heads,
                n_seqs);
    KDA_REQUIRE(t >= 1 && t_pad >= t, KDA_ERR_INVALID_ARG, "%s: need 1 <= t (%d) <= t_pad (%d)",
                fn, t, t_pad);
    KDA_REQUIRE(!cu_seqlens || t_pad == t, KDA_ERR_INVALID_ARG,
                "%s: packed sequences (cu_seqlens) take no padding: t_pad must equal t", fn);
    KDA_REQUIRE(qkv_row_stride >= (int64_t)heads * D, KDA_ERR_INVALID_ARG,
                "%s: qkv_row_stride %lld < heads * 128", fn, (long long)qkv_row_stride);
    const int esz = in_dtype == KDA_BF16 ? 2 : 4;
    KDA_REQUIRE((qkv_row_stride * esz) % 16 == 0, KDA_ERR_INVALID_ARG,
                "%s: qkv_row_stride must be a multiple of 16 bytes", fn);
    const long long rows = cu_seqlens ? (long long)t : (long long)t_pad * n_seqs;
    KDA_REQUIRE(rows <= 0x7fffffffLL, KDA_ERR_INVALID_ARG, "%s: too many token rows", fn);
    return KDA_OK;
}

}  // namespace kda

extern "C" kda_status kda_prefill(float* state, const void* q, const void* k, const void* v,
                                  const void* g, const void* beta, float* o, int t, int t_pad,
                                  int chunk, float pad_fill, int heads, int head_dim,
                                  int in_dtype, int64_t qkv_row_stride, const int* cu_seqlens,
                                  int n_seqs, void* workspace, size_t workspace_bytes,
                                  uint64_t stream) {
    (void)pad_fill;  // the caller's fill of rows [t, t_pad): never read, never written
    const kda_status vs = validate_prefill("kda_prefill", state, q, k, v, g, beta, o, t, t_pad,
                                           chunk, heads, head_dim, in_dtype, qkv_row_stride,
                                           cu_seqlens, n_seqs);
    if (vs != KDA_OK) return vs;
    const long long rows = cu_seqlens ? (long long)t : (long long)t_pad * n_seqs;
    const size_t need = kda_prefill_workspace_size(rows, n_seqs, chunk, heads, head_dim, in_dtype);
    KDA_REQUIRE(workspace_bytes >= need && (need == 0 || workspace), KDA_ERR_WORKSPACE,
                "kda_prefill: workspace of %zu B given, %zu B needed", workspace_bytes, need);
    KDA_REQUIRE(need == 0 || aligned16(workspace), KDA_ERR_INVALID_ARG,
                "kda_prefill: workspace must be 16-byte aligned");
    KDA_REQUIRE(!fault_injected(), KDA_ERR_CUDA, "kda_prefill: injected launch failure");
    cudaStream_t s = as_stream(stream);
    if (in_dtype == KDA_BF16)
        return launch<uint16_t>(state, q, k, v, g, beta, o, t, t_pad, chunk, heads,
                                qkv_row_stride, cu_seqlens, n_seqs, workspace, s);
    return launch<float>(state, q, k, v, g, beta, o, t, t_pad, chunk, heads, qkv_row_stride,
                         cu_seqlens, n_seqs, workspace, s);
}

extern "C" kda_status kda_prefill_gated(float* state, const void* q, const void* k, const void* v,
                                        const uint16_t* g_raw, int64_t g_raw_stride,
                                        const float* dt_bias, const float* a_log,
                                        float gate_lower_bound, const uint16_t* b_raw,
                                        int64_t b_stride, float* o, int t, int t_pad, int heads,
                                        int head_dim, int64_t qkv_row_stride,
                                        const int* cu_seqlens, int n_seqs, void* workspace,
                                        size_t workspace_bytes, uint64_t stream) {
    KDA_REQUIRE(state && q && k && v && g_raw && dt_bias && a_log && b_raw && o,
                KDA_ERR_INVALID_ARG, "kda_prefill_gated: null pointer argument");
    KDA_REQUIRE(aligned16(state) && aligned16(q) && aligned16(k) && aligned16(v) &&
                    aligned16(g_raw) && aligned16(o),
                KDA_ERR_INVALID_ARG,
                "kda_prefill_gated: state, q, k, v, g_raw and o must be 16-byte aligned");
    KDA_REQUIRE(head_dim == D, KDA_ERR_UNSUPPORTED, "kda_prefill_gated: head_dim %d unsupported",
                head_dim);
    KDA_REQUIRE(heads >= 1 && n_seqs >= 1 && heads <= 65535 && n_seqs <= 65535,
                KDA_ERR_INVALID_ARG, "kda_prefill_gated: heads (%d) / n_seqs (%d) out of range",
                heads, n_seqs);
    KDA_REQUIRE(t >= 1 && t_pad >= t, KDA_ERR_INVALID_ARG,
                "kda_prefill_gated: need 1 <= t (%d) <= t_pad (%d)", t, t_pad);
    KDA_REQUIRE(!cu_seqlens || t_pad == t, KDA_ERR_INVALID_ARG,
                "kda_prefill_gated: packed sequences (cu_seqlens) take no padding: t_pad must "
                "equal t");
    KDA_REQUIRE(qkv_row_stride >= (int64_t)heads * D && qkv_row_stride % 8 == 0,
                KDA_ERR_INVALID_ARG,
                "kda_prefill_gated: qkv_row_stride must be >= heads * 128 and a multiple of 8");
    KDA_REQUIRE(g_raw_stride >= (int64_t)heads * D && g_raw_stride % 8 == 0 && b_stride >= heads,
                KDA_ERR_INVALID_ARG,
                "kda_prefill_gated: g_raw_stride must be >= heads*128 and a multiple of 8, "
                "b_stride >= heads");
    KDA_REQUIRE(gate_lower_bound < 0.f && gate_lower_bound > -INFINITY, KDA_ERR_INVALID_ARG,
                "kda_prefill_gated: gate_lower_bound must be finite and negative");
    const long long rows = cu_seqlens ? (long long)t : (long long)t_pad * n_seqs;
    KDA_REQUIRE(rows <= 0x7fffffffLL, KDA_ERR_INVALID_ARG,
                "kda_prefill_gated: too many token rows");
    const size_t need = prefill_tc_workspace_bytes(rows, n_seqs, heads);
    KDA_REQUIRE(workspace && workspace_bytes >= need, KDA_ERR_WORKSPACE,
                "kda_prefill_gated: workspace of %zu B given, %zu B needed", workspace_bytes, need);
    KDA_REQUIRE(aligned16(workspace), KDA_ERR_INVALID_ARG,
                "kda_prefill_gated: workspace must be 16-byte aligned");
    KDA_REQUIRE(!fault_injected(), KDA_ERR_CUDA, "kda_prefill_gated: injected launch failure");
    const PrefillGate gate = {dt_bias, a_log, gate_lower_bound, (long long)g_raw_stride,
                              (long long)b_stride};
    return launch_prefill_tc(state, q, k, v, g_raw, b_raw, o, t, t_pad, heads,
                             (long long)qkv_row_stride, cu_seqlens, n_seqs, workspace,
                             as_stream(stream), &gate);
}

extern "C" kda_status kda_prefill_o_norm(float* state, const void* q, const void* k,
                                         const void* v, const void* g, const void* beta,
                                         const uint16_t* gate, int64_t gate_stride,
                                         const uint16_t* w_norm, float eps, uint16_t* out,
                                         int64_t out_stride, int t, int t_pad, int chunk,
                                         int heads, int head_dim, int in_dtype,
                                         int64_t qkv_row_stride, const int* cu_seqlens,
                                         int n_seqs, void* workspace, size_t workspace_bytes,
                                         uint64_t stream) {
    const char* fn = "kda_prefill_o_norm";
    // the output stands in for o in the shared checks (non-null, 16-byte aligned)
    const kda_status vs = validate_prefill(fn, state, q, k, v, g, beta,
                                           reinterpret_cast<const float*>(out), t, t_pad, chunk,
                                           heads, head_dim, in_dtype, qkv_row_stride, cu_seqlens,
                                           n_seqs);
    if (vs != KDA_OK) return vs;
    KDA_REQUIRE(in_dtype == KDA_BF16 && !simt_pinned(), KDA_ERR_UNSUPPORTED,
                "%s: the fused norm runs on the BF16 tensor-core path only", fn);
    KDA_REQUIRE(gate && w_norm, KDA_ERR_INVALID_ARG, "%s: null gate or o_norm weight", fn);
    KDA_REQUIRE(aligned16(gate) && (reinterpret_cast<uintptr_t>(w_norm) & 7u) == 0,
                KDA_ERR_INVALID_ARG, "%s: gate must be 16-byte and w 8-byte aligned", fn);
    KDA_REQUIRE(gate_stride >= (int64_t)heads * D && gate_stride % 8 == 0 &&
                    out_stride >= (int64_t)heads * D && out_stride % 8 == 0,
                KDA_ERR_INVALID_ARG,
                "%s: gate_stride and out_stride must be >= heads * 128 and multiples of 8", fn);
    KDA_REQUIRE(eps >= 0.f && eps < INFINITY, KDA_ERR_INVALID_ARG,
                "%s: eps must be finite and >= 0", fn);
    const long long rows = cu_seqlens ? (long long)t : (long long)t_pad * n_seqs;
    const size_t need = kda_prefill_workspace_size(rows, n_seqs, chunk, heads, head_dim, in_dtype);
    KDA_REQUIRE(workspace && workspace_bytes >= need, KDA_ERR_WORKSPACE,
                "%s: workspace of %zu B given, %zu B needed", fn, workspace_bytes, need);
    KDA_REQUIRE(aligned16(workspace), KDA_ERR_INVALID_ARG, "%s: workspace must be 16-byte aligned",
                fn);
    KDA_REQUIRE(!fault_injected(), KDA_ERR_CUDA, "%s: injected launch failure", fn);
    const PrefillNorm nrm = {gate, (long long)gate_stride, w_norm, eps, out, (long long)out_stride};
    return launch_prefill_tc(state, q, k, v, g, beta, nullptr, t, t_pad, heads,
                             (long long)qkv_row_stride, cu_seqlens, n_seqs, workspace,
                             as_stream(stream), nullptr, &nrm);
}
