// Tensor-core chunked prefill of the KDA core for BF16 inputs and chunk 64:
// Glm5NextKdaKernels::chunk_prepare and chunk_scan around a caller-owned
// workspace, as two kernels or as one cooperative grid.
//
// For a chunk of L <= 64 tokens (rows r, s; key channels i; value columns j)
// of one head, with Gamma_r = sum_{u<=r} g_u and qh = KDA_Q_SCALE q:
//   A_rs   = beta_s sum_i k_ri k_si e^(Gamma_ri-Gamma_si), s < r
//   P_rs   = beta_s sum_i qh_ri k_si e^(Gamma_ri-Gamma_si), s <= r
//   T      = (I + A)^-1                    (blocked forward substitution)
//   Ktil   = e^Gamma (.) k,  Qtil = e^Gamma (.) qh,
//   Khat_s = beta_s e^(Gamma_{L-1}-Gamma_s) (.) k_s,   dec = e^Gamma_{L-1}
// prepare_kernel computes everything above that does not depend on the
// carried state, for every (chunk, head) item, fully parallel: one persistent
// CTA per SM walks the items, with the next item's q/k/g tiles arriving by
// TMA into a second buffer while the current one is processed.  It writes
// [Ktil; Qtil], [T; P], Khat^T (FP16 tensor-core operands, already in the
// layout the scan consumes) and dec to the workspace: 66,176 bytes per chunk
// and head.
// scan_t_kernel, one CTA per (sequence, head), carries the FP32 state across
// the sequence's chunks in order:
//   X = V - Ktil S;  U = T X;  O = Qtil S + P U;  S <- dec (.) S + Khat^T U
// as three tensor-core round trips per chunk, in transposed form with the
// chain's operands in TMEM; the chunk's operands arrive by bulk copy from the
// workspace and the value tile by TMA.
// prefill_fused_kernel runs both in one cooperative grid when there are few
// (sequence, head) chains: one SM per chain (scan_t_role) while the other SMs
// walk the prepare items in chunk order and release a ready flag per item,
// so the prepare work no longer precedes the scan.
// The <true> instantiations of prepare_kernel and prefill_fused_kernel (the
// gated prefill) read the raw forget-gate projection where the others read
// g and the raw b_proj output where they read beta, and form g and beta as
// they load them (PrepMaps).
//
// Precision: prepare forms A and P from TF32 operands (their decay factors
// span e^(+-8 |g|)); the scan's products take FP16 operands (10 stored
// significand bits, as TF32) with FP32 accumulation.  Every scan operand is
// bounded by the inputs' scale: |Ktil|, |Khat| <= |k|, |Qtil| <= |qh|, P, the
// state S, X = V - Ktil S and U = T X are of the order of v and the initial
// state, far inside FP16's range for normalised q, k; values below 2^-14
// keep an absolute error under 2^-25.
//
// A and P come from tensor-core products over column blocks b with a
// reference token m_b: e^(Gamma_r-Gamma_s) = e^(Gamma_r-Gamma_mb)
// e^(Gamma_mb-Gamma_s).  With four 16-token blocks (m_b = 16b + 8) both
// factors stay within e^(+-8 |g|max) for every (r >= 16b, s in block b), so
// FP32 neither overflows nor loses the product for g >= -10; rows above the
// block are never formed into results.  Chunks whose decays all stay above
// -kWideGMin take two 32-token blocks instead (see kWideGMin).
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <type_traits>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "f32x2.h"
#include "kda_common.h"
#include "sm103_tc.h"
#include "tma_map.h"

namespace kda {
namespace {

__device__ unsigned g_tc_status = 0;

constexpr int C = 64;
constexpr int NTP = 512;  // prepare threads
constexpr int KP = 132;  // pitch (floats) of the FP32 [64][128] Gamma array (16-B rows)
constexpr int AP = 65;   // pitch (floats) of the FP32 [64][64] A / W array
constexpr int TPP = 68;  // pitch (floats) of the FP32 [64][64] T array (16-B rows)

// K-major operand of R rows in the "K-outer" core-matrix layout: the core
// matrices of one K group (the 16 bytes of a row: 4 TF32 or 8 FP16 values)
// are stacked over all rows (128 B per 8 rows); successive K groups are
// LBO = 16 R + PAD bytes apart.  PAD = 16 spreads operands that are written
// one K index per thread over all banks.  One MMA K-step reads 32 bytes of K
// per row (8 TF32 or 16 FP16 values): two K groups.
template <int R, int PAD, int ES = 4>
struct Op {
    static constexpr uint32_t LBO = R * 16 + PAD;
    static constexpr int KG = 16 / ES;  // values per K group
    static __device__ __forceinline__ uint32_t off(int r, int k) {
        return (uint32_t)((k / KG) * LBO + (r >> 3) * 128 + (r & 7) * 16 + (k % KG) * ES);
    }
    static __device__ __forceinline__ uint64_t desc(uint32_t base, int ks) {
        return tc::make_desc(base + (uint32_t)ks * 2u * LBO, LBO, 128u);
    }
    // Descriptor increment of one MMA K-step (two K groups): the start address
    // field holds the byte address / 16 in its low 14 bits, and every operand
    // lies below 228 KB, so adding this never carries out of the field.
    static constexpr uint64_t KSTEP = (2u * LBO) >> 4;
    static __host__ __device__ constexpr uint32_t bytes(int K) { return (uint32_t)(K / KG) * LBO; }
};
// prepare's A/P products (TF32: their decay factors reach e^(+-8 |g|))
using OpX = Op<128, 0>;   // A: [X_b; QX_b], K = 128 channels
using OpY = Op<16, 0>;    // B: Y_b of a 16-token block, K = 128 channels
using OpY32 = Op<32, 0>;  // B: Y_b of a 32-token block, K = 128 channels
using OpKH = Op<128, 16>; // sizes the Y_b region, which later holds Khat^T
using OpX1 = Op<64, 0>;   // A: [X_1; QX_1] of the second 32-token block, rows 32..63 only
// the scan's operands (FP16: every value is bounded by the inputs' scale)
using OpXh = Op<128, 0, 2>;    // [Ktil; Qtil], K = 128 channels
using OpTPh = Op<128, 0, 2>;   // [T; P], K = 64 tokens
using OpKHh = Op<128, 16, 2>;  // Khat^T, rows = key channel, K = 64 tokens (written per K index)

// ------------------------------------------------------------ workspace
// [chunk_off: (n_seqs + 1) int32, padded to 256 B][blob (g, h) for every
// chunk g and head h].  A blob is the byte image of the scan's operands.
constexpr uint32_t BLOB_OPX = 0;
constexpr uint32_t BLOB_TP = BLOB_OPX + OpXh::bytes(128);
constexpr uint32_t BLOB_KH = BLOB_TP + OpTPh::bytes(64);
constexpr uint32_t BLOB_DEC = BLOB_KH + OpKHh::bytes(64);
constexpr uint32_t BLOB_BYTES = BLOB_DEC + 128 * 4;
static_assert(BLOB_BYTES % 128 == 0, "blobs must stay 128-byte aligned");

__host__ __device__ inline size_t header_bytes(int n_seqs) {
    return ((size_t)(n_seqs + 1) * 4 + 255) & ~(size_t)255;
}
__host__ __device__ inline size_t blob_offset(int n_seqs, long long g, int h, int heads) {
    return header_bytes(n_seqs) + ((size_t)g * heads + h) * BLOB_BYTES;
}

// ------------------------------------------------------------ prepare smem
// prepare_kernel is persistent: each CTA walks (chunk, head) items with the
// next item's raw tiles loading into the other of two buffers.  A raw buffer
// holds the BF16 q, k and g tiles [64 tokens][128 channels], each as two TMA
// boxes of 64 channels with the 128-byte swizzle (row r, 16-byte chunk c
// stored at chunk c ^ (r & 7)).
constexpr uint32_t RAW_TILE = 16384;
constexpr uint32_t RAW_BUF = 3 * RAW_TILE;
constexpr uint32_t RAW_Q = 0, RAW_K = RAW_TILE, RAW_G = 2 * RAW_TILE;
// inside the current buffer, once Gamma is formed: reference rows and
// Gamma_{L-1} at the end of the g tile; once the operands are out: the solve
constexpr uint32_t RB_GMID = RAW_G + RAW_TILE - 7 * 128 * 4;  // 6 x 128: 4 + 2 reference rows
constexpr uint32_t RB_GLAST = RB_GMID + 6 * 128 * 4;
// wide path: e^Gamma_17, e^(Gamma_63 - Gamma_17), e^(Gamma_63 - Gamma_49) per channel
constexpr uint32_t RB_PC = RB_GMID - 3 * 128 * 4;
constexpr uint32_t RB_AM = 0;                                 // FP32 A, then W blocks [64][AP]
constexpr uint32_t RB_TM = (RB_AM + 64 * AP * 4 + 15) & ~15u;  // FP32 T [64][TPP]
constexpr uint32_t PS_GAM = 2 * RAW_BUF;                     // FP32 Gamma [64][KP]
constexpr uint32_t PS_OPX = PS_GAM + 64 * KP * 4;            // A operand of the A/P products
constexpr uint32_t PS_Y = PS_OPX + OpX::bytes(128);          // B operands Y_b
constexpr uint32_t PS_BETA = PS_Y + OpKH::bytes(64);
constexpr uint32_t PS_BAR = PS_BETA + 64 * 4;  // bar_tma[2], bar_mma[2], TMEM base, bar_g
// Packed batches of up to SEQ_CACHE sequences keep their chunk map (chunk_off
// and cu_seqlens, n_seqs + 1 entries each) in shared memory: the item lookup
// is a binary search, dependent global loads otherwise.
constexpr int SEQ_CACHE = 128;
constexpr uint32_t PS_SEQ = PS_BAR + 64;
constexpr uint32_t PS_TOTAL = PS_SEQ + ((2 * (SEQ_CACHE + 1) * 4 + 15) & ~15u);
static_assert(RB_TM + 64 * TPP * 4 <= RB_PC, "solve arrays overlap the reference rows");
static_assert(RB_GLAST + 128 * 4 == RAW_G + RAW_TILE, "reference rows must end the g tile");
static_assert(2 * OpY32::bytes(128) <= 4 * OpY::bytes(128), "Y_b operands do not fit");
static_assert(4 * OpY::bytes(128) <= OpKH::bytes(64), "Y_b operands do not fit");
static_assert(PS_OPX % 1024 == 0 && PS_Y % 16 == 0, "operand alignment");
static_assert(OpXh::bytes(128) <= OpX::bytes(128) / 2 && 2 * 64 * 64 * 4 <= OpX::bytes(128) / 2,
              "the steep path's A and P share the A operand region with Ktil and Qtil");

// A chunk whose decays all satisfy g >= -kWideGMin takes 32-token column
// blocks with reference token 32 b + 17: the A-side factor stays below
// e^(17 |g|) < FLT_MAX, the B-side factor above e^(-17 |g|) (a normal
// number), and a flushed A-side factor loses under 1.2e-38 e^(14 |g|) < 2e-7.
constexpr float kWideGMin = 5.1f;
// Four 16-token blocks (reference token 16 b + 8) keep the A-side factor below
// e^(8 |g|) < FLT_MAX and a flushed A-side factor's loss under
// e^(-87.3 + 7 |g|) < 1e-7 while g >= -kNarrowGMin.  A chunk with a steeper
// decay forms A and P on the CUDA cores, each (row, column) pair's factor
// e^(Gamma_r - Gamma_s) <= 1 by its own exponential: exact for any g.
constexpr float kNarrowGMin = 10.0f;
static_assert(PS_TOTAL <= 232448, "shared memory budget exceeded");

constexpr uint32_t SS_OPX = BLOB_OPX, SS_TP = BLOB_TP;

// TMEM columns of prepare: A and P
constexpr uint32_t TC_AP = 0;

// 1/x by the hardware approximation (subnormal results flush to zero); its
// callers use it only for TF32 operands, rounded to 11 bits afterwards.
__device__ __forceinline__ float rcp_fast(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float bf(uint16_t b) {
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

__device__ __forceinline__ void st4(unsigned char* base, uint32_t off, float a, float b, float c,
                                    float d) {
    *reinterpret_cast<float4*>(base + off) =
        make_float4(tc::to_tf32(a), tc::to_tf32(b), tc::to_tf32(c), tc::to_tf32(d));
}

// Four values rounded to FP16, stored as one 8-byte write.
__device__ __forceinline__ void st4h(unsigned char* p, float a, float b, float c, float d) {
    *reinterpret_cast<uint2*>(p) = make_uint2(tc::pack_f16x2(a, b), tc::pack_f16x2(c, d));
}
__device__ __forceinline__ void st1h(unsigned char* p, float a) {
    *reinterpret_cast<uint16_t*>(p) = tc::f16_bits(a);
}

// What prepare reads besides the workspace: TMA maps of the q, k and g tiles,
// beta's row pitch, and (gated calls) the forget-gate parameters.  In the
// gated kernels the g tiles hold the gate projection g_raw and beta the raw
// b_proj output; the first use of each element turns it into the core's input:
//     g = lb * sigmoid(exp(a_log[h]) * (g_raw + dt_bias[h * 128 + i])),
//     beta = sigmoid(b),
// with the FP32 operations, in the same order, of the standalone gate kernel.
struct PrepMaps {
    CUtensorMap q, k, g;
    const float* dt_bias;
    const float* a_log;
    float lb;
    long long b_stride;  // elements between token rows of beta
};

// The sigmoid-gated RMSNorm fused into the scan's epilogue (kda_prefill_o_norm):
// the gate tiles' load map and the BF16 output's store map (both [rows][heads
// x 128], boxes of 128 channels x 64 tokens), the o_norm weight, epsilon, and
// the output again for plain stores (row pitch in elements).
struct NormArgs {
    CUtensorMap gmap, nmap;
    const uint16_t* w;
    uint16_t* out;
    long long out_pitch;
    float eps;
};

constexpr float kLog2e = 1.4426950408889634f;

// sigmoid(z) = 1 / (1 + 2^(-z log2 e)) by the hardware 2^x and 1/x.
__device__ __forceinline__ float sigmoid_hw(float z) {
    return rcp_approx(__fadd_rn(ex2_approx(__fmul_rn(z, -kLog2e)), 1.0f));
}
// sigmoid(z) = (1 + tanh(z / 2)) / 2 by the hardware tanh: one special-
// function operation (absolute error about 2^-11 relative to 1), for the
// fused norm's BF16 output.
__device__ __forceinline__ float sigmoid_tanh(float z) {
    float t;
    asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(0.5f * z));
    return __fmaf_rn(0.5f, t, 0.5f);
}
// lb * sigmoid(c (x + dt)) given nc = -c log2 e.
__device__ __forceinline__ float gate_hw(float x, float dt, float nc, float lb) {
    return __fmul_rn(lb, rcp_approx(__fadd_rn(ex2_approx(__fmul_rn(__fadd_rn(x, dt), nc)), 1.0f)));
}

// D = A . B^T over KS TF32 K-steps of 8, issued by the calling thread.  The
// loop is unrolled and each K-step's descriptors are the first ones plus a
// constant: a single issuing thread otherwise spends tens of cycles per
// instruction rebuilding descriptors, against about 44 cycles per small-N
// instruction of the tensor core itself.
template <class OA, class OB, int KS>
__device__ __forceinline__ void issue_mma(uint32_t d, uint32_t a, uint32_t b, uint32_t idesc) {
    const uint64_t ad = OA::desc(a, 0), bd = OB::desc(b, 0);
#pragma unroll
    for (int ks = 0; ks < KS; ++ks)
        tc::mma_tf32(d, ad + ks * OA::KSTEP, bd + ks * OB::KSTEP, idesc, ks > 0);
}

// Token range [start, end) of sequence n; false when cu_seqlens is malformed.
// kGlobal: cu is device memory read through the read-only path; otherwise a
// generic pointer (shared memory).
template <bool kGlobal = true>
__device__ __forceinline__ bool seq_range(const int* __restrict__ cu, int n, int n_seqs, int t,
                                          int t_pad, int& start, int& end) {
    if (!cu) {
        start = n * t_pad;
        end = start + t;
        return true;
    }
    start = kGlobal ? __ldg(cu + n) : cu[n];
    end = kGlobal ? __ldg(cu + n + 1) : cu[n + 1];
    bool ok = start >= 0 && start <= end && end <= t;
    if (n == 0) ok = ok && start == 0;
    if (n == n_seqs - 1) ok = ok && end == t;
    return ok;
}

// chunk_off[n] = number of chunks of all sequences before n (one CTA).
constexpr int MAP_THREADS = 1024;
__global__ void __launch_bounds__(MAP_THREADS)
chunk_map_kernel(const int* __restrict__ cu, int n_seqs, int t, int* __restrict__ chunk_off,
                 unsigned* __restrict__ ready, long long n_ready) {
    __shared__ int part[MAP_THREADS];
    pdl_wait();
    pdl_release();
    // the fused grid's ready flags start cleared (n_ready is a multiple of 4
    // and `ready` 16-byte aligned)
    for (long long i = threadIdx.x; i < n_ready / 4; i += MAP_THREADS)
        reinterpret_cast<uint4*>(ready)[i] = make_uint4(0u, 0u, 0u, 0u);
    const int per = (n_seqs + MAP_THREADS - 1) / MAP_THREADS;
    const int lo = threadIdx.x * per, hi = min(n_seqs, lo + per);
    int sum = 0;
    for (int n = lo; n < hi; ++n) {
        int len = t;
        if (cu) {
            len = __ldg(cu + n + 1) - __ldg(cu + n);
            if (len < 0) {
                atomicOr(&g_tc_status, STATUS_BAD_CU_SEQLENS);
                len = 0;
            }
        }
        sum += (len + C - 1) / C;
    }
    part[threadIdx.x] = sum;
    __syncthreads();
    for (int off = 1; off < MAP_THREADS; off <<= 1) {  // inclusive scan of the partial sums
        const int v = (threadIdx.x >= off) ? part[threadIdx.x - off] : 0;
        __syncthreads();
        part[threadIdx.x] += v;
        __syncthreads();
    }
    int run = (threadIdx.x == 0) ? 0 : part[threadIdx.x - 1];
    for (int n = lo; n < hi; ++n) {
        chunk_off[n] = run;
        int len = t;
        if (cu) len = max(0, __ldg(cu + n + 1) - __ldg(cu + n));
        run += (len + C - 1) / C;
    }
    if (threadIdx.x == MAP_THREADS - 1) chunk_off[n_seqs] = part[MAP_THREADS - 1];
}

// The two-kernel path's chain order for a packed batch (one CTA): order[rank]
// = the sequence with that rank by decreasing chunk count (equal counts by
// index), so that the scan starts the longest chains first instead of
// wherever they fall in the batch.  n_seqs <= ORDER_MAX ints of dynamic
// shared memory.
constexpr int ORDER_MAX = 1024;
__global__ void __launch_bounds__(MAP_THREADS)
chain_order_kernel(const int* __restrict__ cu, int n_seqs, int* __restrict__ order) {
    extern __shared__ int s_chunks[];
    pdl_wait();
    pdl_release();
    for (int n = threadIdx.x; n < n_seqs; n += MAP_THREADS)
        s_chunks[n] = (max(0, __ldg(cu + n + 1) - __ldg(cu + n)) + C - 1) / C;
    __syncthreads();
    for (int n = threadIdx.x; n < n_seqs; n += MAP_THREADS) {
        const int cn = s_chunks[n];
        int rank = 0;  // sequences ahead of n
        for (int m = 0; m < n_seqs; ++m) {
            const int cm = s_chunks[m];
            rank += (cm > cn || (cm == cn && m < n)) ? 1 : 0;
        }
        order[rank] = n;
    }
}

// Byte offset of channel c of row r inside a raw tile (see above).
__device__ __forceinline__ uint32_t raw_off(int r, int c) {
    return (uint32_t)((c >> 6) * 8192 + r * 128 + ((((c & 63) >> 3) ^ (r & 7)) << 4) + (c & 7) * 2);
}
__device__ __forceinline__ float raw1(const unsigned char* tile, int r, int c) {
    return bf(*reinterpret_cast<const uint16_t*>(tile + raw_off(r, c)));
}
// Channels c .. c + 3 (c a multiple of 4) of row r.
__device__ __forceinline__ float4 raw4(const unsigned char* tile, int r, int c) {
    const uint2 u = *reinterpret_cast<const uint2*>(tile + raw_off(r, c));
    return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u),
                       __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
}
// FP16 bits to FP32 (exact).
__device__ __forceinline__ float h2f(uint16_t h) {
    float f;
    asm("cvt.f32.f16 %0, %1;" : "=f"(f) : "h"(h));
    return f;
}
// raw4 for the FP16 tiles of FP32 inputs (converted to FP16 before the call).
template <bool F16>
__device__ __forceinline__ float4 in4(const unsigned char* tile, int r, int c) {
    if constexpr (F16) {
        const uint2 u = *reinterpret_cast<const uint2*>(tile + raw_off(r, c));
        return make_float4(h2f((uint16_t)u.x), h2f((uint16_t)(u.x >> 16)), h2f((uint16_t)u.y),
                           h2f((uint16_t)(u.y >> 16)));
    } else {
        return raw4(tile, r, c);
    }
}

// A (chunk, head) item of the prepare walk: item = g * heads + h.
struct PrepItem {
    long long g;
    int h, c0, L;
    bool valid;
};

__device__ __forceinline__ PrepItem prep_item(long long item, int heads, const int* __restrict__ cu,
                                              const int* __restrict__ chunk_off, int n_seqs, int t,
                                              int t_pad) {
    PrepItem it;
    if (item < 0x7fffffffLL) {  // 32-bit divisions (a 64-bit one is a long software routine)
        const int g32 = (int)item / heads;
        it.g = g32;
        it.h = (int)item - g32 * heads;
    } else {
        it.g = item / heads;
        it.h = (int)(item - it.g * heads);
    }
    if (!cu) {  // uniform sequences of t tokens, t_pad rows apart: no table lookup
        const int cps = (t + C - 1) / C;
        const long long n = (it.g < 0x7fffffffLL) ? (long long)((int)it.g / cps) : it.g / cps;
        it.c0 = (int)(n * t_pad + (it.g - n * cps) * C);
        it.valid = n < n_seqs;
        it.L = it.valid ? min(C, (int)(n * t_pad) + t - it.c0) : 0;
        return it;
    }
    // chunk_off and cu are generic pointers (the shared-memory copies, or
    // device memory for large batches)
    int lo = 0, hi = n_seqs - 1;  // the sequence holding chunk g: largest n with chunk_off[n] <= g
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (chunk_off[mid] <= it.g) lo = mid;
        else hi = mid - 1;
    }
    int start, end;
    it.valid = seq_range<false>(cu, lo, n_seqs, t, t_pad, start, end);
    it.c0 = start + (int)(it.g - chunk_off[lo]) * C;
    it.valid = it.valid && it.c0 < end;
    it.L = it.valid ? min(C, end - it.c0) : 0;
    return it;
}

// The prepare walk of one CTA: items first, first + stride, ...  When `ready`
// is set, each finished item's flag (ready[item]) is released once its
// operands are in the workspace.
// F16: the inputs were FP32: q and k arrive as FP16 tiles, g as an FP32 tile
// (maps.g) loaded into the Gamma array, which the cumulative sum then
// overwrites in place, and beta as FP32.
template <bool GATED, bool F16, bool TWO_KERNEL>
__device__ __forceinline__ void prepare_role(const PrepMaps& maps, const void* __restrict__ beta,
                                             int t, int t_pad, int heads,
                                             const int* __restrict__ cu, int n_seqs,
                                             unsigned char* __restrict__ ws, long long first,
                                             long long stride, unsigned* __restrict__ ready,
                                             long long ready_pitch, bool publish = true) {
    extern __shared__ __align__(1024) unsigned char sm[];
    const int tid = threadIdx.x, warp = tid >> 5;
    const int ln = tid & 127, ch = tid >> 7;  // TMEM lane and column quarter
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    // Threads 0 and 32 issue the tensor-core products; a thread of another
    // warp issues the tile loads and bulk stores and releases the ready
    // flags, so the stores' completion and the release's fences are waited
    // for while the next item's A/P products run instead of between two items.
    const bool copier = (tid == 128);

    const int* chunk_off = reinterpret_cast<const int*>(ws);
    const long long items = (long long)__ldg(chunk_off + n_seqs) * heads;
    if (first >= items) return;
    if (tc::smem_u32(sm) & 1023u) {  // the swizzled tiles need a 1024-byte aligned base
        if (tid == 0) atomicOr(&g_tc_status, STATUS_SMEM_ALIGN);
        return;
    }

    float* GAM = reinterpret_cast<float*>(sm + PS_GAM);
    float* BETA = reinterpret_cast<float*>(sm + PS_BETA);
    const bool seq_cached = cu && n_seqs <= SEQ_CACHE;
    int* s_off = reinterpret_cast<int*>(sm + PS_SEQ);
    int* s_cu = s_off + SEQ_CACHE + 1;
    if (seq_cached && tid <= n_seqs) {  // visible after the barrier below
        s_off[tid] = __ldg(chunk_off + tid);
        s_cu[tid] = __ldg(cu + tid);
    }
    const int* map_off = seq_cached ? s_off : chunk_off;
    const int* map_cu = seq_cached ? s_cu : cu;
    uint64_t* bar_tma = reinterpret_cast<uint64_t*>(sm + PS_BAR);  // one per raw buffer
    uint64_t* bar_mma = bar_tma + 2;
    uint64_t* bar_mma2 = bar_tma + 3;  // the wide path's second A/P product (its own issuer)
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + PS_BAR + 32);
    uint64_t* bar_g = reinterpret_cast<uint64_t*>(sm + PS_BAR + 40);  // FP32 g tile (F16)
    const uint32_t s_opx = tc::smem_u32(sm + PS_OPX), s_y = tc::smem_u32(sm + PS_Y);

    if (tid == 0) {
        tc::mbar_init(bar_tma, 1);
        tc::mbar_init(bar_tma + 1, 1);
        tc::mbar_init(bar_mma, 1);
        tc::mbar_init(bar_mma2, 1);
        if (F16) tc::mbar_init(bar_g, 1);
        tc::fence_mbar_init();
        tc::prefetch_tmap(&maps.q);
        tc::prefetch_tmap(&maps.k);
        tc::prefetch_tmap(&maps.g);
    }
    if (warp == 0) tc::tmem_alloc(tmem_slot, 64);
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // Per-buffer state is kept as bit masks (bit b): an array indexed by the
    // buffer would live in local memory, whose lines the small L1 left by the
    // shared-memory carve-out does not keep -- an L2 round trip per access.
    uint32_t ph_mma = 0, ph_mma2 = 0, ph_tma = 0, ph_g = 0;
    bool failed = false;

    auto wait_mma = [&]() {
        if (!tc::mbar_wait(bar_mma, ph_mma)) {
            atomicOr(&g_tc_status, STATUS_TIMEOUT);
            failed = true;
        }
        ph_mma ^= 1;
        tc::tc_fence_after();
    };
    auto sync_for_mma = [&]() {  // generic smem writes and TMEM reads before an MMA
        tc::fence_async_smem();
        tc::tc_fence_before();
        __syncthreads();
    };
    // Raw tiles of item `it` into buffer b (thread 0), and its beta (threads
    // 0..63, returned in a register).
    auto load_raw = [&](const PrepItem& it, int b) {
        if (copier && it.valid) {
            unsigned char* dst = sm + b * RAW_BUF;
            tc::fence_async_smem();  // the buffer's previous generic-proxy contents are dead
            tc::mbar_arrive_expect_tx(bar_tma + b, F16 ? 2 * RAW_TILE : RAW_BUF);
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const int x = it.h * D + 64 * half;
                const uint32_t o2 = half * (RAW_TILE / 2);
                tc::tma_load_2d(dst + RAW_Q + o2, &maps.q, bar_tma + b, x, it.c0);
                tc::tma_load_2d(dst + RAW_K + o2, &maps.k, bar_tma + b, x, it.c0);
                if (!F16) tc::tma_load_2d(dst + RAW_G + o2, &maps.g, bar_tma + b, x, it.c0);
            }
        }
    };
    // F16: the FP32 g tile of item `it` ([64][128], dense rows) into the Gamma
    // array, once the previous item's last Gamma reads are behind a barrier.
    auto load_g32 = [&](const PrepItem& it) {
        if (F16 && copier && it.valid) {
            tc::fence_async_smem();
            tc::mbar_arrive_expect_tx(bar_g, 64 * D * 4);
            tc::tma_load_2d(sm + PS_GAM, &maps.g, bar_g, it.h * D, it.c0);
        }
    };
    // beta of item `it` (threads 0..63): the raw BF16 bits, widened only
    // when the item starts.  Every thread loads from a valid address (the
    // tensor's first element where the row is not part of the item) and the
    // mask is kept apart and applied at that point: no operation touches the
    // loaded value, and so waits for it, before then.
    using BetaRaw = typename std::conditional<F16, float, uint16_t>::type;
    const BetaRaw* betap = static_cast<const BetaRaw*>(beta);
    auto beta_live = [&](const PrepItem& it) { return tid < C && it.valid && tid < it.L; };
    auto load_beta = [&](const PrepItem& it) {
        const BetaRaw* src =
            beta_live(it) ? betap + (size_t)(it.c0 + tid) * maps.b_stride + it.h : betap;
        return __ldg(src);
    };
    auto beta_of = [&](BetaRaw raw, bool live) {
        if constexpr (F16) return live ? raw : 0.f;
        else return live ? (GATED ? sigmoid_hw(bf(raw)) : bf(raw)) : 0.f;
    };

    // The item whose ready flag is still to be released (copier thread): an
    // item's flag goes out during the next item's first A/P product, or at
    // the end of an item that has none, or after the walk.
    long long pending = -1;
    auto release_pending = [&]() {
        if (ready && copier && pending >= 0) {
            tc::bulk_wait_all();
            const long long pg = pending / heads;  // flags are head-major: [heads][pitch]
            if (publish) tc::flag_release(ready + (pending - pg * heads) * ready_pitch + pg, 1u);
            pending = -1;
        }
    };

    long long item = first;
    PrepItem cur = prep_item(item, heads, map_cu, map_off, n_seqs, t, t_pad);
    load_raw(cur, 0);
    load_g32(cur);
    BetaRaw beta_cur = load_beta(cur);
    bool blive_cur = beta_live(cur);
    // gated calls: dt_bias of this thread's channel (tid & 127 in the Gamma
    // phase) and a_log of the item's head, loaded one item ahead
    auto load_gate = [&](const PrepItem& it) {
        float2 r = make_float2(0.f, 0.f);
        if (GATED) {  // head 0's parameters stand in for an invalid item (never used)
            const int hh = it.valid ? it.h : 0;
            r = make_float2(__ldg(maps.dt_bias + hh * D + (tid & 127)), __ldg(maps.a_log + hh));
        }
        return r;
    };
    float2 gate_cur = load_gate(cur);

    for (int iter = 0; item < items; ++iter) {
        const int b = iter & 1;
        const long long nitem = item + stride;
        PrepItem nxt = {};
        nxt.valid = false;
        BetaRaw beta_nxt = 0;
        bool blive_nxt = false;
        float2 gate_nxt = make_float2(0.f, 0.f);
        // The next item is resolved (global loads) while the first A/P product
        // runs, and its raw tiles go to the other buffer, which the previous
        // iteration's closing barrier released.
        auto resolve_next = [&]() {  // the item, and its beta and gate loads
            if (nitem < items) nxt = prep_item(nitem, heads, map_cu, map_off, n_seqs, t, t_pad);
            beta_nxt = load_beta(nxt);
            blive_nxt = beta_live(nxt);
            gate_nxt = load_gate(nxt);
        };
        auto fetch_next = [&]() {
            if (nitem < items) nxt = prep_item(nitem, heads, map_cu, map_off, n_seqs, t, t_pad);
            load_raw(nxt, b ^ 1);
            beta_nxt = load_beta(nxt);
            blive_nxt = beta_live(nxt);
            gate_nxt = load_gate(nxt);
        };

        if (!cur.valid) {
            if (tid == 0) atomicOr(&g_tc_status, STATUS_BAD_CU_SEQLENS);
            fetch_next();
            load_g32(nxt);
        } else {
            const int L = cur.L, h = cur.h;
            const unsigned char* RAWQ = sm + b * RAW_BUF + RAW_Q;
            const unsigned char* RAWK = sm + b * RAW_BUF + RAW_K;
            const unsigned char* RAWG = sm + b * RAW_BUF + RAW_G;
            float* GMID = reinterpret_cast<float*>(sm + b * RAW_BUF + RB_GMID);
            float* GLAST = reinterpret_cast<float*>(sm + b * RAW_BUF + RB_GLAST);
            float* PC = reinterpret_cast<float*>(sm + b * RAW_BUF + RB_PC);
            float* AM = reinterpret_cast<float*>(sm + b * RAW_BUF + RB_AM);
            float* TM = reinterpret_cast<float*>(sm + b * RAW_BUF + RB_TM);
            unsigned char* blob = ws + blob_offset(n_seqs, cur.g, h, heads);

            if (tid < C) BETA[tid] = beta_of(beta_cur, blive_cur);
            if (!tc::mbar_wait(bar_tma + b, (ph_tma >> b) & 1u)) {
                atomicOr(&g_tc_status, STATUS_TIMEOUT);
                failed = true;
            }
            ph_tma ^= 1u << b;
            if (F16) {
                if (!tc::mbar_wait(bar_g, ph_g)) {
                    atomicOr(&g_tc_status, STATUS_TIMEOUT);
                    failed = true;
                }
                ph_g ^= 1u;
            }

            // ------------------------------------------------------ P1 Gamma
            // Four 16-token quarters per channel, then each quarter adds the
            // totals of the quarters before it.  The totals sit in the other raw
            // buffer, whose next tiles are requested only after this phase.
            bool wide, steep;
            float* GH = reinterpret_cast<float*>(sm + (b ^ 1) * RAW_BUF);  // [3][128]
            {
                const int i = tid & 127, qt = tid >> 7;
                // gated: -exp(a_log[h]) log2 e, the exponent's factor of this head
                const float nc = -ex2_approx(gate_cur.y * kLog2e) * kLog2e;
                float acc[16];
                if constexpr (GATED) {  // all 16 rows at once (independent), then masked
#pragma unroll
                    for (int rr = 0; rr < 16; ++rr)
                        acc[rr] = gate_hw(raw1(RAWG, 16 * qt + rr, i), gate_cur.x, nc, maps.lb);
                }
                // F16: the FP32 g tile, dense rows, in the Gamma array; every
                // thread reads its rows before the barriers below, and writes
                // Gamma over them only after them
                const float* G32 = GAM;
                float run = 0.f, gmin = 0.f;
#pragma unroll
                for (int rr = 0; rr < 16; ++rr) {
                    const int r = 16 * qt + rr;
                    float gv = 0.f;
                    if (r < L) gv = GATED ? acc[rr] : (F16 ? G32[r * D + i] : raw1(RAWG, r, i));
                    gmin = fminf(gmin, gv);
                    run = __fadd_rn(run, gv);
                    acc[rr] = run;
                }
                if (qt < 3) GH[qt * 128 + i] = run;
                wide = __syncthreads_and(gmin >= -kWideGMin);  // false on NaN too
                steep = __syncthreads_or(!(gmin >= -kNarrowGMin));  // true on NaN
                // the g tile is dead from here on: its end takes the reference rows
                float base = 0.f;
                if (qt > 0) base = GH[i];
                if (qt > 1) base = __fadd_rn(base, GH[128 + i]);
                if (qt > 2) base = __fadd_rn(base, GH[256 + i]);
#pragma unroll
                for (int rr = 0; rr < 16; ++rr) {
                    const float gr = (qt > 0) ? __fadd_rn(acc[rr], base) : acc[rr];
                    GAM[(16 * qt + rr) * KP + i] = gr;
                    if (rr == 8) GMID[qt * 128 + i] = gr;              // rows 8, 24, 40, 56
                    if (rr == 1 && qt == 1) GMID[4 * 128 + i] = gr;    // row 17
                    if (rr == 1 && qt == 3) GMID[5 * 128 + i] = gr;    // row 49
                    if (rr == 15 && qt == 3) {                         // row 63
                        GLAST[i] = gr;
                        if (!failed) reinterpret_cast<float*>(blob + BLOB_DEC)[i] = __expf(gr);
                    }
                }
            }
            if (copier) tc::bulk_wait_read_all();  // the last item's operands left OPX and Y
            __syncthreads();
            if (wide) {  // per-channel constants of the operand build below
                if (tid < 128) {
                    const float g17 = GMID[4 * 128 + tid], g49 = GMID[5 * 128 + tid];
                    PC[tid] = __expf(g17);
                    PC[128 + tid] = __expf(GLAST[tid] - g17);
                    PC[256 + tid] = __expf(GLAST[tid] - g49);
                }
                __syncthreads();
            }

            // ------------------------------------------------------ P2 A and P blocks
            // X_b rows r >= r0: k_r and qh_r times e^(Gamma_r - Gamma_mb).
            auto build_x = [&](int r0, const float* gmb) {
                const int r = tid & 63, qg = tid >> 6;
                if (r >= r0) {
                    const bool live = r < L;
#pragma unroll 1  // the narrow path only: kept compact
                    for (int jj = 0; jj < 32 / (NTP / 64); ++jj) {
                        const int j = qg + (NTP / 64) * jj;
                        const float4 gm = *reinterpret_cast<const float4*>(gmb + 4 * j);
                        const float4 ga = *reinterpret_cast<const float4*>(GAM + r * KP + 4 * j);
                        float4 kf = in4<F16>(RAWK, r, 4 * j), qf = in4<F16>(RAWQ, r, 4 * j);
                        if (!live) kf = qf = make_float4(0.f, 0.f, 0.f, 0.f);
                        const float f0 = __expf(ga.x - gm.x), f1 = __expf(ga.y - gm.y),
                                    f2 = __expf(ga.z - gm.z), f3 = __expf(ga.w - gm.w);
                        st4(sm + PS_OPX, OpX::off(r, 4 * j), kf.x * f0, kf.y * f1, kf.z * f2,
                            kf.w * f3);
                        st4(sm + PS_OPX, OpX::off(64 + r, 4 * j), KDA_Q_SCALE * qf.x * f0,
                            KDA_Q_SCALE * qf.y * f1, KDA_Q_SCALE * qf.z * f2,
                            KDA_Q_SCALE * qf.w * f3);
                    }
                }
            };
            // Both 32-token blocks' operands in one pass: X_0 for every row into
            // OPX, X_1 for rows 32..63 into a compact 64-row operand (k rows, then q
            // rows) in the idle raw buffer (the second product's 64 padding rows
            // read the next K group, or the 1 KB after the operand, and are never
            // used), and Y_b for the rows of block b, whose factor
            // e^(Gamma_mb - Gamma_s) is the reciprocal of the row's own X_b factor
            // (both within e^(+-17 kWideGMin), normal FP32 numbers).
            unsigned char* x1buf = sm + (b ^ 1) * RAW_BUF;
            // The scan's operands of the wide path are formed in the same pass,
            // from the same factors, and held in registers (FP16 pairs) until
            // the A/P products have released their buffers:
            //   Ktil_r = k_r e^(Gamma_r - Gamma_17) e^Gamma_17,
            //   Khat_r = beta_r k_r e^(Gamma_mb - Gamma_r) e^(Gamma_63 - Gamma_mb).
            // A product below 2^-24 (flushed, or FP16 zero) has no FP16 value.
            constexpr int P3J = 32 / (NTP / 64);
            uint32_t p3k[P3J][2], p3q[P3J][2], p3h[P3J][2];
            auto build_xy_wide = [&]() {
                const int r = tid & 63, qg = tid >> 6;
                const bool live = r < L;
                const float br = BETA[r];  // 0 past the chunk's end
                const float* gm0 = GMID + 4 * 128;
                const float* gm1 = GMID + 5 * 128;
                const float* pcl = PC + (r < 32 ? 128 : 256);  // e^(Gamma_63 - Gamma_mb)
                unsigned char* ydst = sm + PS_Y + (r >> 5) * OpY32::bytes(128);
#pragma unroll
                for (int jj = 0; jj < P3J; ++jj) {
                    const int j = qg + (NTP / 64) * jj;
                    const float4 ga = *reinterpret_cast<const float4*>(GAM + r * KP + 4 * j);
                    float4 kf = in4<F16>(RAWK, r, 4 * j), qf = in4<F16>(RAWQ, r, 4 * j);
                    if (!live) kf = qf = make_float4(0.f, 0.f, 0.f, 0.f);
                    qf = make_float4(KDA_Q_SCALE * qf.x, KDA_Q_SCALE * qf.y, KDA_Q_SCALE * qf.z,
                                     KDA_Q_SCALE * qf.w);
                    {
                        const float4 gm = *reinterpret_cast<const float4*>(gm0 + 4 * j);
                        const float f0 = __expf(ga.x - gm.x), f1 = __expf(ga.y - gm.y),
                                    f2 = __expf(ga.z - gm.z), f3 = __expf(ga.w - gm.w);
                        st4(sm + PS_OPX, OpX::off(r, 4 * j), kf.x * f0, kf.y * f1, kf.z * f2,
                            kf.w * f3);
                        st4(sm + PS_OPX, OpX::off(64 + r, 4 * j), qf.x * f0, qf.y * f1, qf.z * f2,
                            qf.w * f3);
                        const float4 c0 = *reinterpret_cast<const float4*>(PC + 4 * j);
                        const float e0 = f0 * c0.x, e1 = f1 * c0.y, e2 = f2 * c0.z, e3 = f3 * c0.w;
                        p3k[jj][0] = tc::pack_f16x2(kf.x * e0, kf.y * e1);
                        p3k[jj][1] = tc::pack_f16x2(kf.z * e2, kf.w * e3);
                        p3q[jj][0] = tc::pack_f16x2(qf.x * e0, qf.y * e1);
                        p3q[jj][1] = tc::pack_f16x2(qf.z * e2, qf.w * e3);
                        if (r < 32) {
                            const float y0 = rcp_fast(f0), y1 = rcp_fast(f1), y2 = rcp_fast(f2),
                                        y3 = rcp_fast(f3);
                            st4(ydst, OpY32::off(r, 4 * j), kf.x * y0, kf.y * y1, kf.z * y2,
                                kf.w * y3);
                            const float4 cl = *reinterpret_cast<const float4*>(pcl + 4 * j);
                            p3h[jj][0] = tc::pack_f16x2(br * kf.x * y0 * cl.x, br * kf.y * y1 * cl.y);
                            p3h[jj][1] = tc::pack_f16x2(br * kf.z * y2 * cl.z, br * kf.w * y3 * cl.w);
                        }
                    }
                    if (r >= 32) {
                        const float4 gm = *reinterpret_cast<const float4*>(gm1 + 4 * j);
                        const float f0 = __expf(ga.x - gm.x), f1 = __expf(ga.y - gm.y),
                                    f2 = __expf(ga.z - gm.z), f3 = __expf(ga.w - gm.w);
                        st4(x1buf, OpX1::off(r - 32, 4 * j), kf.x * f0, kf.y * f1, kf.z * f2,
                            kf.w * f3);
                        st4(x1buf, OpX1::off(r, 4 * j), qf.x * f0, qf.y * f1, qf.z * f2,
                            qf.w * f3);
                        const float y0 = rcp_fast(f0), y1 = rcp_fast(f1), y2 = rcp_fast(f2),
                                    y3 = rcp_fast(f3);
                        st4(ydst, OpY32::off(r - 32, 4 * j), kf.x * y0, kf.y * y1, kf.z * y2,
                            kf.w * y3);
                        const float4 cl = *reinterpret_cast<const float4*>(pcl + 4 * j);
                        p3h[jj][0] = tc::pack_f16x2(br * kf.x * y0 * cl.x, br * kf.y * y1 * cl.y);
                        p3h[jj][1] = tc::pack_f16x2(br * kf.z * y2 * cl.z, br * kf.w * y3 * cl.w);
                    }
                }
            };
            auto p3_store = [&]() {  // the registers above into the freed operand buffers
                const int r = tid & 63, qg = tid >> 6;
                unsigned char* kh = sm + PS_Y;
#pragma unroll
                for (int jj = 0; jj < P3J; ++jj) {
                    const int j = qg + (NTP / 64) * jj;
                    *reinterpret_cast<uint2*>(sm + PS_OPX + OpXh::off(r, 4 * j)) =
                        make_uint2(p3k[jj][0], p3k[jj][1]);
                    *reinterpret_cast<uint2*>(sm + PS_OPX + OpXh::off(64 + r, 4 * j)) =
                        make_uint2(p3q[jj][0], p3q[jj][1]);
                    *reinterpret_cast<uint16_t*>(kh + OpKHh::off(4 * j, r)) = (uint16_t)p3h[jj][0];
                    *reinterpret_cast<uint16_t*>(kh + OpKHh::off(4 * j + 1, r)) =
                        (uint16_t)(p3h[jj][0] >> 16);
                    *reinterpret_cast<uint16_t*>(kh + OpKHh::off(4 * j + 2, r)) = (uint16_t)p3h[jj][1];
                    *reinterpret_cast<uint16_t*>(kh + OpKHh::off(4 * j + 3, r)) =
                        (uint16_t)(p3h[jj][1] >> 16);
                }
            };
            // Y_b row s of block b = s >> bshift: k_s e^(Gamma_mb - Gamma_s).
            auto build_y = [&](int bshift, int gm_row0, uint32_t ybytes, auto op) {
#pragma unroll 1  // the narrow path only: kept compact
                for (int e = tid; e < 64 * 32; e += NTP) {
                    const int s = e & 63, j = e >> 6, bb = s >> bshift;
                    const float4 gm =
                        *reinterpret_cast<const float4*>(GMID + (gm_row0 + bb) * 128 + 4 * j);
                    const float4 ga = *reinterpret_cast<const float4*>(GAM + s * KP + 4 * j);
                    float4 kf = in4<F16>(RAWK, s, 4 * j);
                    if (s >= L) kf = make_float4(0.f, 0.f, 0.f, 0.f);
                    st4(sm + PS_Y + bb * ybytes, decltype(op)::off(s & ((1 << bshift) - 1), 4 * j),
                        kf.x * __expf(gm.x - ga.x), kf.y * __expf(gm.y - ga.y),
                        kf.z * __expf(gm.z - ga.z), kf.w * __expf(gm.w - ga.w));
                }
            };
            // the steep path's A and P, FP32 [64][64] each, in the second half of
            // the A operand region (the first half takes Ktil and Qtil in P3)
            float* SA = reinterpret_cast<float*>(sm + PS_OPX + OpX::bytes(128) / 2);
            float* SPV = SA + 64 * 64;
            if (wide) {
                // Two 32-token column blocks (every g of the chunk is >= -kWideGMin).
                build_xy_wide();
                sync_for_mma();
                // the two blocks' products are independent: two threads of two
                // warps issue them side by side (a single issuing thread spends
                // about 45 cycles per instruction), each with its own barrier
                if (tid == 0) {
                    tc::tc_fence_after();
                    issue_mma<OpX, OpY32, 16>(tmem + TC_AP, s_opx, s_y, tc::idesc_tf32(128, 32));
                    tc::mma_commit(bar_mma);
                } else if (tid == 32) {
                    tc::tc_fence_after();
                    issue_mma<OpX1, OpY32, 16>(tmem + TC_AP + 32, tc::smem_u32(x1buf),
                                               s_y + OpY32::bytes(128), tc::idesc_tf32(128, 32));
                    tc::mma_commit(bar_mma2);
                }
                release_pending();
                // Two-kernel path: the next item is resolved while the products
                // run (in the fused grid that moves no time off its critical
                // path, the copier's, and measured slower)
                if constexpr (TWO_KERNEL) resolve_next();
                wait_mma();
                if (!tc::mbar_wait(bar_mma2, ph_mma2)) {
                    atomicOr(&g_tc_status, STATUS_TIMEOUT);
                    failed = true;
                }
                ph_mma2 ^= 1;
                tc::tc_fence_after();
                // the compact X_1 in the other buffer has been read
                if constexpr (TWO_KERNEL) load_raw(nxt, b ^ 1);
                else fetch_next();
                p3_store();
            } else if (steep) {
                // Exact products on the CUDA cores: thread (column s = tid & 63)
                // forms A_rs and P_rs for rows r = tid / 64 + 8 k.  The results
                // wait in shared memory until the raw tiles and Gamma are dead
                // (P4).  A rare path, kept compact (its loops are not unrolled):
                // code that the common path's instruction stream skips over
                // still costs it time.
                fetch_next();
                const int s2 = tid & 63;
                const bool slive = s2 < L;
#pragma unroll 1
                for (int k8 = 0; k8 < 8; ++k8) {
                    const int r2 = (tid >> 6) + 8 * k8;
                    float a = 0.f, pv = 0.f;
                    if (s2 <= r2) {
                        const bool rlive = r2 < L;
#pragma unroll 1
                        for (int i = 0; i < D; i += 4) {
                            const float4 gr = *reinterpret_cast<const float4*>(GAM + r2 * KP + i);
                            const float4 gs = *reinterpret_cast<const float4*>(GAM + s2 * KP + i);
                            float4 kr = in4<F16>(RAWK, r2, i), qr = in4<F16>(RAWQ, r2, i), ks = in4<F16>(RAWK, s2, i);
                            if (!rlive) kr = qr = make_float4(0.f, 0.f, 0.f, 0.f);
                            if (!slive) ks = make_float4(0.f, 0.f, 0.f, 0.f);
                            const float e0 = __expf(gr.x - gs.x), e1 = __expf(gr.y - gs.y),
                                        e2 = __expf(gr.z - gs.z), e3 = __expf(gr.w - gs.w);
                            a = __fmaf_rn(kr.x * ks.x, e0, a);
                            a = __fmaf_rn(kr.y * ks.y, e1, a);
                            a = __fmaf_rn(kr.z * ks.z, e2, a);
                            a = __fmaf_rn(kr.w * ks.w, e3, a);
                            pv = __fmaf_rn(qr.x * ks.x, e0, pv);
                            pv = __fmaf_rn(qr.y * ks.y, e1, pv);
                            pv = __fmaf_rn(qr.z * ks.z, e2, pv);
                            pv = __fmaf_rn(qr.w * ks.w, e3, pv);
                        }
                    }
                    SA[r2 * 64 + s2] = a;
                    SPV[r2 * 64 + s2] = KDA_Q_SCALE * pv;
                }
            } else {
                // Four 16-token column blocks with reference token 16 b + 8.
                build_y(4, 0, OpY::bytes(128), OpY{});
#pragma unroll 1  // a rare path, kept compact
                for (int bb = 0; bb < 4; ++bb) {
                    build_x(16 * bb, GMID + bb * 128);
                    sync_for_mma();
                    if (tid == 0) {
                        tc::tc_fence_after();
                        issue_mma<OpX, OpY, 16>(tmem + TC_AP + 16 * bb, s_opx,
                                                s_y + bb * OpY::bytes(128),
                                                tc::idesc_tf32(128, 16));
                        tc::mma_commit(bar_mma);
                    }
                    if (bb == 0) {
                        release_pending();
                        fetch_next();
                    }
                    wait_mma();
                }
            }

            // ------------------------------------------------------ P3 [Ktil; Qtil], Khat^T
            // Built in the A/P operand buffers (both products are complete; the
            // wide path has formed them during its operand build) and sent to
            // the workspace by bulk copies that drain during P4 and P5.  Thread
            // (r, qg) forms token r's channels 4 j .. 4 j + 3: Ktil and Qtil as
            // 8-byte rows, Khat^T as four 2-byte column entries.
            if (!wide) {
                const int r = tid & 63, qg = tid >> 6;
                const bool live = r < L;
                const float br = BETA[r];  // 0 past the chunk's end
#pragma unroll 1  // narrow and steep paths only: kept compact
                for (int jj = 0; jj < 32 / (NTP / 64); ++jj) {
                    const int j = qg + (NTP / 64) * jj;
                    const float4 ga = *reinterpret_cast<const float4*>(GAM + r * KP + 4 * j);
                    const float4 gl = *reinterpret_cast<const float4*>(GLAST + 4 * j);
                    float4 kf = in4<F16>(RAWK, r, 4 * j), qf = in4<F16>(RAWQ, r, 4 * j);
                    if (!live) kf = qf = make_float4(0.f, 0.f, 0.f, 0.f);
                    const float f0 = __expf(ga.x), f1 = __expf(ga.y), f2 = __expf(ga.z),
                                f3 = __expf(ga.w);
                    st4h(sm + PS_OPX + OpXh::off(r, 4 * j), kf.x * f0, kf.y * f1, kf.z * f2,
                         kf.w * f3);
                    st4h(sm + PS_OPX + OpXh::off(64 + r, 4 * j), KDA_Q_SCALE * qf.x * f0,
                         KDA_Q_SCALE * qf.y * f1, KDA_Q_SCALE * qf.z * f2, KDA_Q_SCALE * qf.w * f3);
                    unsigned char* kh = sm + PS_Y;
                    st1h(kh + OpKHh::off(4 * j, r), br * kf.x * __expf(gl.x - ga.x));
                    st1h(kh + OpKHh::off(4 * j + 1, r), br * kf.y * __expf(gl.y - ga.y));
                    st1h(kh + OpKHh::off(4 * j + 2, r), br * kf.z * __expf(gl.z - ga.z));
                    st1h(kh + OpKHh::off(4 * j + 3, r), br * kf.w * __expf(gl.w - ga.w));
                }
            }
            tc::fence_async_smem();
            __syncthreads();  // the raw tiles, Gamma and the reference rows are dead from here on
            if (copier && !failed) {
                tc::bulk_store(blob + BLOB_OPX, sm + PS_OPX, OpXh::bytes(128));
                tc::bulk_store(blob + BLOB_KH, sm + PS_Y, OpKHh::bytes(64));
                tc::bulk_commit();
            }
            load_g32(nxt);

            // ------------------------------------------------------ P4 read A, P
            if (steep) {
                const int s2 = tid & 63;
                const float bs = BETA[s2];
#pragma unroll 1
                for (int k8 = 0; k8 < 8; ++k8) {  // each thread reads back its own values
                    const int r2 = (tid >> 6) + 8 * k8;
                    AM[r2 * AP + s2] = (s2 < r2) ? SA[r2 * 64 + s2] * bs : 0.f;
                    if (!failed)
                        *reinterpret_cast<uint16_t*>(blob + BLOB_TP + OpTPh::off(64 + r2, s2)) =
                            tc::f16_bits((s2 <= r2) ? SPV[r2 * 64 + s2] * bs : 0.f);
                }
            } else {   // thread (lane ln, quarter ch) reads columns [16 ch, 16 ch + 16)
                float v[16];
                tc::tmem_ld16(tmem + lane_base + TC_AP + 16 * ch, v);
                tc::tmem_ld_wait();
                if (wide && ch >= 2) {
                    // Second 32-token block from the compact operand: lane l < 32
                    // holds A row 32 + l, lane 32 + l holds P row 32 + l; P rows
                    // 0..31 are zero in these columns (s >= 32 > r).
                    if (ln < 32) {
                        const int r = 32 + ln;
#pragma unroll
                        for (int c = 0; c < 16; ++c) {
                            const int s = 16 * ch + c;
                            AM[r * AP + s] = (s < r) ? v[c] * BETA[s] : 0.f;
                        }
                    } else if (ln < 96 && !failed) {
                        const int r = (ln < 64) ? ln : ln - 64;
                        const bool zero = ln >= 64;
#pragma unroll
                        for (int c4 = 0; c4 < 4; ++c4) {
                            float p[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const int s = 16 * ch + 4 * c4 + e;
                                p[e] = (!zero && s <= r) ? v[4 * c4 + e] * BETA[s] : 0.f;
                            }
                            st4h(blob + BLOB_TP + OpTPh::off(64 + r, 16 * ch + 4 * c4), p[0],
                                 p[1], p[2], p[3]);
                        }
                    }
                } else if (ln < 64) {
                    const int r = ln;
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        const int s = 16 * ch + c;
                        AM[r * AP + s] = (s < r) ? v[c] * BETA[s] : 0.f;
                    }
                } else if (!failed) {
                    const int r = ln - 64;
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4) {
                        float p[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int s = 16 * ch + 4 * c4 + e;
                            p[e] = (s <= r) ? v[4 * c4 + e] * BETA[s] : 0.f;
                        }
                        st4h(blob + BLOB_TP + OpTPh::off(64 + r, 16 * ch + 4 * c4), p[0], p[1],
                             p[2], p[3]);
                    }
                }
            }
            tc::tc_fence_before();
            __syncthreads();

            // ------------------------------------------------------ P5 T = (I + A)^-1
            // The diagonal 16 x 16 blocks by forward substitution, one column per
            // thread with the column in registers: after x_s is final, every later
            // row subtracts A_rs x_s, so each row's terms are added in the order
            // of s.  Below the diagonal, two levels of block inversion: the
            // inverse of [[L11, 0], [L21, L22]] has the lower-left block
            // -L22^-1 L21 L11^-1; first inside the two 32 x 32 diagonal blocks
            // (16 x 16 pieces), then for the whole matrix (32 x 32 pieces).  The
            // products' intermediates sit in T's upper right 32 x 32 block, which
            // the store below replaces by zeros; the two upper 16 x 16 blocks that
            // the level-2 products read as part of T are zeroed here.
            if (tid < 64) {
                const int o0 = 16 * (tid >> 4), cc = tid & 15;
                float x[16];
#pragma unroll
                for (int rr = 0; rr < 16; ++rr) x[rr] = (rr == cc) ? 1.f : 0.f;
#pragma unroll
                for (int ss = 0; ss < 15; ++ss) {
#pragma unroll
                    for (int rr = ss + 1; rr < 16; ++rr)
                        x[rr] = __fmaf_rn(-AM[(o0 + rr) * AP + o0 + ss], x[ss], x[rr]);
                }
#pragma unroll
                for (int rr = 0; rr < 16; ++rr) TM[(o0 + rr) * TPP + o0 + cc] = x[rr];
            } else if (tid < 128) {  // T_01 and T_23 (above the diagonal) are zero
                const int e = tid - 64, blk = e >> 5, rr = (e >> 1) & 15, hh = e & 1;
                float* z = TM + (32 * blk + rr) * TPP + 32 * blk + 16 + 8 * hh;
                *reinterpret_cast<float4*>(z) = make_float4(0.f, 0.f, 0.f, 0.f);
                *reinterpret_cast<float4*>(z + 4) = make_float4(0.f, 0.f, 0.f, 0.f);
            }
            __syncthreads();
            // Both levels run on eight warps, register-tiled (a thread forms
            // 1 x 2 or 2 x 2 outputs per shared-memory row and column load), with
            // warps laid out so that a product's triangular operand bounds its k
            // range uniformly inside a warp; the terms left out are exact zeros,
            // so every sum keeps the order of the full product.
            if (tid < 256) {  // level 1: warps 4 pr .. 4 pr + 3 form T_ab, (a, b) = (2 pr + 1, 2 pr)
                const int w = tid >> 5, ln = tid & 31;
                const int pr = w >> 2, rh = (w >> 1) & 1, chh = w & 1;  // 8 x 8 quadrant
                const int ob = 32 * pr, oa = ob + 16;
                const int r = 8 * rh + (ln >> 2), c = 8 * chh + 2 * (ln & 3);
                float* mscr = TM + 32 + 16 * pr;  // M = A_ab T_bb in rows 0..15
                float m0 = 0.f, m1 = 0.f;
                // T_bb is lower triangular: its rows below 8 chh add nothing here
#pragma unroll 4
                for (int k = 8 * chh; k < 16; ++k) {
                    const float a = AM[(oa + r) * AP + ob + k];
                    const float2 tv = *reinterpret_cast<const float2*>(TM + (ob + k) * TPP + ob + c);
                    m0 = __fmaf_rn(a, tv.x, m0);
                    m1 = __fmaf_rn(a, tv.y, m1);
                }
                *reinterpret_cast<float2*>(mscr + r * TPP + c) = make_float2(m0, m1);
                if (pr == 0) asm volatile("bar.sync 3, 128;" ::: "memory");
                else asm volatile("bar.sync 4, 128;" ::: "memory");
                float t0 = 0.f, t1 = 0.f;
                // T_aa is lower triangular: its columns past 8 rh + 7 add nothing here
#pragma unroll 4
                for (int k = 0; k < 8 * rh + 8; ++k) {
                    const float a = TM[(oa + r) * TPP + oa + k];
                    const float2 mv = *reinterpret_cast<const float2*>(mscr + k * TPP + c);
                    t0 = __fmaf_rn(a, mv.x, t0);
                    t1 = __fmaf_rn(a, mv.y, t1);
                }
                *reinterpret_cast<float2*>(TM + (oa + r) * TPP + ob + c) = make_float2(-t0, -t1);
            }
            __syncthreads();
            if (tid < 256) {  // level 2: rows 32..63, columns 0..31 (eight warps)
                const int w = tid >> 5, ln = tid & 31;
                {   // M1 = A_[23][01] T_[01][01]: warp w takes columns 4 w .. 4 w + 3, all
                    // rows; T_[01][01] is lower triangular, so k starts at 4 w
                    const int r0 = 2 * (ln >> 1), c0 = 4 * w + 2 * (ln & 1);
                    float m00 = 0.f, m01 = 0.f, m10 = 0.f, m11 = 0.f;
#pragma unroll 4
                    for (int k = 4 * w; k < 32; ++k) {
                        const float a0 = AM[(32 + r0) * AP + k], a1 = AM[(33 + r0) * AP + k];
                        const float2 tv = *reinterpret_cast<const float2*>(TM + k * TPP + c0);
                        m00 = __fmaf_rn(a0, tv.x, m00); m01 = __fmaf_rn(a0, tv.y, m01);
                        m10 = __fmaf_rn(a1, tv.x, m10); m11 = __fmaf_rn(a1, tv.y, m11);
                    }
                    *reinterpret_cast<float2*>(TM + r0 * TPP + 32 + c0) = make_float2(m00, m01);
                    *reinterpret_cast<float2*>(TM + (r0 + 1) * TPP + 32 + c0) = make_float2(m10, m11);
                }
                asm volatile("bar.sync 1, 256;" ::: "memory");
                {   // -T_[23][23] M1: warp w takes rows 4 w .. 4 w + 3, all columns;
                    // T_[23][23] is lower triangular, so k stops at 4 w + 3
                    const int r0 = 4 * w + 2 * (ln >> 4), c0 = 2 * (ln & 15);
                    float t00 = 0.f, t01 = 0.f, t10 = 0.f, t11 = 0.f;
#pragma unroll 4
                    for (int k = 0; k < 4 * w + 4; ++k) {
                        const float a0 = TM[(32 + r0) * TPP + 32 + k], a1 = TM[(33 + r0) * TPP + 32 + k];
                        const float2 mv = *reinterpret_cast<const float2*>(TM + k * TPP + 32 + c0);
                        t00 = __fmaf_rn(a0, mv.x, t00); t01 = __fmaf_rn(a0, mv.y, t01);
                        t10 = __fmaf_rn(a1, mv.x, t10); t11 = __fmaf_rn(a1, mv.y, t11);
                    }
                    *reinterpret_cast<float2*>(TM + (32 + r0) * TPP + c0) = make_float2(-t00, -t01);
                    *reinterpret_cast<float2*>(TM + (33 + r0) * TPP + c0) = make_float2(-t10, -t11);
                }
            }
            __syncthreads();
            if (!failed) {  // T into rows 0..63 of [T; P], zeros above the diagonal
                const int r = tid & 63, qg = tid >> 6;
#pragma unroll
                for (int jj = 0; jj < 16 / (NTP / 64); ++jj) {
                    const int j = qg + (NTP / 64) * jj;
                    const float4 tr = *reinterpret_cast<const float4*>(TM + r * TPP + 4 * j);
                    const int c = 4 * j;
                    st4h(blob + BLOB_TP + OpTPh::off(r, c), c <= r ? tr.x : 0.f,
                         c + 1 <= r ? tr.y : 0.f, c + 2 <= r ? tr.z : 0.f, c + 3 <= r ? tr.w : 0.f);
                }
            }
            tc::tc_fence_before();
            __syncthreads();  // buffer b is free for the item after next
        }
        // every thread's stores of this item precede the barrier above (an
        // invalid item stores nothing)
        if (ready && copier) {
            release_pending();  // an item without an A/P product in between
            pending = item;
        }
        item = nitem;
        cur = nxt;
        beta_cur = beta_nxt;
        blive_cur = blive_nxt;
        gate_cur = gate_nxt;
    }
    release_pending();
    if (copier) tc::bulk_wait_all();
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, 64);
    }
}

template <bool GATED, bool F16>
__global__ void __launch_bounds__(NTP, 1)
prepare_kernel(const __grid_constant__ PrepMaps maps, const void* __restrict__ beta, int t,
               int t_pad, int heads, const int* __restrict__ cu, int n_seqs,
               unsigned char* __restrict__ ws) {
    pdl_wait();  // the chunk map (and the callers' inputs) are complete
    pdl_release();
    prepare_role<GATED, F16, true>(maps, beta, t, t_pad, heads, cu, n_seqs, ws, blockIdx.x,
                                   gridDim.x,
                             nullptr, 0);
}

// ------------------------------------------------------------ transposed scan
// One CTA per (sequence, head) carries the whole 128 x 128 state through the
// chunks in transposed form, so that each matrix on the state's chain is the
// A operand of the next product and stays in TMEM (lane = value column j,
// two FP16 values per column along K):
//   X^T = V^T - S^T Ktil^T;  U^T = X^T T^T;  O^T = S^T Qtil^T + U^T P^T;
//   S^T <- S^T diag(dec) + U^T Khat
// The prepared operands are the B operands, in the layouts prepare writes:
// [Ktil; Qtil] (rows = tokens), [T; P] (rows = tokens) and Khat^T (rows = key
// channels).  S^T, X^T and U^T enter TMEM by tcgen05.st from the threads that
// computed them, so no operand passes through shared memory on the chain.
struct ScanT {
    static constexpr int NT = 512;  // 4 lane quarters x 4 column groups
    // shared memory: blob image (OPX | TP | KH | DEC: operand group 0 of
    // [Ktil; Qtil] and of [T; P] | Khat^T | dec), value tile [64][128] BF16
    // (no swizzle), group 1 of [T; P] | Khat^T | dec, group 1 of
    // [Ktil; Qtil], the O staging tile [64][128] FP32, barriers
    static constexpr uint32_t BGRP = BLOB_BYTES - BLOB_TP;  // [T; P] | Khat^T | dec
    static constexpr uint32_t RAWV = (BLOB_BYTES + 127) & ~127u;
    static constexpr uint32_t TP1 = RAWV + 64 * D * 2;
    static constexpr uint32_t OPX1 = (TP1 + BGRP + 127) & ~127u;
    static constexpr uint32_t OST = OPX1 + OpXh::bytes(128);
    static constexpr uint32_t RAWV1 = OST + 64 * D * 4;  // the second value tile
    // two gate tiles ([64][128] BF16, kda_prefill_o_norm) by chunk parity;
    // each is overwritten in place by its chunk's normalised output
    static constexpr uint32_t GATE0 = RAWV1 + 64 * D * 2, GATE1 = GATE0 + 64 * D * 2;
    static constexpr uint32_t BAR = GATE1 + 64 * D * 2;
    static constexpr uint32_t TOTAL = BAR + 128;
    // TMEM columns: S^T (A, FP16 pairs: 64 columns), T X (64); two
    // 128-column chunk regions used alternately: chunk g computes Ktil S |
    // Qtil S, then O, in R_(g mod 2) and keeps X^T / U^T (A, FP16 pairs: 32
    // columns) in the first columns of the other region, whose last 64 still
    // hold chunk g - 1's O until chunk g + 1's first product; the FP32 state
    // S^T itself, which the last product of a chunk accumulates into
    static constexpr uint32_t T_S = 0, T_TX = 64, R0 = 128, R1 = 256, T_SA = 384;
    static constexpr uint32_t TMEM_COLS = 512;
    static_assert(TOTAL <= 232448, "shared memory budget exceeded");
    static_assert(TP1 % 16 == 0 && OST % 128 == 0, "copy alignment");
};

// The chain of (sequence n, head h).  When `ready` is set, chunk g's operands
// are read only after ready[g * heads + h] has been released by the CTA that
// prepared them (the prepare and scan roles then share one cooperative grid).
//
// Per chunk: three tensor-core round trips of 8, 4 and 8 FP16 K-steps (the
// tensor core takes about the same time per instruction for any N <= 128,
// so Qtil S rides with Ktil S and P U with Khat^T U).  Both operand groups
// are double-buffered by chunk parity, so chunk g + 1's are requested (after
// its ready flag) while chunk g's first product runs, a whole chunk ahead;
// the value tile as soon as it is consumed.  O of chunk g - 1 is read from
// TMEM and staged while chunk g's last product runs, by the warps that do
// not issue it (warp 0's rows go to the other warps of its TMEM lane
// quarter), and leaves by one TMA tile store that no thread waits for:
// per-thread global stores of O cost the chain about 1.4K cycles per chunk
// while the prepare CTAs keep the memory system busy.  Rows of a partial
// chunk go out by plain stores.
// NORM (kda_prefill_o_norm): O is not written.  The staged O tile of chunk
// g - 1 is normalised at the start of chunk g + 1, while its first product
// runs, by warps 8..15 (the sigmoid-gated RMSNorm with the tile's BF16 gate,
// loaded by TMA a chunk ahead), and the BF16 result leaves by one TMA tile
// store; the last chunk's tile is normalised after the loop and written by
// plain stores.
// F16: the value tiles hold FP16 (FP32 inputs, converted before the call).
template <bool NORM, bool F16, bool TWO_KERNEL>
__device__ __forceinline__ void scan_t_role(const CUtensorMap& vmap, const CUtensorMap& omap,
                                            float* __restrict__ state,
                                            float* __restrict__ o, int t, int t_pad, int heads,
                                            const int* __restrict__ cu, int n_seqs,
                                            const unsigned char* __restrict__ ws, int h, int n,
                                            const unsigned* __restrict__ ready,
                                            long long ready_pitch, const NormArgs* na,
                                            uint32_t acquire_iters = 1u << 22) {
    extern __shared__ __align__(1024) unsigned char sm[];
    const int tid = threadIdx.x, warp = tid >> 5;
    const int qd = warp & 3, cg = warp >> 2;  // TMEM lane quarter, column group
    const int j = 32 * qd + (tid & 31);       // value column = TMEM lane
    const uint32_t lane_base = (uint32_t)(32 * qd) << 16;
    // Thread 0 issues the tensor-core products; a thread of another warp
    // issues every copy (the ready-flag acquire alone is a global-memory
    // round trip), so neither waits on the other's latency.
    const bool copier = (tid == 128);

    int start, end;
    if (!seq_range(cu, n, n_seqs, t, t_pad, start, end)) {
        if (tid == 0) atomicOr(&g_tc_status, STATUS_BAD_CU_SEQLENS);
        return;
    }
    const long long g0 = __ldg(reinterpret_cast<const int*>(ws) + n);
    if (tc::smem_u32(sm) & 1023u) {
        if (tid == 0) atomicOr(&g_tc_status, STATUS_SMEM_ALIGN);
        return;
    }

    // buffers by chunk parity (selects, not arrays: see prepare_role)
    auto rawv_off = [](int b) { return b ? ScanT::RAWV1 : ScanT::RAWV; };  // value tiles
    float* OST = reinterpret_cast<float*>(sm + ScanT::OST);
    uint64_t* bar_x = reinterpret_cast<uint64_t*>(sm + ScanT::BAR);  // [2]: [Ktil; Qtil] groups
    uint64_t* bar_b = bar_x + 2;                                     // [2]: [T; P] | Khat^T | dec
    uint64_t* bar_v = bar_x + 4;                                     // [2]: value tiles
    uint64_t* bar_mma = bar_x + 6;
    uint64_t* bar_gt = bar_x + 7;  // [2]: the gate tiles (NORM)
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + ScanT::BAR + 80);
    int* abort_flag = reinterpret_cast<int*>(sm + ScanT::BAR + 84);
    auto opx_off = [](int b) { return b ? ScanT::OPX1 : (uint32_t)SS_OPX; };
    auto tp_off = [](int b) { return b ? ScanT::TP1 : (uint32_t)SS_TP; };  // group b: TP, KH, DEC follow

    if (tid == 0) {
        for (int i = 0; i < 9; ++i) tc::mbar_init(bar_x + i, 1);
        tc::fence_mbar_init();
        tc::prefetch_tmap(&vmap);
        if (NORM) {
            tc::prefetch_tmap(&na->gmap);
            tc::prefetch_tmap(&na->nmap);
        } else {
            tc::prefetch_tmap(&omap);
        }
        *abort_flag = 0;
    }
    if (warp == 0) tc::tmem_alloc(tmem_slot, ScanT::TMEM_COLS);
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t my = tmem + lane_base;  // this thread's TMEM lane

    // state: thread (j, cg) moves S[32 cg + i][j], i < 32, between TMEM and
    // registers; the FP32 state lives in TMEM (T_SA) for the whole sequence
    float* Sg = state + ((size_t)n * heads + h) * D * D + (size_t)(32 * cg) * D + j;
    {
        uint32_t sa[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) sa[i] = __float_as_uint(Sg[(size_t)i * D]);
        // S^T: K index 32 cg + i in column 16 cg + i / 2
        uint32_t sv[16];
#pragma unroll
        for (int m = 0; m < 16; ++m)
            sv[m] = tc::pack_f16x2(__uint_as_float(sa[2 * m]), __uint_as_float(sa[2 * m + 1]));
        tc::tmem_st16u(my + ScanT::T_S + 16 * cg, sv);
        tc::tmem_st32u(my + ScanT::T_SA + 32 * cg, sa);
        tc::tmem_st_wait();
    }

    uint32_t ph_mma = 0, ph_v = 0, ph_x = 0, ph_b = 0;  // ph_v, ph_x, ph_b: bit per buffer
    auto wait_bar = [&](uint64_t* bar, uint32_t parity) {
        if (!tc::mbar_wait(bar, parity)) {
            atomicOr(&g_tc_status, STATUS_TIMEOUT);
            *abort_flag = 1;
        }
    };
    // Copies (the copier thread).  Outstanding ones are tracked so an early
    // exit can let them land before the shared memory is released.
    uint32_t out_x = 0, out_b = 0;  // bit per group
    uint32_t out_v = 0;  // bit per value tile
    // Ready flags (fused grid): head h's flags are consecutive words, read four
    // at a time with one acquire load, so one global round trip usually covers
    // several chunks; acq_hi is the last chunk known to be ready.
    long long acq_hi = -1;
    auto acquire = [&](long long gg) {
        if (!ready || gg <= acq_hi) return true;
        const unsigned* fh = ready + (size_t)h * ready_pitch;
        const long long g4 = gg & ~3LL;
        for (uint32_t it = 0; it < acquire_iters; ++it) {
            const uint4 f = tc::flags4_acquire(fh + g4);
            // the four flags as a bit mask (a runtime-indexed array would live
            // in local memory)
            const uint32_t fm = (f.x ? 1u : 0u) | (f.y ? 2u : 0u) | (f.z ? 4u : 0u) | (f.w ? 8u : 0u);
            int k = (int)(gg - g4);
            if ((fm >> k) & 1u) {
                while (k + 1 < 4 && ((fm >> (k + 1)) & 1u)) ++k;
                tc::flags_proxy_fence();
                acq_hi = g4 + k;
                return true;
            }
            __nanosleep(64);
        }
        return false;
    };
    // chunk gg's operands into group b, after its flag.  Two-kernel path
    // (every blob written before the scan starts, most of them gone from L2):
    // with next_too, chunk gg + 1's blob is also pulled into L2, so that its
    // copies, a chunk later, need not wait on DRAM (in the fused grid the
    // chains read blobs soon after prepare wrote them, and this measured slower)
    auto load_ops = [&](long long gg, int b, bool next_too) {
        if (!acquire(gg)) {
            atomicOr(&g_tc_status, STATUS_TIMEOUT);
            *abort_flag = 1;
        }
        const unsigned char* blob = ws + blob_offset(n_seqs, gg, h, heads);
        tc::mbar_arrive_expect_tx(bar_x + b, OpXh::bytes(128));
        tc::bulk_load(sm + opx_off(b), blob + BLOB_OPX, OpXh::bytes(128), bar_x + b);
        tc::mbar_arrive_expect_tx(bar_b + b, ScanT::BGRP);
        tc::bulk_load(sm + tp_off(b), blob + BLOB_TP, ScanT::BGRP, bar_b + b);
        out_x |= 1u << b;
        out_b |= 1u << b;
        if constexpr (TWO_KERNEL) {
            if (next_too) tc::bulk_prefetch_l2(blob + BLOB_BYTES * (size_t)heads, BLOB_BYTES);
        }
    };
    // Value tiles are double-buffered by chunk parity and requested two chunks
    // ahead, as soon as the X phase has consumed the buffer.
    auto load_v = [&](int cc0, int vb) {
        tc::mbar_arrive_expect_tx(bar_v + vb, 64 * D * 2);
        tc::tma_load_2d(sm + rawv_off(vb), &vmap, bar_v + vb, h * D, cc0);
        out_v |= 1u << vb;
    };
    if (copier && start < end) {
        load_ops(g0, 0, start + C < end);
        load_v(start, 0);
        if (start + C < end) load_v(start + C, 1);
    }

    // NORM: the staged O tile of a chunk is normalised in two halves of 32
    // token rows, each by warps 8..15: thread tt = tid - 256 takes row
    // 32 half + tt / 8, channels 4 cb + 32 k (k < 4, cb = tt % 8: a quarter
    // warp reads a row's 128 consecutive bytes), with the o_norm weight of
    // those channels kept in registers.
    uint32_t ph_g = 0, out_g = 0;  // gate buffers: phase, load in flight (bit per buffer)
    float wn[16];
    if (NORM && tid >= 256) {
        const int cb = (tid - 256) & 7;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint2 wv = __ldg(reinterpret_cast<const uint2*>(na->w + 4 * cb + 32 * k));
            wn[4 * k] = __uint_as_float(wv.x << 16);
            wn[4 * k + 1] = __uint_as_float(wv.x & 0xffff0000u);
            wn[4 * k + 2] = __uint_as_float(wv.y << 16);
            wn[4 * k + 3] = __uint_as_float(wv.y & 0xffff0000u);
        }
    }
    auto gate_off = [](int b) { return b ? ScanT::GATE1 : ScanT::GATE0; };
    // the gate tile of the chunk at token row cc0 into buffer b (copier), once
    // the buffer's last output tile has left
    auto load_gate = [&](int cc0, int b) {
        tc::bulk_wait_read_all();
        tc::mbar_arrive_expect_tx(bar_gt + b, 64 * D * 2);
        tc::tma_load_2d(sm + gate_off(b), &na->gmap, bar_gt + b, h * D, cc0);
        out_g |= 1u << b;
    };
    // Half hf of the sigmoid-gated RMSNorm of the staged O tile (OST, FP32
    // [64][128]) with the gate tile in buffer b,
    //     out[j] = o[j] / sqrt(mean_j o[j]^2 + eps) * w[j] * sigmoid(gate[j]),
    // in FP32 (the sigmoid by the hardware 2^x and reciprocal), rounded once
    // to BF16: in place over the gate tile (to_tile: each thread overwrites the
    // gate values it read), or to `out` for the chunk's first `rows` rows at
    // token row oc0.  Called by every thread (all track the gate's phase).
    auto norm_half = [&](int hf, int b, bool to_tile, int rows, int oc0) {
        if (tid >= 256) {
            if (hf == 0) {
                if (tid == 256 && !tc::mbar_wait(bar_gt + b, (ph_g >> b) & 1u)) {
                    atomicOr(&g_tc_status, STATUS_TIMEOUT);
                    *abort_flag = 1;
                }
                asm volatile("bar.sync 2, 256;" ::: "memory");
            }
            const int tt = tid - 256, cb = tt & 7, r = 32 * hf + (tt >> 3);
            uint16_t* GT = reinterpret_cast<uint16_t*>(sm + gate_off(b));
            float y[16];
            uint2 gv[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float4 f = *reinterpret_cast<const float4*>(OST + r * D + 4 * cb + 32 * k);
                y[4 * k] = f.x;
                y[4 * k + 1] = f.y;
                y[4 * k + 2] = f.z;
                y[4 * k + 3] = f.w;
                gv[k] = *reinterpret_cast<const uint2*>(GT + r * D + 4 * cb + 32 * k);
            }
            float s4[4] = {0.f, 0.f, 0.f, 0.f};  // four independent chains
#pragma unroll
            for (int e = 0; e < 16; ++e) s4[e & 3] = __fmaf_rn(y[e], y[e], s4[e & 3]);
            float ss = (s4[0] + s4[1]) + (s4[2] + s4[3]);
            ss += __shfl_xor_sync(0xffffffffu, ss, 1);
            ss += __shfl_xor_sync(0xffffffffu, ss, 2);
            ss += __shfl_xor_sync(0xffffffffu, ss, 4);
            const float rr = rsqrtf(ss * (1.0f / D) + na->eps);
            uint2 ob[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float gg[4] = {__uint_as_float(gv[k].x << 16),
                                     __uint_as_float(gv[k].x & 0xffff0000u),
                                     __uint_as_float(gv[k].y << 16),
                                     __uint_as_float(gv[k].y & 0xffff0000u)};
                float z[4];
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    z[e] = y[4 * k + e] * rr * wn[4 * k + e] * sigmoid_hw(gg[e]);
                ob[k] = make_uint2(tc::pack_bf16x2(z[0], z[1]), tc::pack_bf16x2(z[2], z[3]));
            }
            if (to_tile) {
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    *reinterpret_cast<uint2*>(GT + r * D + 4 * cb + 32 * k) = ob[k];
                tc::fence_async_smem();
            } else if (r < rows) {
                uint16_t* orow = na->out + (size_t)(oc0 + r) * na->out_pitch + h * D;
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    *reinterpret_cast<uint2*>(orow + 4 * cb + 32 * k) = ob[k];
            }
        }
        if (hf == 1) {
            ph_g ^= 1u << b;
            if (copier) out_g &= ~(1u << b);
        }
    };
    bool n_active = false;  // this chunk normalises the staged tile of chunk n_c0 (NORM)
    int n_c0 = -1, st_b = 0, o_b = 0;  // gate buffers of the staged and the last chunk

    int o_c0 = -1, o_L = 0;  // the chunk whose O is still in TMEM (region o_reg)
    uint32_t o_reg = 0;
    bool o_staged = false;  // a staged O (chunk st_c0) waits for its store
    int st_c0 = -1;
    long long g = g0;
    int xb = 0;
    for (int c0 = start; c0 < end; c0 += C, ++g, xb ^= 1) {
        const int L = min(C, end - c0);
        const bool more = c0 + C < end;
        const uint32_t r_d1 = xb ? ScanT::R1 : ScanT::R0;  // Ktil S, then Qtil S / O at +64
        const uint32_t r_a = xb ? ScanT::R0 : ScanT::R1;   // X^T / U^T (A), then T X at +64
        const uint32_t s_tp = tc::smem_u32(sm + tp_off(xb));
        const uint32_t s_kh = s_tp + (BLOB_KH - BLOB_TP);
        const float* DEC = reinterpret_cast<const float*>(sm + tp_off(xb) + (BLOB_DEC - BLOB_TP));
        tc::tc_fence_before();
        if (__syncthreads_or(*abort_flag)) break;  // every thread takes the same exit
        if (NORM) {
            // chunk g - 2's O, staged during the last chunk: its first half now,
            // the second while this chunk's second product runs
            n_active = o_staged;
            if (n_active) {
                n_c0 = st_c0;
                norm_half(0, st_b, true, C, n_c0);
            }
            // the gate of chunk g - 1, whose O is staged in this chunk
            if (copier && c0 > start) load_gate(c0 - C, xb ^ 1);
        } else if (copier && o_staged) {  // chunk g - 2's O, staged during the last chunk
            tc::tma_store_2d(&omap, OST, h * D, st_c0);
            tc::bulk_commit();
        }
        o_staged = false;
        wait_bar(bar_x + xb, (ph_x >> xb) & 1u);
        ph_x ^= 1u << xb;
        if (copier) out_x &= ~(1u << xb);
        wait_bar(bar_v + xb, (ph_v >> xb) & 1u);
        ph_v ^= 1u << xb;
        if (copier) out_v &= ~(1u << xb);
        const uint16_t* RAWV = reinterpret_cast<const uint16_t*>(sm + rawv_off(xb));

        // ---------------------------------------------------------- S^T [Ktil; Qtil]^T
        // (one N = 128 product: Ktil S into r_d1, Qtil S into r_d1 + 64)
        if (tid == 0) {
            tc::tc_fence_after();
            const uint64_t bd = OpXh::desc(tc::smem_u32(sm + opx_off(xb)), 0);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
                tc::mma_f16_ta(tmem + r_d1, tmem + ScanT::T_S + 8 * ks, bd + ks * OpXh::KSTEP,
                               tc::idesc_f16(128, 128), ks > 0);
            tc::mma_commit(bar_mma);
        }
        // the next chunk's operands into the other groups, whose last products
        // completed in the previous chunk
        if (copier && more) load_ops(g + 1, xb ^ 1, c0 + 2 * C < end);
        float vr[16];  // V[16 cg + i][j], read while the product runs
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const uint16_t e = RAWV[(16 * cg + i) * D + j];
            vr[i] = F16 ? h2f(e) : bf(e);
        }
        wait_bar(bar_mma, ph_mma);
        ph_mma ^= 1;
        tc::tc_fence_after();
        {   // X^T[j][r] = V[r][j] - (Ktil S)[r][j], r = 16 cg + i
            float v[16];
            tc::tmem_ld16(my + r_d1 + 16 * cg, v);
            tc::tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int r = 16 * cg + i;
                v[i] = (r < L) ? vr[i] - v[i] : 0.f;
            }
            uint32_t xv[8];  // X^T: token 16 cg + i in column 8 cg + i / 2
#pragma unroll
            for (int m = 0; m < 8; ++m) xv[m] = tc::pack_f16x2(v[2 * m], v[2 * m + 1]);
            tc::tmem_st8u(my + r_a + 8 * cg, xv);
            tc::tmem_st_wait();
        }
        tc::tc_fence_before();
        __syncthreads();
        if (copier && c0 + 2 * C < end) load_v(c0 + 2 * C, xb);  // this tile is consumed
        wait_bar(bar_b + xb, (ph_b >> xb) & 1u);
        ph_b ^= 1u << xb;
        if (copier) out_b &= ~(1u << xb);

        // ---------------------------------------------------------- U^T = X^T T^T
        if (tid == 0) {
            tc::tc_fence_after();
            const uint64_t bd = OpTPh::desc(s_tp, 0);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                tc::mma_f16_ta(tmem + ScanT::T_TX, tmem + r_a + 8 * ks, bd + ks * OpTPh::KSTEP,
                               tc::idesc_f16(128, 64), ks > 0);
            tc::mma_commit(bar_mma);
        }
        {   // while it runs: S^T <- S^T diag(dec) in TMEM, which the chunk's last
            // product then accumulates into
            const float4* dec4 = reinterpret_cast<const float4*>(DEC + 32 * cg);
            float sv[32];
            tc::tmem_ld32(my + ScanT::T_SA + 32 * cg, sv);
            tc::tmem_ld_wait();
            uint32_t su[32];
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4) {
                const float4 d4 = dec4[q4];
                su[4 * q4] = __float_as_uint(__fmul_rn(sv[4 * q4], d4.x));
                su[4 * q4 + 1] = __float_as_uint(__fmul_rn(sv[4 * q4 + 1], d4.y));
                su[4 * q4 + 2] = __float_as_uint(__fmul_rn(sv[4 * q4 + 2], d4.z));
                su[4 * q4 + 3] = __float_as_uint(__fmul_rn(sv[4 * q4 + 3], d4.w));
            }
            tc::tmem_st32u(my + ScanT::T_SA + 32 * cg, su);
        }
        if (NORM && n_active) norm_half(1, st_b, true, C, n_c0);
        wait_bar(bar_mma, ph_mma);
        ph_mma ^= 1;
        tc::tc_fence_after();
        {
            float v[16];
            tc::tmem_ld16(my + ScanT::T_TX + 16 * cg, v);
            tc::tmem_ld_wait();
            uint32_t uv[8];
#pragma unroll
            for (int m = 0; m < 8; ++m) uv[m] = tc::pack_f16x2(v[2 * m], v[2 * m + 1]);
            tc::tmem_st8u(my + r_a + 8 * cg, uv);
            tc::tmem_st_wait();
        }
        if (copier) tc::bulk_wait_read_all();  // the staging tile's last store has read it
        tc::tc_fence_before();
        __syncthreads();
        if (NORM && copier && n_active) {  // chunk n_c0's normalised tile, over its gate
            tc::tma_store_2d(&na->nmap, sm + gate_off(st_b), h * D, n_c0);
            tc::bulk_commit();
        }
        n_active = false;

        // ---------------------------------------------------------- U^T Khat; O^T += U^T P^T
        if (tid == 0) {
            tc::tc_fence_after();
            const uint64_t bk = OpKHh::desc(s_kh, 0), bp = OpTPh::desc(s_tp + 8 * 128, 0);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                tc::mma_f16_ta(tmem + ScanT::T_SA, tmem + r_a + 8 * ks, bk + ks * OpKHh::KSTEP,
                               tc::idesc_f16(128, 128), true);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)  // P = rows 64..127 of [T; P]
                tc::mma_f16_ta(tmem + r_d1 + 64, tmem + r_a + 8 * ks, bp + ks * OpTPh::KSTEP,
                               tc::idesc_f16(128, 64), true);
            tc::mma_commit(bar_mma);
        }
        // chunk g - 1's O (the last 64 columns of r_a) into the staging tile
        // while this product runs, or straight out if partial
        if (o_c0 >= 0 && warp != 0) {
            float ov[16];
            tc::tmem_ld16(my + o_reg + 16 * cg, ov);
            float ow[8];  // warps 4 and 8 also take rows 0..7 and 8..15 of warp 0
            const bool extra = (qd == 0) && (cg == 1 || cg == 2);
            const int wr = (cg == 1) ? 0 : 8;
            if (extra) tc::tmem_ld8(my + o_reg + wr, ow);
            tc::tmem_ld_wait();
            if (NORM || o_L == C) {  // (inside the loop every chunk but the last is whole)
#pragma unroll
                for (int i = 0; i < 16; ++i) OST[(16 * cg + i) * D + j] = ov[i];
                if (extra) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) OST[(wr + i) * D + j] = ow[i];
                }
                tc::fence_async_smem();
            } else {
                float* orow = o + ((size_t)o_c0 * heads + h) * D + j;
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int r = 16 * cg + i;
                    if (r < o_L) orow[(size_t)r * heads * D] = ov[i];
                }
                if (extra) {
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        if (wr + i < o_L) orow[(size_t)(wr + i) * heads * D] = ow[i];
                }
            }
        }
        if (o_c0 >= 0 && (NORM || o_L == C)) {
            o_staged = true;
            st_c0 = o_c0;
            st_b = o_b;
        }
        wait_bar(bar_mma, ph_mma);
        ph_mma ^= 1;
        tc::tc_fence_after();
        {   // S^T (FP32, updated in TMEM) into the next chunk's FP16 A operand
            float sv[32];
            tc::tmem_ld32(my + ScanT::T_SA + 32 * cg, sv);
            tc::tmem_ld_wait();
            uint32_t sh[16];
#pragma unroll
            for (int m = 0; m < 16; ++m) sh[m] = tc::pack_f16x2(sv[2 * m], sv[2 * m + 1]);
            tc::tmem_st16u(my + ScanT::T_S + 16 * cg, sh);
            tc::tmem_st_wait();
        }
        o_c0 = c0;
        o_b = xb;
        o_L = L;
        o_reg = r_d1 + 64;
    }
    // every thread leaves the loop through the same iteration; agree on the flag
    const bool aborted = __syncthreads_or(*abort_flag);
    if (NORM) {
        if (!aborted) {
            // the staged O of the chunk before the last, then the last chunk's:
            // normalised and written by plain stores
            if (o_staged) {
                norm_half(0, st_b, false, C, st_c0);
                norm_half(1, st_b, false, C, st_c0);
            }
            __syncthreads();  // OST is free
            if (o_c0 >= 0) {
                float ov[16];
                tc::tmem_ld16(my + o_reg + 16 * cg, ov);
                tc::tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 16; ++i) OST[(16 * cg + i) * D + j] = ov[i];
                if (copier) load_gate(o_c0, o_b);
            }
            __syncthreads();
            if (o_c0 >= 0) {
                norm_half(0, o_b, false, o_L, o_c0);
                norm_half(1, o_b, false, o_L, o_c0);
            }
        }
    } else {
        if (copier && o_staged && !aborted) {  // the staged O of the chunk before the last
            tc::tma_store_2d(&omap, OST, h * D, st_c0);
            tc::bulk_commit();
        }
        if (o_c0 >= 0 && !aborted) {  // the last chunk's O, by plain stores
            float ov[16];
            tc::tmem_ld16(my + o_reg + 16 * cg, ov);
            tc::tmem_ld_wait();
            float* orow = o + ((size_t)o_c0 * heads + h) * D + j;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int r = 16 * cg + i;
                if (r < o_L) orow[(size_t)r * heads * D] = ov[i];
            }
        }
    }
    if (copier) {  // copies still in flight land before the exit (bounded waits)
        tc::bulk_wait_all();
        for (int b2 = 0; b2 < 2; ++b2)
            if ((out_g >> b2) & 1u) tc::mbar_wait(bar_gt + b2, (ph_g >> b2) & 1u, 1u << 20);
        for (int b2 = 0; b2 < 2; ++b2) {
            if ((out_x >> b2) & 1u) tc::mbar_wait(bar_x + b2, (ph_x >> b2) & 1u, 1u << 20);
            if ((out_b >> b2) & 1u) tc::mbar_wait(bar_b + b2, (ph_b >> b2) & 1u, 1u << 20);
        }
        for (int b2 = 0; b2 < 2; ++b2)
            if ((out_v >> b2) & 1u) tc::mbar_wait(bar_v + b2, (ph_v >> b2) & 1u, 1u << 20);
    }
    if (!aborted) {
        float sv[32];
        tc::tmem_ld32(my + ScanT::T_SA + 32 * cg, sv);
        tc::tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) Sg[(size_t)i * D] = sv[i];
    }
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, ScanT::TMEM_COLS);
    }
}

// prepare and the transposed scan in one cooperative grid: CTAs [0, chains)
// run the (sequence, head) chains, the others walk the prepare items in
// chunk-major order and release each item's ready flag, so a chain consumes
// chunk g as soon as its operands are out, with the rest of the sequence
// still being prepared on the other SMs.  All CTAs are resident at once
// (cooperative launch), so every wait on a flag ends.
static_assert(ScanT::NT == NTP, "the two roles share the block size");
static_assert(ScanT::TOTAL <= PS_TOTAL, "the two roles share the shared-memory size");
template <bool GATED, bool NORM, bool F16>
__global__ void __launch_bounds__(NTP, 1)
prefill_fused_kernel(const __grid_constant__ PrepMaps maps, const __grid_constant__ CUtensorMap vmap,
                     const __grid_constant__ CUtensorMap omap, const __grid_constant__ NormArgs na,
                     const void* __restrict__ beta, float* __restrict__ state,
                     float* __restrict__ o, int t, int t_pad, int heads,
                     const int* __restrict__ cu, int n_seqs, unsigned char* __restrict__ ws,
                     unsigned* __restrict__ ready, long long ready_pitch, uint32_t fault) {
    // fault == FAULT_READY_WAIT (a test of the bounded flag wait, set only
    // through KDA_FAULT_INJECT): prepare releases no flag and each chain's
    // wait gives up after a few milliseconds, so every chain records
    // STATUS_TIMEOUT and returns without writing o or the state.
    const bool inject = fault == FAULT_READY_WAIT;
    const int chains = n_seqs * heads;
    if ((int)blockIdx.x < chains)
        scan_t_role<NORM, F16, false>(vmap, omap, state, o, t, t_pad, heads, cu, n_seqs, ws,
                               (int)blockIdx.x % heads, (int)blockIdx.x / heads, ready,
                               ready_pitch, &na, inject ? 1u << 12 : 1u << 22);
    else
        prepare_role<GATED, F16, false>(maps, beta, t, t_pad, heads, cu, n_seqs, ws,
                                 (long long)blockIdx.x - chains, (long long)gridDim.x - chains,
                                 ready, ready_pitch, !inject);
}

// The chains of the two-kernel path: one CTA per (sequence, head), after
// prepare_kernel has written every chunk's operands.
template <bool NORM, bool F16>
__global__ void __launch_bounds__(NTP, 1)
scan_t_kernel(const __grid_constant__ CUtensorMap vmap, const __grid_constant__ CUtensorMap omap,
              const __grid_constant__ NormArgs na, float* __restrict__ state, float* __restrict__ o,
              int t, int t_pad, int heads, const int* __restrict__ cu, int n_seqs,
              const unsigned char* __restrict__ ws, const int* __restrict__ order) {
    pdl_wait();  // the prepared operands (and the callers' state) are complete
    pdl_release();
    // a packed batch's chains in chain_order_kernel's order, longest first
    const int n = order ? __ldg(order + (int)blockIdx.x / heads) : (int)blockIdx.x / heads;
    scan_t_role<NORM, F16, true>(vmap, omap, state, o, t, t_pad, heads, cu, n_seqs, ws,
                                 (int)blockIdx.x % heads, n, nullptr, 0, &na);
}

// BF16 (FP16 with f16) [rows][cols] with a row pitch of `pitch_elems`; boxes
// of `box_cols` channels x 64 tokens with the given shared-memory swizzle.
bool make_map(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint64_t pitch_elems,
              uint32_t box_cols, CUtensorMapSwizzle swizzle, bool f16 = false) {
    return tma_map_bf16(m, base, cols, rows, pitch_elems, box_cols, (uint32_t)C, swizzle,
                        f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16);
}

// FP32 inputs: q, k and v rounded to FP16 (round to nearest even; 11
// significant bits, the precision of the TF32 and FP16 operands they become)
// into the workspace, [rows][hd] each and contiguous, for the kernels' 16-bit
// tiles.  A warp per row; lane l converts channels 8 (l + 32 m) .. + 7.
// Input rows are 16-byte aligned (checked by the callers).
constexpr int CVT_THREADS = 256;
__global__ void __launch_bounds__(CVT_THREADS)
f32_to_f16_kernel(const float* __restrict__ q, const float* __restrict__ k,
                  const float* __restrict__ v, long long stride, uint16_t* __restrict__ out,
                  int rows, int hd) {
    pdl_wait();
    pdl_release();
    const float* src_t = blockIdx.y == 0 ? q : (blockIdx.y == 1 ? k : v);
    uint16_t* dst_t = out + (size_t)blockIdx.y * rows * hd;
    const int warps = CVT_THREADS / 32, lane = threadIdx.x & 31;
    for (int row = blockIdx.x * warps + (int)(threadIdx.x >> 5); row < rows;
         row += gridDim.x * warps) {
        const float4* src = reinterpret_cast<const float4*>(src_t + (size_t)row * stride);
        uint4* dst = reinterpret_cast<uint4*>(dst_t + (size_t)row * hd);
#pragma unroll 4
        for (int c8 = lane; c8 < hd / 8; c8 += 32) {
            const float4 a = __ldcs(src + 2 * c8), b = __ldcs(src + 2 * c8 + 1);
            dst[c8] = make_uint4(tc::pack_f16x2(a.x, a.y), tc::pack_f16x2(a.z, a.w),
                                 tc::pack_f16x2(b.x, b.y), tc::pack_f16x2(b.z, b.w));
        }
    }
}

// Ready flags of the fused grid: one 32-bit word per (chunk, head) blob,
// after the blobs, head-major with each head's run of chunks padded to a
// multiple of 4 words (16-byte groups), the whole padded to 256 bytes.
size_t ready_offset(long long chunks, int n_seqs, int heads) {
    return header_bytes(n_seqs) + (size_t)chunks * heads * BLOB_BYTES;
}
long long ready_pitch(long long chunks) { return (chunks + 3) & ~3LL; }
size_t ready_words(long long chunks, int heads) {
    return (((size_t)ready_pitch(chunks) * heads * 4 + 255) & ~(size_t)255) / 4;
}

}  // namespace

// The chains' launch order (n_seqs int32, padded to 256 B), after the flags.
size_t order_offset(long long chunks, int n_seqs, int heads) {
    return ready_offset(chunks, n_seqs, heads) + ready_words(chunks, heads) * 4;
}

size_t prefill_tc_workspace_bytes(long long rows, int n_seqs, int heads, bool f32_in) {
    const long long chunks = (rows + C - 1) / C + n_seqs;
    const size_t base =
        order_offset(chunks, n_seqs, heads) + (((size_t)n_seqs * 4 + 255) & ~(size_t)255);
    if (!f32_in) return base;
    // the FP16 copies of q, k and v, 256-byte aligned after the rest
    return ((base + 255) & ~(size_t)255) + 3 * (size_t)rows * heads * D * 2;
}

// Per-SM cost figures measured on GB300 (T = 8192, 32 heads) that choose
// between the fused grid and the two kernels: a prepare item, and a chunk of
// the transposed scan's chain.
constexpr double kPrepItemUs = 8.3, kScanTChunkUs = 2.3;

// Launches the tensor-core prefill (BF16 inputs, or FP32 inputs converted to
// FP16 tiles first; chunk 64); arguments, including the workspace size, are
// validated by kda_prefill.
kda_status launch_prefill_tc(float* state, const void* q, const void* k, const void* v,
                             const void* g, const void* beta, float* o, int t, int t_pad,
                             int heads, long long stride, const int* cu, int n_seqs,
                             void* workspace, cudaStream_t s, const PrefillGate* gate,
                             const PrefillNorm* norm, bool f32_in) {
    const uint64_t rows = cu ? (uint64_t)t : (uint64_t)t_pad * n_seqs;
    const int sms = sm_count();
    if (sms <= 0) {
        set_error("kda_prefill: cannot query the multiprocessor count");
        return KDA_ERR_CUDA;
    }
    // Every (sequence, head) chain runs on one SM for its whole length.  The
    // fused grid (one SM per chain, the other SMs preparing just ahead of the
    // chains) when, per chunk of a chain, max(chains x item / (sms - chains),
    // chain) beats the two kernels' chains x item / sms + chain (prepare on
    // every SM, then the chains in one wave).
    const long long chains = (long long)n_seqs * heads;
    const char* impl = getenv("KDA_PREFILL_IMPL");
    const bool fused_allowed = !(impl && strcmp(impl, "unfused") == 0);
    bool fused = false;
    if (fused_allowed && chains < sms) {
        const double per_chunk_fused =
            std::max((double)chains * kPrepItemUs / (double)(sms - chains), kScanTChunkUs);
        const double per_chunk_two = (double)chains * kPrepItemUs / sms + kScanTChunkUs;
        fused = per_chunk_fused < per_chunk_two;
    }
    if (f32_in && (gate || norm)) {
        set_error("kda_prefill: FP32 inputs take neither the fused gate nor the fused norm");
        return KDA_ERR_UNSUPPORTED;
    }
    PrepMaps maps;
    CUtensorMap vmap, omap;
    NormArgs na;
    memset(&na, 0, sizeof(na));
    const uint64_t hd = (uint64_t)heads * D;
    maps.dt_bias = gate ? gate->dt_bias : nullptr;
    maps.a_log = gate ? gate->a_log : nullptr;
    maps.lb = gate ? gate->lb : 0.f;
    maps.b_stride = gate ? gate->b_stride : heads;
    const uint64_t g_pitch = gate ? (uint64_t)gate->g_stride : hd;
    // FP32 inputs: the kernels read FP16 copies of q, k and v (written below,
    // after the other host steps) and the FP32 g in place
    const float* q32 = static_cast<const float*>(q);
    const float* k32 = static_cast<const float*>(k);
    const float* v32 = static_cast<const float*>(v);
    const long long stride32 = stride;
    uint16_t* f16 = nullptr;
    if (f32_in) {
        f16 = reinterpret_cast<uint16_t*>(
            static_cast<unsigned char*>(workspace) +
            ((prefill_tc_workspace_bytes((long long)rows, n_seqs, heads) + 255) & ~(size_t)255));
        q = f16;
        k = f16 + rows * hd;
        v = f16 + 2 * rows * hd;
        stride = (long long)hd;
    }
    const bool gmap_ok =
        f32_in ? tma_map_f32(&maps.g, g, hd, rows, hd, D, (uint32_t)C)
               : make_map(&maps.g, g, hd, rows, g_pitch, 64, CU_TENSOR_MAP_SWIZZLE_128B);
    if (!make_map(&maps.q, q, hd, rows, (uint64_t)stride, 64, CU_TENSOR_MAP_SWIZZLE_128B, f32_in) ||
        !make_map(&maps.k, k, hd, rows, (uint64_t)stride, 64, CU_TENSOR_MAP_SWIZZLE_128B, f32_in) ||
        !gmap_ok ||
        !make_map(&vmap, v, hd, rows, (uint64_t)stride, D, CU_TENSOR_MAP_SWIZZLE_NONE, f32_in) ||
        (norm ? !make_map(&na.gmap, norm->gate, hd, rows, (uint64_t)norm->gate_stride, D,
                          CU_TENSOR_MAP_SWIZZLE_NONE) ||
                    !make_map(&na.nmap, norm->out, hd, rows, (uint64_t)norm->out_stride, D,
                              CU_TENSOR_MAP_SWIZZLE_NONE)
              : !tma_map_f32(&omap, o, hd, rows, hd, D, (uint32_t)C))) {
        set_error("kda_prefill: cannot encode TMA tensor maps");
        return KDA_ERR_CUDA;
    }
    if (norm) {
        na.w = norm->w;
        na.out = norm->out;
        na.out_pitch = norm->out_stride;
        na.eps = norm->eps;
        memset(&omap, 0, sizeof(omap));
    }
    auto* prep_k = f32_in ? prepare_kernel<false, true>
                          : (gate ? prepare_kernel<true, false> : prepare_kernel<false, false>);
    auto* fused_k = f32_in ? prefill_fused_kernel<false, false, true>
                    : norm ? prefill_fused_kernel<false, true, false>
                           : (gate ? prefill_fused_kernel<true, false, false>
                                   : prefill_fused_kernel<false, false, false>);
    auto* scan_k = f32_in ? scan_t_kernel<false, true>
                          : (norm ? scan_t_kernel<true, false> : scan_t_kernel<false, false>);
    cudaError_t e = cudaFuncSetAttribute(prep_k,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)PS_TOTAL);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(scan_k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)ScanT::TOTAL);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(fused_k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)PS_TOTAL);
    if (e != cudaSuccess) {
        set_error("kda_prefill: cannot reserve shared memory: %s", cudaGetErrorString(e));
        return KDA_ERR_CUDA;
    }
    unsigned char* ws = static_cast<unsigned char*>(workspace);
    const long long chunk_bound = ((long long)rows + C - 1) / C + n_seqs;
    unsigned* ready = reinterpret_cast<unsigned*>(ws + ready_offset(chunk_bound, n_seqs, heads));
    const long long n_ready = fused ? (long long)ready_words(chunk_bound, heads) : 0;
    if (f32_in) {
        const long long blocks = std::min<long long>(((long long)rows + 7) / 8, 16LL * sms);
        launch_pdl(f32_to_f16_kernel, dim3((unsigned)blocks, 3), dim3(CVT_THREADS), 0, s, q32, k32,
                   v32, stride32, f16, (int)rows, (int)hd);
        const kda_status cs = launch_result("kda_prefill (FP16 copies)");
        if (cs != KDA_OK) return cs;
    }
    launch_pdl(chunk_map_kernel, dim3(1), dim3(MAP_THREADS), 0, s, cu, n_seqs, cu ? 0 : t,
               reinterpret_cast<int*>(ws), ready, n_ready);
    kda_status st = launch_result("kda_prefill (chunk map)");
    if (st != KDA_OK) return st;
    if (fused) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)sms);
        cfg.blockDim = dim3(NTP);
        cfg.dynamicSmemBytes = PS_TOTAL;
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, fused_k, maps, vmap, omap, na, beta,
                               state, o, t, t_pad, heads, cu, n_seqs, ws, ready,
                               ready_pitch(chunk_bound),
                               fault_injected("ready_wait") ? (uint32_t)FAULT_READY_WAIT : 0u);
        if (e == cudaSuccess) return launch_result("kda_prefill (fused)");
        // the grid could not be made resident (e.g. SMs held by other work):
        // run the two kernels instead
        (void)cudaGetLastError();
    }
    // A packed batch's chains start longest first (see chain_order_kernel).
    int* order = nullptr;
    if (cu && n_seqs > 1 && n_seqs <= ORDER_MAX) {
        order = reinterpret_cast<int*>(ws + order_offset(chunk_bound, n_seqs, heads));
        launch_pdl(chain_order_kernel, dim3(1), dim3(MAP_THREADS), (size_t)n_seqs * 4, s, cu,
                   n_seqs, order);
        st = launch_result("kda_prefill (chain order)");
        if (st != KDA_OK) return st;
    }
    // Persistent prepare: one CTA per SM (shared memory allows no more),
    // never more CTAs than (chunk, head) items.
    const long long items = (((long long)rows + C - 1) / C + n_seqs) * heads;
    const unsigned grid = (unsigned)(items < sms ? items : sms);
    launch_pdl(prep_k, dim3(grid), dim3(NTP), PS_TOTAL, s, maps, beta, t,
               t_pad, heads, cu, n_seqs, ws);
    st = launch_result("kda_prefill (prepare)");
    if (st != KDA_OK) return st;
    launch_pdl(scan_k, dim3((unsigned)chains), dim3(NTP), ScanT::TOTAL, s, vmap, omap, na,
               state, o, t, t_pad, heads, cu, n_seqs, (const unsigned char*)ws,
               (const int*)order);
    return launch_result("kda_prefill (scan)");
}

cudaError_t read_and_clear_status_prefill_tc(unsigned* out) {
    unsigned zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(out, g_tc_status, sizeof(unsigned));
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_tc_status, &zero, sizeof(unsigned));
    return e;
}

}  // namespace kda
