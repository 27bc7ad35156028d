// Tensor-core chunked prefill of the KDA core for BF16 inputs and chunk 64
// (Glm5NextKdaKernels::chunk_prepare + chunk_scan fused in one kernel).
//
// One CTA of 256 threads per (sequence, head, 32-column value slice); it walks
// the sequence's chunks in order, keeping its 128 x 32 slice of the FP32
// state in registers (and a TF32 copy in shared memory as an MMA operand).
//
// Per chunk of L <= 64 tokens (rows r, s; key channels i; value columns j):
//   Gamma_r  = sum_{u<=r} g_u                                  (FP32, SIMT)
//   A_rs     = beta_s sum_i k_ri k_si e^(Gamma_ri-Gamma_si), s < r
//   P_rs     = beta_s sum_i qh_ri k_si e^(Gamma_ri-Gamma_si), s <= r
//   T        = (I + A)^-1                    (blocked forward substitution)
//   X        = V - Ktil S,   Ktil = e^Gamma (.) k,  Qtil = e^Gamma (.) qh
//   U        = T X,   O = Qtil S + P U
//   S       <- diag(e^Gamma_{L-1}) S + Khat^T U,
//              Khat_s = beta_s e^(Gamma_{L-1}-Gamma_s) (.) k_s
// A and P are formed on the tensor cores one 16-column block b at a time:
// with m_b = 16b + 8, e^(Gamma_r-Gamma_s) = e^(Gamma_r-Gamma_mb) e^(Gamma_mb-Gamma_s),
// and for every (r >= 16b, s in block b) both factors stay within
// e^(+-8 |g|_max), so FP32 neither overflows nor loses the product for
// g >= -10; rows above the block (where the first factor would overflow) are
// never formed into results.
//
// Tensor-core products (tcgen05.mma kind::tf32, FP32 accumulate in TMEM):
//   [X_b; QX_b] (128x128) . Y_b^T     -> A, P column block b   (x4)
//   [Ktil; Qtil] (128x128) . S        -> Ktil S, Qtil S
//   [T; P] (128x64) . X               -> U = T X (rows 0..63)
//   Khat^T (128x64) . U               -> state increment
//   [T; P] (128x64) . U               -> P U (rows 64..127)
// Raw q, k, g and the value slice arrive by TMA (cp.async.bulk.tensor).
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "kda_common.h"
#include "sm103_tc.h"

namespace kda {
namespace {

__device__ unsigned g_tc_status = 0;

constexpr int C = 64;
constexpr int DV = 32;
constexpr int NT = 256;
constexpr int KP = 129;  // pitch (floats) of FP32 [64][128] staging arrays
constexpr int AP = 65;   // pitch (floats) of FP32 [64][64] arrays

// K-major operand of R rows in the "K-outer" core-matrix layout: the core
// matrices of one K group of 4 columns are stacked over all rows (128 B per 8
// rows); successive K groups are LBO = 16 R + PAD bytes apart.  PAD = 16
// spreads operands that are written one K index per thread over all banks.
template <int R, int PAD>
struct Op {
    static constexpr uint32_t LBO = R * 16 + PAD;
    static __device__ __forceinline__ uint32_t off(int r, int k) {
        return (uint32_t)((k >> 2) * LBO + (r >> 3) * 128 + (r & 7) * 16 + (k & 3) * 4);
    }
    static __device__ __forceinline__ uint64_t desc(uint32_t base, int ks) {
        return tc::make_desc(base + (uint32_t)ks * 2u * LBO, LBO, 128u);
    }
    static constexpr uint32_t bytes(int K) { return (uint32_t)(K / 4) * LBO; }
};
using OpX = Op<128, 0>;   // A: [Xb; QXb] then [Ktil; Qtil], K = 128 channels
using OpY = Op<16, 0>;    // B: Y_b, 16 rows, K = 128 channels
using OpKH = Op<128, 0>;  // A: Khat^T, rows = key channel, K = 64 tokens
using OpTP = Op<128, 0>;  // A: [T; P], K = 64 tokens
using OpXV = Op<32, 16>;  // B: X^T and U^T, rows = value column, K = 64 tokens
using OpS = Op<32, 16>;   // B: S^T, rows = value column, K = 128 key channels

// ------------------------------------------------------------ smem layout
constexpr uint32_t SM_OPX = 0;                       // 65536 (raw TMA tiles alias it)
constexpr uint32_t SM_RAWQ = 0, SM_RAWK = 16384, SM_RAWG = 32768, SM_RAWV = 49152;
constexpr uint32_t SM_KF = 65536;                    // FP32 k       [64][KP]
constexpr uint32_t SM_QF = SM_KF + 64 * KP * 4;      // FP32 qh      [64][KP]
constexpr uint32_t SM_GAM = SM_QF + 64 * KP * 4;     // FP32 Gamma   [64][KP]
constexpr uint32_t SM_STAGE_END = SM_GAM + 64 * KP * 4;
// reused after the prepare operands are built
constexpr uint32_t SM_AM = SM_KF;                    // FP32 A [64][AP]
constexpr uint32_t SM_TM = SM_AM + 64 * AP * 4;      // FP32 T [64][AP]
constexpr uint32_t SM_TP = (SM_TM + 64 * AP * 4 + 15) & ~15u;
constexpr uint32_t SM_XV = SM_TP + OpTP::bytes(64);
constexpr uint32_t SM_ZS = SM_XV + OpXV::bytes(64);  // solve scratch [3][16][17]
constexpr uint32_t SM_OPKH = SM_STAGE_END;
constexpr uint32_t SM_OPY = SM_OPKH + OpKH::bytes(64);  // Y_b, later U^T
constexpr uint32_t SM_OPS = SM_OPY + OpXV::bytes(64);
constexpr uint32_t SM_BETA = SM_OPS + OpS::bytes(128);
constexpr uint32_t SM_GH = SM_BETA + 64 * 4;
constexpr uint32_t SM_GMID = SM_GH + 128 * 4;
constexpr uint32_t SM_GLAST = SM_GMID + 4 * 128 * 4;
constexpr uint32_t SM_DEC = SM_GLAST + 128 * 4;
constexpr uint32_t SM_BAR = SM_DEC + 128 * 4;        // 2 mbarriers + TMEM base + flag
constexpr uint32_t SM_TOTAL = SM_BAR + 64;

static_assert(SM_ZS + 3 * 16 * 17 * 4 <= SM_STAGE_END, "solve scratch overlaps");
static_assert(OpY::bytes(128) <= OpXV::bytes(64), "Y_b does not fit its slot");
static_assert(SM_TOTAL <= 232448, "shared memory budget exceeded");

// TMEM columns (256 allocated)
constexpr uint32_t TC_AP = 0, TC_PU = 64, TC_Y = 128, TC_U = 160, TC_E = 192;

__device__ __forceinline__ float bf(uint16_t b) {
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

__device__ __forceinline__ void st4(unsigned char* base, uint32_t off, float a, float b, float c,
                                    float d) {
    *reinterpret_cast<float4*>(base + off) =
        make_float4(tc::to_tf32(a), tc::to_tf32(b), tc::to_tf32(c), tc::to_tf32(d));
}

struct TmaMaps {
    CUtensorMap q, k, g, v;
};

// D = A . B^T over `ksteps` K-steps of 8, issued by the calling thread.
template <class OA, class OB>
__device__ __forceinline__ void issue_mma(uint32_t d, uint32_t a, uint32_t b, int ksteps,
                                          uint32_t idesc) {
    for (int ks = 0; ks < ksteps; ++ks)
        tc::mma_tf32(d, OA::desc(a, ks), OB::desc(b, ks), idesc, ks > 0);
}

__global__ void __launch_bounds__(NT, 1)
prefill_tc_kernel(const __grid_constant__ TmaMaps maps, float* __restrict__ state,
                  const uint16_t* __restrict__ beta, float* __restrict__ o, int t, int t_pad,
                  int heads, const int* __restrict__ cu, int n_seqs) {
    extern __shared__ __align__(1024) unsigned char sm[];
    const int slice = blockIdx.x, h = blockIdx.y, n = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5;
    const int ln = tid & 127, ch = tid >> 7;  // TMEM lane and column half
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;

    float* KF = reinterpret_cast<float*>(sm + SM_KF);
    float* QF = reinterpret_cast<float*>(sm + SM_QF);
    float* GAM = reinterpret_cast<float*>(sm + SM_GAM);
    float* AM = reinterpret_cast<float*>(sm + SM_AM);
    float* TM = reinterpret_cast<float*>(sm + SM_TM);
    float* ZS = reinterpret_cast<float*>(sm + SM_ZS);
    float* BETA = reinterpret_cast<float*>(sm + SM_BETA);
    float* GH = reinterpret_cast<float*>(sm + SM_GH);
    float* GMID = reinterpret_cast<float*>(sm + SM_GMID);
    float* GLAST = reinterpret_cast<float*>(sm + SM_GLAST);
    float* DEC = reinterpret_cast<float*>(sm + SM_DEC);
    uint64_t* bar_tma = reinterpret_cast<uint64_t*>(sm + SM_BAR);
    uint64_t* bar_mma = bar_tma + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + SM_BAR + 16);
    int* abort_flag = reinterpret_cast<int*>(sm + SM_BAR + 20);
    const uint16_t* RAWQ = reinterpret_cast<const uint16_t*>(sm + SM_RAWQ);
    const uint16_t* RAWK = reinterpret_cast<const uint16_t*>(sm + SM_RAWK);
    const uint16_t* RAWG = reinterpret_cast<const uint16_t*>(sm + SM_RAWG);
    const uint16_t* RAWV = reinterpret_cast<const uint16_t*>(sm + SM_RAWV);
    const uint32_t s_opx = tc::smem_u32(sm + SM_OPX), s_opy = tc::smem_u32(sm + SM_OPY),
                   s_opkh = tc::smem_u32(sm + SM_OPKH), s_tp = tc::smem_u32(sm + SM_TP),
                   s_xv = tc::smem_u32(sm + SM_XV),
                   s_ops = tc::smem_u32(sm + SM_OPS);

    int start, end;
    if (!cu) {
        start = n * t_pad;
        end = start + t;
    } else {
        start = __ldg(cu + n);
        end = __ldg(cu + n + 1);
        bool ok = start >= 0 && start <= end && end <= t;
        if (n == 0) ok = ok && start == 0;
        if (n == n_seqs - 1) ok = ok && end == t;
        if (!ok) {
            if (tid == 0) atomicOr(&g_tc_status, STATUS_BAD_CU_SEQLENS);
            return;
        }
    }

    if (tid == 0) {
        tc::mbar_init(bar_tma, 1);
        tc::mbar_init(bar_mma, 1);
        tc::fence_mbar_init();
        tc::prefetch_tmap(&maps.q);
        tc::prefetch_tmap(&maps.k);
        tc::prefetch_tmap(&maps.g);
        tc::prefetch_tmap(&maps.v);
        *abort_flag = 0;
    }
    if (warp == 0) tc::tmem_alloc(tmem_slot, 256);
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    uint32_t ph_tma = 0, ph_mma = 0;

    // state slice: thread (key ln, half ch) owns S[ln][16 ch .. 16 ch + 15]
    float* Sg = state + ((size_t)n * heads + h) * D * D + (size_t)ln * D + slice * DV + ch * 16;
    float sreg[16];
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4) {
        const float4 v4 = *reinterpret_cast<const float4*>(Sg + 4 * q4);
        sreg[4 * q4] = v4.x;
        sreg[4 * q4 + 1] = v4.y;
        sreg[4 * q4 + 2] = v4.z;
        sreg[4 * q4 + 3] = v4.w;
    }
#pragma unroll
    for (int jj = 0; jj < 16; ++jj)
        *reinterpret_cast<float*>(sm + SM_OPS + OpS::off(ch * 16 + jj, ln)) = tc::to_tf32(sreg[jj]);

    auto wait_mma = [&]() {
        if (!tc::mbar_wait(bar_mma, ph_mma)) {
            atomicOr(&g_tc_status, STATUS_TIMEOUT);
            *abort_flag = 1;
        }
        ph_mma ^= 1;
        tc::tc_fence_after();
    };
    auto sync_for_mma = [&]() {  // generic smem writes and TMEM reads before an MMA
        tc::fence_async_smem();
        tc::tc_fence_before();
        __syncthreads();
    };

    for (int c0 = start; c0 < end; c0 += C) {
        const int L = min(C, end - c0);
        // ---------------------------------------------------------- P0 loads
        sync_for_mma();
        if (*abort_flag) break;
        if (tid == 0) {
            tc::mbar_arrive_expect_tx(bar_tma, 3 * 16384 + 64 * DV * 2);
            tc::tma_load_2d(sm + SM_RAWQ, &maps.q, bar_tma, h * D, c0);
            tc::tma_load_2d(sm + SM_RAWK, &maps.k, bar_tma, h * D, c0);
            tc::tma_load_2d(sm + SM_RAWG, &maps.g, bar_tma, h * D, c0);
            tc::tma_load_2d(sm + SM_RAWV, &maps.v, bar_tma, h * D + slice * DV, c0);
        }
        if (tid < C) BETA[tid] = (tid < L) ? bf(__ldg(beta + (size_t)(c0 + tid) * heads + h)) : 0.f;
        if (!tc::mbar_wait(bar_tma, ph_tma)) {
            atomicOr(&g_tc_status, STATUS_TIMEOUT);
            *abort_flag = 1;
        }
        ph_tma ^= 1;

        // ---------------------------------------------------------- P1 Gamma, staging
        {
            const int i = tid & 127, hf = tid >> 7;
            float acc = 0.f;
#pragma unroll
            for (int rr = 0; rr < 32; ++rr) {
                const int r = 32 * hf + rr;
                float gv = 0.f, kv = 0.f, qv = 0.f;
                if (r < L) {
                    gv = bf(RAWG[r * D + i]);
                    kv = bf(RAWK[r * D + i]);
                    qv = __fmul_rn(KDA_Q_SCALE, bf(RAWQ[r * D + i]));
                }
                acc = __fadd_rn(acc, gv);
                GAM[r * KP + i] = acc;
                KF[r * KP + i] = kv;
                QF[r * KP + i] = qv;
            }
            if (hf == 0) GH[i] = acc;
        }
        float vreg[16];
        if (ln < C) {
#pragma unroll
            for (int jj = 0; jj < 16; ++jj)
                vreg[jj] = (ln < L) ? bf(RAWV[ln * DV + ch * 16 + jj]) : 0.f;
        }
        __syncthreads();
        if (tid >= 128) {
            const int i = tid & 127;
            const float base = GH[i];
#pragma unroll
            for (int rr = 0; rr < 32; ++rr) GAM[(32 + rr) * KP + i] += base;
        }
        __syncthreads();
        if (tid < 128) {
#pragma unroll
            for (int a = 0; a < 4; ++a) GMID[a * 128 + tid] = GAM[(16 * a + 8) * KP + tid];
            GLAST[tid] = GAM[63 * KP + tid];
            DEC[tid] = __expf(GAM[63 * KP + tid]);
        }
        __syncthreads();

        // ---------------------------------------------------------- P2 A and P blocks
        for (int b = 0; b < 4; ++b) {
            {
                const int r = tid & 63, qg = tid >> 6;
                if (r >= 16 * b) {
                    const float* gm = GMID + b * 128;
                    for (int jj = 0; jj < 8; ++jj) {
                        const int j = qg + 4 * jj;
                        float f[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) f[e] = __expf(GAM[r * KP + 4 * j + e] - gm[4 * j + e]);
                        const float* kr = KF + r * KP + 4 * j;
                        const float* qr = QF + r * KP + 4 * j;
                        st4(sm + SM_OPX, OpX::off(r, 4 * j), kr[0] * f[0], kr[1] * f[1],
                            kr[2] * f[2], kr[3] * f[3]);
                        st4(sm + SM_OPX, OpX::off(64 + r, 4 * j), qr[0] * f[0], qr[1] * f[1],
                            qr[2] * f[2], qr[3] * f[3]);
                    }
                }
                const float* gm = GMID + b * 128;
                for (int q2 = 0; q2 < 2; ++q2) {
                    const int sr = tid & 15, j = (tid >> 4) + 16 * q2, s = 16 * b + sr;
                    float y[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        y[e] = KF[s * KP + 4 * j + e] * __expf(gm[4 * j + e] - GAM[s * KP + 4 * j + e]);
                    st4(sm + SM_OPY, OpY::off(sr, 4 * j), y[0], y[1], y[2], y[3]);
                }
            }
            sync_for_mma();
            if (tid == 0) {
                tc::tc_fence_after();
                issue_mma<OpX, OpY>(tmem + TC_AP + 16 * b, s_opx, s_opy, 16, tc::idesc_tf32(128, 16));
                tc::mma_commit(bar_mma);
            }
            wait_mma();
        }

        // ---------------------------------------------------------- P3 Ktil/Qtil, Khat^T
        {
            const int r = tid & 63, qg = tid >> 6;
            for (int jj = 0; jj < 8; ++jj) {
                const int j = qg + 4 * jj;
                float f[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) f[e] = __expf(GAM[r * KP + 4 * j + e]);
                const float* kr = KF + r * KP + 4 * j;
                const float* qr = QF + r * KP + 4 * j;
                st4(sm + SM_OPX, OpX::off(r, 4 * j), kr[0] * f[0], kr[1] * f[1], kr[2] * f[2],
                    kr[3] * f[3]);
                st4(sm + SM_OPX, OpX::off(64 + r, 4 * j), qr[0] * f[0], qr[1] * f[1],
                    qr[2] * f[2], qr[3] * f[3]);
            }
            const int i = tid & 127, hq = tid >> 7;
            const float gl = GLAST[i];
            for (int qq = 0; qq < 8; ++qq) {
                const int q4 = 2 * qq + hq;  // token quad
                float kh[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int s = 4 * q4 + e;
                    kh[e] = BETA[s] * KF[s * KP + i] * __expf(gl - GAM[s * KP + i]);
                }
                st4(sm + SM_OPKH, OpKH::off(i, 4 * q4), kh[0], kh[1], kh[2], kh[3]);
            }
        }
        __syncthreads();  // staging arrays are dead from here on

        // ---------------------------------------------------------- P4 read A, P
        {
            float v[32];
            tc::tmem_ld16(tmem + lane_base + TC_AP + 32 * ch, *reinterpret_cast<float(*)[16]>(v));
            tc::tmem_ld16(tmem + lane_base + TC_AP + 32 * ch + 16,
                          *reinterpret_cast<float(*)[16]>(v + 16));
            tc::tmem_ld_wait();
            if (ln < 64) {
                const int r = ln;
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    const int s = 32 * ch + c;
                    AM[r * AP + s] = (s < r) ? v[c] * BETA[s] : 0.f;
                }
            } else {
                const int r = ln - 64;
#pragma unroll
                for (int c4 = 0; c4 < 8; ++c4) {
                    float p[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int s = 32 * ch + 4 * c4 + e;
                        p[e] = (s <= r) ? v[4 * c4 + e] * BETA[s] : 0.f;
                    }
                    st4(sm + SM_TP, OpTP::off(64 + r, 32 * ch + 4 * c4), p[0], p[1], p[2], p[3]);
                }
            }
        }
        for (int e = tid; e < 64 * 64; e += NT) TM[(e >> 6) * AP + (e & 63)] = 0.f;
        tc::tc_fence_before();
        __syncthreads();

        // ---------------------------------------------------------- P5 T = (I + A)^-1
        if (tid < 64) {  // diagonal 16 x 16 blocks: one column per thread
            const int a = tid >> 4, cc = tid & 15, o0 = 16 * a;
            float col[16];
#pragma unroll
            for (int rr = 0; rr < 16; ++rr) {
                float x = (rr == cc) ? 1.f : 0.f;
#pragma unroll
                for (int ss = 0; ss < rr; ++ss)
                    x = __fmaf_rn(-AM[(o0 + rr) * AP + o0 + ss], col[ss], x);
                col[rr] = (rr < cc) ? 0.f : x;
            }
#pragma unroll
            for (int rr = 0; rr < 16; ++rr) TM[(o0 + rr) * AP + o0 + cc] = col[rr];
        }
        __syncthreads();
        for (int d = 1; d < 4; ++d) {  // block sub-diagonal d: T_ab = -T_aa sum_c A_ac T_cb
            const int np = 4 - d;
            for (int e = tid; e < np * 256; e += NT) {
                const int pb = e >> 8, rr = (e >> 4) & 15, cc = e & 15;
                const int b = pb, a = pb + d;
                float z = 0.f;
                for (int c = b; c < a; ++c)
#pragma unroll
                    for (int kk = 0; kk < 16; ++kk)
                        z = __fmaf_rn(AM[(16 * a + rr) * AP + 16 * c + kk],
                                      TM[(16 * c + kk) * AP + 16 * b + cc], z);
                ZS[(pb * 16 + rr) * 17 + cc] = z;
            }
            __syncthreads();
            for (int e = tid; e < np * 256; e += NT) {
                const int pb = e >> 8, rr = (e >> 4) & 15, cc = e & 15;
                const int b = pb, a = pb + d;
                float x = 0.f;
#pragma unroll
                for (int kk = 0; kk < 16; ++kk)
                    x = __fmaf_rn(TM[(16 * a + rr) * AP + 16 * a + kk], ZS[(pb * 16 + kk) * 17 + cc], x);
                TM[(16 * a + rr) * AP + 16 * b + cc] = -x;
            }
            __syncthreads();
        }
        {   // T into rows 0..63 of [T; P]
            const int r = tid & 63, qg = tid >> 6;
            for (int jj = 0; jj < 4; ++jj) {
                const int j = qg + 4 * jj;
                const float* tr = TM + r * AP + 4 * j;
                st4(sm + SM_TP, OpTP::off(r, 4 * j), tr[0], tr[1], tr[2], tr[3]);
            }
        }
        sync_for_mma();

        // ---------------------------------------------------------- P6 state scan
        if (tid == 0) {
            tc::tc_fence_after();
            issue_mma<OpX, OpS>(tmem + TC_Y, s_opx, s_ops, 16, tc::idesc_tf32(128, DV));
            tc::mma_commit(bar_mma);
        }
        wait_mma();
        float qs[16];
        {
            float v[16];
            tc::tmem_ld16(tmem + lane_base + TC_Y + 16 * ch, v);
            tc::tmem_ld_wait();
            if (ln < 64) {
                const int r = ln;
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) {
                    const float x = (r < L) ? vreg[jj] - v[jj] : 0.f;
                    *reinterpret_cast<float*>(sm + SM_XV + OpXV::off(16 * ch + jj, r)) = tc::to_tf32(x);
                }
            } else {
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) qs[jj] = v[jj];
            }
        }
        sync_for_mma();
        if (tid == 0) {
            tc::tc_fence_after();
            issue_mma<OpTP, OpXV>(tmem + TC_U, s_tp, s_xv, 8, tc::idesc_tf32(128, DV));
            tc::mma_commit(bar_mma);
        }
        wait_mma();
        if (ln < 64) {
            float v[16];
            tc::tmem_ld16(tmem + lane_base + TC_U + 16 * ch, v);
            tc::tmem_ld_wait();
            const int r = ln;
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
                const float u = (r < L) ? v[jj] : 0.f;
                *reinterpret_cast<float*>(sm + SM_OPY + OpXV::off(16 * ch + jj, r)) = tc::to_tf32(u);
            }
        }
        sync_for_mma();
        if (tid == 0) {
            tc::tc_fence_after();
            issue_mma<OpKH, OpXV>(tmem + TC_E, s_opkh, s_opy, 8, tc::idesc_tf32(128, DV));
            issue_mma<OpTP, OpXV>(tmem + TC_PU, s_tp, s_opy, 8, tc::idesc_tf32(128, DV));
            tc::mma_commit(bar_mma);
        }
        wait_mma();
        if (ln >= 64) {  // O = Qtil S + P U for the chunk's rows
            float v[16];
            tc::tmem_ld16(tmem + lane_base + TC_PU + 16 * ch, v);
            tc::tmem_ld_wait();
            const int r = ln - 64;
            if (r < L) {
                float* orow = o + ((size_t)(c0 + r) * heads + h) * D + slice * DV + 16 * ch;
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4)
                    *reinterpret_cast<float4*>(orow + 4 * q4) =
                        make_float4(qs[4 * q4] + v[4 * q4], qs[4 * q4 + 1] + v[4 * q4 + 1],
                                    qs[4 * q4 + 2] + v[4 * q4 + 2], qs[4 * q4 + 3] + v[4 * q4 + 3]);
            }
        }
        {
            float v[16];
            tc::tmem_ld16(tmem + lane_base + TC_E + 16 * ch, v);
            tc::tmem_ld_wait();
            const float dk = DEC[ln];
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
                sreg[jj] = __fmaf_rn(dk, sreg[jj], v[jj]);
                *reinterpret_cast<float*>(sm + SM_OPS + OpS::off(16 * ch + jj, ln)) = tc::to_tf32(sreg[jj]);
            }
        }
    }

    if (!*abort_flag) {
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4)
            *reinterpret_cast<float4*>(Sg + 4 * q4) =
                make_float4(sreg[4 * q4], sreg[4 * q4 + 1], sreg[4 * q4 + 2], sreg[4 * q4 + 3]);
    }
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, 256);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                            cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

bool make_map(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint64_t pitch_elems,
              uint32_t box_cols) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t gdim[2] = {cols, rows};
    cuuint64_t gstride[1] = {pitch_elems * 2};
    cuuint32_t box[2] = {box_cols, (cuuint32_t)C};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), gdim, gstride, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// Launches the tensor-core prefill (BF16 inputs, chunk 64); arguments are
// validated by kda_prefill.
kda_status launch_prefill_tc(float* state, const void* q, const void* k, const void* v,
                             const void* g, const void* beta, float* o, int t, int t_pad,
                             int heads, long long stride, const int* cu, int n_seqs,
                             cudaStream_t s) {
    const uint64_t rows = cu ? (uint64_t)t : (uint64_t)t_pad * n_seqs;
    TmaMaps maps;
    const uint64_t hd = (uint64_t)heads * D;
    if (!make_map(&maps.q, q, hd, rows, (uint64_t)stride, D) ||
        !make_map(&maps.k, k, hd, rows, (uint64_t)stride, D) ||
        !make_map(&maps.g, g, hd, rows, hd, D) ||
        !make_map(&maps.v, v, hd, rows, (uint64_t)stride, DV)) {
        set_error("kda_prefill: cannot encode TMA tensor maps");
        return KDA_ERR_CUDA;
    }
    cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SM_TOTAL);
    if (e != cudaSuccess) {
        set_error("kda_prefill: cannot reserve %u B of shared memory: %s", SM_TOTAL,
                  cudaGetErrorString(e));
        return KDA_ERR_CUDA;
    }
    dim3 grid(D / DV, heads, n_seqs);
    prefill_tc_kernel<<<grid, NT, SM_TOTAL, s>>>(maps, state, (const uint16_t*)beta, o, t, t_pad,
                                                 heads, cu, n_seqs);
    return launch_result("kda_prefill (tensor cores)");
}

cudaError_t read_and_clear_status_prefill_tc(unsigned* out) {
    unsigned zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(out, g_tc_status, sizeof(unsigned));
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_tc_status, &zero, sizeof(unsigned));
    return e;
}

}  // namespace kda
