// Front end of the KDA block: depthwise causal conv1d + SiLU, then L2 over the
// q and k channels (block pipeline "conv1d + SiLU -> L2(q,k only)"; fused at
// decode as causal_conv1d_update_l2norm, split at prefill into conv_prefill
// and l2_norm_bf16; config.rs: conv state of conv_kernel slots, L2 applied as
// 1/sqrt(sum + eps)).
//
// Kernel 1 (conv_silu_l2_kernel): one CTA of 128 threads per (group of 1024
// channels = 8 heads, span of consecutive tokens), about three CTAs per SM in
// one wave.  The span's x rows arrive by TMA in blocks of 16 tokens, double
// buffered behind an mbarrier each, so the next block is in flight while the
// current one is computed.  A thread owns 8 adjacent channels (16-byte shared
// loads and global stores) and carries a register window of the last
// conv_kernel - 1 inputs from block to block.  History before a sequence's
// first token comes from the conv state, which this kernel only reads.  A
// q/k head's 128 channels are one half-warp, so its L2 sum is a 4-step
// shuffle reduction within the half-warp, per token, with no shared memory;
// the conv taps run as packed FP32 pairs (fma.rn.f32x2).
// Kernel 2 (conv_state_kernel): after kernel 1, each thread rewrites one
// (sequence, channel) state row to hold that sequence's last conv_kernel
// inputs, reading the old row first; separating it from kernel 1 keeps any
// CTA from reading a state row another CTA has already replaced.
// Kernel 3 (conv_rows_kernel) replaces the pair for uniform batches of short
// sequences (decode, the k-row form): one thread per (sequence, 8 channels)
// walks the rows and rewrites its own state rows, and writes the snapshots.
#include <cuda_bf16.h>

#include "f32x2.h"
#include "kda_common.h"
#include "sm103_tc.h"
#include "tma_map.h"

namespace kda {
namespace {

__device__ unsigned g_conv_status = 0;

constexpr int kTok = 16;                   // tokens per x block
constexpr int kThreads = 128;              // per CTA
constexpr int kCh = 8;                     // channels per thread
constexpr int kCtaCh = kThreads * kCh;     // channels per CTA (8 heads)

__device__ __forceinline__ float bf16_to_f32(uint16_t b) {
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

__device__ __forceinline__ float2 bf16x2_to_f32(uint32_t u) {
    return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
}

__device__ __forceinline__ uint32_t f32x2_to_bf16x2(float a, float b) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);  // one packed conversion
    return *reinterpret_cast<const uint32_t*>(&v);
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


// SiLU of a channel pair, a / (1 + e^-a) with e^-a = 2^(-a log2 e), in FP32
// (rounded to BF16 by the caller).
__device__ __forceinline__ float2 silu2(float2 a) {
    constexpr float kNegLog2e = -1.4426950408889634f;
    const float2 t = mul2(a, make_float2(kNegLog2e, kNegLog2e));
    const float2 d = add2(make_float2(ex2_approx(t.x), ex2_approx(t.y)), make_float2(1.f, 1.f));
    return mul2(a, make_float2(rcp_approx(d.x), rcp_approx(d.y)));
}

// The end of one token for a thread's 8 channels, given the conv sums a:
// SiLU, then (q and k heads) the head's L2 scale from a half-warp reduction,
// then one rounding to BF16.  Both conv kernels go through this function, so
// the same token gives the same bits whichever kernel computes it.
__device__ __forceinline__ uint4 silu_l2_bf16(const float2 (&a)[kCh / 2], bool normalise,
                                              unsigned hmask, float l2_eps) {
    float2 y[kCh / 2];
#pragma unroll
    for (int e = 0; e < kCh / 2; ++e) y[e] = silu2(a[e]);
    if (normalise) {  // uniform per half-warp
        float2 p2 = mul2(y[0], y[0]);
#pragma unroll
        for (int e = 1; e < kCh / 2; ++e) p2 = fma2(y[e], y[e], p2);
        float p = p2.x + p2.y;
#pragma unroll
        for (int off = 8; off > 0; off >>= 1) p += __shfl_xor_sync(hmask, p, off);
        const float inv = rsqrtf(p + l2_eps);
#pragma unroll
        for (int e = 0; e < kCh / 2; ++e) y[e] = mul2(y[e], make_float2(inv, inv));
    }
    uint4 o;
    o.x = f32x2_to_bf16x2(y[0].x, y[0].y);
    o.y = f32x2_to_bf16x2(y[1].x, y[1].y);
    o.z = f32x2_to_bf16x2(y[2].x, y[2].y);
    o.w = f32x2_to_bf16x2(y[3].x, y[3].y);
    return o;
}

// x arrives in blocks of kTok tokens x 1024 channels through TMA, as four
// boxes of 256 channels ([box][token][256] in shared memory), in a ring of
// kStages buffers with one mbarrier each.
constexpr int kBoxCh = 256;
constexpr int kStages = 2;
constexpr int kCtasPerSm = 3;                                  // shared memory allows three
constexpr uint32_t kBlkBytes = kTok * kCtaCh * 2;              // 32 KB
constexpr uint32_t kConvSmem = kStages * kBlkBytes + 8 * kStages;

template <int K>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
conv_silu_l2_kernel(const __grid_constant__ CUtensorMap xmap, const float* __restrict__ conv_state,
                    const uint16_t* __restrict__ x, const uint16_t* __restrict__ w,
                    uint16_t* __restrict__ out, int total, int t_per_seq,
                    const int* __restrict__ cu, int n_seqs, int heads, float l2_eps, int span) {
    extern __shared__ __align__(128) unsigned char sm[];
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + kStages * kBlkBytes);
    pdl_wait();
    pdl_release();
    const int tid = threadIdx.x, lane = tid & 31;
    const int ch0 = blockIdx.x * kCtaCh;
    const int c = ch0 + kCh * tid;  // first of this thread's 8 channels
    const size_t conv_dim = (size_t)3 * heads * D;
    // conv_dim is a multiple of 128, so a head (16 threads, a half-warp) is
    // either wholly present or wholly absent; absent threads stay for the barriers.
    const bool active = (size_t)c < conv_dim;
    const bool normalise = c < 2 * heads * D;            // a q or k head
    const unsigned hmask = 0xffffu << (lane & 16);       // this half-warp
    const int tok0 = blockIdx.y * span;
    if (tok0 >= total) return;  // the whole CTA
    const int tok_end = min(total, tok0 + span);
    const int nblk = (tok_end - tok0 + kTok - 1) / kTok;

    if (tid == 0) {
        for (int b = 0; b < kStages; ++b) tc::mbar_init(bar + b, 1);
        tc::fence_mbar_init();
    }
    __syncthreads();
    // boxes holding at least one channel of this group (conv_dim is a
    // multiple of 384, so the last group may cover fewer than four)
    const int nbox = min(kCtaCh / kBoxCh, (int)((conv_dim - ch0 + kBoxCh - 1) / kBoxCh));
    auto load_block = [&](int i) {  // block i into buffer i % kStages (thread 0)
        uint64_t* b = bar + i % kStages;
        tc::mbar_arrive_expect_tx(b, (uint32_t)nbox * (kTok * kBoxCh * 2));
        for (int bx = 0; bx < nbox; ++bx)
            tc::tma_load_2d(sm + (i % kStages) * kBlkBytes + bx * (kTok * kBoxCh * 2), &xmap, b,
                            ch0 + bx * kBoxCh, tok0 + i * kTok);
    };
    if (tid == 0)
        for (int i = 0; i < kStages - 1 && i < nblk; ++i) load_block(i);

    float2 wv[K][kCh / 2];  // tap j of channel pairs
#pragma unroll
    for (int j = 0; j < K; ++j)
#pragma unroll
        for (int e = 0; e < kCh / 2; ++e)
            wv[j][e] = active ? make_float2(bf16_to_f32(__ldg(w + (size_t)(c + 2 * e) * K + j)),
                                            bf16_to_f32(__ldg(w + (size_t)(c + 2 * e + 1) * K + j)))
                              : make_float2(0.f, 0.f);

    // The span's tokens are consecutive: find the first one's sequence once,
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
    // hv[j][e]: channel pair e's inputs at token tau - (K - 1) + j.
    float2 hv[K > 1 ? K - 1 : 1][kCh / 2];
    auto state_slot = [&](int e2, int slot) {  // the state's slot for channel pair e2
        const float* st = conv_state + ((size_t)n * conv_dim + c + 2 * e2) * K;
        return make_float2(__ldg(st + slot), __ldg(st + K + slot));
    };
    auto state_history = [&]() {  // a sequence's first token: history from its state
#pragma unroll
        for (int j = 0; j < K - 1; ++j)
#pragma unroll
            for (int e = 0; e < kCh / 2; ++e)
                hv[j][e] = active ? state_slot(e, j + 1) : make_float2(0.f, 0.f);
    };
#pragma unroll
    for (int j = 0; j < K - 1; ++j) {
        const int src = tok0 - (K - 1) + j;
#pragma unroll
        for (int e = 0; e < kCh / 2; ++e) hv[j][e] = make_float2(0.f, 0.f);
        if (ok && active) {
            if (src >= start) {
                const uint4 u = __ldg(reinterpret_cast<const uint4*>(x + (size_t)src * conv_dim + c));
                hv[j][0] = bf16x2_to_f32(u.x);
                hv[j][1] = bf16x2_to_f32(u.y);
                hv[j][2] = bf16x2_to_f32(u.z);
                hv[j][3] = bf16x2_to_f32(u.w);
            } else {
#pragma unroll
                for (int e = 0; e < kCh / 2; ++e) hv[j][e] = state_slot(e, K + (src - start));
            }
        }
    }
    // this thread's 16 bytes of token row m inside a block buffer
    const uint32_t xoff = (uint32_t)(tid / (kBoxCh / kCh)) * (kTok * kBoxCh * 2) +
                          (uint32_t)((kCh * tid) % kBoxCh) * 2;
    bool timed_out = false;
    for (int i = 0; i < nblk; ++i) {
        const int tb = tok0 + i * kTok;
        // block i + kStages - 1 reuses the buffer released at the end of iteration i - 1
        if (tid == 0 && i + kStages - 1 < nblk) load_block(i + kStages - 1);
        if (!tc::mbar_wait(bar + i % kStages, (uint32_t)(i / kStages) & 1u)) timed_out = true;
        const unsigned char* xb = sm + (i % kStages) * kBlkBytes + xoff;
        uint4* op = reinterpret_cast<uint4*>(out + (size_t)tb * conv_dim + c);
        // One token: conv over the window, SiLU, the head's L2 scale, BF16 store.
        auto token = [&](int m) {
            const uint4 xm = *reinterpret_cast<const uint4*>(xb + m * (kBoxCh * 2));
            const float2 xv[kCh / 2] = {bf16x2_to_f32(xm.x), bf16x2_to_f32(xm.y),
                                        bf16x2_to_f32(xm.z), bf16x2_to_f32(xm.w)};
            float2 a[kCh / 2];
#pragma unroll
            for (int e = 0; e < kCh / 2; ++e) {
                if constexpr (K > 1) {
                    a[e] = mul2(wv[0][e], hv[0][e]);
#pragma unroll
                    for (int j = 1; j < K - 1; ++j) a[e] = fma2(wv[j][e], hv[j][e], a[e]);
                    a[e] = fma2(wv[K - 1][e], xv[e], a[e]);
                } else {
                    a[e] = mul2(wv[0][e], xv[e]);
                }
#pragma unroll
                for (int j = 0; j + 1 < K - 1; ++j) hv[j][e] = hv[j + 1][e];
                if constexpr (K > 1) hv[K - 2][e] = xv[e];
            }
            const uint4 o = silu_l2_bf16(a, normalise, hmask, l2_eps);
            if (active) op[(size_t)m * (conv_dim / kCh)] = o;
        };
        if (ok && tb + kTok <= tok_end && tb + kTok <= end) {
            // Common case: the block's tokens lie in one sequence; straight-line
            // code lets the tokens' independent work overlap.
#pragma unroll
            for (int m = 0; m < kTok; ++m) token(m);
        } else {
#pragma unroll 1
            for (int m = 0; m < kTok; ++m) {  // uniform over the CTA
                const int tau = tb + m;
                if (!ok || tau >= tok_end) break;
                if (tau >= end) {  // a new sequence starts at tau (skipping empty ones)
                    if (cu) {
                        while (n + 1 < n_seqs && __ldg(cu + n + 1) <= tau) ++n;
                        start = __ldg(cu + n);
                        end = __ldg(cu + n + 1);
                        if (!(start == tau && tau < end)) {
                            ok = false;
                            break;
                        }
                    } else {
                        ++n;
                        start = n * t_per_seq;
                        end = start + t_per_seq;
                    }
                    state_history();
                }
                token(m);
            }
        }
        __syncthreads();  // every thread is done with buffer i % kStages
    }
    if (tid == 0 && (!ok || timed_out))
        atomicOr(&g_conv_status, timed_out ? STATUS_TIMEOUT : STATUS_BAD_CU_SEQLENS);
}

// Up to KDA_MAX_K snapshot targets, each [n_seqs][conv_dim][K] FP32.
struct ConvSnaps {
    float* p[KDA_MAX_K];
};

template <int K>
__global__ void conv_state_kernel(float* __restrict__ conv_state, const uint16_t* __restrict__ x,
                                  int total, int t_per_seq, const int* __restrict__ cu,
                                  int n_seqs, int heads) {
    pdl_wait();  // the conv kernel has read the old state
    pdl_release();
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
    // a state row of 4 slots moves as one 16-byte access (rows are 16-byte
    // aligned: conv_state is, and K = 4 makes every row 16 bytes)
    if constexpr (K == 4) {
        const float4 o4 = *reinterpret_cast<const float4*>(st);
        old[0] = o4.x;
        old[1] = o4.y;
        old[2] = o4.z;
        old[3] = o4.w;
    } else {
#pragma unroll
        for (int j = 0; j < K; ++j) old[j] = st[j];
    }
#pragma unroll
    for (int j = 0; j < K; ++j) {
        const int rel = len - K + j;  // position relative to the sequence start
        float kept = old[K - 1];  // old[min(j + len, K - 1)], selected without indexing
#pragma unroll
        for (int jj = 0; jj < K - 1; ++jj)
            if (jj == j + len) kept = old[jj];
        nw[j] = (rel >= 0) ? bf16_to_f32(__ldg(x + (size_t)(start + rel) * conv_dim + c)) : kept;
    }
    if constexpr (K == 4) {
        *reinterpret_cast<float4*>(st) = make_float4(nw[0], nw[1], nw[2], nw[3]);
    } else {
#pragma unroll
        for (int j = 0; j < K; ++j) st[j] = nw[j];
    }
}

// Uniform batches of short sequences (rows <= KDA_MAX_K tokens each: the
// decode-time update and the k-row form).  One thread per (sequence, 8
// channels) takes its window from the sequence's conv state, runs the rows in
// order and writes the outputs, snapshot t (the window ending at row t) and
// the new state.  A state row is read and rewritten by the thread that owns
// it, so this one launch replaces the conv and state-rewrite pair.
// With K = 4 a warp's 32 threads own 256 consecutive channels, whose windows
// are one contiguous 4 KB span of a state array: each window goes out through
// a per-warp shared-memory tile (XOR-swizzled by 16-byte chunk, so neither
// side conflicts on banks) as eight 512-byte warp stores, instead of eight
// 16-byte stores per thread that each touch 32 different lines.
constexpr int kRowsThreads = 256;

template <int K>
__global__ void __launch_bounds__(kRowsThreads, 2)
conv_rows_kernel(float* __restrict__ conv_state, const uint16_t* __restrict__ x,
                 const uint16_t* __restrict__ w, uint16_t* __restrict__ out, int rows, int n_seqs,
                 int heads, float l2_eps, ConvSnaps snaps, int n_snap) {
    pdl_wait();
    pdl_release();
    const int conv_dim = 3 * heads * D;
    const int per_seq = conv_dim / kCh;  // threads per sequence, a multiple of 16
    const long long total = (long long)n_seqs * per_seq;
    const long long idx0 = (long long)blockIdx.x * kRowsThreads + threadIdx.x;
    // total is a multiple of 16: a half-warp is wholly in or out.  With K = 4
    // the idle half of the last warp stays (its windows are staged but not
    // stored) so that the warp's tile copies keep all 32 lanes.
    if (idx0 >= total && (K != 4 || (idx0 & ~31LL) >= total)) return;
    const bool live = idx0 < total;
    const long long idx = live ? idx0 : total - 1;  // idle lanes compute on a valid copy
    const int n = (int)(idx / per_seq);
    const int c = (int)(idx % per_seq) * kCh;
    const bool normalise = c < 2 * heads * D;
    const unsigned hmask = 0xffffu << (threadIdx.x & 16);

    float2 wv[K][kCh / 2];
    bool w_vec = false;
    if constexpr (K == 4) w_vec = (reinterpret_cast<uintptr_t>(w) & 15) == 0;
    if (w_vec) {
        // the 8 channels' taps are 64 contiguous bytes: four 16-byte loads
        const uint4* w4 = reinterpret_cast<const uint4*>(w + (size_t)c * K);
#pragma unroll
        for (int q = 0; q < 4; ++q) {  // q covers channels 2q and 2q + 1
            const uint4 u = __ldg(w4 + q);
            const float2 lo0 = bf16x2_to_f32(u.x), lo1 = bf16x2_to_f32(u.y);  // channel 2q
            const float2 hi0 = bf16x2_to_f32(u.z), hi1 = bf16x2_to_f32(u.w);  // channel 2q+1
            wv[0][q] = make_float2(lo0.x, hi0.x);
            wv[1 % K][q] = make_float2(lo0.y, hi0.y);  // (K == 4 here)
            wv[2 % K][q] = make_float2(lo1.x, hi1.x);
            wv[3 % K][q] = make_float2(lo1.y, hi1.y);
        }
    } else {
#pragma unroll
        for (int j = 0; j < K; ++j)
#pragma unroll
            for (int e = 0; e < kCh / 2; ++e)
                wv[j][e] = make_float2(bf16_to_f32(__ldg(w + (size_t)(c + 2 * e) * K + j)),
                                       bf16_to_f32(__ldg(w + (size_t)(c + 2 * e + 1) * K + j)));
    }
    // win[j][e]: channel pair e's input at row r - (K - 1) + j; before row 0,
    // slots 1..K-1 of the state are the inputs before the sequence.
    float* st = conv_state + ((size_t)n * conv_dim + c) * K;  // 8 channels x K slots
    float2 win[K][kCh / 2];
    if constexpr (K == 4) {
#pragma unroll
        for (int e = 0; e < kCh / 2; ++e) {
            const float4 s0 = __ldg(reinterpret_cast<const float4*>(st) + 2 * e);
            const float4 s1 = __ldg(reinterpret_cast<const float4*>(st) + 2 * e + 1);
            win[0][e] = make_float2(s0.y, s1.y);
            win[1][e] = make_float2(s0.z, s1.z);
            win[2][e] = make_float2(s0.w, s1.w);
        }
    } else {
#pragma unroll
        for (int j = 0; j < K - 1; ++j)
#pragma unroll
            for (int e = 0; e < kCh / 2; ++e)
                win[j][e] = make_float2(__ldg(st + (2 * e) * K + j + 1),
                                        __ldg(st + (2 * e + 1) * K + j + 1));
    }
    // window of K slots of 8 channels to a [channel][slot] state row; `base`
    // is the state array (state, or a snapshot), dst this thread's rows in it
    __shared__ float4 tile[kRowsThreads / 32][256];  // K = 4: one 4 KB tile per warp
    const int lane = threadIdx.x & 31;
    float4* wt = tile[threadIdx.x >> 5];
    auto store_window = [&](float* base, float* dst) {
        if constexpr (K == 4) {
            // channel 8 lane + e of the warp -> chunk 8 lane + (e ^ (lane & 7))
#pragma unroll
            for (int e = 0; e < kCh / 2; ++e) {
                wt[8 * lane + ((2 * e) ^ (lane & 7))] =
                    make_float4(win[0][e].x, win[1][e].x, win[2][e].x, win[3][e].x);
                wt[8 * lane + ((2 * e + 1) ^ (lane & 7))] =
                    make_float4(win[0][e].y, win[1][e].y, win[2][e].y, win[3][e].y);
            }
            __syncwarp();
            // the warp's 256 channels start at its first thread's channel
            const long long wfirst = idx0 - lane;
            float4* wdst = reinterpret_cast<float4*>(base) + wfirst * kCh;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int L = 32 * k + lane, tq = L >> 3;  // channel L belongs to lane tq
                if (wfirst + tq < total) wdst[L] = wt[8 * tq + ((L & 7) ^ (tq & 7))];
            }
            __syncwarp();  // the tile is read before the next window overwrites it
            (void)dst;
        } else {
#pragma unroll
            for (int j = 0; j < K; ++j)
#pragma unroll
                for (int e = 0; e < kCh / 2; ++e) {
                    dst[(2 * e) * K + j] = win[j][e].x;
                    dst[(2 * e + 1) * K + j] = win[j][e].y;
                }
        }
    };
    const size_t row0 = (size_t)n * rows;
    uint4 xn = __ldg(reinterpret_cast<const uint4*>(x + row0 * conv_dim + c));
#pragma unroll
    for (int r = 0; r < KDA_MAX_K; ++r) {  // unrolled: snaps.p[r] stays a parameter read
        if (r >= rows) continue;
        const uint4 xm = xn;
        if (r + 1 < rows)  // the next row's load overlaps this row's arithmetic
            xn = __ldg(reinterpret_cast<const uint4*>(x + (row0 + r + 1) * conv_dim + c));
        win[K - 1][0] = bf16x2_to_f32(xm.x);
        win[K - 1][1] = bf16x2_to_f32(xm.y);
        win[K - 1][2] = bf16x2_to_f32(xm.z);
        win[K - 1][3] = bf16x2_to_f32(xm.w);
        float2 a[kCh / 2];
#pragma unroll
        for (int e = 0; e < kCh / 2; ++e) {  // the same operations as the span kernel
            a[e] = mul2(wv[0][e], win[0][e]);
#pragma unroll
            for (int j = 1; j < K; ++j) a[e] = fma2(wv[j][e], win[j][e], a[e]);
        }
        const uint4 o = silu_l2_bf16(a, normalise, hmask, l2_eps);
        if (live) *reinterpret_cast<uint4*>(out + (row0 + r) * conv_dim + c) = o;
        if (r < n_snap) store_window(snaps.p[r], snaps.p[r] + ((size_t)n * conv_dim + c) * K);
        if (r + 1 == rows) store_window(conv_state, st);
#pragma unroll
        for (int j = 0; j + 1 < K; ++j)
#pragma unroll
            for (int e = 0; e < kCh / 2; ++e) win[j][e] = win[j + 1][e];
    }
}

template <int K>
kda_status launch(float* conv_state, const uint16_t* x, const uint16_t* w, uint16_t* out,
                  int total, int t_per_seq, const int* cu, int n_seqs, int heads, float eps,
                  cudaStream_t s, ConvSnaps snaps = {}, int n_snap = 0) {
    const int conv_dim = 3 * heads * D;
    if (!cu && t_per_seq <= KDA_MAX_K) {
        const long long threads = (long long)n_seqs * (conv_dim / kCh);
        launch_pdl(conv_rows_kernel<K>,
                   dim3((unsigned)((threads + kRowsThreads - 1) / kRowsThreads)),
                   dim3(kRowsThreads), 0, s, conv_state, x, w, out, t_per_seq, n_seqs, heads, eps,
                   snaps, n_snap);
        return launch_result("kda_conv_silu_l2 (rows)");
    }
    const int groups = (conv_dim + kCtaCh - 1) / kCtaCh;
    const int sms = sm_count();
    if (sms <= 0) {
        set_error("kda_conv_silu_l2: cannot query the multiprocessor count");
        return KDA_ERR_CUDA;
    }
    // Token spans sized for one wave of kCtasPerSm resident CTAs per SM, in
    // whole blocks of kTok tokens.
    const long long target = (long long)kCtasPerSm * sms;
    long long span = ((long long)total * groups + target - 1) / target;
    span = (span + kTok - 1) / kTok * kTok;
    if (span < kTok) span = kTok;
    const long long spans = (total + span - 1) / span;
    CUtensorMap xmap;
    if (!tma_map_bf16(&xmap, x, (uint64_t)conv_dim, (uint64_t)total, (uint64_t)conv_dim, kBoxCh,
                      kTok, CU_TENSOR_MAP_SWIZZLE_NONE)) {
        set_error("kda_conv_silu_l2: cannot encode the TMA tensor map");
        return KDA_ERR_CUDA;
    }
    cudaError_t e = cudaFuncSetAttribute(conv_silu_l2_kernel<K>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kConvSmem);
    if (e != cudaSuccess) {
        set_error("kda_conv_silu_l2: cannot reserve shared memory: %s", cudaGetErrorString(e));
        return KDA_ERR_CUDA;
    }
    launch_pdl(conv_silu_l2_kernel<K>, dim3((unsigned)groups, (unsigned)spans), dim3(kThreads),
               kConvSmem, s, xmap, conv_state, x, w, out, total, t_per_seq, cu, n_seqs, heads,
               eps, (int)span);
    kda_status st = launch_result("kda_conv_silu_l2 (conv)");
    if (st != KDA_OK) return st;
    const size_t rows = (size_t)n_seqs * 3 * heads * D;
    // A plain launch: under programmatic dependent launch its CTAs became
    // resident while the conv grid still ran, and back-to-back calls on many
    // sequences (768 CTAs for 16) slowed from 656 to 821 us per call.
    conv_state_kernel<K><<<dim3((unsigned)((rows + 255) / 256)), dim3(256), 0, s>>>(
        conv_state, x, total, t_per_seq, cu, n_seqs, heads);
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

extern "C" kda_status kda_conv_silu_l2_k(float* conv_state, const uint16_t* x, const uint16_t* w,
                                         uint16_t* out, int n_seqs, int krows, int conv_kernel,
                                         float l2_eps, int heads, int head_dim,
                                         float* const* snapshots, int n_snap, uint64_t stream) {
    KDA_REQUIRE(krows >= 1 && krows <= KDA_MAX_K, KDA_ERR_INVALID_ARG,
                "kda_conv_silu_l2_k: k = %d outside [1, %d]", krows, KDA_MAX_K);
    KDA_REQUIRE(n_snap >= 0 && n_snap <= krows, KDA_ERR_INVALID_ARG,
                "kda_conv_silu_l2_k: n_snap = %d outside [0, k = %d]", n_snap, krows);
    KDA_REQUIRE(n_snap == 0 || snapshots, KDA_ERR_INVALID_ARG,
                "kda_conv_silu_l2_k: snapshots is NULL with n_snap = %d", n_snap);
    KDA_REQUIRE(conv_state && x && w && out, KDA_ERR_INVALID_ARG,
                "kda_conv_silu_l2_k: null pointer argument");
    KDA_REQUIRE(aligned16(conv_state) && aligned16(x) && aligned16(out), KDA_ERR_INVALID_ARG,
                "kda_conv_silu_l2_k: conv_state, x and out must be 16-byte aligned");
    KDA_REQUIRE(head_dim == D, KDA_ERR_UNSUPPORTED,
                "kda_conv_silu_l2_k: head_dim %d unsupported (only 128)", head_dim);
    KDA_REQUIRE(heads >= 1 && n_seqs >= 1, KDA_ERR_INVALID_ARG,
                "kda_conv_silu_l2_k: heads (%d) and n_seqs (%d) must be >= 1", heads, n_seqs);
    KDA_REQUIRE(conv_kernel >= 1 && conv_kernel <= KDA_MAX_CONV_KERNEL, KDA_ERR_UNSUPPORTED,
                "kda_conv_silu_l2_k: conv_kernel %d outside [1, %d]", conv_kernel,
                KDA_MAX_CONV_KERNEL);
    KDA_REQUIRE(l2_eps >= 0.f, KDA_ERR_INVALID_ARG, "kda_conv_silu_l2_k: l2_eps must be >= 0");
    const long long total = (long long)krows * n_seqs;
    KDA_REQUIRE(total <= 0x7fffffffLL && (long long)3 * heads * D * total < (1LL << 46),
                KDA_ERR_INVALID_ARG, "kda_conv_silu_l2_k: problem too large");
    ConvSnaps sn = {};
    for (int t = 0; t < n_snap; ++t) {
        KDA_REQUIRE(snapshots[t] && aligned16(snapshots[t]) && snapshots[t] != conv_state,
                    KDA_ERR_INVALID_ARG,
                    "kda_conv_silu_l2_k: snapshot %d is NULL, misaligned or the conv state", t);
        sn.p[t] = snapshots[t];
    }
    KDA_REQUIRE(!fault_injected(), KDA_ERR_CUDA, "kda_conv_silu_l2_k: injected launch failure");
    cudaStream_t s = as_stream(stream);
    const int tot = (int)total;
    switch (conv_kernel) {
        case 1: return launch<1>(conv_state, x, w, out, tot, krows, nullptr, n_seqs, heads, l2_eps, s, sn, n_snap);
        case 2: return launch<2>(conv_state, x, w, out, tot, krows, nullptr, n_seqs, heads, l2_eps, s, sn, n_snap);
        case 3: return launch<3>(conv_state, x, w, out, tot, krows, nullptr, n_seqs, heads, l2_eps, s, sn, n_snap);
        default: return launch<4>(conv_state, x, w, out, tot, krows, nullptr, n_seqs, heads, l2_eps, s, sn, n_snap);
    }
}
