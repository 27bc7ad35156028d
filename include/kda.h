/*
 * kda.h -- C ABI of libkda: the KDA (Kimi-style delta attention) core of the
 * GLM-5.3-Flash attention block on one GB300 (sm_103a).
 *
 * The method (rustdoc pages of the glm5next_kda module: the block pipeline
 * in the module index, Glm5NextKdaLayer's decode / decode_k / prefill /
 * prefill_with_pad_fill, Glm5NextKdaKernels' chunk_prepare / chunk_scan /
 * recurrent, and config.rs): per head, an FP32 state S[i][j] of
 * KDA_HEAD_DIM x KDA_HEAD_DIM, i = key channel (outer, "K-major"),
 * j = value channel.  For each token t with inputs q_t, k_t, v_t, g_t (one
 * value per key channel) and beta_t (one per head):
 *
 *     S[i][j] <- exp(g_t[i]) * S[i][j]
 *     u[j]     = v_t[j] - sum_i S[i][j] * k_t[i]
 *     S[i][j] += beta_t * k_t[i] * u[j]
 *     o_t[j]   = sum_i S[i][j] * (KDA_Q_SCALE * q_t[i])
 *
 * q and k arrive L2-normalised (kda_conv_silu_l2 produces them that way);
 * the core itself does not normalise.
 *
 * Conventions for every call:
 *  - Pointers are device pointers unless stated; buffers are caller-owned,
 *    contiguous in the stated layout and 16-byte aligned.  The library never
 *    allocates, frees or keeps a pointer after the call returns.
 *  - `stream` is a cudaStream_t cast to uint64_t (0 = legacy default stream).
 *    Work is enqueued and the call returns without synchronising.
 *  - Arguments are validated before anything is enqueued; on any error the
 *    call returns a non-zero kda_status, launches nothing, and
 *    kda_last_error() describes the problem.
 *  - Faults the host cannot see (malformed device-side cu_seqlens) are
 *    recorded in a device status word and reported by kda_sync_status().
 *  - Calls on one stream are ordered; calls that touch the same state buffer
 *    from different streams must be ordered by the caller.
 */
#ifndef KDA_H
#define KDA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Fixed geometry: head_dim is 128 (config.rs validate refuses any other). */
#define KDA_HEAD_DIM 128
/* The query scale 1/sqrt(KDA_HEAD_DIM), applied as q_hat = KDA_Q_SCALE * q in
 * FP32 before any use of q.  The pages print no scale; this is the library's
 * fixed reading (the conventional attention scale). */
#define KDA_Q_SCALE 0.08838834764831845f
/* decode_k row limit: Glm5NextKdaKernels::gemv_batchm serves 2..=8 rows. */
#define KDA_MAX_K 8
/* Depthwise conv taps: the conv kernels keep the window in 4 registers
 * (config.rs validate). */
#define KDA_MAX_CONV_KERNEL 4

typedef enum {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARG = 1, /* null / misaligned pointer, bad size or count    */
    KDA_ERR_UNSUPPORTED = 2, /* valid in principle, not built (head_dim, chunk) */
    KDA_ERR_WORKSPACE = 3,   /* workspace smaller than kda_prefill_workspace_size */
    KDA_ERR_CUDA = 4,        /* a CUDA runtime call or launch failed            */
    KDA_ERR_DEVICE = 5       /* device-side check failed (kda_sync_status)     */
} kda_status;

typedef enum { KDA_F32 = 0, KDA_BF16 = 1 } kda_dtype;

/*
 * kda_decode -- one token for each of n_seqs independent sequences
 * (Glm5NextKdaLayer::decode; Glm5NextKdaKernels::recurrent_smem, the 1R+1W
 * single-token recurrence).  Reads and writes the state exactly once.
 *
 *   state : FP32 [n_seqs][heads][128][128], updated in place
 *   q,k,v,g : FP32 [n_seqs][heads][128]      beta : FP32 [n_seqs][heads]
 *   o     : FP32 [n_seqs][heads][128], written
 *   heads >= 1, head_dim == 128, n_seqs >= 1.
 * The result is deterministic: the same inputs give the same bits.
 */
kda_status kda_decode(float* state, const float* q, const float* k, const float* v,
                      const float* g, const float* beta, float* o, int n_seqs, int heads,
                      int head_dim, uint64_t stream);

/*
 * kda_decode_k -- krows tokens of each of n_seqs sequences, walked in row
 * order with the state held on chip (Glm5NextKdaLayer::decode_k: the
 * speculative-verify row walk).  The output is bit-identical to krows serial
 * kda_decode calls on the same rows.
 *
 *   state : FP32 [n_seqs][heads][128][128], updated in place to the state
 *           after the last row
 *   q,k,v,g : FP32 [n_seqs][krows][heads][128]   beta : FP32 [n_seqs][krows][heads]
 *   o     : FP32 [n_seqs][krows][heads][128]
 *   snapshots : HOST array of n_snap device pointers; snapshots[t] (FP32
 *           [n_seqs][heads][128][128]) receives the state after row t.  Rows
 *           at or after n_snap write no snapshot (Glm5NextKdaLayer::decode_k).
 *           May be NULL when n_snap == 0.
 *   Refused: krows of 0 or less, or above KDA_MAX_K, the row capacity of the
 *   walk (Glm5NextKdaLayer::decode_k); n_snap < 0 or n_snap > krows; a null
 *   snapshot pointer.
 */
kda_status kda_decode_k(float* state, const float* q, const float* k, const float* v,
                        const float* g, const float* beta, float* o, int n_seqs, int krows,
                        int heads, int head_dim, float* const* snapshots, int n_snap,
                        uint64_t stream);

/*
 * kda_prefill -- chunked prefill from the carried state
 * (Glm5NextKdaLayer::prefill_with_pad_fill; Glm5NextKdaKernels::chunk_prepare
 * for the intra-chunk solve and cumulative decay, chunk_scan for the
 * inter-chunk state carry).
 *
 * Two batch forms:
 *  - cu_seqlens == NULL: n_seqs sequences of t valid tokens each, stored as
 *    [n_seqs][t_pad] token rows (t <= t_pad).  Rows [t, t_pad) of q, k, v, g
 *    and beta are the caller's padded tail, filled with pad_fill
 *    (Glm5NextKdaLayer::prefill_with_pad_fill): the library never writes them
 *    and never reads them into arithmetic, so o and the final state do not
 *    depend on their contents (NaN included).  pad_fill itself is not used.
 *  - cu_seqlens != NULL: DEVICE int32 [n_seqs + 1] offsets of n_seqs packed
 *    sequences; t is the total token count (== cu_seqlens[n_seqs]); t_pad
 *    must equal t and no fill happens.  Offsets are checked on the device
 *    (non-decreasing, cu_seqlens[0] == 0, last == t); a violation makes the
 *    kernel skip that sequence and sets KDA_ERR_DEVICE for kda_sync_status.
 *
 *   state : FP32 [n_seqs][heads][128][128], in place (state after the last
 *           valid token of each sequence)
 *   q,k,v : in_dtype, token row r of head h at ptr + r*qkv_row_stride + h*128
 *           (qkv_row_stride >= heads*128, in elements; lets q/k/v be views of
 *           one [T][3*heads*128] buffer such as kda_conv_silu_l2's output)
 *   g     : in_dtype [rows][heads][128]   beta : in_dtype [rows][heads]
 *   o     : FP32 [rows][heads][128]; rows of padding are not written
 *   chunk : 16, 32, 64 or 128 (config.rs chunk).  The chunked form equals the
 *           token recurrence for any width, up to rounding, so the width is a
 *           performance choice: the tensor-core kernels step 64 tokens at a
 *           time for every width, the SIMT kernel min(chunk, 64).
 *   in_dtype : KDA_F32 or KDA_BF16 (applies to q, k, v, g, beta)
 * Routing: inputs in the uniform form with t <= KDA_MAX_K and
 * qkv_row_stride == heads*128 run decode_k's row walk (the pages' dispatch
 * for pieces that do not take the chunked arm: state read once, t token steps
 * in FP32 arithmetic, BF16 inputs widened exactly, state written once); every
 * other call runs the tensor-core prepare and scan
 * kernels -- as one cooperative grid (the scan consuming each chunk as soon
 * as another SM has prepared it) when there are few (sequence, head) chains
 * relative to the SMs, e.g. one sequence of 32 heads.  FP32 inputs reach
 * those kernels through FP16 copies of q, k and v that a conversion kernel
 * writes into the workspace first; g and beta are read in FP32.  The
 * environment variable KDA_PREFILL_IMPL=simt pins the FP32 SIMT chunk kernel
 * (FP32 arithmetic throughout, no workspace) and KDA_PREFILL_IMPL=unfused the
 * two-kernel tensor-core path (for comparisons).
 * Precision of the tensor-core path: A and P from TF32 operands; the scan's
 * products from FP16 operands with FP32 accumulation; the state, T, the
 * decays and all sums in FP32.  FP32 inputs: q, k and v rounded to FP16 (11
 * significant bits, the precision of the TF32 and FP16 operands they feed),
 * g and beta exact.  Chunks whose steepest decay is below -10 form A and P on
 * the CUDA cores in FP32 (exact factors for any g).
 * Valid domain of the tensor-core path (the FP16 operands): q and k of unit
 * norm or less (as kda_conv_silu_l2 leaves them), and |v| and the entries of
 * the carried state below about 6e4 (FP16's largest value is 65504; larger
 * values turn into inf); values far below 2^-14 keep an absolute error under
 * 2^-25 but lose relative precision.  Inputs with v and the initial state
 * scaled by 1e-4 and by 1e3 are tested within the 2e-3 tolerance, BF16 and
 * FP32.  The row walk and the SIMT kernel have no such limits.
 *
 *   workspace : device scratch, 16-byte aligned, of at least
 *           kda_prefill_workspace_size(...) bytes (may be NULL when that
 *           size is 0).  Its contents on entry do not matter; calls that
 *           share one workspace must be ordered on the GPU.
 */
kda_status kda_prefill(float* state, const void* q, const void* k, const void* v,
                       const void* g, const void* beta, float* o,
                       int t, int t_pad, int chunk, float pad_fill, int heads, int head_dim,
                       int in_dtype, int64_t qkv_row_stride, const int* cu_seqlens, int n_seqs,
                       void* workspace, size_t workspace_bytes, uint64_t stream);

/* Bytes of device workspace kda_prefill needs for `rows` token rows in total
 * (n_seqs * t_pad in the uniform form, t in the packed form) over n_seqs
 * sequences with the given chunk width and input dtype.  Returns 0 when the
 * call needs none (KDA_PREFILL_IMPL=simt pins the SIMT kernel) or when an
 * argument is invalid.  The tensor-core path stores the state-independent
 * operands of every (chunk, head) there: 66,176 bytes per chunk of 64 tokens
 * and head (with one chunk of slack per sequence), plus (n_seqs + 1) * 4
 * bytes rounded up to 256, plus a 4-byte ready flag per chunk and head
 * rounded up to 256 bytes, plus n_seqs * 4 bytes rounded up to 256 (the order
 * in which a packed batch's chains start); FP32 inputs add, 256-byte aligned
 * after that, the
 * FP16 copies of q, k and v: 3 * rows * heads * 128 * 2 bytes.  (The row walk
 * of short FP32 sequences uses none of it.) */
size_t kda_prefill_workspace_size(int64_t rows, int n_seqs, int chunk, int heads, int head_dim,
                                  int in_dtype);

/*
 * kda_prefill_gated -- kda_prefill on the tensor-core path (BF16 q, k, v;
 * chunk 64) with the forget gate and beta formed inside the prepare kernel
 * from their raw inputs: the block pipeline's gate step (the forget gate and
 * the sigmoid of the b projection) fused into the core's g and beta loads (glm5next_kda module index;
 * Glm5NextKdaWeights dt_bias and a_log; config.rs gate_lower_bound).  Each
 * g element is read once, as BF16, and becomes
 *     g[r][h][i] = lb * sigmoid(exp(a_log[h]) * (g_raw[r][h*128 + i] + dt_bias[h*128 + i]))
 *     beta[r][h] = sigmoid(b_raw[r][h])
 * in FP32 (the hardware 2^x and 1/x; the same operations, in the same order,
 * as kda_gate's FP32 output), never stored.  The pages give the gate's inputs
 * and its bound, not this formula: it is the reading kda_gate states.
 *
 *   state, q, k, v, o, t, t_pad, heads, head_dim, qkv_row_stride,
 *   cu_seqlens, n_seqs : as kda_prefill (q, k, v BF16); in the uniform form
 *           rows [t, t_pad) are not written to (no pad fill) and never read
 *           into arithmetic
 *   g_raw : BF16, token row r at g_raw + r * g_raw_stride, head h's channels
 *           at + h*128 (g_raw_stride >= heads*128, a multiple of 8)
 *   dt_bias : FP32 [heads*128]      a_log : FP32 [heads]
 *   gate_lower_bound : finite and negative
 *   b_raw : BF16, token row r at b_raw + r * b_stride (b_stride >= heads)
 *   workspace : at least kda_prefill_workspace_size(rows, n_seqs, 64, heads,
 *           128, KDA_BF16) bytes, 16-byte aligned (never NULL)
 * Refused (nothing launched): null pointers, misaligned state/q/k/v/g_raw/o,
 * head_dim != 128, strides out of range, a gate_lower_bound that is not
 * finite and negative, too small a workspace.  Device-side cu_seqlens checks
 * and KDA_PREFILL_IMPL=unfused are as for kda_prefill; KDA_PREFILL_IMPL=simt
 * does not apply (this call has no SIMT form), and while it is set
 * kda_prefill_workspace_size answers 0 for the SIMT kernel, so size the
 * workspace without it.
 */
kda_status kda_prefill_gated(float* state, const void* q, const void* k, const void* v,
                             const uint16_t* g_raw, int64_t g_raw_stride, const float* dt_bias,
                             const float* a_log, float gate_lower_bound, const uint16_t* b_raw,
                             int64_t b_stride, float* o, int t, int t_pad, int heads,
                             int head_dim, int64_t qkv_row_stride, const int* cu_seqlens,
                             int n_seqs, void* workspace, size_t workspace_bytes,
                             uint64_t stream);

/*
 * kda_conv_silu_l2 -- depthwise causal conv1d + SiLU, then L2 over the q and k
 * channels (the block pipeline's front end: causal conv1d and SiLU, then L2
 * normalisation of the q and k channels only;
 * causal_conv1d_update_l2norm at decode, conv_prefill + l2_norm_bf16 at
 * prefill; config.rs: the L2 epsilon is applied as 1/sqrt(sum + eps)).
 *
 * Channels: conv_dim = 3*heads*128, laid out q | k | v.  Per sequence and
 * channel the conv state holds conv_kernel slots, slot conv_kernel-1 the
 * newest input; each token shifts it left, inserts x, and convolves:
 * y = sum_j w[c][j] * state[c][j]; y <- y * sigmoid(y).  Each q and k head is
 * then scaled by 1/sqrt(sum y^2 + l2_eps); v channels are not normalised.
 *
 *   conv_state : FP32 [n_seqs][conv_dim][conv_kernel], in place
 *   x          : BF16 [tokens][conv_dim]     out : BF16 [tokens][conv_dim]
 *   w          : BF16 [conv_dim][conv_kernel]
 *   cu_seqlens == NULL: n_seqs sequences of t tokens each, packed
 *       ([n_seqs][t][conv_dim]); decode is t == 1.
 *   cu_seqlens != NULL: DEVICE int32 [n_seqs + 1] offsets, t = total tokens;
 *       checked on the device like kda_prefill's.
 *   1 <= conv_kernel <= KDA_MAX_CONV_KERNEL.
 * With cu_seqlens == NULL and t <= KDA_MAX_K (decode and other short uniform
 * batches) one kernel is enqueued: each thread carries 8 channels of one
 * sequence through its t rows and rewrites that sequence's state rows itself.
 * Otherwise two: the conv over spans of tokens (reads the old state) and the
 * state update (writes the last conv_kernel inputs of each sequence).  Both
 * forms give the same bits for the same tokens.
 */
kda_status kda_conv_silu_l2(float* conv_state, const uint16_t* x, const uint16_t* w,
                            uint16_t* out, int t, int n_seqs, const int* cu_seqlens,
                            int conv_kernel, float l2_eps, int heads, int head_dim,
                            uint64_t stream);

/*
 * kda_gate -- the forget gate and beta of the core, the block pipeline's step
 * before it (the forget gate and the sigmoid of the b projection,
 * glm5next_kda module index;
 * Glm5NextKdaWorkspace g_raw [T, qkv], the forget-gate projection that
 * kda_gate reads, gate [T_pad, heads, head_dim], the log-decay it produces,
 * bounded below, and beta [T_pad, heads], stored after its sigmoid;
 * Glm5NextKdaWeights dt_bias
 * [heads * head_dim] F32 one per channel, a_log [heads] F32 one per head;
 * config.rs gate_lower_bound).  The pages give these inputs and that the
 * decay is bounded below by gate_lower_bound, not the formula; this library's
 * reading, for channel c = h * 128 + i of token row r:
 *     g[r][h][i] = gate_lower_bound * sigmoid(exp(a_log[h]) * (g_raw[r][c] + dt_bias[c]))
 *     beta[r][h] = sigmoid(b_raw[r][h])
 * in FP32, rounded once to out_dtype; gate_lower_bound < g < 0.  The results
 * are kda_prefill's g and beta (in_dtype = out_dtype) or, in FP32, decode's.
 *
 *   g_raw        : BF16 [rows][g_raw_stride], channels in the first heads*128
 *                  columns (16-byte aligned; g_raw_stride a multiple of 8)
 *   dt_bias      : FP32 [heads * 128] (16-byte aligned)
 *   a_log        : FP32 [heads]
 *   b_raw        : BF16 [rows][b_stride], the b_proj output in the first heads
 *                  columns
 *   g_out        : [rows][heads][128] of out_dtype (16-byte aligned)
 *   beta_out     : [rows][heads] of out_dtype
 *   out_dtype    : KDA_F32 or KDA_BF16
 *   rows >= 0 (0 launches nothing and the pointers may then be NULL),
 *   heads >= 1, head_dim == 128, gate_lower_bound finite and negative.
 * One kernel is enqueued on `stream`; the outputs may not alias the inputs.
 */
kda_status kda_gate(const uint16_t* g_raw, int64_t g_raw_stride, const float* dt_bias,
                    const float* a_log, float gate_lower_bound, const uint16_t* b_raw,
                    int64_t b_stride, void* g_out, void* beta_out, int out_dtype, int64_t rows,
                    int heads, int head_dim, uint64_t stream);

/*
 * kda_o_norm_gated -- sigmoid-gated RMSNorm of the core output, the block
 * pipeline's step after the core (an RMSNorm with the o_norm weight, gated by
 * the sigmoid of a two-stage projection of the hidden state, glm5next_kda
 * module index; Glm5NextKdaWorkspace core,
 * out_gate and o_norm_out; config.rs o_norm [head_dim] BF16, rms_norm_eps).
 * Per token row and head, over the head's 128 channels j:
 *     out[j] = core[j] / sqrt(mean_j core[j]^2 + eps) * w[j] * sigmoid(gate[j])
 * computed in FP32, rounded once to BF16 (the pages fix the inputs and the
 * sigmoid gate; the exact composition is this library's reading).
 *
 *   core : FP32 [rows][heads][128], e.g. kda_prefill's o or kda_decode's o
 *          (16-byte aligned)
 *   gate : BF16 [rows][heads * 128], the output-gate projection (8-byte aligned)
 *   w    : BF16 [128], shared by all heads (8-byte aligned)
 *   out  : BF16 [rows][heads * 128] (8-byte aligned); may not alias core
 *   rows >= 0 (0 launches nothing and the pointers may then be NULL),
 *   heads >= 1, head_dim == 128, eps >= 0.
 * One kernel is enqueued on `stream`.
 */
kda_status kda_o_norm_gated(const float* core, const uint16_t* gate, const uint16_t* w,
                            uint16_t* out, int64_t rows, int heads, int head_dim, float eps,
                            uint64_t stream);

/*
 * kda_prefill_o_norm -- kda_prefill with the sigmoid-gated RMSNorm of
 * kda_o_norm_gated fused into the scan's epilogue: the core output never
 * leaves the chip in FP32; what is written is the BF16 normalised output
 * (glm5next_kda module index, block pipeline: the core, then the gated
 * RMSNorm with the o_norm weight; Glm5NextKdaWorkspace core and o_norm_out).
 * Per token row and head, over the head's 128 channels j:
 *     out[j] = o[j] / sqrt(mean_j o[j]^2 + eps) * w[j] * sigmoid(gate[j])
 * with o the core output kda_prefill would write, in FP32, rounded once to
 * BF16 (the same reading as kda_o_norm_gated).
 *
 *   state, q, k, v, g, beta, t, t_pad, chunk, heads, head_dim, qkv_row_stride,
 *   cu_seqlens, n_seqs, workspace, workspace_bytes: as kda_prefill (the same
 *           argument checks, statuses and workspace size); in_dtype must be
 *           KDA_BF16: the fused norm exists on the tensor-core path only
 *           (KDA_ERR_UNSUPPORTED otherwise, and with KDA_PREFILL_IMPL=simt).
 *   gate  : BF16, token row r of head h at gate + r * gate_stride + h * 128
 *           (16-byte aligned, gate_stride >= heads * 128, a multiple of 8)
 *   w_norm: BF16 [128], shared by all heads (8-byte aligned)
 *   eps   : rms_norm_eps, finite and >= 0
 *   out   : BF16, token row r of head h at out + r * out_stride + h * 128
 *           (16-byte aligned, out_stride >= heads * 128, a multiple of 8);
 *           rows of padding are not written
 */
kda_status kda_prefill_o_norm(float* state, const void* q, const void* k, const void* v,
                              const void* g, const void* beta, const uint16_t* gate,
                              int64_t gate_stride, const uint16_t* w_norm, float eps,
                              uint16_t* out, int64_t out_stride, int t, int t_pad, int chunk,
                              int heads, int head_dim, int in_dtype, int64_t qkv_row_stride,
                              const int* cu_seqlens, int n_seqs, void* workspace,
                              size_t workspace_bytes, uint64_t stream);

/*
 * kda_conv_silu_l2_k -- the front end's half of decode_k: k rows of each of
 * n_seqs sequences through the conv + SiLU + L2 of kda_conv_silu_l2, with
 * optional conv-state snapshots (Glm5NextKdaLayer::decode_k: snapshots[t] is
 * the pair (h_dst, conv_dst) receiving the state after row t; kda_decode_k
 * fills h_dst, this call conv_dst).  Rows are walked in order, so the output
 * and the final conv state equal k single-token kda_conv_silu_l2 calls bit
 * for bit, and snapshots[t] equals the conv state after the t + 1-th.
 *
 *   conv_state : FP32 [n_seqs][conv_dim][conv_kernel], in place
 *   x, out     : BF16 [n_seqs][krows][conv_dim];  w : BF16 [conv_dim][conv_kernel]
 *   snapshots  : HOST array of n_snap DEVICE pointers, each FP32
 *                [n_seqs][conv_dim][conv_kernel], 16-byte aligned, distinct from
 *                conv_state (read on the host during the call only)
 *   1 <= krows <= KDA_MAX_K; 0 <= n_snap <= krows; other limits as
 *   kda_conv_silu_l2.  One kernel is enqueued (kda_conv_silu_l2's short-rows
 *   form, which also writes the snapshots).
 */
kda_status kda_conv_silu_l2_k(float* conv_state, const uint16_t* x, const uint16_t* w,
                              uint16_t* out, int n_seqs, int krows, int conv_kernel, float l2_eps,
                              int heads, int head_dim, float* const* snapshots, int n_snap,
                              uint64_t stream);

/* Size of the library-owned device array kda_prefill_static_ws uses as its
 * workspace: 64 MiB on every GPU that loads the library, held until exit. */
#define KDA_STATIC_WORKSPACE_BYTES (64u << 20)

/*
 * kda_prefill_static_ws -- kda_prefill without a caller workspace: the
 * workspace is a fixed array of KDA_STATIC_WORKSPACE_BYTES that the library
 * owns, so the call allocates nothing and the caller passes only inputs and
 * outputs.  The source pages have no counterpart; it serves callers that
 * cannot allocate device memory themselves, such as a plugin that receives
 * only input and output pointers from its host application, or a serving
 * loop that forbids cudaMalloc because it can synchronise the device.
 *
 *   Arguments, layouts and results are those of kda_prefill, and so are its
 *   refusals of invalid arguments (checked first, with the same statuses).
 *   Refused with KDA_ERR_WORKSPACE when kda_prefill_workspace_size(...) for
 *   the call exceeds KDA_STATIC_WORKSPACE_BYTES: at 32 heads that is 30
 *   chunks of 64 tokens in total (one BF16 sequence of up to 1,920 tokens;
 *   17 chunks, 1,088 tokens, for FP32 inputs, whose FP16 copies sit there
 *   too); fewer heads allow proportionally more.
 *   The first call on a device resolves the array's device address for that
 *   device (cudaGetSymbolAddress, with the device current); make that first
 *   call before any stream capture.
 *   All calls on a device share the one array and it keeps the last call's
 *   contents; nothing in it needs to start at zero (each call rewrites what it
 *   reads).  Calls that overlap on the GPU (other streams, other threads)
 *   race on it: order them.
 */
kda_status kda_prefill_static_ws(float* state, const void* q, const void* k, const void* v,
                                 const void* g, const void* beta, float* o, int t, int t_pad,
                                 int chunk, float pad_fill, int heads, int head_dim, int in_dtype,
                                 int64_t qkv_row_stride, const int* cu_seqlens, int n_seqs,
                                 uint64_t stream);

/* Synchronises `stream`, then reads and clears the device status words of the
 * calling thread's current device.  Returns KDA_OK, KDA_ERR_DEVICE (a
 * device-side check failed since the last call; kda_last_error says which),
 * or KDA_ERR_CUDA (the stream reported an error). */
kda_status kda_sync_status(uint64_t stream);

/* Thread-local description of the last error returned on this thread. */
const char* kda_last_error(void);

/* Library version string. */
const char* kda_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H */
