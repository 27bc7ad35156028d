/*
 * kda_oracle.c -- plain FP64 CPU oracle for the KDA (gated delta-rule) core.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library links, includes or calls
 * this file; only the tests, the smoke check and the benchmark's CPU-baseline
 * leg load it.  It shares no code, header, table or constant with the CUDA
 * path.
 *
 * Source of the method: the rustdoc pages of the GLM-5.3-Flash KDA block
 * ("glm5next_kda" module index: the block pipeline and its invariants;
 * Glm5NextKdaLayer: decode / decode_k / prefill_with_pad_fill;
 * Glm5NextKdaKernels: chunk_prepare, chunk_scan, recurrent; config.rs:
 * recurrent_state_elems, an FP32 [heads, head_dim, head_dim] state laid out
 * K-major, conv_state_elems, and the L2 epsilon added under the square root).
 *
 * Notation.  D = head_dim, H = heads.  The state of one head is S[i][j], i the
 * key channel (row), j the value channel (column): "K-major" read as the key
 * index outer.  For one token with inputs q, k, v, g (length D), beta:
 *
 *     S[i][j] <- exp(g[i]) * S[i][j]                 (decay per key channel)
 *     u[j]     = v[j] - sum_i S[i][j] k[i]            (delta-rule residual)
 *     S[i][j] += beta * k[i] * u[j]                   (rank-1 update)
 *     o[j]     = sum_i S[i][j] * scale * q[i]         (read-out, updated S)
 *
 * with scale = 1/sqrt(D), the query scale this oracle fixes (the pages print
 * none).  Every function below is plain loops in double precision, compiled
 * without FP contraction so the result is the same on x86-64 and aarch64.
 *
 * Parity status: every function here is pinned by the CPU tests (closed forms,
 * special cases, brute force and a library-routine cross-check); the unpinned
 * choices are conventions the pages leave open: the value of the query scale,
 * and the formula of the forget gate (kda_oracle_gate, parity unpinned: its
 * inputs are on the pages, its formula is a reading).
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

double kda_oracle_default_q_scale(int head_dim) { return 1.0 / sqrt((double)head_dim); }

int kda_oracle_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* One token of the recurrence on one head (the per-token step of the
 * Glm5NextKdaLayer::decode call).  S is [D][D], in place; o is [D]. */
static void token_step(int D, double scale, const double* q, const double* k,
                       const double* v, const double* g, double beta, double* S,
                       double* o, double* u) {
    for (int i = 0; i < D; ++i) {
        double a = exp(g[i]);
        for (int j = 0; j < D; ++j) S[(size_t)i * D + j] *= a;
    }
    for (int j = 0; j < D; ++j) {
        double acc = 0.0;
        for (int i = 0; i < D; ++i) acc += S[(size_t)i * D + j] * k[i];
        u[j] = v[j] - acc;
    }
    for (int i = 0; i < D; ++i) {
        double bk = beta * k[i];
        for (int j = 0; j < D; ++j) S[(size_t)i * D + j] += bk * u[j];
    }
    for (int j = 0; j < D; ++j) {
        double acc = 0.0;
        for (int i = 0; i < D; ++i) acc += S[(size_t)i * D + j] * (scale * q[i]);
        o[j] = acc;
    }
}

/*
 * Token-by-token recurrence over N independent sequences of T tokens each.
 *   q, k, v, g : [N][T][H][D]      beta : [N][T][H]
 *   S          : [N][H][D][D]      in place (state before -> after token T-1)
 *   o          : [N][T][H][D]
 *   snaps      : NULL, or [T][N][H][D][D]: the state after token t
 *                (decode_k's snapshot t holds the state once row t is applied).
 * Single-token decode is T = 1; decode_k is T = k; a prefill is N = 1.
 */
void kda_oracle_recurrent(int N, int T, int H, int D, double scale, const double* q,
                          const double* k, const double* v, const double* g,
                          const double* beta, double* S, double* o, double* snaps) {
    const size_t dd = (size_t)D * D;
#pragma omp parallel for schedule(dynamic, 1)
    for (int nh = 0; nh < N * H; ++nh) {
        int n = nh / H, h = nh % H;
        double* u = (double*)malloc(sizeof(double) * D);
        double* Sh = S + (size_t)nh * dd;
        for (int t = 0; t < T; ++t) {
            size_t row = ((size_t)n * T + t) * H + h;
            token_step(D, scale, q + row * D, k + row * D, v + row * D, g + row * D,
                       beta[row], Sh, o + row * D, u);
            if (snaps) memcpy(snaps + (((size_t)t * N + n) * H + h) * dd, Sh, sizeof(double) * dd);
        }
        free(u);
    }
}

/*
 * Chunked form, intra-chunk part (Glm5NextKdaKernels::chunk_prepare, the
 * "kda_chunk (prefill)" stage of the block pipeline): everything about one
 * chunk of L tokens of one head that does not depend on the carried state.
 * Inputs are the chunk's rows: q, k, v, g [L][D] (row stride ld elements),
 * beta [L] (stride ldb).  Outputs (row-major, dense):
 *   Gam [L][D]  Gamma_r = sum_{s<=r} g_s                (cumulative log-decay)
 *   A   [L][L]  A_rs = beta_s sum_i k_ri k_si exp(Gamma_ri - Gamma_si), s < r
 *   Tm  [L][L]  (I + A)^-1, unit lower triangular
 *   W   [L][D]  Tm * Ktil,  Ktil_r = exp(Gamma_r) (.) k_r
 *   Ut  [L][D]  Tm * V
 *   P   [L][L]  P_rs = beta_s sum_i qh_ri k_si exp(Gamma_ri - Gamma_si), s <= r
 *   Qt  [L][D]  exp(Gamma_r) (.) qh_r,   qh = scale * q
 *   Kh  [L][D]  exp(Gamma_{L-1} - Gamma_s) (.) k_s
 *   dec [D]     exp(Gamma_{L-1})
 * Derivation: unrolling the token step over the chunk from a state S gives
 * u_r = v_r - S^T Ktil_r - sum_{s<r} A_rs u_s, i.e. (I + A) U = V - Ktil S.
 */
void kda_oracle_chunk_prepare(int L, int D, double scale, const double* q, const double* k,
                              const double* v, const double* g, const double* beta,
                              int ld, int ldb, double* Gam, double* A, double* Tm,
                              double* W, double* Ut, double* P, double* Qt, double* Kh,
                              double* dec) {
    for (int i = 0; i < D; ++i) {
        double acc = 0.0;
        for (int r = 0; r < L; ++r) {
            acc += g[(size_t)r * ld + i];
            Gam[(size_t)r * D + i] = acc;
        }
    }
    for (int r = 0; r < L; ++r)
        for (int s = 0; s < L; ++s) {
            double a = 0.0, p = 0.0;
            if (s <= r) {
                for (int i = 0; i < D; ++i) {
                    double e = exp(Gam[(size_t)r * D + i] - Gam[(size_t)s * D + i]);
                    double ks = k[(size_t)s * ld + i];
                    a += k[(size_t)r * ld + i] * ks * e;
                    p += scale * q[(size_t)r * ld + i] * ks * e;
                }
                a *= beta[(size_t)s * ldb];
                p *= beta[(size_t)s * ldb];
            }
            A[(size_t)r * L + s] = (s < r) ? a : 0.0;
            P[(size_t)r * L + s] = (s <= r) ? p : 0.0;
        }
    /* (I + A) Tm = I by forward substitution, one column at a time. */
    for (int c = 0; c < L; ++c)
        for (int r = 0; r < L; ++r) {
            double x = (r == c) ? 1.0 : 0.0;
            for (int s = 0; s < r; ++s) x -= A[(size_t)r * L + s] * Tm[(size_t)s * L + c];
            Tm[(size_t)r * L + c] = x;
        }
    for (int r = 0; r < L; ++r)
        for (int i = 0; i < D; ++i) {
            double gr = Gam[(size_t)r * D + i];
            Qt[(size_t)r * D + i] = exp(gr) * scale * q[(size_t)r * ld + i];
            Kh[(size_t)r * D + i] = exp(Gam[(size_t)(L - 1) * D + i] - gr) * k[(size_t)r * ld + i];
        }
    for (int i = 0; i < D; ++i) dec[i] = exp(Gam[(size_t)(L - 1) * D + i]);
    for (int r = 0; r < L; ++r)
        for (int i = 0; i < D; ++i) {
            double w = 0.0, ut = 0.0;
            for (int s = 0; s < L; ++s) {
                double t = Tm[(size_t)r * L + s];
                w += t * exp(Gam[(size_t)s * D + i]) * k[(size_t)s * ld + i];
                ut += t * v[(size_t)s * ld + i];
            }
            W[(size_t)r * D + i] = w;
            Ut[(size_t)r * D + i] = ut;
        }
}

/*
 * Chunked form, inter-chunk part (Glm5NextKdaKernels::chunk_scan): carries the
 * state of one head across one chunk.  S [D][D] in place; o [L][D] (row
 * stride ldo).
 *   U = Ut - W S;   O = Qt S + P U;   S <- diag(dec) S + Kh^T diag(beta) U
 */
void kda_oracle_chunk_scan(int L, int D, const double* W, const double* Ut, const double* P,
                           const double* Qt, const double* Kh, const double* dec,
                           const double* beta, int ldb, double* S, double* o, int ldo) {
    double* U = (double*)malloc(sizeof(double) * (size_t)L * D);
    for (int r = 0; r < L; ++r)
        for (int j = 0; j < D; ++j) {
            double acc = 0.0;
            for (int i = 0; i < D; ++i) acc += W[(size_t)r * D + i] * S[(size_t)i * D + j];
            U[(size_t)r * D + j] = Ut[(size_t)r * D + j] - acc;
        }
    for (int r = 0; r < L; ++r)
        for (int j = 0; j < D; ++j) {
            double acc = 0.0;
            for (int i = 0; i < D; ++i) acc += Qt[(size_t)r * D + i] * S[(size_t)i * D + j];
            for (int s = 0; s < L; ++s) acc += P[(size_t)r * L + s] * U[(size_t)s * D + j];
            o[(size_t)r * ldo + j] = acc;
        }
    for (int i = 0; i < D; ++i)
        for (int j = 0; j < D; ++j) {
            double acc = dec[i] * S[(size_t)i * D + j];
            for (int s = 0; s < L; ++s)
                acc += Kh[(size_t)s * D + i] * beta[(size_t)s * ldb] * U[(size_t)s * D + j];
            S[(size_t)i * D + j] = acc;
        }
    free(U);
}

/*
 * Chunked prefill of one sequence of T tokens, chunk width C: prepare + scan
 * chunk after chunk; the last chunk holds T - C*floor((T-1)/C) tokens.  Same
 * layouts as kda_oracle_recurrent with N = 1.  Used to pin the chunked
 * derivation against the recurrence; the result is the same up to rounding.
 */
void kda_oracle_chunked(int T, int H, int D, int C, double scale, const double* q,
                        const double* k, const double* v, const double* g,
                        const double* beta, double* S, double* o) {
#pragma omp parallel for schedule(dynamic, 1)
    for (int h = 0; h < H; ++h) {
        size_t LD = (size_t)C * D, LL = (size_t)C * C;
        double* buf = (double*)malloc(sizeof(double) * (5 * LD + 3 * LL + D));
        double *Gam = buf, *W = Gam + LD, *Ut = W + LD, *Qt = Ut + LD, *Kh = Qt + LD,
               *A = Kh + LD, *Tm = A + LL, *P = Tm + LL, *dec = P + LL;
        double* Sh = S + (size_t)h * D * D;
        for (int c0 = 0; c0 < T; c0 += C) {
            int L = (T - c0 < C) ? (T - c0) : C;
            size_t base = (size_t)c0 * H + h;
            int ld = H * D;
            kda_oracle_chunk_prepare(L, D, scale, q + base * D, k + base * D, v + base * D,
                                     g + base * D, beta + base, ld, H, Gam, A, Tm, W, Ut, P,
                                     Qt, Kh, dec);
            kda_oracle_chunk_scan(L, D, W, Ut, P, Qt, Kh, dec, beta + base, H, Sh,
                                  o + base * D, ld);
        }
        free(buf);
    }
}

/*
 * Depthwise causal conv1d + SiLU + L2 over the q and k channels (the front end
 * of the block pipeline: "conv1d + SiLU -> L2(q,k only)", fused at decode in
 * causal_conv1d_update_l2norm).  Channels: conv_dim = 3*H*D laid out q | k | v.
 *   x          : [T_total][conv_dim]     packed tokens of all sequences
 *   cu_seqlens : [N+1] token offsets of each sequence in x
 *   w          : [conv_dim][K]           tap K-1 multiplies the current token
 *   conv_state : [N][conv_dim][K]        in place; slot K-1 is the newest input
 *   out        : [T_total][conv_dim]
 * Per token and channel, as the decode kernel does it: shift the state left by
 * one slot, insert x into slot K-1, y = sum_j w[c][j] * state[c][j],
 * y <- y * sigmoid(y).  Then each q and k head (D channels) is scaled by
 * 1/sqrt(sum y^2 + l2_eps); v channels are left as they are.  A prefill is
 * this token step applied in order, which is its definition.
 */
void kda_oracle_conv_silu_l2(int N, const int* cu_seqlens, int H, int D, int K, double l2_eps,
                             const double* x, const double* w, double* conv_state,
                             double* out) {
    const int conv_dim = 3 * H * D;
    const int groups = 3 * H; /* one group = the D channels of one head */
#pragma omp parallel for schedule(dynamic, 1)
    for (int ng = 0; ng < N * groups; ++ng) {
        int n = ng / groups, grp = ng % groups;
        int normalise = grp < 2 * H; /* q heads then k heads */
        double* y = (double*)malloc(sizeof(double) * D);
        for (int t = cu_seqlens[n]; t < cu_seqlens[n + 1]; ++t) {
            double ss = 0.0;
            for (int d = 0; d < D; ++d) {
                int c = grp * D + d;
                double* st = conv_state + ((size_t)n * conv_dim + c) * K;
                for (int j = 0; j + 1 < K; ++j) st[j] = st[j + 1];
                st[K - 1] = x[(size_t)t * conv_dim + c];
                double acc = 0.0;
                for (int j = 0; j < K; ++j) acc += w[(size_t)c * K + j] * st[j];
                double sv = acc / (1.0 + exp(-acc));
                y[d] = sv;
                ss += sv * sv;
            }
            double inv = normalise ? 1.0 / sqrt(ss + l2_eps) : 1.0;
            for (int d = 0; d < D; ++d) out[(size_t)t * conv_dim + grp * D + d] = y[d] * inv;
        }
        free(y);
    }
}

/*
 * Sigmoid-gated RMSNorm of the core output (module index, block pipeline:
 * "sigmoid-gated RMSNorm(o_norm, g_b(g_a(h)))"; Glm5NextKdaWorkspace: core
 * [T, heads, head_dim] FP32 pre-norm, out_gate [T, qkv], o_norm_out [T, qkv];
 * config.rs: o_norm [head_dim], rms_norm_eps read by o_norm).  The pages fix
 * the inputs, not the formula; the reading taken here: per token and head,
 *     out[j] = core[j] / sqrt(mean_j core[j]^2 + eps) * w[j] * sigmoid(gate[j])
 * with the norm over the head's D channels and w shared by all heads.
 */
void kda_oracle_o_norm_gated(long rows, int H, int D, double eps, const double* core,
                             const double* gate, const double* w, double* out) {
#pragma omp parallel for schedule(static)
    for (long rh = 0; rh < rows * H; ++rh) {
        const double* y = core + (size_t)rh * D;
        double ss = 0.0;
        for (int d = 0; d < D; ++d) ss += y[d] * y[d];
        const double r = 1.0 / sqrt(ss / D + eps);
        for (int d = 0; d < D; ++d) {
            const double gt = gate[(size_t)rh * D + d];
            out[(size_t)rh * D + d] = y[d] * r * w[d] * (1.0 / (1.0 + exp(-gt)));
        }
    }
}

/*
 * Forget gate and beta of the core (module index, block pipeline:
 * "kda_gate / sigmoid(b_proj)"; Glm5NextKdaWorkspace: gate [T_pad, heads,
 * head_dim] FP32, the log-decay kda_gate produces, g_raw [T, qkv] the
 * forget-gate projection kda_gate reads, beta [T_pad, heads] stored after its
 * sigmoid; Glm5NextKdaWeights: dt_bias [heads * head_dim] one value per
 * channel, a_log [heads] one value per head; config.rs: gate_lower_bound).
 * The pages give the gate's inputs and that its result is a log-decay bounded
 * below by gate_lower_bound, not its formula (parity unpinned).  The reading
 * taken here, for channel c = h * D + d of row r:
 *     g[r][c]    = lb * sigmoid(exp(a_log[h]) * (g_raw[r][c] + dt_bias[c]))
 *     beta[r][h] = sigmoid(b[r][h])
 * so that lb < g < 0 for every finite input.
 */
void kda_oracle_gate(long rows, int H, int D, double lb, const double* g_raw,
                     const double* dt_bias, const double* a_log, const double* b,
                     double* g, double* beta) {
#pragma omp parallel for schedule(static)
    for (long r = 0; r < rows; ++r) {
        for (int h = 0; h < H; ++h) {
            const double rate = exp(a_log[h]);
            for (int d = 0; d < D; ++d) {
                const size_t c = (size_t)h * D + d;
                const double z = rate * (g_raw[(size_t)r * H * D + c] + dt_bias[c]);
                g[(size_t)r * H * D + c] = lb / (1.0 + exp(-z));
            }
            beta[(size_t)r * H + h] = 1.0 / (1.0 + exp(-b[(size_t)r * H + h]));
        }
    }
}
