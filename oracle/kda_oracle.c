/*
 * kda_oracle.c -- float64 CPU oracle for the Kimi Delta Attention (KDA) core
 * recurrence.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously-correct
 * definition that the CUDA library is checked against.  Only the tests, the
 * smoke check and the benchmark's CPU-baseline leg may load it.  It shares no
 * code, header, table or helper with the CUDA path and must never be linked
 * into it.
 *
 * Sources (web pages on the subject; none prints the recurrence as a formula,
 * so the formula below is their verbal description written out):
 *   [EN]  "Kimi K3 reconstructs long-context inference efficiency through KDA,
 *          cross-depth attention, and latent expert routing" (xxquant,
 *          English), section "Methodology notes":
 *            - "Memory update: DeltaNet and Delta Rule": the state is updated
 *              by minimising the L2 norm of the value-retrieval error;
 *            - "Memory control: Kimi Delta Attention": the forgetting factor
 *              of Gated DeltaNet becomes a diagonal matrix (per-channel
 *              decay); queries and keys are L2-normalised;
 *            - "System optimization: FlashKDA": the token recurrence unrolled
 *              into blocks (K1 tensor preparation, K2 blockwise recurrence).
 *          section "Key data": decode state is fp32, read and written once.
 *   [ZH2] "SemiAnalysis对月之暗面（Moonshot）发布的Kimi K3开源前沿模型进行了
 *          深度架构解读..." (zsxq post), section "一、Kimi Delta Attention
 *          （KDA）" (GDN forget gate alpha extended to a diagonal matrix; UT
 *          transform for chunk-level parallelism) and section "五、KV缓存效率
 *          与服务性能" (recurrent state saved every 32K tokens and at prompt
 *          boundaries).
 *
 * The recurrence, per sequence and head, with S a Dk x Dv state:
 *     qh = q / sqrt(sum q^2 + eps),  kh = k / sqrt(sum k^2 + eps)
 *     S' = Diag(exp g_t) S_{t-1}                  (per-channel decay of key rows)
 *     u  = v_t - S'^T kh                          (value-retrieval error)
 *     S_t = S' + beta_t kh u^T                    (= (I - b k k^T) Diag(a) S + b k v^T)
 *     o_t = S_t^T qh                              (reads the updated state)
 * The delta step is one gradient step with rate beta_t on
 * 0.5 * || S'^T kh - v_t ||^2, which is the [EN] "Memory update" description.
 *
 * Readings where the pages are silent: eps = 1e-6 inside the square root; no
 * query scale; g is the log-decay (alpha = exp g) applied before the delta
 * correction; a NULL initial state means zeros; checkpoint j of a sequence is
 * the state after its first j*stride tokens.
 *
 * Layouts (all contiguous, row-major):
 *   q, k, g : [T, H, Dk]     v, out : [T, H, Dv]     beta : [T, H]
 *   states  : [num_seqs, H, Dk, Dv]   ckpts : [n_ckpt, H, Dk, Dv]
 *   cu_seqlens : [num_seqs + 1], token offsets of the packed sequences.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define KDA_ORACLE_EPS 1e-6

/* y = x / sqrt(sum x^2 + eps): the L2 normalisation of [EN] "Memory control". */
static void l2_normalise(const double *x, double *y, int n)
{
    double ss = 0.0;
    for (int i = 0; i < n; ++i) ss += x[i] * x[i];
    double inv = 1.0 / sqrt(ss + KDA_ORACLE_EPS);
    for (int i = 0; i < n; ++i) y[i] = x[i] * inv;
}

/*
 * One token of the recurrence on state S (Dk x Dv, row-major), in place.
 * Writes o (Dv) if o != NULL.  Scratch: qh, kh (Dk), u (Dv).
 */
static void token_step(double *S, const double *q, const double *k, const double *v,
                       const double *g, double beta, int Dk, int Dv, double *o,
                       double *qh, double *kh, double *u)
{
    l2_normalise(q, qh, Dk);
    l2_normalise(k, kh, Dk);
    /* S' = Diag(exp g) S : decay scales the key rows. */
    for (int i = 0; i < Dk; ++i) {
        double a = exp(g[i]);
        for (int j = 0; j < Dv; ++j) S[(size_t)i * Dv + j] *= a;
    }
    /* u = v - S'^T kh */
    for (int j = 0; j < Dv; ++j) {
        double r = 0.0;
        for (int i = 0; i < Dk; ++i) r += S[(size_t)i * Dv + j] * kh[i];
        u[j] = v[j] - r;
    }
    /* S = S' + beta kh u^T */
    for (int i = 0; i < Dk; ++i) {
        double bk = beta * kh[i];
        for (int j = 0; j < Dv; ++j) S[(size_t)i * Dv + j] += bk * u[j];
    }
    /* o = S^T qh, on the updated state */
    if (o) {
        for (int j = 0; j < Dv; ++j) {
            double r = 0.0;
            for (int i = 0; i < Dk; ++i) r += S[(size_t)i * Dv + j] * qh[i];
            o[j] = r;
        }
    }
}

/* Number of checkpoints each sequence emits, and the slot offsets. Returns total. */
static int64_t ckpt_offsets(const int64_t *cu, int num_seqs, int stride, int64_t *first_slot)
{
    int64_t total = 0;
    for (int n = 0; n < num_seqs; ++n) {
        first_slot[n] = total;
        if (stride > 0) total += (cu[n + 1] - cu[n]) / stride;
    }
    return total;
}

/*
 * Token-by-token prefill over packed sequences.  Returns 0, or -1 if the
 * checkpoint buffer is too small (nothing is written in that case).
 */
int oracle_prefill(const double *q, const double *k, const double *v, const double *g,
                   const double *beta, const double *init_state, const int64_t *cu_seqlens,
                   int num_seqs, int H, int Dk, int Dv, double *out, double *final_state,
                   int ckpt_stride, double *ckpts, int64_t ckpt_capacity)
{
    int64_t *first = (int64_t *)malloc(sizeof(int64_t) * (size_t)(num_seqs > 0 ? num_seqs : 1));
    int64_t need = ckpt_offsets(cu_seqlens, num_seqs, ckpt_stride, first);
    if (ckpt_stride > 0 && need > ckpt_capacity) { free(first); return -1; }
    const size_t SS = (size_t)Dk * Dv;

#pragma omp parallel for collapse(2) schedule(dynamic)
    for (int n = 0; n < num_seqs; ++n) {
        for (int h = 0; h < H; ++h) {
            double *S = (double *)malloc(sizeof(double) * SS);
            double *qh = (double *)malloc(sizeof(double) * (size_t)Dk);
            double *kh = (double *)malloc(sizeof(double) * (size_t)Dk);
            double *u = (double *)malloc(sizeof(double) * (size_t)Dv);
            if (init_state) memcpy(S, init_state + ((size_t)n * H + h) * SS, sizeof(double) * SS);
            else memset(S, 0, sizeof(double) * SS);
            int64_t t0 = cu_seqlens[n], t1 = cu_seqlens[n + 1];
            for (int64_t t = t0; t < t1; ++t) {
                size_t th = (size_t)t * H + h;
                token_step(S, q + th * Dk, k + th * Dk, v + th * Dv, g + th * Dk, beta[th],
                           Dk, Dv, out ? out + th * Dv : NULL, qh, kh, u);
                int64_t done = t - t0 + 1;
                if (ckpt_stride > 0 && ckpts && done % ckpt_stride == 0) {
                    int64_t slot = first[n] + done / ckpt_stride - 1;
                    memcpy(ckpts + ((size_t)slot * H + h) * SS, S, sizeof(double) * SS);
                }
            }
            if (final_state) memcpy(final_state + ((size_t)n * H + h) * SS, S, sizeof(double) * SS);
            free(S); free(qh); free(kh); free(u);
        }
    }
    free(first);
    return 0;
}

/*
 * One decode step for N independent sequences: the same token body, applied
 * to state [N, H, Dk, Dv] in place.  q, k, g : [N, H, Dk]; v, out : [N, H, Dv];
 * beta : [N, H].  [EN] "Key data": constant cost per token, fp32 state read
 * and written once.
 */
void oracle_decode(const double *q, const double *k, const double *v, const double *g,
                   const double *beta, double *state, double *out, int N, int H, int Dk, int Dv)
{
    const size_t SS = (size_t)Dk * Dv;
#pragma omp parallel for schedule(static)
    for (long nh = 0; nh < (long)N * H; ++nh) {
        double *qh = (double *)malloc(sizeof(double) * (size_t)Dk);
        double *kh = (double *)malloc(sizeof(double) * (size_t)Dk);
        double *u = (double *)malloc(sizeof(double) * (size_t)Dv);
        token_step(state + (size_t)nh * SS, q + (size_t)nh * Dk, k + (size_t)nh * Dk,
                   v + (size_t)nh * Dv, g + (size_t)nh * Dk, beta[nh], Dk, Dv,
                   out ? out + (size_t)nh * Dv : NULL, qh, kh, u);
        free(qh); free(kh); free(u);
    }
}

/*
 * Gated DeltaNet with a scalar forget gate a_t (log-decay, one per token and
 * head), [ZH2] section "一": S_t = alpha_t (I - beta k k^T) S_{t-1} + beta k v^T,
 * o_t = S_t^T qh.  Written in that order (projection first, then the scalar
 * decay) so that it is an arrangement independent of token_step(); with g
 * constant over channels the two must agree.  a : [T, H].
 */
void oracle_gdn_prefill(const double *q, const double *k, const double *v, const double *a,
                        const double *beta, const double *init_state, const int64_t *cu_seqlens,
                        int num_seqs, int H, int Dk, int Dv, double *out, double *final_state)
{
    const size_t SS = (size_t)Dk * Dv;
#pragma omp parallel for collapse(2) schedule(dynamic)
    for (int n = 0; n < num_seqs; ++n) {
        for (int h = 0; h < H; ++h) {
            double *S = (double *)malloc(sizeof(double) * SS);
            double *qh = (double *)malloc(sizeof(double) * (size_t)Dk);
            double *kh = (double *)malloc(sizeof(double) * (size_t)Dk);
            double *ktS = (double *)malloc(sizeof(double) * (size_t)Dv);
            if (init_state) memcpy(S, init_state + ((size_t)n * H + h) * SS, sizeof(double) * SS);
            else memset(S, 0, sizeof(double) * SS);
            for (int64_t t = cu_seqlens[n]; t < cu_seqlens[n + 1]; ++t) {
                size_t th = (size_t)t * H + h;
                l2_normalise(q + th * Dk, qh, Dk);
                l2_normalise(k + th * Dk, kh, Dk);
                double al = exp(a[th]), b = beta[th];
                for (int j = 0; j < Dv; ++j) {
                    double r = 0.0;
                    for (int i = 0; i < Dk; ++i) r += kh[i] * S[(size_t)i * Dv + j];
                    ktS[j] = r;
                }
                const double *vv = v + th * Dv;
                for (int i = 0; i < Dk; ++i)
                    for (int j = 0; j < Dv; ++j) {
                        size_t ij = (size_t)i * Dv + j;
                        S[ij] = al * (S[ij] - b * kh[i] * ktS[j]) + b * kh[i] * vv[j];
                    }
                if (out) {
                    for (int j = 0; j < Dv; ++j) {
                        double r = 0.0;
                        for (int i = 0; i < Dk; ++i) r += S[(size_t)i * Dv + j] * qh[i];
                        out[th * Dv + j] = r;
                    }
                }
            }
            if (final_state) memcpy(final_state + ((size_t)n * H + h) * SS, S, sizeof(double) * SS);
            free(S); free(qh); free(kh); free(ktS);
        }
    }
}

/*
 * Chunked reformulation ([EN] "System optimization: FlashKDA"; [ZH2] "一":
 * chunk-level parallelism through the UT transform), in float64, chunk C.
 * Chunks restart at each sequence start; a partial last chunk uses only its
 * valid rows.  Per chunk with start state S0 and rows r = 0..L-1:
 *   K1: qh, kh; b_r = sum_{s<=r} g_s (per channel); gamma_r = exp(b_r)
 *       Qg = qh*gamma, Kg = kh*gamma, Kd = kh/gamma, Ke = kh*exp(b_{L-1} - b)
 *       Lmat[r][i] = beta_r (Kg_r . Kd_i) for i < r          (strictly lower)
 *       Tm = (I + Lmat)^-1                                    (UT transform)
 *       Wk = Tm diag(beta) Kg,  Uv = Tm diag(beta) V
 *       Mc[r][i] = Qg_r . Kd_i for i <= r                     (causal, inclusive)
 *   K2: W = Uv - Wk S0;  O = Qg S0 + Mc W;  S1 = Diag(gamma_{L-1}) S0 + Ke^T W
 * Tm is formed column by column by forward substitution on (I + Lmat).
 * Checkpoints are written at chunk ends that fall on multiples of stride
 * (stride must then be a multiple of C).
 */
int oracle_prefill_chunked(const double *q, const double *k, const double *v, const double *g,
                           const double *beta, const double *init_state,
                           const int64_t *cu_seqlens, int num_seqs, int H, int Dk, int Dv,
                           int C, double *out, double *final_state, int ckpt_stride,
                           double *ckpts, int64_t ckpt_capacity)
{
    if (C <= 0 || (ckpt_stride > 0 && ckpt_stride % C != 0)) return -2;
    int64_t *first = (int64_t *)malloc(sizeof(int64_t) * (size_t)(num_seqs > 0 ? num_seqs : 1));
    int64_t need = ckpt_offsets(cu_seqlens, num_seqs, ckpt_stride, first);
    if (ckpt_stride > 0 && need > ckpt_capacity) { free(first); return -1; }
    const size_t SS = (size_t)Dk * Dv;

#pragma omp parallel for collapse(2) schedule(dynamic)
    for (int n = 0; n < num_seqs; ++n) {
        for (int h = 0; h < H; ++h) {
            double *S = (double *)malloc(sizeof(double) * SS);
            double *Qg = (double *)malloc(sizeof(double) * (size_t)C * Dk);
            double *Kg = (double *)malloc(sizeof(double) * (size_t)C * Dk);
            double *Kd = (double *)malloc(sizeof(double) * (size_t)C * Dk);
            double *Ke = (double *)malloc(sizeof(double) * (size_t)C * Dk);
            double *b = (double *)malloc(sizeof(double) * (size_t)C * Dk);
            double *Lm = (double *)malloc(sizeof(double) * (size_t)C * C);
            double *Tm = (double *)malloc(sizeof(double) * (size_t)C * C);
            double *Mc = (double *)malloc(sizeof(double) * (size_t)C * C);
            double *Wk = (double *)malloc(sizeof(double) * (size_t)C * Dk);
            double *Uv = (double *)malloc(sizeof(double) * (size_t)C * Dv);
            double *W = (double *)malloc(sizeof(double) * (size_t)C * Dv);
            double *S1 = (double *)malloc(sizeof(double) * SS);
            double *qh = (double *)malloc(sizeof(double) * (size_t)Dk);
            double *kh = (double *)malloc(sizeof(double) * (size_t)Dk);
            if (init_state) memcpy(S, init_state + ((size_t)n * H + h) * SS, sizeof(double) * SS);
            else memset(S, 0, sizeof(double) * SS);
            int64_t t0 = cu_seqlens[n], len = cu_seqlens[n + 1] - t0;
            for (int64_t c0 = 0; c0 < len; c0 += C) {
                int L = (int)((len - c0) < C ? (len - c0) : C);
                /* K1: normalisation, cumulative log-decay, decayed q/k */
                for (int r = 0; r < L; ++r) {
                    size_t th = (size_t)(t0 + c0 + r) * H + h;
                    l2_normalise(q + th * Dk, qh, Dk);
                    l2_normalise(k + th * Dk, kh, Dk);
                    for (int d = 0; d < Dk; ++d) {
                        b[(size_t)r * Dk + d] = g[th * Dk + d] + (r > 0 ? b[(size_t)(r - 1) * Dk + d] : 0.0);
                        double gm = exp(b[(size_t)r * Dk + d]);
                        Qg[(size_t)r * Dk + d] = qh[d] * gm;
                        Kg[(size_t)r * Dk + d] = kh[d] * gm;
                        Kd[(size_t)r * Dk + d] = kh[d] / gm;
                    }
                }
                for (int r = 0; r < L; ++r) {
                    size_t th = (size_t)(t0 + c0 + r) * H + h;
                    l2_normalise(k + th * Dk, kh, Dk);
                    for (int d = 0; d < Dk; ++d)
                        Ke[(size_t)r * Dk + d] = kh[d] * exp(b[(size_t)(L - 1) * Dk + d] - b[(size_t)r * Dk + d]);
                }
                /* strictly-lower Lmat and inclusive-lower Mc */
                for (int r = 0; r < L; ++r) {
                    double br = beta[(size_t)(t0 + c0 + r) * H + h];
                    for (int i = 0; i < L; ++i) {
                        double kk = 0.0, qk = 0.0;
                        for (int d = 0; d < Dk; ++d) {
                            kk += Kg[(size_t)r * Dk + d] * Kd[(size_t)i * Dk + d];
                            qk += Qg[(size_t)r * Dk + d] * Kd[(size_t)i * Dk + d];
                        }
                        Lm[(size_t)r * C + i] = (i < r) ? br * kk : 0.0;
                        Mc[(size_t)r * C + i] = (i <= r) ? qk : 0.0;
                    }
                }
                /* Tm = (I + Lmat)^-1 by forward substitution, one column e_j at a time */
                for (int j = 0; j < L; ++j) {
                    for (int r = 0; r < L; ++r) {
                        double x = (r == j) ? 1.0 : 0.0;
                        for (int i = 0; i < r; ++i) x -= Lm[(size_t)r * C + i] * Tm[(size_t)i * C + j];
                        Tm[(size_t)r * C + j] = x;
                    }
                }
                /* Wk = Tm diag(beta) Kg ; Uv = Tm diag(beta) V */
                for (int r = 0; r < L; ++r) {
                    for (int d = 0; d < Dk; ++d) {
                        double s = 0.0;
                        for (int i = 0; i < L; ++i)
                            s += Tm[(size_t)r * C + i] * beta[(size_t)(t0 + c0 + i) * H + h] * Kg[(size_t)i * Dk + d];
                        Wk[(size_t)r * Dk + d] = s;
                    }
                    for (int e = 0; e < Dv; ++e) {
                        double s = 0.0;
                        for (int i = 0; i < L; ++i) {
                            size_t ti = (size_t)(t0 + c0 + i) * H + h;
                            s += Tm[(size_t)r * C + i] * beta[ti] * v[ti * Dv + e];
                        }
                        Uv[(size_t)r * Dv + e] = s;
                    }
                }
                /* K2: W = Uv - Wk S0 */
                for (int r = 0; r < L; ++r)
                    for (int e = 0; e < Dv; ++e) {
                        double s = 0.0;
                        for (int d = 0; d < Dk; ++d) s += Wk[(size_t)r * Dk + d] * S[(size_t)d * Dv + e];
                        W[(size_t)r * Dv + e] = Uv[(size_t)r * Dv + e] - s;
                    }
                /* O = Qg S0 + Mc W */
                if (out) {
                    for (int r = 0; r < L; ++r) {
                        size_t th = (size_t)(t0 + c0 + r) * H + h;
                        for (int e = 0; e < Dv; ++e) {
                            double s = 0.0;
                            for (int d = 0; d < Dk; ++d) s += Qg[(size_t)r * Dk + d] * S[(size_t)d * Dv + e];
                            for (int i = 0; i <= r; ++i) s += Mc[(size_t)r * C + i] * W[(size_t)i * Dv + e];
                            out[th * Dv + e] = s;
                        }
                    }
                }
                /* S1 = Diag(gamma_{L-1}) S0 + Ke^T W */
                for (int d = 0; d < Dk; ++d) {
                    double gl = exp(b[(size_t)(L - 1) * Dk + d]);
                    for (int e = 0; e < Dv; ++e) {
                        double s = gl * S[(size_t)d * Dv + e];
                        for (int r = 0; r < L; ++r) s += Ke[(size_t)r * Dk + d] * W[(size_t)r * Dv + e];
                        S1[(size_t)d * Dv + e] = s;
                    }
                }
                memcpy(S, S1, sizeof(double) * SS);
                int64_t done = c0 + L;
                if (ckpt_stride > 0 && ckpts && done % ckpt_stride == 0) {
                    int64_t slot = first[n] + done / ckpt_stride - 1;
                    memcpy(ckpts + ((size_t)slot * H + h) * SS, S, sizeof(double) * SS);
                }
            }
            if (final_state) memcpy(final_state + ((size_t)n * H + h) * SS, S, sizeof(double) * SS);
            free(S); free(Qg); free(Kg); free(Kd); free(Ke); free(b); free(Lm); free(Tm); free(Mc);
            free(Wk); free(Uv); free(W); free(S1); free(qh); free(kh);
        }
    }
    free(first);
    return 0;
}

/* Number of checkpoint slots the given packing needs (host cu_seqlens). */
int64_t oracle_ckpt_count(const int64_t *cu_seqlens, int num_seqs, int ckpt_stride)
{
    int64_t total = 0;
    if (ckpt_stride <= 0) return 0;
    for (int n = 0; n < num_seqs; ++n) total += (cu_seqlens[n + 1] - cu_seqlens[n]) / ckpt_stride;
    return total;
}

/* Threads the OpenMP runtime will use (for the CPU-baseline report). */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}
