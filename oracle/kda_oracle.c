/*
 * kda_oracle.c -- plain, slow, double-precision CPU oracle for the KDA mixer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or calls
 * this file: only the tests, the package's smoke check and the benchmark's CPU
 * baseline leg do.  It shares no code, header, table or constant with the CUDA
 * library under hybrid_linear_attention_rule_gb300/csrc.
 *
 * What it computes (sources, by page title and section):
 *   - "Experimental Native Vulkan Backend for Kimi K3" (Hugging Face discussion
 *     #187), feature list: independent Q/K/V short convolutions, recurrent KDA
 *     state, KDA output gating.
 *   - metrale_model_arch::kimi_k3 docs, Structs: KdaConfig ("production is
 *     128/4": head dim 128, conv width 4) and KdaState ("both buffers are FP32,
 *     read-modify-write": the recurrent state and the conv state);
 *     Constants: KDA_L2_EPS (the eps of the in-kernel q/k L2 norm; the page
 *     gives no number, the value used is passed in by the caller);
 *     Functions: kda_decode_token ("conv update then recurrent step").
 *   - The KDA (Kimi Delta Attention) gated delta rule itself, which none of the
 *     pages writes out: per head a state S (dk x dv) evolves as
 *         S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T,
 *         o_t = scale * S_t^T q_t,      alpha_t = exp(g_t)   (per channel),
 *     and the mixer output is o_t * sigmoid(gate_t) when a gate is given.
 *
 * Readings where the pages are silent:
 *   conv: depthwise, no bias, w[c, W-1] multiplies the current token, history
 *         before a sequence start comes from the conv state (oldest row first)
 *         or is zero; SiLU after the conv; the conv state keeps the last W-1
 *         PRE-conv inputs.
 *   norm: x * (sum x^2 + eps)^(-1/2) over dk, for q and k, after conv+SiLU.
 *   decay: natural log; decay applied before the delta-rule erase; the output
 *         reads the updated state.
 *   varlen: state, conv history and chunking restart at every cu_seqlens
 *         boundary.
 *
 * Layouts (row-major, last index fastest):
 *   q, k [T, H, dk]; v [T, H, dv]; g [T, H, dk]; beta [T, H]; gate [T, H, dv];
 *   states [N, H, dk, dv]; o [T, H, dv]; conv weights [D, W];
 *   conv state [N, W-1, D].
 *
 * Every entry returns 0 on success and -1 on an invalid argument.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static double sigm(double z) { return 1.0 / (1.0 + exp(-z)); }

static int check_cu(const int *cu, int N, int T)
{
    if (!cu || N < 0 || T < 0 || cu[0] != 0 || cu[N] != T) return -1;
    for (int n = 0; n < N; ++n)
        if (cu[n + 1] < cu[n]) return -1;
    return 0;
}

int kda_oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Causal depthwise short convolution over packed sequences.
 *   y[t, c] = act( sum_{i=0}^{W-1} w[c, i] * x[t - (W-1) + i, c] )
 * where positions before the sequence start read the conv state (row W-1+tau
 * for offset tau < 0) or zero.  When cs_out is given it receives the last W-1
 * pre-conv inputs of each sequence, oldest first (shifting in the old state
 * when the sequence is shorter than W-1).  cs_in and cs_out may alias. */
int kda_oracle_short_conv(const double *x, const double *w, const double *cs_in,
                          const int *cu, int N, int T, int D, int W, int apply_silu,
                          double *y, double *cs_out)
{
    if (check_cu(cu, N, T) || D <= 0 || W <= 0 || !x || !w || !y) return -1;
    const int R = W - 1;
    double *hist = NULL;
    if (R > 0 && cs_in) {
        hist = (double *)malloc(sizeof(double) * (size_t)N * R * D);
        if (!hist) return -1;
        memcpy(hist, cs_in, sizeof(double) * (size_t)N * R * D);
    }
    for (int n = 0; n < N; ++n) {
        const long s = cu[n];
        const long L = cu[n + 1] - cu[n];
        for (long t = 0; t < L; ++t) {
            for (int c = 0; c < D; ++c) {
                double acc = 0.0;
                for (int i = 0; i < W; ++i) {
                    long tau = t - R + i;
                    double xv;
                    if (tau >= 0) xv = x[(s + tau) * D + c];
                    else xv = hist ? hist[((size_t)n * R + (R + tau)) * D + c] : 0.0;
                    acc += w[(size_t)c * W + i] * xv;
                }
                y[(s + t) * D + c] = apply_silu ? acc * sigm(acc) : acc;
            }
        }
        if (cs_out) {
            for (int r = 0; r < R; ++r) {
                long tau = L - R + r;
                for (int c = 0; c < D; ++c) {
                    double xv;
                    if (tau >= 0) xv = x[(s + tau) * D + c];
                    else xv = hist ? hist[((size_t)n * R + (R + tau)) * D + c] : 0.0;
                    cs_out[((size_t)n * R + r) * D + c] = xv;
                }
            }
        }
    }
    free(hist);
    return 0;
}

/* In-place L2 normalisation of R rows of length d: x <- x / sqrt(sum x^2 + eps). */
int kda_oracle_l2norm(double *x, long R, int d, double eps)
{
    if (!x || R < 0 || d <= 0) return -1;
    for (long r = 0; r < R; ++r) {
        double ss = 0.0;
        for (int c = 0; c < d; ++c) ss += x[r * d + c] * x[r * d + c];
        double inv = 1.0 / sqrt(ss + eps);
        for (int c = 0; c < d; ++c) x[r * d + c] *= inv;
    }
    return 0;
}

/* Per-token recurrence, the definition itself.  For each token:
 *   S <- Diag(alpha) S;  u = S^T k;  S <- S + beta k (v - u)^T;  o = scale S^T q.
 * The middle two lines are (I - beta k k^T) applied to Diag(alpha) S plus
 * beta k v^T, written as a rank-1 update. */
int kda_oracle_recurrent(const double *q, const double *k, const double *v,
                         const double *g, const double *beta, const double *S0,
                         const double *gate, const int *cu, int N, int T, int H,
                         int dk, int dv, double scale, double *o, double *Sfin)
{
    if (check_cu(cu, N, T) || H <= 0 || dk <= 0 || dv <= 0) return -1;
    if (!q || !k || !v || !g || !beta || !o) return -1;
    int bad = 0;
#pragma omp parallel for collapse(2) schedule(dynamic)
    for (int n = 0; n < N; ++n) {
        for (int h = 0; h < H; ++h) {
            double *S = (double *)malloc(sizeof(double) * (size_t)dk * dv);
            double *u = (double *)malloc(sizeof(double) * (size_t)dv);
            if (!S || !u) {
                free(S); free(u);
#pragma omp atomic write
                bad = 1;
                continue;
            }
            const size_t so = ((size_t)n * H + h) * dk * dv;
            for (size_t e = 0; e < (size_t)dk * dv; ++e) S[e] = S0 ? S0[so + e] : 0.0;
            for (long t = cu[n]; t < cu[n + 1]; ++t) {
                const double *qt = q + ((size_t)t * H + h) * dk;
                const double *kt = k + ((size_t)t * H + h) * dk;
                const double *gt = g + ((size_t)t * H + h) * dk;
                const double *vt = v + ((size_t)t * H + h) * dv;
                const double bt = beta[(size_t)t * H + h];
                for (int c = 0; c < dk; ++c) {
                    const double a = exp(gt[c]);
                    for (int j = 0; j < dv; ++j) S[(size_t)c * dv + j] *= a;
                }
                for (int j = 0; j < dv; ++j) u[j] = 0.0;
                for (int c = 0; c < dk; ++c)
                    for (int j = 0; j < dv; ++j) u[j] += S[(size_t)c * dv + j] * kt[c];
                for (int c = 0; c < dk; ++c) {
                    const double bk = bt * kt[c];
                    for (int j = 0; j < dv; ++j) S[(size_t)c * dv + j] += bk * (vt[j] - u[j]);
                }
                double *ot = o + ((size_t)t * H + h) * dv;
                for (int j = 0; j < dv; ++j) u[j] = 0.0;
                for (int c = 0; c < dk; ++c)
                    for (int j = 0; j < dv; ++j) u[j] += S[(size_t)c * dv + j] * qt[c];
                for (int j = 0; j < dv; ++j) {
                    double r = scale * u[j];
                    if (gate) r *= sigm(gate[((size_t)t * H + h) * dv + j]);
                    ot[j] = r;
                }
            }
            if (Sfin)
                for (size_t e = 0; e < (size_t)dk * dv; ++e) Sfin[so + e] = S[e];
            free(S);
            free(u);
        }
    }
    return bad ? -1 : 0;
}

/* Reverse-mode derivative of the recurrence above, without the gate ("native forward +
 * backward" in the feature list of "Experimental Native Vulkan Backend for Kimi K3", Hugging
 * Face discussion #187, names the backward; none of the pages writes it out, so this is the
 * derivative of the definition, by the chain rule, token by token).  Given dO (the gradient
 * of a loss with respect to o = scale S_t^T q_t) and dSfin (with respect to each sequence's
 * final state; may be null), it returns the gradients with respect to q, k, v, g, beta and
 * the initial state.  The forward states S_0 .. S_L of a sequence are kept for the reverse
 * sweep.  For t = L .. 1, with P = Diag(alpha_t) S_{t-1}, u = v_t - P^T k_t and G the gradient
 * reaching S_t (dSfin before the last token):
 *   G  += scale q_t dO_t^T              (o_t reads S_t)
 *   gq  = scale S_t dO_t
 *   h   = G^T k_t;   gv = beta_t h;   gbeta = h . u
 *   gk  = beta_t (G u - P h)            (S_t = P + beta k u^T with u depending on k)
 *   dP  = G - beta_t k_t h^T;   gg[c] = sum_j P[c][j] dP[c][j]   (dP/dg = P row-wise)
 *   G   = Diag(alpha_t) dP              (the gradient reaching S_{t-1})
 * and after the sweep G is the initial-state gradient.  Tiny inputs only. */
int kda_oracle_recurrent_backward(const double *q, const double *k, const double *v, const double *g,
                                  const double *beta, const double *S0, const double *dO, const double *dSfin,
                                  const int *cu, int N, int T, int H, int dk, int dv, double scale,
                                  double *gq, double *gk, double *gv, double *gg, double *gbeta, double *gS0)
{
    if (check_cu(cu, N, T) || H <= 0 || dk <= 0 || dv <= 0) return -1;
    if (!q || !k || !v || !g || !beta || !dO || !gq || !gk || !gv || !gg || !gbeta || !gS0) return -1;
    const size_t M = (size_t)dk * dv;
    int bad = 0;
#pragma omp parallel for collapse(2) schedule(dynamic)
    for (int n = 0; n < N; ++n) {
        for (int h = 0; h < H; ++h) {
            const long L = cu[n + 1] - cu[n];
            double *S = (double *)malloc(sizeof(double) * M * (size_t)(L + 1));
            double *G = (double *)malloc(sizeof(double) * M);
            double *P = (double *)malloc(sizeof(double) * M);
            double *u = (double *)malloc(sizeof(double) * dv);
            double *hv = (double *)malloc(sizeof(double) * dv);
            if (!S || !G || !P || !u || !hv) {
                free(S); free(G); free(P); free(u); free(hv);
#pragma omp atomic write
                bad = 1;
                continue;
            }
            const size_t so = ((size_t)n * H + h) * M;
            for (size_t e = 0; e < M; ++e) S[e] = S0 ? S0[so + e] : 0.0;
            /* forward, keeping every state */
            for (long i = 0; i < L; ++i) {
                const long t = cu[n] + i;
                const double *kt = k + ((size_t)t * H + h) * dk, *gt = g + ((size_t)t * H + h) * dk;
                const double *vt = v + ((size_t)t * H + h) * dv;
                const double bt = beta[(size_t)t * H + h];
                const double *Sp = S + (size_t)i * M;
                double *Sn = S + (size_t)(i + 1) * M;
                for (int c = 0; c < dk; ++c)
                    for (int j = 0; j < dv; ++j) P[(size_t)c * dv + j] = exp(gt[c]) * Sp[(size_t)c * dv + j];
                for (int j = 0; j < dv; ++j) {
                    double w = 0.0;
                    for (int c = 0; c < dk; ++c) w += P[(size_t)c * dv + j] * kt[c];
                    u[j] = vt[j] - w;
                }
                for (int c = 0; c < dk; ++c)
                    for (int j = 0; j < dv; ++j) Sn[(size_t)c * dv + j] = P[(size_t)c * dv + j] + bt * kt[c] * u[j];
            }
            /* reverse sweep */
            for (size_t e = 0; e < M; ++e) G[e] = dSfin ? dSfin[so + e] : 0.0;
            for (long i = L - 1; i >= 0; --i) {
                const long t = cu[n] + i;
                const size_t tk = ((size_t)t * H + h) * dk, tv = ((size_t)t * H + h) * dv;
                const double *qt = q + tk, *kt = k + tk, *gt = g + tk, *vt = v + tv, *dOt = dO + tv;
                const double bt = beta[(size_t)t * H + h];
                const double *Sp = S + (size_t)i * M, *St = S + (size_t)(i + 1) * M;
                for (int c = 0; c < dk; ++c)
                    for (int j = 0; j < dv; ++j) G[(size_t)c * dv + j] += scale * qt[c] * dOt[j];
                for (int c = 0; c < dk; ++c) {
                    double a = 0.0;
                    for (int j = 0; j < dv; ++j) a += St[(size_t)c * dv + j] * dOt[j];
                    gq[tk + c] = scale * a;
                }
                for (int c = 0; c < dk; ++c)
                    for (int j = 0; j < dv; ++j) P[(size_t)c * dv + j] = exp(gt[c]) * Sp[(size_t)c * dv + j];
                for (int j = 0; j < dv; ++j) {
                    double w = 0.0, x = 0.0;
                    for (int c = 0; c < dk; ++c) {
                        w += P[(size_t)c * dv + j] * kt[c];
                        x += G[(size_t)c * dv + j] * kt[c];
                    }
                    u[j] = vt[j] - w;
                    hv[j] = x;
                }
                double db = 0.0;
                for (int j = 0; j < dv; ++j) {
                    gv[tv + j] = bt * hv[j];
                    db += hv[j] * u[j];
                }
                gbeta[(size_t)t * H + h] = db;
                for (int c = 0; c < dk; ++c) {
                    double gu = 0.0, ph = 0.0, pd = 0.0;
                    for (int j = 0; j < dv; ++j) {
                        gu += G[(size_t)c * dv + j] * u[j];
                        ph += P[(size_t)c * dv + j] * hv[j];
                    }
                    gk[tk + c] = bt * (gu - ph);
                    const double al = exp(gt[c]);
                    for (int j = 0; j < dv; ++j) {
                        const double dP = G[(size_t)c * dv + j] - bt * kt[c] * hv[j];
                        pd += P[(size_t)c * dv + j] * dP;
                        G[(size_t)c * dv + j] = al * dP;
                    }
                    gg[tk + c] = pd;
                }
            }
            for (size_t e = 0; e < M; ++e) gS0[so + e] = G[e];
            free(S); free(G); free(P); free(u); free(hv);
        }
    }
    return bad ? -1 : 0;
}

/* Brute force: build the dense dk x dk transition M_t = (I - beta k k^T) Diag(alpha)
 * and form S_t = M_t S_{t-1} + beta k v^T with plain matrix products.  Tiny
 * inputs only (O(dk^2 dv) per token). */
int kda_oracle_bruteforce(const double *q, const double *k, const double *v,
                          const double *g, const double *beta, const double *S0,
                          const double *gate, const int *cu, int N, int T, int H,
                          int dk, int dv, double scale, double *o, double *Sfin)
{
    if (check_cu(cu, N, T) || H <= 0 || dk <= 0 || dv <= 0) return -1;
    if (!q || !k || !v || !g || !beta || !o) return -1;
    double *S = (double *)malloc(sizeof(double) * (size_t)dk * dv);
    double *Sn = (double *)malloc(sizeof(double) * (size_t)dk * dv);
    double *M = (double *)malloc(sizeof(double) * (size_t)dk * dk);
    if (!S || !Sn || !M) { free(S); free(Sn); free(M); return -1; }
    for (int n = 0; n < N; ++n) {
        for (int h = 0; h < H; ++h) {
            const size_t so = ((size_t)n * H + h) * dk * dv;
            for (size_t e = 0; e < (size_t)dk * dv; ++e) S[e] = S0 ? S0[so + e] : 0.0;
            for (long t = cu[n]; t < cu[n + 1]; ++t) {
                const double *qt = q + ((size_t)t * H + h) * dk;
                const double *kt = k + ((size_t)t * H + h) * dk;
                const double *gt = g + ((size_t)t * H + h) * dk;
                const double *vt = v + ((size_t)t * H + h) * dv;
                const double bt = beta[(size_t)t * H + h];
                for (int a = 0; a < dk; ++a)
                    for (int b = 0; b < dk; ++b)
                        M[(size_t)a * dk + b] = ((a == b ? 1.0 : 0.0) - bt * kt[a] * kt[b]) * exp(gt[b]);
                for (int a = 0; a < dk; ++a)
                    for (int j = 0; j < dv; ++j) {
                        double acc = 0.0;
                        for (int b = 0; b < dk; ++b) acc += M[(size_t)a * dk + b] * S[(size_t)b * dv + j];
                        Sn[(size_t)a * dv + j] = acc + bt * kt[a] * vt[j];
                    }
                memcpy(S, Sn, sizeof(double) * (size_t)dk * dv);
                double *ot = o + ((size_t)t * H + h) * dv;
                for (int j = 0; j < dv; ++j) {
                    double acc = 0.0;
                    for (int a = 0; a < dk; ++a) acc += S[(size_t)a * dv + j] * qt[a];
                    double r = scale * acc;
                    if (gate) r *= sigm(gate[((size_t)t * H + h) * dv + j]);
                    ot[j] = r;
                }
            }
            if (Sfin)
                for (size_t e = 0; e < (size_t)dk * dv; ++e) Sfin[so + e] = S[e];
        }
    }
    free(S); free(Sn); free(M);
    return 0;
}

/* Chunked form of the same recurrence (the algebra a chunk-parallel kernel
 * uses), written naively with exponentials of differences, never of single
 * cumulative sums.  Within a chunk of Lc tokens, G[i] = sum_{s<=i} g_s:
 *   Akk[i,j] = beta_i sum_c k_ic k_jc exp(G_ic - G_jc)          (j < i)
 *   Aqk[i,j] = sum_c q_ic k_jc exp(G_ic - G_jc)                 (j <= i)
 *   (I + Akk) Wm = beta * k * exp(G),  (I + Akk) U = beta * v   (forward subst.)
 *   Vp = U - Wm S
 *   O  = scale ((q * exp(G)) S + Aqk Vp)
 *   S  = Diag(exp(G_last)) S + sum_i (k_i * exp(G_last - G_i)) Vp_i^T
 * It is used by the tests to check the chunk algebra against the per-token
 * definition; it is not the parity oracle. */
int kda_oracle_chunked(const double *q, const double *k, const double *v,
                       const double *g, const double *beta, const double *S0,
                       const double *gate, const int *cu, int N, int T, int H,
                       int dk, int dv, double scale, int chunk, double *o, double *Sfin)
{
    if (check_cu(cu, N, T) || H <= 0 || dk <= 0 || dv <= 0 || chunk <= 0) return -1;
    if (!q || !k || !v || !g || !beta || !o) return -1;
    const int C = chunk;
    double *S = (double *)malloc(sizeof(double) * (size_t)dk * dv);
    double *G = (double *)malloc(sizeof(double) * (size_t)C * dk);
    double *Akk = (double *)malloc(sizeof(double) * (size_t)C * C);
    double *Aqk = (double *)malloc(sizeof(double) * (size_t)C * C);
    double *Wm = (double *)malloc(sizeof(double) * (size_t)C * dk);
    double *U = (double *)malloc(sizeof(double) * (size_t)C * dv);
    double *Sn = (double *)malloc(sizeof(double) * (size_t)dk * dv);
    if (!S || !G || !Akk || !Aqk || !Wm || !U || !Sn) {
        free(S); free(G); free(Akk); free(Aqk); free(Wm); free(U); free(Sn);
        return -1;
    }
    for (int n = 0; n < N; ++n) {
        const long s0 = cu[n], L = cu[n + 1] - cu[n];
        for (int h = 0; h < H; ++h) {
            const size_t so = ((size_t)n * H + h) * dk * dv;
            for (size_t e = 0; e < (size_t)dk * dv; ++e) S[e] = S0 ? S0[so + e] : 0.0;
#define QX(t, c) q[((size_t)(t) * H + h) * dk + (c)]
#define KX(t, c) k[((size_t)(t) * H + h) * dk + (c)]
#define GX(t, c) g[((size_t)(t) * H + h) * dk + (c)]
#define VX(t, j) v[((size_t)(t) * H + h) * dv + (j)]
#define BX(t) beta[(size_t)(t) * H + h]
            for (long cs = 0; cs < L; cs += C) {
                const int Lc = (int)((L - cs) < C ? (L - cs) : C);
                const long tb = s0 + cs;
                for (int c = 0; c < dk; ++c) {
                    double acc = 0.0;
                    for (int i = 0; i < Lc; ++i) {
                        acc += GX(tb + i, c);
                        G[(size_t)i * dk + c] = acc;
                    }
                }
                for (int i = 0; i < Lc; ++i)
                    for (int j = 0; j < Lc; ++j) {
                        double skk = 0.0, sqk = 0.0;
                        if (j <= i)
                            for (int c = 0; c < dk; ++c) {
                                double e = exp(G[(size_t)i * dk + c] - G[(size_t)j * dk + c]);
                                skk += KX(tb + i, c) * KX(tb + j, c) * e;
                                sqk += QX(tb + i, c) * KX(tb + j, c) * e;
                            }
                        Akk[(size_t)i * C + j] = (j < i) ? BX(tb + i) * skk : 0.0;
                        Aqk[(size_t)i * C + j] = (j <= i) ? sqk : 0.0;
                    }
                for (int i = 0; i < Lc; ++i) {
                    const double bi = BX(tb + i);
                    for (int c = 0; c < dk; ++c) {
                        double r = bi * KX(tb + i, c) * exp(G[(size_t)i * dk + c]);
                        for (int j = 0; j < i; ++j) r -= Akk[(size_t)i * C + j] * Wm[(size_t)j * dk + c];
                        Wm[(size_t)i * dk + c] = r;
                    }
                    for (int jj = 0; jj < dv; ++jj) {
                        double r = bi * VX(tb + i, jj);
                        for (int j = 0; j < i; ++j) r -= Akk[(size_t)i * C + j] * U[(size_t)j * dv + jj];
                        U[(size_t)i * dv + jj] = r;
                    }
                }
                /* U <- U - Wm S  (this is Vp) */
                for (int i = 0; i < Lc; ++i)
                    for (int jj = 0; jj < dv; ++jj) {
                        double acc = 0.0;
                        for (int c = 0; c < dk; ++c) acc += Wm[(size_t)i * dk + c] * S[(size_t)c * dv + jj];
                        U[(size_t)i * dv + jj] -= acc;
                    }
                for (int i = 0; i < Lc; ++i)
                    for (int jj = 0; jj < dv; ++jj) {
                        double acc = 0.0;
                        for (int c = 0; c < dk; ++c)
                            acc += QX(tb + i, c) * exp(G[(size_t)i * dk + c]) * S[(size_t)c * dv + jj];
                        for (int j = 0; j <= i; ++j) acc += Aqk[(size_t)i * C + j] * U[(size_t)j * dv + jj];
                        double r = scale * acc;
                        if (gate) r *= sigm(gate[((size_t)(tb + i) * H + h) * dv + jj]);
                        o[((size_t)(tb + i) * H + h) * dv + jj] = r;
                    }
                const double *Gl = G + (size_t)(Lc - 1) * dk;
                for (int c = 0; c < dk; ++c)
                    for (int jj = 0; jj < dv; ++jj) {
                        double acc = exp(Gl[c]) * S[(size_t)c * dv + jj];
                        for (int i = 0; i < Lc; ++i)
                            acc += KX(tb + i, c) * exp(Gl[c] - G[(size_t)i * dk + c]) * U[(size_t)i * dv + jj];
                        Sn[(size_t)c * dv + jj] = acc;
                    }
                memcpy(S, Sn, sizeof(double) * (size_t)dk * dv);
            }
#undef QX
#undef KX
#undef GX
#undef VX
#undef BX
            if (Sfin)
                for (size_t e = 0; e < (size_t)dk * dv; ++e) Sfin[so + e] = S[e];
        }
    }
    free(S); free(G); free(Akk); free(Aqk); free(Wm); free(U); free(Sn);
    return 0;
}

/* The whole mixer on packed sequences: optional causal conv (+SiLU) over the
 * concatenated channels [q | k | v] (D = 2*H*dk + H*dv, weights [D, W], conv
 * state [N, W-1, D]), optional q/k L2 norm, then the recurrence with the
 * optional gate.  conv_w == NULL skips the conv; then cs_in/cs_out are unused. */
int kda_oracle_mixer(const double *q_in, const double *k_in, const double *v_in,
                     const double *g, const double *beta, const double *S0,
                     const double *gate, const double *conv_w, int W,
                     const double *cs_in, double *cs_out,
                     const int *cu, int N, int T, int H, int dk, int dv,
                     double scale, int use_l2, double eps, double *o, double *Sfin)
{
    if (check_cu(cu, N, T) || H <= 0 || dk <= 0 || dv <= 0) return -1;
    const size_t nq = (size_t)T * H * dk, nv = (size_t)T * H * dv;
    double *qq = (double *)malloc(sizeof(double) * (nq ? nq : 1));
    double *kk = (double *)malloc(sizeof(double) * (nq ? nq : 1));
    double *vv = (double *)malloc(sizeof(double) * (nv ? nv : 1));
    int rc = 0;
    if (!qq || !kk || !vv) { rc = -1; goto done; }
    if (conv_w) {
        const int Dq = H * dk, Dv = H * dv, D = 2 * Dq + Dv;
        double *x = (double *)malloc(sizeof(double) * ((size_t)T * D + 1));
        double *y = (double *)malloc(sizeof(double) * ((size_t)T * D + 1));
        if (!x || !y) { free(x); free(y); rc = -1; goto done; }
        for (long t = 0; t < T; ++t) {
            memcpy(x + (size_t)t * D, q_in + (size_t)t * Dq, sizeof(double) * Dq);
            memcpy(x + (size_t)t * D + Dq, k_in + (size_t)t * Dq, sizeof(double) * Dq);
            memcpy(x + (size_t)t * D + 2 * Dq, v_in + (size_t)t * Dv, sizeof(double) * Dv);
        }
        rc = kda_oracle_short_conv(x, conv_w, cs_in, cu, N, T, D, W, 1, y, cs_out);
        for (long t = 0; t < T && rc == 0; ++t) {
            memcpy(qq + (size_t)t * Dq, y + (size_t)t * D, sizeof(double) * Dq);
            memcpy(kk + (size_t)t * Dq, y + (size_t)t * D + Dq, sizeof(double) * Dq);
            memcpy(vv + (size_t)t * Dv, y + (size_t)t * D + 2 * Dq, sizeof(double) * Dv);
        }
        free(x); free(y);
        if (rc) goto done;
    } else {
        memcpy(qq, q_in, sizeof(double) * nq);
        memcpy(kk, k_in, sizeof(double) * nq);
        memcpy(vv, v_in, sizeof(double) * nv);
    }
    if (use_l2) {
        kda_oracle_l2norm(qq, (long)T * H, dk, eps);
        kda_oracle_l2norm(kk, (long)T * H, dk, eps);
    }
    rc = kda_oracle_recurrent(qq, kk, vv, g, beta, S0, gate, cu, N, T, H, dk, dv, scale, o, Sfin);
done:
    free(qq); free(kk); free(vv);
    return rc;
}

/* One decode token for each of N sequences ("conv update then recurrent
 * step"): the mixer on N sequences of length one, starting from and writing
 * back the recurrent state [N, H, dk, dv] and the conv state [N, W-1, D].
 * state and conv_state are updated in place. */
int kda_oracle_decode_step(const double *q, const double *k, const double *v,
                           const double *g, const double *beta, const double *gate,
                           const double *conv_w, int W, double *conv_state,
                           double *state, int N, int H, int dk, int dv,
                           double scale, int use_l2, double eps, double *o)
{
    if (N < 0 || !state) return -1;
    int *cu = (int *)malloc(sizeof(int) * (size_t)(N + 1));
    if (!cu) return -1;
    for (int n = 0; n <= N; ++n) cu[n] = n;
    int rc = kda_oracle_mixer(q, k, v, g, beta, state, gate, conv_w, W, conv_state, conv_state,
                              cu, N, N, H, dk, dv, scale, use_l2, eps, o, state);
    free(cu);
    return rc;
}
