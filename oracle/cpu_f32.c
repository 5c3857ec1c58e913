/*
 * cpu_f32.c -- the FP32 CPU baseline of the KDA mixer: the oracle's per-token
 * loop, in single precision, with the same threading (OpenMP over sequences x
 * heads).
 *
 * TEST INFRASTRUCTURE ONLY.  It is timed by the benchmark's CPU-baseline leg
 * beside the FP64 oracle, as the plain CPU implementation a user without a GPU
 * would run; no test takes it as a reference and nothing on the product path
 * links, loads or calls it.  It shares no code with the CUDA library.
 *
 * What it computes is kda_oracle_mixer's composition (see kda_oracle.c for the
 * sources and readings): causal depthwise conv of width W over [q | k | v]
 * (no bias, tap W-1 on the current token, zero history), SiLU, q/k L2 norm
 * x (sum x^2 + eps)^(-1/2), then per token S <- Diag(exp g) S; u = S^T k;
 * S <- S + beta k (v - u)^T; o = scale S^T q, times sigmoid(gate) when given.
 * One sequence (B = 1) of T tokens; the conv runs per (head, channel) inside
 * the head's loop, so every thread touches only its head's channels.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int kda_cpu_f32_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

static float silu_f(float z) { return z / (1.0f + expf(-z)); }
static float sigm_f(float z) { return 1.0f / (1.0f + expf(-z)); }

/* conv (+SiLU) of one channel sequence x[t * stride] into y[t] (zero history) */
static void conv_channel(const float *x, long stride, const float *w, int W, int T, float *y)
{
    for (int t = 0; t < T; ++t) {
        float acc = 0.0f;
        for (int i = 0; i < W; ++i) {
            const int s = t - W + 1 + i;
            if (s >= 0) acc += w[i] * x[(long)s * stride];
        }
        y[t] = silu_f(acc);
    }
}

int kda_cpu_f32_mixer(const float *q, const float *k, const float *v, const float *g, const float *beta,
                      const float *gate, const float *conv_w, int W, int T, int H, int d, float scale,
                      float eps, float *o, float *Sfin)
{
    if (T < 0 || H <= 0 || d <= 0 || !q || !k || !v || !g || !beta || !o) return -1;
    int bad = 0;
#pragma omp parallel for schedule(dynamic)
    for (int h = 0; h < H; ++h) {
        float *S = (float *)calloc((size_t)d * d, sizeof(float));
        float *u = (float *)malloc(sizeof(float) * (size_t)d);
        float *xq = (float *)malloc(sizeof(float) * ((size_t)T * d + 1));
        float *xk = (float *)malloc(sizeof(float) * ((size_t)T * d + 1));
        float *xv = (float *)malloc(sizeof(float) * ((size_t)T * d + 1));
        float *col = (float *)malloc(sizeof(float) * ((size_t)T + 1));
        if (!S || !u || !xq || !xk || !xv || !col) {
            free(S); free(u); free(xq); free(xk); free(xv); free(col);
#pragma omp atomic write
            bad = 1;
            continue;
        }
        const long rs = (long)H * d;
        for (int c = 0; c < d; ++c) {
            const float *src[3] = {q + (long)h * d + c, k + (long)h * d + c, v + (long)h * d + c};
            float *dst[3] = {xq, xk, xv};
            for (int which = 0; which < 3; ++which) {
                if (conv_w) {
                    conv_channel(src[which], rs, conv_w + ((long)which * H * d + (long)h * d + c) * W, W, T, col);
                    for (int t = 0; t < T; ++t) dst[which][(long)t * d + c] = col[t];
                } else {
                    for (int t = 0; t < T; ++t) dst[which][(long)t * d + c] = src[which][(long)t * rs];
                }
            }
        }
        for (int t = 0; t < T; ++t) {
            float *qt = xq + (long)t * d, *kt = xk + (long)t * d, *vt = xv + (long)t * d;
            float sq = 0.0f, sk = 0.0f;
            for (int c = 0; c < d; ++c) { sq += qt[c] * qt[c]; sk += kt[c] * kt[c]; }
            const float iq = 1.0f / sqrtf(sq + eps), ik = 1.0f / sqrtf(sk + eps);
            for (int c = 0; c < d; ++c) { qt[c] *= iq; kt[c] *= ik; }
            const float *gt = g + ((long)t * H + h) * d;
            const float bt = beta[(long)t * H + h];
            for (int c = 0; c < d; ++c) {
                const float a = expf(gt[c]);
                for (int j = 0; j < d; ++j) S[(size_t)c * d + j] *= a;
            }
            for (int j = 0; j < d; ++j) u[j] = 0.0f;
            for (int c = 0; c < d; ++c)
                for (int j = 0; j < d; ++j) u[j] += S[(size_t)c * d + j] * kt[c];
            for (int c = 0; c < d; ++c) {
                const float bk = bt * kt[c];
                for (int j = 0; j < d; ++j) S[(size_t)c * d + j] += bk * (vt[j] - u[j]);
            }
            for (int j = 0; j < d; ++j) u[j] = 0.0f;
            for (int c = 0; c < d; ++c)
                for (int j = 0; j < d; ++j) u[j] += S[(size_t)c * d + j] * qt[c];
            float *ot = o + ((long)t * H + h) * d;
            for (int j = 0; j < d; ++j) {
                float r = scale * u[j];
                if (gate) r *= sigm_f(gate[((long)t * H + h) * d + j]);
                ot[j] = r;
            }
        }
        if (Sfin) memcpy(Sfin + (size_t)h * d * d, S, sizeof(float) * (size_t)d * d);
        free(S); free(u); free(xq); free(xk); free(xv); free(col);
    }
    return bad ? -1 : 0;
}
