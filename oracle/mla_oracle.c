/*
 * mla_oracle.c -- plain, slow, double-precision CPU oracle for one decode token
 * of the hybrid's gated attention (MLA) layers.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or calls
 * this file: only the tests and the package's smoke check do.  It shares no
 * code, header, table or constant with the CUDA library under
 * hybrid_linear_attention_rule_gb300/csrc, nor with kda_oracle.c.
 *
 * What it computes (sources, by page title and section):
 *   - metrale_model_arch::kimi_k3 docs, Functions: mla_decode_token -- one
 *     decode token is "optional RoPE, append K/V, SDPA, optional output gate",
 *     with the projections kept outside (in the mixer);
 *   - metrale_model_arch::kimi_k3 docs, Modules: mla ("gated NoPE MLA": the
 *     production layers use no positional rotation, so RoPE is optional);
 *   - mlite-k3 README, "What this repository is": the 69 KDA + 24 gated-MLA
 *     layer schedule of the hybrid.
 *
 * Readings where the pages are silent:
 *   heads: one key and one value row per query head (no sharing across heads),
 *         the decompressed form of the layer, since the token step receives
 *         projected q, k, v;
 *   RoPE: rotate-half form on the first rd dims of q and of the new key, pair
 *         (i, i + rd/2) turned by the angle pos * theta^(-2i/rd), pos = the
 *         number of tokens already cached for the sequence; keys are stored
 *         rotated, so cached keys are never rotated again; rd = 0 is NoPE;
 *   SDPA: softmax over the scores scale * q . k_j for every cached key
 *         j = 0 .. pos (the new key included), no mask beyond that, output the
 *         softmax-weighted sum of the value rows;
 *   gate: out = o * sigmoid(gate) elementwise when a gate is given;
 *   storage: the appended key and value rows are stored in the cache's type
 *         (rounded to the nearest bfloat16, ties to even, for a bf16 cache) and
 *         the attention reads them back from the cache;
 *   full cache: a sequence whose cache already holds L_max tokens (or whose
 *         length is negative) gets NaN outputs; its cache and length are left
 *         as they were.
 *
 * Layouts (row-major, last index fastest):
 *   q, k_new [N, H, dqk]; v_new, gate, out [N, H, dv];
 *   k_cache [N, H, L_max, dqk]; v_cache [N, H, L_max, dv]; cache_len [N].
 *
 * Every entry returns 0 on success and -1 on an invalid argument.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Nearest bfloat16 of a double, ties to even, returned as a double.  A bf16
 * has float32's 8 exponent bits and 7 stored fraction bits, so a normal bf16
 * carries 8 significant bits.  The double is rounded once, straight to that
 * grid: write x = m * 2^e with 0.5 <= |m| < 1, scale m to an integer of
 * 8 bits and round half to even. */
static double round_bf16(double x)
{
    if (isnan(x)) return x;
    int e;
    double m = frexp(x, &e);
    if (m == 0.0) return x;
    double s = ldexp(m, 8);               /* |s| in [128, 256) */
    double r = nearbyint(s);              /* default rounding mode: half to even */
    double y = ldexp(r, e - 8);
    if (fabs(y) > 3.3895313892515355e38) y = copysign(INFINITY, x);   /* above the largest bf16 */
    /* bf16 has float32's exponent range; values below 2^-126 would be subnormal:
     * round them on the subnormal grid of spacing 2^-133. */
    if (fabs(x) < ldexp(1.0, -126)) y = ldexp(nearbyint(ldexp(x, 133)), -133);
    return y;
}

/* Rotate-half RoPE of one row x[0..rd) at position pos (mla_decode_token's
 * "optional RoPE"; the rotate-half pairing is the reading used). */
static void rope_row(double *x, int rd, long pos, double theta)
{
    const int half = rd / 2;
    for (int i = 0; i < half; ++i) {
        const double ang = (double)pos * pow(theta, -2.0 * i / rd);
        const double c = cos(ang), s = sin(ang);
        const double a = x[i], b = x[i + half];
        x[i] = a * c - b * s;
        x[i + half] = b * c + a * s;
    }
}

/* RoPE applied to rows of x [rows, d] in place, row r at position pos[r]. */
int mla_oracle_rope(double *x, long rows, int d, int rd, const long *pos, double theta)
{
    if (!x || rows < 0 || d <= 0 || rd < 0 || rd > d || (rd & 1) || (rd > 0 && (!pos || !(theta > 0))))
        return -1;
    if (rd == 0) return 0;
    for (long r = 0; r < rows; ++r) rope_row(x + r * d, rd, pos[r], theta);
    return 0;
}

/* One decode token for N sequences and H heads (mla_decode_token: optional
 * RoPE, append K/V, SDPA, optional output gate). */
int mla_oracle_decode_step(const double *q, const double *k_new, const double *v_new, const double *gate,
                           double *k_cache, double *v_cache, int *cache_len,
                           int N, int H, int dqk, int dv, int L_max, int rd, double theta, double scale,
                           int cache_bf16, double *out)
{
    if (N < 0 || H <= 0 || dqk <= 0 || dv <= 0 || L_max <= 0 || rd < 0 || rd > dqk || (rd & 1))
        return -1;
    if (rd > 0 && !(theta > 0)) return -1;
    if (N == 0) return 0;
    if (!q || !k_new || !v_new || !k_cache || !v_cache || !cache_len || !out) return -1;

    double *qr = malloc(sizeof(double) * dqk);
    double *kr = malloc(sizeof(double) * dqk);
    double *sc = malloc(sizeof(double) * ((size_t)L_max + 1));
    if (!qr || !kr || !sc) { free(qr); free(kr); free(sc); return -1; }

    for (int n = 0; n < N; ++n) {
        const int pos = cache_len[n];
        const int valid = pos >= 0 && pos < L_max;
        for (int h = 0; h < H; ++h) {
            const size_t nh = (size_t)n * H + h;
            double *o = out + nh * dv;
            if (!valid) {
                for (int j = 0; j < dv; ++j) o[j] = NAN;
                continue;
            }
            double *Kc = k_cache + nh * (size_t)L_max * dqk;
            double *Vc = v_cache + nh * (size_t)L_max * dv;
            /* optional RoPE of the query and the new key at position pos */
            memcpy(qr, q + nh * dqk, sizeof(double) * dqk);
            memcpy(kr, k_new + nh * dqk, sizeof(double) * dqk);
            if (rd > 0) { rope_row(qr, rd, pos, theta); rope_row(kr, rd, pos, theta); }
            /* append the new key and value at row pos, in the cache's type */
            for (int c = 0; c < dqk; ++c) Kc[(size_t)pos * dqk + c] = cache_bf16 ? round_bf16(kr[c]) : kr[c];
            for (int j = 0; j < dv; ++j)
                Vc[(size_t)pos * dv + j] = cache_bf16 ? round_bf16(v_new[nh * dv + j]) : v_new[nh * dv + j];
            /* scaled dot-product attention over rows 0..pos */
            double mx = -INFINITY;
            for (int t = 0; t <= pos; ++t) {
                double s = 0.0;
                for (int c = 0; c < dqk; ++c) s += qr[c] * Kc[(size_t)t * dqk + c];
                sc[t] = scale * s;
                if (sc[t] > mx) mx = sc[t];
            }
            double den = 0.0;
            for (int t = 0; t <= pos; ++t) { sc[t] = exp(sc[t] - mx); den += sc[t]; }
            for (int j = 0; j < dv; ++j) {
                double acc = 0.0;
                for (int t = 0; t <= pos; ++t) acc += sc[t] * Vc[(size_t)t * dv + j];
                double r = acc / den;
                if (gate) r *= 1.0 / (1.0 + exp(-gate[nh * dv + j]));
                o[j] = r;
            }
        }
        if (valid) cache_len[n] = pos + 1;
    }
    free(qr);
    free(kr);
    free(sc);
    return 0;
}

/* Nearest bfloat16 of each value (exposed so that the tests can pin it). */
int mla_oracle_round_bf16(double *x, long n)
{
    if (!x || n < 0) return -1;
    for (long i = 0; i < n; ++i) x[i] = round_bf16(x[i]);
    return 0;
}
