// mla_decode.cu -- one decode token of the hybrid's gated attention (MLA) layers on sm_103a.
//
// Source (by page title and section): metrale_model_arch::kimi_k3 docs, Functions:
// mla_decode_token -- "optional RoPE, append K/V, SDPA, optional output gate", projections
// kept in the mixer; Modules: mla (the layers are gated NoPE MLA, so RoPE is optional);
// mlite-k3 README, "What this repository is" (24 of the hybrid's 93 layers are this kind).
//
// Three launches on the caller's stream:
//   1. mla_append_kernel   (one CTA per sequence): reads the cached length pos, turns the
//      query and the new key by RoPE at position pos (angles in double precision, once per
//      frequency), stores the new key/value row at pos in the cache's type, and leaves the
//      query pre-multiplied by scale*log2(e) in the workspace together with the number of
//      keys to attend (pos + 1, or 0 when the cache is full or the length negative).
//   2. mla_attend_kernel   (one 4-warp CTA per (sequence, head, 512-key split)): streams the
//      split's key and value rows from HBM once with evict-first vector loads, each warp
//      owning 128 keys and keeping an online-softmax partial (max, sum, weighted values);
//      the CTA merges its four warps and writes one partial per split.
//   3. mla_combine_kernel  (one CTA per (sequence, head)): merges the splits, normalises,
//      applies sigmoid(gate), stores the output and advances the cached length.
// The work is HBM-bound (one multiply-add per cached element read): no tensor cores; the
// design point is full-bandwidth streaming of the head-major caches [N, H, L_max, dq | dv].
// Keys and queries may be wider than values (dq in {64, 128, 192, 256}, dv in {64, 128, 256}),
// e.g. 128 rotation-free dims beside a 64-dim RoPE part.
#include <math.h>

#include <type_traits>

#include "common.cuh"

namespace k3kda {
namespace {

constexpr int kSplit = 512;                 // keys per attention CTA
constexpr int kWarps = 4;
constexpr int kWarpKeys = kSplit / kWarps;  // keys per warp
constexpr float kLog2e = 1.4426950408889634f;

struct MlaArgs {
    const void *q, *k_new, *v_new;   // [N, H, d]
    int in_bf16;
    const void *gate;                // [N, H, d] or null
    void *k_cache, *v_cache;         // [N, H, L_max, d]
    int cache_bf16;
    int32_t *cache_len;              // [N] (or [num_slots] with a slot map)
    const int32_t *slot;             // [N] cache slot of each sequence, or null (slot n)
    int num_slots;
    int N, H, dq, dv, L_max, rope_dim;   // dq: query/key width, dv: value width
    float theta, scale;
    void *out;                       // [N, H, d]
    int out_bf16;
    int S;                           // splits per (sequence, head)
    int32_t *vlen;                   // workspace [N]: keys to attend, 0 = cache full or slot invalid
    int32_t *vslot;                  // workspace [N]: the cache slot of each sequence
    float *qs;                       // workspace [N, H, dq]: rotated query * scale * log2(e)
    float2 *ml;                      // workspace [N, H, S]: (max, sum) of each split, base-2 scores
    float *po;                       // workspace [N, H, S, dv]: unnormalised weighted values
};

// ---- 1. RoPE + append -------------------------------------------------------------------------

__global__ void __launch_bounds__(256) mla_append_kernel(const __grid_constant__ MlaArgs A) {
    __shared__ float cs[128], sn[128];                  // rope_dim <= dq <= 256
    const int n = blockIdx.x;
    const int sl = seq_slot(A.slot, A.num_slots, n);
    const int pos = sl >= 0 ? A.cache_len[sl] : -1;
    const bool valid = pos >= 0 && pos < A.L_max;
    if (threadIdx.x == 0) {
        A.vlen[n] = valid ? pos + 1 : 0;
        A.vslot[n] = sl;
    }
    if (!valid) return;
    const int half = A.rope_dim / 2;
    for (int i = threadIdx.x; i < half; i += blockDim.x) {
        // angle pos * theta^(-2i/rd), formed and reduced in double so that large positions keep
        // their accuracy; the rotation itself runs in fp32
        const double ang = (double)pos * pow((double)A.theta, -2.0 * i / A.rope_dim);
        double s, c;
        sincos(ang, &s, &c);
        cs[i] = (float)c;
        sn[i] = (float)s;
    }
    __syncthreads();
    const int dq = A.dq, dv = A.dv;
    const size_t HQ = (size_t)A.H * dq, HV = (size_t)A.H * dv;
    const float qmul = A.scale * kLog2e;
    for (size_t e = threadIdx.x; e < HQ; e += blockDim.x) {
        const int h = (int)(e / dq), c = (int)(e - (size_t)h * dq);
        const size_t src = (size_t)n * HQ + e;
        float qv = load_elt(A.q, src, A.in_bf16), kv = load_elt(A.k_new, src, A.in_bf16);
        if (c < A.rope_dim) {
            const bool lo = c < half;
            const int i = lo ? c : c - half;
            const size_t pr = lo ? src + half : src - half;
            const float qp = load_elt(A.q, pr, A.in_bf16), kp = load_elt(A.k_new, pr, A.in_bf16);
            const float sgn = lo ? -sn[i] : sn[i];
            qv = qv * cs[i] + qp * sgn;
            kv = kv * cs[i] + kp * sgn;
        }
        A.qs[src] = qv * qmul;
        store_elt(A.k_cache, (((size_t)sl * A.H + h) * A.L_max + pos) * dq + c, kv, A.cache_bf16);
    }
    for (size_t e = threadIdx.x; e < HV; e += blockDim.x) {
        const int h = (int)(e / dv), c = (int)(e - (size_t)h * dv);
        store_elt(A.v_cache, (((size_t)sl * A.H + h) * A.L_max + pos) * dv + c,
                  load_elt(A.v_new, (size_t)n * HV + e, A.in_bf16), A.cache_bf16);
    }
}

// ---- 2. split attention -----------------------------------------------------------------------

// W 32-bit words of one lane's slice of a key or value row
template <int W> struct Raw { uint32_t w[W]; };

// a lane's slice starts at lane * W words: 16-byte pieces when W is a multiple of 4, 8-byte
// pieces when W is even, else 4-byte ones
template <int W> __device__ __forceinline__ void ld_stream(Raw<W> &r, const void *p) {
    if constexpr (W % 4 == 0) {
#pragma unroll
        for (int i = 0; i < W / 4; ++i) {
            const uint4 x = __ldcs(reinterpret_cast<const uint4 *>(p) + i);
            r.w[4 * i] = x.x; r.w[4 * i + 1] = x.y; r.w[4 * i + 2] = x.z; r.w[4 * i + 3] = x.w;
        }
    } else if constexpr (W % 2 == 0) {
#pragma unroll
        for (int i = 0; i < W / 2; ++i) {
            const uint2 x = __ldcs(reinterpret_cast<const uint2 *>(p) + i);
            r.w[2 * i] = x.x; r.w[2 * i + 1] = x.y;
        }
    } else {
#pragma unroll
        for (int i = 0; i < W; ++i) r.w[i] = __ldcs(reinterpret_cast<const unsigned int *>(p) + i);
    }
}

template <int W> __device__ __forceinline__ void zero(Raw<W> &r) {
#pragma unroll
    for (int i = 0; i < W; ++i) r.w[i] = 0u;
}

// element e of a lane slice: bf16 pairs sit low half first in each word
template <bool BF, int W> __device__ __forceinline__ float elt(const Raw<W> &r, int e) {
    if constexpr (BF) return __uint_as_float((e & 1) ? (r.w[e >> 1] & 0xffff0000u) : (r.w[e >> 1] << 16));
    else return __uint_as_float(r.w[e]);
}

// EQ, EV elements per lane of a key and of a value row (dq = 32 EQ, dv = 32 EV); R keys per
// warp round, chosen so that a round keeps 40 to 80 words of key and value rows in flight per lane.
template <int EQ, int EV, bool BF>
__global__ void __launch_bounds__(kWarps * 32, 4) mla_attend_kernel(const __grid_constant__ MlaArgs A) {
    constexpr int DQ = 32 * EQ, DV = 32 * EV;
    constexpr int WQ = BF ? EQ / 2 : EQ, WV = BF ? EV / 2 : EV;   // words per lane slice
    constexpr int R = (WQ + WV) <= 5 ? 16 : (WQ + WV) <= 10 ? 8 : 4;   // keys per round
    constexpr int SH = (R == 16) ? 1 : (R == 8) ? 2 : 3;             // lanes per key = 1 << SH
    static_assert((1 << SH) * R == 32 && EQ % 2 == 0 && EV % 2 == 0, "round shape");
    using T = typename std::conditional<BF, __nv_bfloat16, float>::type;

    const size_t blk = blockIdx.x;
    const int s = (int)(blk % A.S);
    const size_t nh = blk / A.S;
    const int n = (int)(nh / A.H);
    const int len = A.vlen[n];
    const int k0 = s * kSplit;
    if (k0 >= len) return;
    const int k1 = min(len, k0 + kSplit);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    float q[EQ];
    {
        const float *qp = A.qs + nh * DQ + lane * EQ;
#pragma unroll
        for (int e = 0; e < EQ; e += 2) {
            const float2 x = *reinterpret_cast<const float2 *>(qp + e);
            q[e] = x.x; q[e + 1] = x.y;
        }
    }
    const size_t ch = (size_t)A.vslot[n] * A.H + (nh - (size_t)n * A.H);   // the cache's (slot, head)
    const T *Kc = reinterpret_cast<const T *>(A.k_cache) + ch * (size_t)A.L_max * DQ + lane * EQ;
    const T *Vc = reinterpret_cast<const T *>(A.v_cache) + ch * (size_t)A.L_max * DV + lane * EV;

    float m = -INFINITY, l = 0.f, o[EV];
#pragma unroll
    for (int e = 0; e < EV; ++e) o[e] = 0.f;

    const int wb = k0 + warp * kWarpKeys, we = min(k1, wb + kWarpKeys);
    const int mykey = lane >> SH;
    for (int j0 = wb; j0 < we; j0 += R) {
        const int nk = min(R, we - j0);
        Raw<WQ> kr[R];
        Raw<WV> vr[R];
#pragma unroll
        for (int j = 0; j < R; ++j) {
            if (j < nk) {
                ld_stream(kr[j], Kc + (size_t)(j0 + j) * DQ);
                ld_stream(vr[j], Vc + (size_t)(j0 + j) * DV);
            } else {
                zero(kr[j]);
                zero(vr[j]);
            }
        }
        float part[R];
#pragma unroll
        for (int j = 0; j < R; ++j) {
            float acc = 0.f;
#pragma unroll
            for (int e = 0; e < EQ; ++e) acc = fmaf(q[e], elt<BF>(kr[j], e), acc);
            part[j] = acc;
        }
        // reduce-scatter the R partial dot products over the warp: after the step with offset
        // o a lane keeps the half of its keys selected by its bit o, so at the end lane L holds
        // the sum for key L >> SH over 32 >> SH lanes; the remaining SH steps finish the sum
#pragma unroll
        for (int st = 0; st < 5 - SH; ++st) {
            const int off = 16 >> st, cnt = R >> (st + 1);
            const bool up = (lane & off) != 0;
#pragma unroll
            for (int i = 0; i < cnt; ++i) {
                const float send = up ? part[i] : part[i + cnt];
                const float keep = up ? part[i + cnt] : part[i];
                part[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
            }
        }
#pragma unroll
        for (int off = (1 << SH) >> 1; off > 0; off >>= 1) part[0] += __shfl_xor_sync(0xffffffffu, part[0], off);
        const float sc = mykey < nk ? part[0] : -INFINITY;
        float mr = sc;
#pragma unroll
        for (int off = 16; off >= (1 << SH); off >>= 1) mr = fmaxf(mr, __shfl_xor_sync(0xffffffffu, mr, off));
        const float mn = fmaxf(m, mr);
        const float corr = exp2f(m - mn);
        const float p = exp2f(sc - mn);
        l = l * corr + p;
#pragma unroll
        for (int e = 0; e < EV; ++e) o[e] *= corr;
#pragma unroll
        for (int j = 0; j < R; ++j) {
            const float pj = __shfl_sync(0xffffffffu, p, j << SH);
#pragma unroll
            for (int e = 0; e < EV; ++e) o[e] = fmaf(pj, elt<BF>(vr[j], e), o[e]);
        }
        m = mn;
    }
    // every key's weight sits in 1 << SH lanes
    l = warp_sum(l) * (1.f / (1 << SH));

    __shared__ float sm_m[kWarps], sm_l[kWarps];
    __shared__ __align__(16) float sm_o[kWarps][DV];
    if (lane == 0) { sm_m[warp] = m; sm_l[warp] = l; }
#pragma unroll
    for (int e = 0; e < EV; ++e) sm_o[warp][lane * EV + e] = o[e];
    __syncthreads();
    float M = sm_m[0];
#pragma unroll
    for (int w = 1; w < kWarps; ++w) M = fmaxf(M, sm_m[w]);
    float f[kWarps];
#pragma unroll
    for (int w = 0; w < kWarps; ++w) f[w] = sm_m[w] == -INFINITY ? 0.f : exp2f(sm_m[w] - M);
    const size_t ps = nh * A.S + s;
    for (int c = threadIdx.x; c < DV; c += kWarps * 32) {
        float acc = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) acc = fmaf(f[w], sm_o[w][c], acc);
        A.po[ps * DV + c] = acc;
    }
    if (threadIdx.x == 0) {
        float L = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) L = fmaf(f[w], sm_l[w], L);
        A.ml[ps] = make_float2(M, L);
    }
}

// ---- 3. combine splits, gate, store -------------------------------------------------------------

__global__ void __launch_bounds__(128) mla_combine_kernel(const __grid_constant__ MlaArgs A) {
    const size_t nh = blockIdx.x;
    const int n = (int)(nh / A.H), h = (int)(nh - (size_t)n * A.H);
    const int len = A.vlen[n];
    const int D = A.dv;
    if (len == 0) {
        for (int c = threadIdx.x; c < D; c += blockDim.x) store_elt(A.out, nh * D + c, __int_as_float(0x7fc00000), A.out_bf16);
        return;
    }
    const int ns = (len + kSplit - 1) / kSplit;
    const float2 *ml = A.ml + nh * A.S;
    float M = -INFINITY;
    for (int s = 0; s < ns; ++s) M = fmaxf(M, ml[s].x);
    float L = 0.f;
    for (int s = 0; s < ns; ++s) L = fmaf(exp2f(ml[s].x - M), ml[s].y, L);
    const float inv = 1.f / L;
    for (int c = threadIdx.x; c < D; c += blockDim.x) {
        float acc = 0.f;
        for (int s = 0; s < ns; ++s) acc = fmaf(exp2f(ml[s].x - M), A.po[(nh * A.S + s) * D + c], acc);
        float r = acc * inv;
        if (A.gate) r *= sigmoidf_(load_elt(A.gate, nh * D + c, A.in_bf16));
        store_elt(A.out, nh * D + c, r, A.out_bf16);
    }
    if (h == 0 && threadIdx.x == 0) A.cache_len[A.vslot[n]] = len;
}

template <int EQ, int EV, bool BF> void *attend_fn() { return (void *)mla_attend_kernel<EQ, EV, BF>; }

template <int EQ, bool BF> void *attend_fn_v(int ev) {
    return ev == 2 ? attend_fn<EQ, 2, BF>() : ev == 4 ? attend_fn<EQ, 4, BF>() : attend_fn<EQ, 8, BF>();
}
template <bool BF> void *attend_fn_qv(int eq, int ev) {
    return eq == 2 ? attend_fn_v<2, BF>(ev) : eq == 4 ? attend_fn_v<4, BF>(ev) : eq == 6 ? attend_fn_v<6, BF>(ev)
                                                                                      : attend_fn_v<8, BF>(ev);
}

}  // namespace

size_t mla_splits(int L_max) { return ((size_t)L_max + kSplit - 1) / kSplit; }

size_t mla_workspace(int N, int H, int dq, int dv, int L_max) {
    auto r256 = [](size_t b) { return (b + 255) & ~size_t(255); };
    const size_t S = mla_splits(L_max), NH = (size_t)N * H;
    return 2 * r256((size_t)N * 4) + r256(NH * dq * 4) + r256(NH * S * 8) + r256(NH * S * dv * 4);
}

cudaError_t launch_mla_decode(const void *q, const void *k_new, const void *v_new, int in_bf16, const void *gate,
                              void *k_cache, void *v_cache, int cache_bf16, int32_t *cache_len, int N, int H, int dq,
                              int dv, int L_max, int rope_dim, float theta, float scale, void *out, int out_bf16,
                              void *ws, cudaStream_t st, const int32_t *slot, int num_slots) {
    if (N == 0) return cudaSuccess;
    auto r256 = [](size_t b) { return (b + 255) & ~size_t(255); };
    MlaArgs A;
    A.q = q; A.k_new = k_new; A.v_new = v_new; A.in_bf16 = in_bf16; A.gate = gate;
    A.k_cache = k_cache; A.v_cache = v_cache; A.cache_bf16 = cache_bf16; A.cache_len = cache_len;
    A.N = N; A.H = H; A.dq = dq; A.dv = dv; A.L_max = L_max; A.rope_dim = rope_dim; A.theta = theta; A.scale = scale;
    A.out = out; A.out_bf16 = out_bf16;
    A.slot = slot; A.num_slots = num_slots;
    A.S = (int)mla_splits(L_max);
    const size_t NH = (size_t)N * H;
    char *p = static_cast<char *>(ws);
    A.vlen = reinterpret_cast<int32_t *>(p);  p += r256((size_t)N * 4);
    A.vslot = reinterpret_cast<int32_t *>(p); p += r256((size_t)N * 4);
    A.qs = reinterpret_cast<float *>(p);      p += r256(NH * dq * 4);
    A.ml = reinterpret_cast<float2 *>(p);     p += r256(NH * A.S * 8);
    A.po = reinterpret_cast<float *>(p);

    mla_append_kernel<<<N, 256, 0, st>>>(A);
    count_launch();
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;

    void *fn = cache_bf16 ? attend_fn_qv<true>(dq / 32, dv / 32) : attend_fn_qv<false>(dq / 32, dv / 32);
    void *args[] = {&A};
    e = cudaLaunchKernel(fn, dim3((unsigned)(NH * A.S)), dim3(kWarps * 32), args, 0, st);
    count_launch();
    if (e != cudaSuccess) return e;

    mla_combine_kernel<<<(unsigned)NH, 128, 0, st>>>(A);
    count_launch();
    return cudaGetLastError();
}

}  // namespace k3kda
