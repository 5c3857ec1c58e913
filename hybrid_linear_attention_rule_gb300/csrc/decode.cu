// decode.cu -- one KDA decode token for N independent sequences.
//
// metrale kimi_k3 docs, Functions: kda_decode_token ("One decode token: conv
// update then recurrent step"); Structs: KdaState (both buffers FP32,
// read-modify-write).  Per (sequence n, head h):
//   conv (+SiLU) of the new q, k, v channels against the conv window, window
//   shifted in place; q, k L2-normalised; then with alpha = exp(g):
//     a = k^T (Diag(alpha) S),  b = q^T (Diag(alpha) S)
//     d = beta (v - a)
//     S' = Diag(alpha) S + k d^T          (= (I - beta k k^T) Diag(alpha) S + beta k v^T)
//     o  = scale (b + (q . k) d)  [* sigmoid(gate)]   (= scale S'^T q)
// so one read pass and one write pass over S suffice.
//
// Roofline: HBM.  Per (n, h) the FP32 state is 4*dk*dv bytes read and the
// same written; everything else is < 10 % of that.  One CTA of 256 threads
// per (n, h): warp w owns state rows w, w+8, ..., lane l owns columns
// 4l..4l+3, so each warp load is one contiguous 512-byte row (dv = 128) and
// all 16 row loads of a thread are issued before the conv/norm work, which
// hides their latency.  The column sums over rows are reduced across the 8
// warps through shared memory.
#include "common.cuh"

namespace k3kda {
namespace {

constexpr int kDecThreads = 256;
constexpr int kDecWarps = kDecThreads / 32;
constexpr int kMaxD = 128;
constexpr int kRowsPerWarp = kMaxD / kDecWarps;   // 16

struct DecodeArgs {
    const void *q, *k, *v;
    int bf16;
    const float *g, *beta;
    const void *gate;
    const float *conv_w;
    float *conv_state;
    float *state;
    int N, H, dk, dv, W;
    float scale;
    int l2;
    void *out;
    int out_bf16;
};

__global__ void __launch_bounds__(kDecThreads, 2) decode_kernel(DecodeArgs a) {
    const int nh = blockIdx.x;
    const int n = nh / a.H, h = nh - (nh / a.H) * a.H;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int dk = a.dk, dv = a.dv;

    __shared__ float sq[kMaxD], sk[kMaxD], sv[kMaxD], salpha[kMaxD], sd[kMaxD];
    __shared__ float red[2][kDecWarps][kMaxD];
    __shared__ float sred[3];

    // 1. stream the state rows in (read once; evict-first)
    float *Sp = a.state + (size_t)nh * dk * dv;
    const bool colok = 4 * lane < dv;
    float4 s[kRowsPerWarp];
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
        const int c = warp + kDecWarps * r;
        if (c < dk && colok) s[r] = __ldcs(reinterpret_cast<const float4 *>(Sp + (size_t)c * dv + 4 * lane));
        else s[r] = make_float4(0.f, 0.f, 0.f, 0.f);
    }

    // 2. conv update + SiLU for this head's q, k, v channels
    const int D = 2 * a.H * dk + a.H * dv;
    const int W = a.W;
    for (int i = tid; i < 2 * dk + dv; i += kDecThreads) {
        int ch;
        float x;
        if (i < dk) { ch = h * dk + i; x = load_elt(a.q, (size_t)nh * dk + i, a.bf16); }
        else if (i < 2 * dk) { ch = a.H * dk + h * dk + (i - dk); x = load_elt(a.k, (size_t)nh * dk + (i - dk), a.bf16); }
        else { ch = 2 * a.H * dk + h * dv + (i - 2 * dk); x = load_elt(a.v, (size_t)nh * dv + (i - 2 * dk), a.bf16); }
        float y = x;
        if (a.conv_w != nullptr) {
            const float *w = a.conv_w + (size_t)ch * W;
            float *cs = a.conv_state + (size_t)n * (W - 1) * D + ch;
            float acc = w[W - 1] * x;
            float prev[3];
#pragma unroll
            for (int r = 0; r < 3; ++r)
                if (r < W - 1) { prev[r] = cs[(size_t)r * D]; acc = fmaf(w[r], prev[r], acc); }
#pragma unroll
            for (int r = 0; r < 2; ++r)
                if (r < W - 2) cs[(size_t)r * D] = prev[r + 1];
            if (W > 1) cs[(size_t)(W - 2) * D] = x;
            y = acc / (1.0f + expf(-acc));
        }
        if (i < dk) sq[i] = y;
        else if (i < 2 * dk) sk[i - dk] = y;
        else sv[i - 2 * dk] = y;
    }
    for (int c = tid; c < dk; c += kDecThreads) salpha[c] = expf(a.g[(size_t)nh * dk + c]);
    __syncthreads();

    // 3. |q|^2, |k|^2, q.k
    if (warp < 3) {
        float acc = 0.f;
        for (int c = lane; c < dk; c += 32) {
            const float x = warp == 1 ? sk[c] : sq[c];
            const float y = warp == 0 ? sq[c] : sk[c];
            acc = fmaf(x, y, acc);
        }
        acc = warp_sum(acc);
        if (lane == 0) sred[warp] = acc;
    }
    __syncthreads();
    float rq = 1.f, rk = 1.f;
    if (a.l2) {
        rq = 1.0f / sqrtf(sred[0] + K3KDA_L2_EPS);
        rk = 1.0f / sqrtf(sred[1] + K3KDA_L2_EPS);
    }
    const float qk = sred[2] * rq * rk;

    // 4. decay in registers; per-thread partial column sums of k^T S and q^T S
    float pa[4] = {0.f, 0.f, 0.f, 0.f}, pb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
        const int c = warp + kDecWarps * r;
        if (c < dk) {
            const float al = salpha[c], kc = sk[c] * rk, qc = sq[c] * rq;
            s[r].x *= al; s[r].y *= al; s[r].z *= al; s[r].w *= al;
            pa[0] = fmaf(kc, s[r].x, pa[0]); pa[1] = fmaf(kc, s[r].y, pa[1]);
            pa[2] = fmaf(kc, s[r].z, pa[2]); pa[3] = fmaf(kc, s[r].w, pa[3]);
            pb[0] = fmaf(qc, s[r].x, pb[0]); pb[1] = fmaf(qc, s[r].y, pb[1]);
            pb[2] = fmaf(qc, s[r].z, pb[2]); pb[3] = fmaf(qc, s[r].w, pb[3]);
        }
    }
    if (colok) {
        *reinterpret_cast<float4 *>(&red[0][warp][4 * lane]) = make_float4(pa[0], pa[1], pa[2], pa[3]);
        *reinterpret_cast<float4 *>(&red[1][warp][4 * lane]) = make_float4(pb[0], pb[1], pb[2], pb[3]);
    }
    __syncthreads();

    // 5. per column: d = beta (v - a), o = scale (b + qk d) [* sigmoid(gate)]
    if (tid < dv) {
        float av = 0.f, bv = 0.f;
#pragma unroll
        for (int w = 0; w < kDecWarps; ++w) { av += red[0][w][tid]; bv += red[1][w][tid]; }
        const float d = a.beta[nh] * (sv[tid] - av);
        sd[tid] = d;
        float o = a.scale * fmaf(qk, d, bv);
        if (a.gate != nullptr) {
            const float z = load_elt(a.gate, (size_t)nh * dv + tid, a.bf16);
            o = o / (1.0f + expf(-z));
        }
        store_elt(a.out, (size_t)nh * dv + tid, o, a.out_bf16);
    }
    __syncthreads();

    // 6. rank-1 update and write back (evict-first)
    if (colok) {
        const float4 dd = *reinterpret_cast<const float4 *>(&sd[4 * lane]);
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r) {
            const int c = warp + kDecWarps * r;
            if (c < dk) {
                const float kc = sk[c] * rk;
                float4 x = s[r];
                x.x = fmaf(kc, dd.x, x.x); x.y = fmaf(kc, dd.y, x.y);
                x.z = fmaf(kc, dd.z, x.z); x.w = fmaf(kc, dd.w, x.w);
                __stcs(reinterpret_cast<float4 *>(Sp + (size_t)c * dv + 4 * lane), x);
            }
        }
    }
}

}  // namespace

cudaError_t launch_decode(const void *q, const void *k, const void *v, int in_bf16, const float *g,
                          const float *beta, const void *gate, const float *conv_w, float *conv_state,
                          float *state, int N, int H, int dk, int dv, int W, float scale, int l2,
                          void *out, int out_bf16, cudaStream_t s) {
    if (N == 0) return cudaSuccess;
    DecodeArgs a{q, k, v, in_bf16, g, beta, gate, conv_w, conv_state, state, N, H, dk, dv, W, scale,
                 l2, out, out_bf16};
    decode_kernel<<<N * H, kDecThreads, 0, s>>>(a);
    count_launch();
    return cudaGetLastError();
}

}  // namespace k3kda
