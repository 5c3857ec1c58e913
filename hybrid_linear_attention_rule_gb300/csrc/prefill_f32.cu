// prefill_f32.cu -- chunked KDA prefill in FP32 on CUDA cores (any supported
// head dim, chunk 16/32/64, FP32 or BF16 inputs).
//
// The recurrence ("recurrent KDA state", HF discussion #187 feature list; FP32
// KdaState, metrale kimi_k3 docs) computed chunk by chunk.  Within a chunk of
// Lc tokens, G_i = sum_{s<=i} g_s (per channel) and
//   Akk[i,j] = beta_i sum_c k_ic k_jc exp(G_ic - G_jc)         (j < i)
//   Aqk[i,j] = sum_c q_ic k_jc exp(G_ic - G_jc)                (j <= i)
//   (I + Akk) [Wm | U] = [beta k exp(G) | beta v]             (forward substitution)
//   V' = U - Wm S
//   O  = scale ((q exp(G)) S + Aqk V')  [* sigmoid(gate)]
//   S  = Diag(exp(G_last)) S + (k exp(G_last - G))^T V'
// which is the per-token recurrence reorganised (the WY/UT form of the delta
// rule with per-channel decay).  The exponentials are always of differences
// of cumulative log-decays inside one chunk, so nothing overflows for any
// g <= 0.
//
// One CTA per (sequence, head, dv block of BV columns); the CTA walks its
// sequence's chunks in order and keeps its S block in shared memory.  This
// kernel is the reference-grade path (fp32 everywhere, errors ~1e-7
// relative); the tensor-core kernel takes the bf16 d=128 chunk-64 shapes.
#include "common.cuh"

namespace k3kda {
namespace {

constexpr int kPfThreads = 256;

struct Smem {
    // all row-major with a +1 pad on the fast dim to keep column walks conflict-free
    int DKP, BVP, CP;
    size_t q, k, G, W, U, Akk, Aqk, S, beta, total;
};

__host__ __device__ inline Smem smem_plan(int C, int dk, int BV) {
    Smem p;
    p.DKP = dk + 1; p.BVP = BV + 1; p.CP = C + 1;
    size_t o = 0;
    p.q = o; o += (size_t)C * p.DKP;
    p.k = o; o += (size_t)C * p.DKP;
    p.G = o; o += (size_t)C * p.DKP;
    p.W = o; o += (size_t)C * p.DKP;
    p.U = o; o += (size_t)C * p.BVP;
    p.Akk = o; o += (size_t)C * p.CP;
    p.Aqk = o; o += (size_t)C * p.CP;
    p.S = o; o += (size_t)dk * p.BVP;
    p.beta = o; o += C;
    p.total = o * sizeof(float);
    return p;
}

template <int C>
__global__ void __launch_bounds__(kPfThreads, 1) prefill_f32_kernel(PrefillArgs a, int BV, int nvb) {
    extern __shared__ float sm[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int vb = blockIdx.x % nvb;
    const int nh = blockIdx.x / nvb;
    const int h = nh % a.H, n = nh / a.H;
    const int sn = seq_slot(a.slot, a.num_slots, n);           // state row of this sequence (-1: none)
    const size_t snh = (size_t)(sn < 0 ? 0 : sn) * a.H + h;
    const int dk = a.dk, dv = a.dv, H = a.H;
    const Smem P = smem_plan(C, dk, BV);
    float *sQ = sm + P.q, *sK = sm + P.k, *sG = sm + P.G, *sW = sm + P.W, *sU = sm + P.U;
    float *sAkk = sm + P.Akk, *sAqk = sm + P.Aqk, *sS = sm + P.S, *sB = sm + P.beta;
    const int DKP = P.DKP, BVP = P.BVP, CP = P.CP;
    const int j0 = vb * BV;

    int tb, te;
    seq_bounds(a.cu, n, a.T, tb, te);

    // state block S[:, j0:j0+BV]
    for (int e = tid; e < dk * BV; e += kPfThreads) {
        const int c = e / BV, j = e % BV;
        sS[c * BVP + j] = (a.S0 && sn >= 0) ? a.S0[(snh * dk + c) * dv + j0 + j] : 0.f;
    }

    for (int cs = tb; cs < te; cs += C) {
        const int Lc = min(C, te - cs);
        __syncthreads();
        // ---- load the chunk (zero rows past Lc: they then contribute nothing) ----
        for (int e = tid; e < C * dk; e += kPfThreads) {
            const int i = e / dk, c = e % dk;
            float qv = 0.f, kv = 0.f, gv = 0.f;
            if (i < Lc) {
                const size_t t = (size_t)(cs + i);
                qv = load_elt(a.q, t * a.q_row + (size_t)h * dk + c, a.in_bf16);
                kv = load_elt(a.k, t * a.k_row + (size_t)h * dk + c, a.in_bf16);
                gv = a.g[(t * H + h) * dk + c];
            }
            sQ[i * DKP + c] = qv; sK[i * DKP + c] = kv; sG[i * DKP + c] = gv;
        }
        for (int i = tid; i < C; i += kPfThreads) sB[i] = i < Lc ? a.beta[(size_t)(cs + i) * H + h] : 0.f;
        for (int e = tid; e < C * BV; e += kPfThreads) {
            const int i = e / BV, j = e % BV;
            sU[i * BVP + j] = i < Lc ? load_elt(a.v, (size_t)(cs + i) * a.v_row + (size_t)h * dv + j0 + j, a.in_bf16) : 0.f;
        }
        __syncthreads();
        // ---- L2 norm of q and k rows; cumulative log-decay per channel ----
        if (a.l2) {
            for (int r = warp; r < 2 * C; r += kPfThreads / 32) {
                float *row = (r < C ? sQ : sK) + (r % C) * DKP;
                float ss = 0.f;
                for (int c = lane; c < dk; c += 32) ss = fmaf(row[c], row[c], ss);
                ss = warp_sum(ss);
                const float inv = 1.0f / sqrtf(ss + K3KDA_L2_EPS);
                for (int c = lane; c < dk; c += 32) row[c] *= inv;
            }
        }
        for (int c = tid; c < dk; c += kPfThreads) {
            float acc = 0.f;
            for (int i = 0; i < C; ++i) { acc += sG[i * DKP + c]; sG[i * DKP + c] = acc; }
        }
        for (int i = tid; i < C; i += kPfThreads)
            for (int j = 0; j < BV; ++j) sU[i * BVP + j] *= sB[i];     // U rhs = beta v
        __syncthreads();
        // ---- Akk, Aqk ----
        for (int e = tid; e < C * C; e += kPfThreads) {
            const int i = e / C, j = e % C;
            float kk = 0.f, qk = 0.f;
            if (j <= i) {
                const float *Gi = sG + i * DKP, *Gj = sG + j * DKP;
                const float *Ki = sK + i * DKP, *Kj = sK + j * DKP, *Qi = sQ + i * DKP;
                for (int c = 0; c < dk; ++c) {
                    const float ex = __expf(Gi[c] - Gj[c]);
                    const float kj = Kj[c] * ex;
                    kk = fmaf(Ki[c], kj, kk);
                    qk = fmaf(Qi[c], kj, qk);
                }
            }
            sAkk[i * CP + j] = j < i ? sB[i] * kk : 0.f;
            sAqk[i * CP + j] = j <= i ? qk : 0.f;
        }
        __syncthreads();
        // ---- rhs of W; scale q by exp(G) and k by exp(G_last - G) for the state products ----
        for (int e = tid; e < C * dk; e += kPfThreads) {
            const int i = e / dk, c = e % dk;
            const float Gi = sG[i * DKP + c], Gl = sG[(C - 1) * DKP + c];
            const float kv = sK[i * DKP + c];
            sW[i * DKP + c] = sB[i] * kv * __expf(Gi);
            sQ[i * DKP + c] *= __expf(Gi);
            sK[i * DKP + c] = kv * __expf(Gl - Gi);
        }
        __syncthreads();
        // ---- forward substitution: thread per column of [W | U] ----
        for (int col = tid; col < dk + BV; col += kPfThreads) {
            float *X = col < dk ? sW + col : sU + (col - dk);
            const int ld = col < dk ? DKP : BVP;
            for (int i = 1; i < Lc; ++i) {
                float acc = X[i * ld];
                const float *Ai = sAkk + i * CP;
                for (int j = 0; j < i; ++j) acc = fmaf(-Ai[j], X[j * ld], acc);
                X[i * ld] = acc;
            }
        }
        __syncthreads();
        // ---- V' = U - W S (in place in sU) ----
        for (int e = tid; e < C * BV; e += kPfThreads) {
            const int i = e / BV, j = e % BV;
            float acc = sU[i * BVP + j];
            const float *Wi = sW + i * DKP;
            for (int c = 0; c < dk; ++c) acc = fmaf(-Wi[c], sS[c * BVP + j], acc);
            sU[i * BVP + j] = acc;
        }
        __syncthreads();
        // ---- O = scale ((q e^G) S + Aqk V') [* sigmoid(gate)] ----
        for (int e = tid; e < Lc * BV; e += kPfThreads) {
            const int i = e / BV, j = e % BV;
            float acc = 0.f;
            const float *Qi = sQ + i * DKP;
            for (int c = 0; c < dk; ++c) acc = fmaf(Qi[c], sS[c * BVP + j], acc);
            const float *Ai = sAqk + i * CP;
            for (int jj = 0; jj <= i; ++jj) acc = fmaf(Ai[jj], sU[jj * BVP + j], acc);
            float o = a.scale * acc;
            const size_t oi = ((size_t)(cs + i) * H + h) * dv + j0 + j;
            if (a.gate) o = o * sigmoidf_(load_elt(a.gate, oi, a.gate_bf16));
            store_elt(a.out, oi, o, a.out_bf16);
        }
        __syncthreads();
        // ---- S = Diag(e^{G_last}) S + (k e^{G_last - G})^T V' ----
        for (int e = tid; e < dk * BV; e += kPfThreads) {
            const int c = e / BV, j = e % BV;
            float acc = __expf(sG[(C - 1) * DKP + c]) * sS[c * BVP + j];
            for (int i = 0; i < Lc; ++i) acc = fmaf(sK[i * DKP + c], sU[i * BVP + j], acc);
            sS[c * BVP + j] = acc;
        }
    }
    __syncthreads();
    if (a.Sfin && sn >= 0)
        for (int e = tid; e < dk * BV; e += kPfThreads) {
            const int c = e / BV, j = e % BV;
            a.Sfin[(snh * dk + c) * dv + j0 + j] = sS[c * BVP + j];
        }
}

template <int C>
cudaError_t launch_c(const PrefillArgs &a, cudaStream_t s) {
    const int BV = (a.dv % 32 == 0) ? 32 : 16;
    const int nvb = a.dv / BV;
    const Smem P = smem_plan(C, a.dk, BV);
    cudaError_t e = cudaFuncSetAttribute(prefill_f32_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)P.total);
    if (e != cudaSuccess) return e;
    const long long blocks = (long long)a.N * a.H * nvb;
    if (blocks == 0) return cudaSuccess;
    prefill_f32_kernel<C><<<(unsigned)blocks, kPfThreads, P.total, s>>>(a, BV, nvb);
    count_launch();
    return cudaGetLastError();
}

}  // namespace

size_t prefill_f32_smem_bytes(int chunk, int dk, int dv) {
    const int BV = (dv % 32 == 0) ? 32 : 16;
    return smem_plan(chunk, dk, BV).total;
}

cudaError_t launch_prefill_f32(const PrefillArgs &a, cudaStream_t s) {
    switch (a.chunk) {
        case 16: return launch_c<16>(a, s);
        case 32: return launch_c<32>(a, s);
        case 64: return launch_c<64>(a, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace k3kda
