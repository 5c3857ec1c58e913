// backward.cu -- reverse-mode gradients of the KDA recurrence (the ungated core of the mixer):
// dq, dk, dv, dg, dbeta and dS0 for given gradients dO (of o = scale S_t^T q_t) and dS_final.
//
// The recurrence S_t = (I - beta_t k_t k_t^T) Diag(exp g_t) S_{t-1} + beta_t k_t v_t^T is
// separable in the dv columns of S, and so is its reverse sweep, except for the quantities
// that sum over dv (dq, dk, dg, dbeta), which each CTA adds into the outputs with atomics.
// So a CTA owns one (sequence, head, 32-column block): 4 CTAs per head at dv = 128.
//
// Pass 1 runs the recurrence forward and stores the state before every 64-token chunk.
// Pass 2 walks the chunks backwards: it recomputes the chunk's states from its checkpoint
// (kept in a per-CTA scratch buffer), then sweeps the chunk's tokens in reverse.  With
// P = Diag(alpha) S_{t-1}, u = v - P^T k and G the gradient reaching S_t:
//   G += scale q dO^T;  dq = scale S_t dO;  h = G^T k;  dv = beta h;  dbeta = h.u;
//   dk = beta (G u - P h);  dP = G - beta k h^T;  dg = rowsum(P o dP);  G <- Diag(alpha) dP,
// and G after the first token is dS0.  This is the chain rule on the per-token definition
// (the backward named in the feature list of "Experimental Native Vulkan Backend for Kimi K3",
// Hugging Face discussion #187); CUDA cores, fp32 throughout.
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include <atomic>

#include "common.cuh"

namespace k3kda {
namespace {

constexpr int kD = 128;           // dk = dv
constexpr int kBV = 32;           // dv columns per CTA
constexpr int kNV = kD / kBV;     // CTAs per (sequence, head)
constexpr int kThreads = 256;     // thread (row r = tid / 2, half) owns 16 columns of row r
constexpr int kCols = 16;
constexpr int kChunk = 64;        // tokens per checkpoint
constexpr int kWarps = kThreads / 32;
constexpr size_t kBlockFloats = (size_t)kD * kBV;   // one CTA's share of a state

struct BwdArgs {
    const void *q, *k, *v;
    int bf16;
    const float *g, *beta, *S0, *dO, *dSfin;
    const int32_t *cu;
    int N, T, H;
    float scale;
    const int32_t *chunk_off;     // [N + 1] 64-token chunks before each sequence
    float *ckpt;                  // [(chunk) * H * kNV][kD][kBV]: state before each chunk
    float *scratch;               // [N * H * kNV][kChunk][kD][kBV]: states after each token of a chunk
    float *dq, *dk, *dv, *dg, *dbeta, *dS0;
};

__global__ void __launch_bounds__(1024) chunk_offsets_kernel(const int32_t *cu, int N, int T, int32_t *off) {
    // sequential prefix over the sequences (N is small next to the passes that follow)
    if (threadIdx.x == 0) {
        int acc = 0;
        off[0] = 0;
        for (int n = 0; n < N; ++n) {
            int b, e;
            seq_bounds(cu, n, T, b, e);
            acc += (e - b + kChunk - 1) / kChunk;
            off[n + 1] = acc;
        }
    }
}

// Sum over the block's 128 rows of this thread's 16 column values (x), for two vectors at once:
// a reduce-scatter over the 16 rows of the warp (lane bits 1-4) leaves lane (i, half) with
// column half*16 + i, then the warps' partials meet in shared memory.  The 32 column sums of
// vector a are returned in red[0][0][...] .. (read after the barrier inside) -- see below.
__device__ __forceinline__ void warp_rows_reduce(float (&x)[kCols], float &out) {
    const int lane = threadIdx.x & 31;
    // step over lane bit 4 (rows i and i^8): keep columns 8..15 when the bit is set
    float y8[8];
    {
        const bool hi = (lane >> 4) & 1;
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            const float send = hi ? x[m] : x[m + 8];
            const float keep = hi ? x[m + 8] : x[m];
            y8[m] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
        }
    }
    float y4[4];
    {
        const bool hi = (lane >> 3) & 1;
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const float send = hi ? y8[m] : y8[m + 4];
            const float keep = hi ? y8[m + 4] : y8[m];
            y4[m] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
        }
    }
    float y2[2];
    {
        const bool hi = (lane >> 2) & 1;
#pragma unroll
        for (int m = 0; m < 2; ++m) {
            const float send = hi ? y4[m] : y4[m + 2];
            const float keep = hi ? y4[m + 2] : y4[m];
            y2[m] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
        }
    }
    {
        const bool hi = (lane >> 1) & 1;
        const float send = hi ? y2[0] : y2[1];
        const float keep = hi ? y2[1] : y2[0];
        out = keep + __shfl_xor_sync(0xffffffffu, send, 2);
    }
    // lane (i = lane >> 1, half = lane & 1) now holds column half*16 + (bit-reversed... ) :
    // the kept index is 8*b4 + 4*b3 + 2*b2 + b1 of the lane, i.e. lane >> 1
}

struct Shared {
    float red[2][kWarps][kBV];    // warp partial column sums of two vectors
    float u[kBV], h[kBV];         // the column vectors of the current token
    float wsum[kWarps];
};

// One CTA's view of a token: per-row scalars of this thread's row, and its 16 dO columns.
struct Tok {
    float q, k, a, beta;          // q[r], k[r], alpha[r] = exp(g[r]), beta
};

__device__ __forceinline__ Tok load_tok(const BwdArgs &A, int t, int h, int r) {
    const size_t row = ((size_t)t * A.H + h) * kD + r;
    Tok x;
    x.q = load_elt(A.q, row, A.bf16);
    x.k = load_elt(A.k, row, A.bf16);
    x.a = __expf(A.g[row]);
    x.beta = A.beta[(size_t)t * A.H + h];
    return x;
}

// S <- Diag(alpha) S + beta k (v - (Diag(alpha) S)^T k)^T for this CTA's columns
__device__ __forceinline__ void forward_step(const BwdArgs &A, Shared &sh, float (&S)[kCols], const Tok &x, int t,
                                             int h, int cb) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    float p[kCols], kp[kCols];
#pragma unroll
    for (int u = 0; u < kCols; ++u) {
        p[u] = x.a * S[u];
        kp[u] = x.k * p[u];
    }
    float part;
    warp_rows_reduce(kp, part);
    sh.red[0][warp][(lane & 1) * kCols + (lane >> 1)] = part;
    __syncthreads();
    if (tid < kBV) {
        float w = 0.f;
#pragma unroll
        for (int i = 0; i < kWarps; ++i) w += sh.red[0][i][tid];
        sh.u[tid] = load_elt(A.v, ((size_t)t * A.H + h) * kD + cb + tid, A.bf16) - w;
    }
    __syncthreads();
    const int c0 = (tid & 1) * kCols;
#pragma unroll
    for (int u = 0; u < kCols; ++u) S[u] = p[u] + x.beta * x.k * sh.u[c0 + u];
}

__device__ __forceinline__ void ld_block(const float *src, int r, int c0, float (&S)[kCols]) {
#pragma unroll
    for (int u = 0; u < kCols; u += 4) {
        const float4 v4 = *reinterpret_cast<const float4 *>(src + (size_t)r * kBV + c0 + u);
        S[u] = v4.x; S[u + 1] = v4.y; S[u + 2] = v4.z; S[u + 3] = v4.w;
    }
}
__device__ __forceinline__ void st_block(float *dst, int r, int c0, const float (&S)[kCols]) {
#pragma unroll
    for (int u = 0; u < kCols; u += 4)
        *reinterpret_cast<float4 *>(dst + (size_t)r * kBV + c0 + u) = make_float4(S[u], S[u + 1], S[u + 2], S[u + 3]);
}

// Pass 1: the state before every chunk of the sequence.
__global__ void __launch_bounds__(kThreads) kda_bwd_checkpoint_kernel(const __grid_constant__ BwdArgs A) {
    __shared__ Shared sh;
    const int tid = threadIdx.x, r = tid >> 1, c0 = (tid & 1) * kCols;
    const int blk = blockIdx.x % kNV, nh = blockIdx.x / kNV, n = nh / A.H, h = nh % A.H;
    const int cb = blk * kBV;
    int tb, te;
    seq_bounds(A.cu, n, A.T, tb, te);
    float S[kCols];
#pragma unroll
    for (int u = 0; u < kCols; ++u) S[u] = A.S0 ? A.S0[((size_t)nh * kD + r) * kD + cb + c0 + u] : 0.f;
    const int q0 = A.chunk_off[n], nq = A.chunk_off[n + 1] - q0;
    for (int c = 0; c < nq; ++c) {
        st_block(A.ckpt + ((size_t)(q0 + c) * A.H * kNV + (size_t)h * kNV + blk) * kBlockFloats, r, c0, S);
        const int cs = tb + c * kChunk, ce = min(te, cs + kChunk);
        for (int t = cs; t < ce; ++t) forward_step(A, sh, S, load_tok(A, t, h, r), t, h, cb);
    }
}

// Pass 2: the reverse sweep.
__global__ void __launch_bounds__(kThreads) kda_bwd_sweep_kernel(const __grid_constant__ BwdArgs A) {
    __shared__ Shared sh;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, r = tid >> 1, c0 = (tid & 1) * kCols;
    const int blk = blockIdx.x % kNV, nh = blockIdx.x / kNV, n = nh / A.H, h = nh % A.H;
    const int cb = blk * kBV;
    const int H = A.H;
    int tb, te;
    seq_bounds(A.cu, n, A.T, tb, te);
    float G[kCols];
#pragma unroll
    for (int u = 0; u < kCols; ++u) G[u] = A.dSfin ? A.dSfin[((size_t)nh * kD + r) * kD + cb + c0 + u] : 0.f;
    float *scr = A.scratch + (size_t)blockIdx.x * kChunk * kBlockFloats;
    const int q0 = A.chunk_off[n], nq = A.chunk_off[n + 1] - q0;
    for (int c = nq - 1; c >= 0; --c) {
        const float *ck = A.ckpt + ((size_t)(q0 + c) * H * kNV + (size_t)h * kNV + blk) * kBlockFloats;
        const int cs = tb + c * kChunk, Lc = min(te, cs + kChunk) - cs;
        // recompute the chunk's states: scr[i] = state after token cs + i
        float S[kCols];
        ld_block(ck, r, c0, S);
        for (int i = 0; i < Lc; ++i) {
            forward_step(A, sh, S, load_tok(A, cs + i, h, r), cs + i, h, cb);
            st_block(scr + (size_t)i * kBlockFloats, r, c0, S);
        }
        // reverse sweep over the chunk; S holds the state after token cs + i
        for (int i = Lc - 1; i >= 0; --i) {
            const int t = cs + i;
            const Tok x = load_tok(A, t, h, r);
            float Sp[kCols];
            ld_block(i > 0 ? scr + (size_t)(i - 1) * kBlockFloats : ck, r, c0, Sp);
            float dO[kCols];
            const float *dOt = A.dO + ((size_t)t * H + h) * kD + cb + c0;
#pragma unroll
            for (int u = 0; u < kCols; u += 4) {
                const float4 v4 = *reinterpret_cast<const float4 *>(dOt + u);
                dO[u] = v4.x; dO[u + 1] = v4.y; dO[u + 2] = v4.z; dO[u + 3] = v4.w;
            }
            // G += scale q dO^T;  dq = scale S_t dO (this CTA's columns)
            float sdo = 0.f;
#pragma unroll
            for (int u = 0; u < kCols; ++u) {
                G[u] = fmaf(A.scale * x.q, dO[u], G[u]);
                sdo = fmaf(S[u], dO[u], sdo);
            }
            sdo += __shfl_xor_sync(0xffffffffu, sdo, 1);
            if ((tid & 1) == 0) atomicAdd(A.dq + ((size_t)t * H + h) * kD + r, A.scale * sdo);
            // column sums w = P^T k and h = G^T k
            float p[kCols], kp[kCols], kg[kCols];
#pragma unroll
            for (int u = 0; u < kCols; ++u) {
                p[u] = x.a * Sp[u];
                kp[u] = x.k * p[u];
                kg[u] = x.k * G[u];
            }
            float pw, ph;
            warp_rows_reduce(kp, pw);
            warp_rows_reduce(kg, ph);
            const int col = (lane & 1) * kCols + (lane >> 1);
            sh.red[0][warp][col] = pw;
            sh.red[1][warp][col] = ph;
            __syncthreads();
            if (tid < kBV) {
                float w = 0.f, hh = 0.f;
#pragma unroll
                for (int wi = 0; wi < kWarps; ++wi) {
                    w += sh.red[0][wi][tid];
                    hh += sh.red[1][wi][tid];
                }
                const size_t vi = ((size_t)t * H + h) * kD + cb + tid;
                const float uu = load_elt(A.v, vi, A.bf16) - w;
                sh.u[tid] = uu;
                sh.h[tid] = hh;
                A.dv[vi] = x.beta * hh;
                const float db = warp_sum(hh * uu);
                if (tid == 0) atomicAdd(A.dbeta + (size_t)t * H + h, db);
            }
            __syncthreads();
            // dk = beta (G u - P h);  dP = G - beta k h^T;  dg = rowsum(P o dP);  G <- alpha dP
            float gu = 0.f, phh = 0.f, pdp = 0.f;
#pragma unroll
            for (int u = 0; u < kCols; ++u) {
                const float uu = sh.u[c0 + u], hh = sh.h[c0 + u];
                gu = fmaf(G[u], uu, gu);
                phh = fmaf(p[u], hh, phh);
                const float dP = G[u] - x.beta * x.k * hh;
                pdp = fmaf(p[u], dP, pdp);
                G[u] = x.a * dP;
            }
            float dkp = x.beta * (gu - phh);
            dkp += __shfl_xor_sync(0xffffffffu, dkp, 1);
            pdp += __shfl_xor_sync(0xffffffffu, pdp, 1);
            if ((tid & 1) == 0) {
                atomicAdd(A.dk + ((size_t)t * H + h) * kD + r, dkp);
                atomicAdd(A.dg + ((size_t)t * H + h) * kD + r, pdp);
            }
#pragma unroll
            for (int u = 0; u < kCols; ++u) S[u] = Sp[u];
            __syncthreads();                           // sh.u / sh.h are rewritten by the next token
        }
    }
    float *d0 = A.dS0 + ((size_t)nh * kD + r) * kD + cb + c0;
#pragma unroll
    for (int u = 0; u < kCols; u += 4) *reinterpret_cast<float4 *>(d0 + u) = make_float4(G[u], G[u + 1], G[u + 2], G[u + 3]);
    (void)warp;
}

size_t round256b(size_t b) { return (b + 255) & ~size_t(255); }
size_t bwd_chunks(int N, int T) { return ((size_t)T + (size_t)(kChunk - 1) * (size_t)N) / kChunk; }

}  // namespace

size_t backward_workspace(int N, int T, int H) {
    return round256b((size_t)(N + 1) * sizeof(int32_t)) +
           round256b(bwd_chunks(N, T) * H * kNV * kBlockFloats * sizeof(float)) +
           (size_t)N * H * kNV * kChunk * kBlockFloats * sizeof(float);
}

cudaError_t launch_backward(const void *q, const void *k, const void *v, int bf16, const float *g, const float *beta,
                            const float *S0, const int32_t *cu, int N, int T, int H, float scale, const float *dO,
                            const float *dSfin, float *dq, float *dk, float *dv, float *dg, float *dbeta, float *dS0,
                            void *ws, cudaStream_t s) {
    cudaError_t e;
    const size_t tk = (size_t)T * H * kD * sizeof(float);
    if (T > 0 &&
        ((e = cudaMemsetAsync(dq, 0, tk, s)) != cudaSuccess || (e = cudaMemsetAsync(dk, 0, tk, s)) != cudaSuccess ||
         (e = cudaMemsetAsync(dg, 0, tk, s)) != cudaSuccess ||
         (e = cudaMemsetAsync(dbeta, 0, (size_t)T * H * sizeof(float), s)) != cudaSuccess))
        return e;
    if ((long long)N * H == 0) return cudaSuccess;
    uint8_t *w = static_cast<uint8_t *>(ws);
    BwdArgs A{};
    A.q = q; A.k = k; A.v = v; A.bf16 = bf16;
    A.g = g; A.beta = beta; A.S0 = S0; A.dO = dO; A.dSfin = dSfin;
    A.cu = cu; A.N = N; A.T = T; A.H = H; A.scale = scale;
    A.chunk_off = reinterpret_cast<int32_t *>(w);
    w += round256b((size_t)(N + 1) * sizeof(int32_t));
    A.ckpt = reinterpret_cast<float *>(w);
    w += round256b(bwd_chunks(N, T) * H * kNV * kBlockFloats * sizeof(float));
    A.scratch = reinterpret_cast<float *>(w);
    A.dq = dq; A.dk = dk; A.dv = dv; A.dg = dg; A.dbeta = dbeta; A.dS0 = dS0;
    chunk_offsets_kernel<<<1, 32, 0, s>>>(cu, N, T, const_cast<int32_t *>(A.chunk_off));
    count_launch();
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const unsigned grid = (unsigned)((size_t)N * H * kNV);
    kda_bwd_checkpoint_kernel<<<grid, kThreads, 0, s>>>(A);
    count_launch();
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    kda_bwd_sweep_kernel<<<grid, kThreads, 0, s>>>(A);
    count_launch();
    return cudaGetLastError();
}

}  // namespace k3kda
