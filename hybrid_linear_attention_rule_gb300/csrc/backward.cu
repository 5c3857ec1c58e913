// backward.cu -- reverse-mode gradients of the KDA recurrence (the ungated core of the mixer):
// dq, dk, dv, dg, dbeta and dS0 for given gradients dO (of o = scale S_t^T q_t) and dS_final.
//
// The recurrence S_t = (I - beta_t k_t k_t^T) Diag(exp g_t) S_{t-1} + beta_t k_t v_t^T is
// separable in the dv columns of S, and so is its reverse sweep, except for the quantities
// that sum over dv (dq, dk, dg, dbeta), which each CTA adds into the outputs with atomics.
// So a CTA owns one (sequence, head, 16-column block): 8 CTAs per head at dv = 128.
//
// Pass 1 runs the recurrence forward and stores the state before every 16-token block.
// Pass 2 walks the blocks backwards: it recomputes the block's states from its checkpoint
// into a per-CTA scratch buffer (256 KB, small enough to stay in L2), then sweeps the
// block's tokens in reverse.  Each token's inputs (and the state it starts from) are loaded
// one token ahead, so the loads' latency hides behind the previous token's arithmetic.  With
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
constexpr int kBV = 16;           // dv columns per CTA
constexpr int kNV = kD / kBV;     // CTAs per (sequence, head)
constexpr int kThreads = 256;     // thread (row r = tid / 2, half) owns kCols columns of row r
constexpr int kCols = kBV / 2;
constexpr int kColShift = kCols == 16 ? 1 : kCols == 8 ? 2 : 3;   // lane >> kColShift = kept column
constexpr int kChunk = 16;        // tokens per checkpoint
constexpr int kWarps = kThreads / 32;
constexpr size_t kBlockFloats = (size_t)kD * kBV;   // one CTA's share of a state

struct BwdArgs {
    const void *q, *k, *v;
    int bf16;
    const float *g, *beta, *S0, *dO, *dSfin;
    const int32_t *cu;
    int N, T, H;
    float scale;
    const int32_t *chunk_off;     // [N + 1] 16-token blocks before each sequence
    float *ckpt;                  // [(block) * H * kNV][kD][kBV]: state before each block
    float *scratch;               // [N * H * kNV][kChunk][kD][kBV]: states after each token of a block
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

// Sum over the warp's 16 rows of this thread's kCols column values: a reduce-scatter over the
// row bits of the lane (bits 4, 3, ... : each step keeps half of the remaining columns, chosen
// by the lane's bit) leaves one column per lane, finished by all-reduce steps over the row bits
// that remain; lane L then holds column (L & 1) * kCols + (L >> kColShift) summed over the warp's
// rows, and the warps' partials meet in shared memory.
__device__ __forceinline__ float warp_rows_reduce(const float (&x)[kCols]) {
    const int lane = threadIdx.x & 31;
    float y[kCols];
#pragma unroll
    for (int m = 0; m < kCols; ++m) y[m] = x[m];
#pragma unroll
    for (int st = 0; (kCols >> (st + 1)) >= 1; ++st) {
        const int off = 16 >> st, cnt = kCols >> (st + 1);
        const bool hi = (lane & off) != 0;
#pragma unroll
        for (int m = 0; m < cnt; ++m) {
            const float send = hi ? y[m] : y[m + cnt];
            const float keep = hi ? y[m + cnt] : y[m];
            y[m] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
    }
#pragma unroll
    for (int off = 16 / kCols; off >= 2; off >>= 1) y[0] += __shfl_xor_sync(0xffffffffu, y[0], off);
    return y[0];
}

__device__ __forceinline__ int kept_column(int lane) { return (lane & 1) * kCols + (lane >> kColShift); }

struct __align__(16) Shared {
    float red[2][kWarps][kBV];    // warp partial column sums of two vectors
    float u[2][kBV], h[2][kBV];   // the column vectors of a token (alternating buffers)
};

// this thread's kCols columns of a kBV-float shared vector (16-byte loads)
__device__ __forceinline__ void ldc(const float *v, int c0, float (&x)[kCols]) {
#pragma unroll
    for (int u = 0; u < kCols; u += 4) {
        const float4 f = *reinterpret_cast<const float4 *>(v + c0 + u);
        x[u] = f.x; x[u + 1] = f.y; x[u + 2] = f.z; x[u + 3] = f.w;
    }
}

// A 16-token block's inputs in shared memory, raw (q, k, v in the input dtype; g, beta, dO
// fp32), copied in by every thread with 16-byte cp.async while the previous block is worked
// on (two buffers).  Row pitches are those of fp32 so that both dtypes fit.
struct BlockIn {
    uint8_t q[kChunk][kD * 4], k[kChunk][kD * 4];   // a row of q or k: 128 elements
    float g[kChunk][kD];
    uint8_t v[kChunk][kBV * 4];                     // this CTA's 32 v columns
    float dO[kChunk][kBV];
    float beta[kChunk];
};
constexpr size_t kBwdSmem = 2 * sizeof(BlockIn);

__device__ __forceinline__ void cp16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)), "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp4(void *dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)), "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// issue the copies of tokens [t0, t0 + L) into `in` (all threads), then commit one group
__device__ __forceinline__ void stage_block(const BwdArgs &A, BlockIn &in, int t0, int L, int h, int cb, bool with_dO) {
    const int tid = threadIdx.x;
    const int es = A.bf16 ? 2 : 4;
    const int qc = kD * es / 16;                    // 16-byte pieces of a q/k row
    const uint8_t *qb = static_cast<const uint8_t *>(A.q), *kb = static_cast<const uint8_t *>(A.k);
    const uint8_t *vb = static_cast<const uint8_t *>(A.v);
    for (int e = tid; e < L * qc; e += kThreads) {
        const int i = e / qc, p = e - i * qc;
        const size_t off = (((size_t)(t0 + i) * A.H + h) * kD) * es + (size_t)p * 16;
        cp16(&in.q[i][p * 16], qb + off);
        cp16(&in.k[i][p * 16], kb + off);
    }
    for (int e = tid; e < L * (kD / 4); e += kThreads) {
        const int i = e / (kD / 4), p = e - i * (kD / 4);
        cp16(&in.g[i][p * 4], A.g + ((size_t)(t0 + i) * A.H + h) * kD + p * 4);
    }
    const int vc = kBV * es / 16;
    for (int e = tid; e < L * vc; e += kThreads) {
        const int i = e / vc, p = e - i * vc;
        cp16(&in.v[i][p * 16], vb + (((size_t)(t0 + i) * A.H + h) * kD + cb) * es + (size_t)p * 16);
    }
    if (with_dO)
        for (int e = tid; e < L * (kBV / 4); e += kThreads) {
            const int i = e / (kBV / 4), p = e - i * (kBV / 4);
            cp16(&in.dO[i][p * 4], A.dO + ((size_t)(t0 + i) * A.H + h) * kD + cb + p * 4);
        }
    if (tid < L) cp4(&in.beta[tid], A.beta + (size_t)(t0 + tid) * A.H + h);
    cp_commit();
}

// One token's per-row scalars for this thread's row r: q[r], k[r], alpha[r] = exp(g[r]), beta.
struct Tok {
    float q, k, a, beta;
};

__device__ __forceinline__ float ld_in(const uint8_t *row, int c, int bf16) {
    return bf16 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(row)[c]) : reinterpret_cast<const float *>(row)[c];
}

__device__ __forceinline__ Tok tok_of(const BlockIn &in, int i, int r, int bf16) {
    Tok x;
    x.q = ld_in(in.q[i], r, bf16);
    x.k = ld_in(in.k[i], r, bf16);
    x.a = __expf(in.g[i][r]);
    x.beta = in.beta[i];
    return x;
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

// Add this CTA's per-row partial x (held by both lanes of a row) into dst[r] for the warp's
// 16 rows: lanes 0, 8, 16, 24 gather four consecutive rows and issue one 16-byte vector
// reduction each (a quarter of the scalar atomics).
__device__ __forceinline__ void add_rows(float *dst_row0, float x) {
    const int lane = threadIdx.x & 31;
    const float x1 = __shfl_down_sync(0xffffffffu, x, 2);
    const float x2 = __shfl_down_sync(0xffffffffu, x, 4);
    const float x3 = __shfl_down_sync(0xffffffffu, x, 6);
    if ((lane & 7) == 0) {
        float *d = dst_row0 + (lane >> 1);
        asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(d), "f"(x), "f"(x1), "f"(x2), "f"(x3)
                     : "memory");
    }
}

// S <- Diag(alpha) S + beta k (v - (Diag(alpha) S)^T k)^T for this CTA's columns; vj is this
// thread's v column (threads tid < kBV); buf alternates between consecutive calls
__device__ __forceinline__ void forward_step(Shared &sh, float (&S)[kCols], const Tok &x, float vj, int buf) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    float p[kCols], kp[kCols];
#pragma unroll
    for (int u = 0; u < kCols; ++u) {
        p[u] = x.a * S[u];
        kp[u] = x.k * p[u];
    }
    sh.red[0][warp][kept_column(lane)] = warp_rows_reduce(kp);
    __syncthreads();
    if (tid < kBV) {
        float w = 0.f;
#pragma unroll
        for (int i = 0; i < kWarps; ++i) w += sh.red[0][i][tid];
        sh.u[buf][tid] = vj - w;
    }
    __syncthreads();
    const int c0 = (tid & 1) * kCols;
    float uv[kCols];
    ldc(sh.u[buf], c0, uv);
    const float bk = x.beta * x.k;
#pragma unroll
    for (int u = 0; u < kCols; ++u) S[u] = fmaf(bk, uv[u], p[u]);
}

// the forward over the block's first L tokens from S; when store is given, the state after
// token i goes to store + i * kBlockFloats
__device__ __forceinline__ void forward_run(const BwdArgs &A, Shared &sh, const BlockIn &in, float (&S)[kCols], int L,
                                            int r, int c0, float *store) {
    const int tid = threadIdx.x;
    for (int i = 0; i < L; ++i) {
        const float vj = tid < kBV ? ld_in(in.v[i], tid, A.bf16) : 0.f;
        forward_step(sh, S, tok_of(in, i, r, A.bf16), vj, i & 1);
        if (store) st_block(store + (size_t)i * kBlockFloats, r, c0, S);
    }
}

// Pass 1: the state before every block of the sequence.
__global__ void __launch_bounds__(kThreads) kda_bwd_checkpoint_kernel(const __grid_constant__ BwdArgs A) {
    __shared__ Shared sh;
    extern __shared__ __align__(16) uint8_t dyn[];
    BlockIn *in = reinterpret_cast<BlockIn *>(dyn);
    const int tid = threadIdx.x, r = tid >> 1, c0 = (tid & 1) * kCols;
    const int blk = blockIdx.x % kNV, nh = blockIdx.x / kNV, n = nh / A.H, h = nh % A.H;
    const int cb = blk * kBV;
    int tb, te;
    seq_bounds(A.cu, n, A.T, tb, te);
    float S[kCols];
#pragma unroll
    for (int u = 0; u < kCols; ++u) S[u] = A.S0 ? A.S0[((size_t)nh * kD + r) * kD + cb + c0 + u] : 0.f;
    const int q0 = A.chunk_off[n], nq = A.chunk_off[n + 1] - q0;
    if (nq > 0) stage_block(A, in[0], tb, min(te - tb, kChunk), h, cb, false);
    for (int c = 0; c < nq; ++c) {
        const int cs = tb + c * kChunk, L = min(te, cs + kChunk) - cs;
        if (c + 1 < nq) {
            const int ns = cs + kChunk;
            stage_block(A, in[(c + 1) & 1], ns, min(te, ns + kChunk) - ns, h, cb, false);
            cp_wait<1>();
        } else {
            cp_wait<0>();
        }
        __syncthreads();
        st_block(A.ckpt + ((size_t)(q0 + c) * A.H * kNV + (size_t)h * kNV + blk) * kBlockFloats, r, c0, S);
        forward_run(A, sh, in[c & 1], S, L, r, c0, nullptr);
        __syncthreads();                               // buffer c & 1 is refilled two blocks on
    }
}

// Pass 2: the reverse sweep.
__global__ void __launch_bounds__(kThreads) kda_bwd_sweep_kernel(const __grid_constant__ BwdArgs A) {
    __shared__ Shared sh;
    extern __shared__ __align__(16) uint8_t dyn[];
    BlockIn *in = reinterpret_cast<BlockIn *>(dyn);
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
    auto block_len = [&](int c) { const int cs = tb + c * kChunk; return min(te, cs + kChunk) - cs; };
    if (nq > 0) stage_block(A, in[(nq - 1) & 1], tb + (nq - 1) * kChunk, block_len(nq - 1), h, cb, true);
    for (int c = nq - 1; c >= 0; --c) {
        if (c > 0) {
            stage_block(A, in[(c - 1) & 1], tb + (c - 1) * kChunk, block_len(c - 1), h, cb, true);
            cp_wait<1>();
        } else {
            cp_wait<0>();
        }
        __syncthreads();
        const BlockIn &bi = in[c & 1];
        const float *ck = A.ckpt + ((size_t)(q0 + c) * H * kNV + (size_t)h * kNV + blk) * kBlockFloats;
        const int cs = tb + c * kChunk, Lc = block_len(c);
        // recompute the block's states: scr[i] = state after token cs + i
        float S[kCols];
        ld_block(ck, r, c0, S);
        forward_run(A, sh, bi, S, Lc, r, c0, scr);
        // reverse sweep over the block; S holds the state after token cs + i, and the state
        // before token i is loaded from the scratch while token i + 1 is processed
        float Spn[kCols];
        ld_block(Lc > 1 ? scr + (size_t)(Lc - 2) * kBlockFloats : ck, r, c0, Spn);
        for (int i = Lc - 1; i >= 0; --i) {
            const int t = cs + i;
            const Tok x = tok_of(bi, i, r, A.bf16);
            float Sp[kCols];
#pragma unroll
            for (int u = 0; u < kCols; ++u) Sp[u] = Spn[u];
            if (i > 0) ld_block(i > 1 ? scr + (size_t)(i - 2) * kBlockFloats : ck, r, c0, Spn);
            const int buf = i & 1;
            // G += scale q dO^T;  dq = scale S_t dO (this CTA's columns)
            float sdo = 0.f, dO[kCols];
            ldc(bi.dO[i], c0, dO);
            const float sq = A.scale * x.q;
#pragma unroll
            for (int u = 0; u < kCols; ++u) {
                G[u] = fmaf(sq, dO[u], G[u]);
                sdo = fmaf(S[u], dO[u], sdo);
            }
            sdo += __shfl_xor_sync(0xffffffffu, sdo, 1);
            add_rows(A.dq + ((size_t)t * H + h) * kD + 16 * warp, A.scale * sdo);
            // column sums w = P^T k and h = G^T k
            float p[kCols], kp[kCols], kg[kCols];
#pragma unroll
            for (int u = 0; u < kCols; ++u) {
                p[u] = x.a * Sp[u];
                kp[u] = x.k * p[u];
                kg[u] = x.k * G[u];
            }
            const int col = kept_column(lane);
            sh.red[0][warp][col] = warp_rows_reduce(kp);
            sh.red[1][warp][col] = warp_rows_reduce(kg);
            __syncthreads();
            if (warp == 0) {
                float db = 0.f;
                if (lane < kBV) {
                    float w = 0.f, hh = 0.f;
#pragma unroll
                    for (int wi = 0; wi < kWarps; ++wi) {
                        w += sh.red[0][wi][lane];
                        hh += sh.red[1][wi][lane];
                    }
                    const float uu = ld_in(bi.v[i], lane, A.bf16) - w;
                    sh.u[buf][lane] = uu;
                    sh.h[buf][lane] = hh;
                    A.dv[((size_t)t * H + h) * kD + cb + lane] = x.beta * hh;
                    db = hh * uu;
                }
                db = warp_sum(db);
                if (lane == 0) atomicAdd(A.dbeta + (size_t)t * H + h, db);
            }
            __syncthreads();
            // dk = beta (G u - P h);  dP = G - beta k h^T;  dg = rowsum(P o dP);  G <- alpha dP
            float gu = 0.f, phh = 0.f, pdp = 0.f, uv[kCols], hv[kCols];
            ldc(sh.u[buf], c0, uv);
            ldc(sh.h[buf], c0, hv);
            const float bk = x.beta * x.k;
#pragma unroll
            for (int u = 0; u < kCols; ++u) {
                gu = fmaf(G[u], uv[u], gu);
                phh = fmaf(p[u], hv[u], phh);
                const float dP = fmaf(-bk, hv[u], G[u]);
                pdp = fmaf(p[u], dP, pdp);
                G[u] = x.a * dP;
            }
            float dkp = x.beta * (gu - phh);
            dkp += __shfl_xor_sync(0xffffffffu, dkp, 1);
            pdp += __shfl_xor_sync(0xffffffffu, pdp, 1);
            add_rows(A.dk + ((size_t)t * H + h) * kD + 16 * warp, dkp);
            add_rows(A.dg + ((size_t)t * H + h) * kD + 16 * warp, pdp);
#pragma unroll
            for (int u = 0; u < kCols; ++u) S[u] = Sp[u];
        }
        __syncthreads();                               // buffer c & 1 is refilled two blocks on
    }
    float *d0 = A.dS0 + ((size_t)nh * kD + r) * kD + cb + c0;
#pragma unroll
    for (int u = 0; u < kCols; u += 4) *reinterpret_cast<float4 *>(d0 + u) = make_float4(G[u], G[u + 1], G[u + 2], G[u + 3]);
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
    static std::atomic<uint64_t> ck_attr{0}, sw_attr{0};
    if ((e = smem_attr_once((const void *)kda_bwd_checkpoint_kernel, (int)kBwdSmem, ck_attr)) != cudaSuccess ||
        (e = smem_attr_once((const void *)kda_bwd_sweep_kernel, (int)kBwdSmem, sw_attr)) != cudaSuccess)
        return e;
    kda_bwd_checkpoint_kernel<<<grid, kThreads, kBwdSmem, s>>>(A);
    count_launch();
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    kda_bwd_sweep_kernel<<<grid, kThreads, kBwdSmem, s>>>(A);
    count_launch();
    return cudaGetLastError();
}

}  // namespace k3kda
