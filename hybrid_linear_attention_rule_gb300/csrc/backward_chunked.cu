// backward_chunked.cu -- reverse-mode gradients of the KDA recurrence in chunked form.
//
// The recurrence S_t = (I - beta_t k_t k_t^T) Diag(exp g_t) S_{t-1} + beta_t k_t v_t^T,
// o_t = scale S_t^T q_t (the ungated core of the mixer, "Experimental Native Vulkan Backend for
// Kimi K3", Hugging Face discussion #187, feature list) is written per chunk of kC tokens in the
// WY form the forward uses.  With Gamma the in-chunk cumulative log decay (per channel), Gamma_L
// its value at the chunk's last token, and
//   Q0 = q e^{Gamma},  K0 = k e^{Gamma},  Kd = k e^{Gamma_L - Gamma}            (all factors <= 1)
//   B_ij = sum_c k_ic k_jc e^{Gamma_ic - Gamma_jc} (j < i),  Aqk_ij = sum_c q_ic k_jc e^{...} (j <= i),
//   Tm = (I + diag(beta) B)^-1,  W = Tm diag(beta) K0,  U = Tm diag(beta) V,
//   Delta = U - W S,  O = scale (Q0 S + Aqk Delta),  S_next = e^{Gamma_L} S + Kd^T Delta.
// Differentiating these products (the chain rule on the chunk algebra) gives, for the gradient
// Dout reaching S_next and dO of the chunk's outputs (dOs = scale dO):
//   dDelta = Kd Dout + Aqk^T dOs,  dR = Tm^T dDelta,
//   Din = e^{Gamma_L} Dout + Q0^T dOs - K0^T diag(beta) dR        (the gradient reaching S),
//   dA = -strict_lower(dR Delta^T),  dAqk = lower(dOs Delta^T),  dv = diag(beta) dR,
//   dq  = (dOs S^T) e^{Gamma} + P1,          P1_ic = sum_{j <= i} dAqk_ij k_jc e^{Gamma_ic - Gamma_jc}
//   dkt = beta (P2 - (dR S^T) e^{Gamma}),    P2_ic = sum_{j < i}  dA_ij  k_jc e^{Gamma_ic - Gamma_jc}
//   dkh = (Delta Dout^T) e^{Gamma_L - Gamma} + P3 + P4,
//         P3_jc = sum_{i >= j} dAqk_ij q_ic e^{Gamma_ic - Gamma_jc},
//         P4_jc = sum_{i > j} dA_ij beta_i k_ic e^{Gamma_ic - Gamma_jc},
//   dk = dkt + dkh,  dbeta = rowsum((V - K0 S) o dR) + rowsum(dA o B),
//   dGamma = q o dq + k o dkt - k o dkh  (+ rowsum(S_next o Dout) on the chunk's last row),
//   dg = the in-chunk suffix sum of dGamma.
// Every exponential is of a non-positive argument (Gamma is non-increasing), so nothing overflows
// whatever the decay: the pairwise products B, Aqk and P1..P4 take e^{-|Gamma_i - Gamma_j|}
// element by element instead of factoring it through a reference.  Launches, after the chunk table
// (its offsets per sequence, then first token, length and sequence of each chunk):
//   1. prep    one CTA per (chunk, head): the tiles above, Tm by forward substitution;
//   2. forward one CTA per (sequence, head): the states at chunk starts and Delta;
//   3. chain   one CTA per (sequence, head), chunks in reverse: Dout, dR and Din, with dS0 at the
//              sequence start; it needs no forward state, so 2 and 3 are one launch whose CTAs
//              run side by side;
//   4. grads   two CTAs per (chunk, head), one per half of the dk columns: dq, dk, dv, dg and
//              each half's share of dbeta.
// Prep and grads run in fp32 on CUDA cores; the two chains keep their carried matrix in tensor
// memory and run their products on the tensor cores (kind::tf32, operands split in two parts).
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include <atomic>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace k3kda {
namespace {

constexpr int kD = 128;
constexpr int kC = 16;             // tokens per chunk
constexpr int kThreads = 256;
constexpr int LD = kD + 1;         // padded row of a 128-wide tile in shared memory
constexpr int LC = kC + 1;         // padded row of a 16-wide tile

struct CbArgs {
    const void *q, *k, *v;
    int bf16;
    const float *g, *beta, *S0, *dO, *dSfin;
    const int32_t *cu;
    int N, T, H, Q;                // Q: chunks over all sequences
    float scale;
    int32_t *chunk_off;            // [N + 1]
    int32_t *ck_t0, *ck_len, *ck_seq;   // [Q]: first token, length and sequence of each chunk
    // per (chunk, head) item, fp32
    float *Q0, *K0, *Kd, *Gm, *W, *U;  // [item][kC][kD]  (Gm: the in-chunk cumulative log decay)
    float *Tm, *Aqk, *Bm;              // [item][kC][kC]
    float *gl;                         // [item][kD]      Gamma_L
    float *Dl, *dR;                    // [item][kC][kD]
    float *Dn;                         // [item][kD][kD]  Dout: the gradient reaching the chunk's S_next
    float *St;                         // [(Q + N) * H][kD][kD]: state at each chunk start, then the final
    float *dq, *dk, *dv, *dg, *dbeta, *dS0;
    unsigned *status;              // the workspace's status word: set when a bounded wait gave up
    unsigned test_limit;           // 0; else the armed test hook's tries (see TestTimeout)
    int *ready;                    // [item]: the chains that have written the item's rows (2: both)
    int *abort;                    // set by a chain that gave up: the grads stop waiting
};

__device__ __forceinline__ float ld_x(const void *p, size_t i, int bf16) {
    return bf16 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(p)[i]) : reinterpret_cast<const float *>(p)[i];
}
// Elements i .. i + 7 of an input (i a multiple of 8; the inputs are 16-byte aligned) in 16-byte
// pieces, or zeros when !ok.
__device__ __forceinline__ void ld_x8(const void *p, size_t i, int bf16, bool ok, float (&o)[8]) {
    if (!ok) {
#pragma unroll
        for (int x = 0; x < 8; ++x) o[x] = 0.f;
    } else if (bf16) {
        const uint4 r = __ldg(reinterpret_cast<const uint4 *>(reinterpret_cast<const __nv_bfloat16 *>(p) + i));
        const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int x = 0; x < 4; ++x) {
            const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w[x]));
            o[2 * x] = f.x;
            o[2 * x + 1] = f.y;
        }
    } else {
        const float4 a = __ldg(reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(p) + i));
        const float4 b = __ldg(reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(p) + i) + 1);
        o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w;
        o[4] = b.x; o[5] = b.y; o[6] = b.z; o[7] = b.w;
    }
}

// chunk offsets of the sequences (a prefix over N, one thread)
__global__ void __launch_bounds__(32) cb_offsets_kernel(CbArgs A) {
    if (threadIdx.x != 0) return;
    int acc = 0;
    A.chunk_off[0] = 0;
    for (int n = 0; n < A.N; ++n) {
        int b, e;
        seq_bounds(A.cu, n, A.T, b, e);
        acc += (e - b + kC - 1) / kC;
        A.chunk_off[n + 1] = acc;
    }
}

// the chunk table, one thread per chunk: its sequence by binary search over the offsets
__global__ void __launch_bounds__(256) cb_chunks_kernel(CbArgs A) {
    const int q = blockIdx.x * blockDim.x + threadIdx.x;
    if (q >= A.chunk_off[A.N]) return;
    int lo = 0, hi = A.N - 1;                          // the last n with chunk_off[n] <= q
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (A.chunk_off[mid] <= q) lo = mid;
        else hi = mid - 1;
    }
    int b, e;
    seq_bounds(A.cu, lo, A.T, b, e);
    const int t = b + (q - A.chunk_off[lo]) * kC;
    A.ck_t0[q] = t;
    A.ck_len[q] = min(kC, e - t);
    A.ck_seq[q] = lo;
}


template <int TM, int TN>
__device__ __forceinline__ void zero(float (&acc)[TM][TN]) {
#pragma unroll
    for (int v = 0; v < TM; ++v)
#pragma unroll
        for (int u = 0; u < TN; ++u) acc[v][u] = 0.f;
}

// Element (i, j) of a 16 x 16 tile for thread t: t < 136 takes element t of the lower triangle
// (j <= i) in row order, the other 120 threads the elements above the diagonal, so that the work on
// the lower triangle fills whole warps.
constexpr int kLow = kC * (kC + 1) / 2;
static_assert(kC * kC == kThreads, "one element of a 16 x 16 tile per thread");
__device__ __forceinline__ void tri_pair(int t, int &i, int &j) {
    if (t < kLow) {                                    // t = i (i + 1) / 2 + j, j <= i
        i = (int)((sqrtf(8.f * t + 1.f) - 1.f) * 0.5f);
        if ((i + 1) * (i + 2) / 2 <= t) ++i;
        if (i * (i + 1) / 2 > t) --i;
        j = t - i * (i + 1) / 2;
    } else {                                           // q = a (a - 1) / 2 + b, b < a: element (b, a)
        const int q = t - kLow;
        int a = (int)((sqrtf(8.f * q + 1.f) + 1.f) * 0.5f);
        if (a * (a - 1) / 2 > q) --a;
        if ((a + 1) * a / 2 <= q) ++a;
        i = q - a * (a - 1) / 2;
        j = a;
    }
}

// ---- 1. prep: one CTA per (chunk, head) ---------------------------------------------------------

__global__ void __launch_bounds__(kThreads, 6) cb_prep_kernel(const __grid_constant__ CbArgs A) {
    __shared__ float sG[kC][LD], sQ[kC][LD], sK[kC][LD], sX[kC][LD];
    __shared__ float sB[kC][LC], sT[kC][LC];
    __shared__ float sBeta[kC];
    const int tid = threadIdx.x;
    const int item = blockIdx.x, qc = item / A.H, h = item % A.H, H = A.H;
    // the grid covers an upper bound of the chunks (the tables have that many entries): the table
    // reads go out together, before the bound is known
    const int nq = A.chunk_off[A.N], t0 = A.ck_t0[qc], L = A.ck_len[qc];
    if (qc >= nq) return;
    // every load of the chunk's g, q and k rows goes out before the first store (one round trip
    // instead of one per element): 16-byte pieces, thread tid taking row i8 and channels c8 .. c8 + 7
    // of q and k (and later v) and two 4-channel pieces of g
    static_assert(kC * kD == 8 * kThreads, "one 8-channel piece of each row tensor per thread");
    const int i8 = tid >> 4, c8 = (tid & 15) * 8;
    const size_t src8 = ((size_t)(t0 + i8) * H + h) * kD + c8;
    float qv[8], kv[8];
    ld_x8(A.q, src8, A.bf16, i8 < L, qv);
    ld_x8(A.k, src8, A.bf16, i8 < L, kv);
    float4 gv[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        const int e = tid + u * kThreads, i = e >> 5, c = (e & 31) * 4;
        gv[u] = i < L ? __ldg(reinterpret_cast<const float4 *>(A.g + ((size_t)(t0 + i) * H + h) * kD + c))
                      : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    const float bv = tid < kC && tid < L ? A.beta[(size_t)(t0 + tid) * H + h] : 0.f;
#pragma unroll
    for (int x = 0; x < 8; ++x) {
        sQ[i8][c8 + x] = qv[x];
        sK[i8][c8 + x] = kv[x];
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        const int e = tid + u * kThreads, i = e >> 5, c = (e & 31) * 4;
        sG[i][c] = gv[u].x; sG[i][c + 1] = gv[u].y; sG[i][c + 2] = gv[u].z; sG[i][c + 3] = gv[u].w;
    }
    if (tid < kC) sBeta[tid] = bv;
    __syncthreads();
    if (tid < kD) {
        float run = 0.f;
        for (int i = 0; i < kC; ++i) { run += sG[i][tid]; sG[i][tid] = run; }
        A.gl[(size_t)item * kD + tid] = sG[L - 1][tid];
    }
    __syncthreads();
    const size_t tile = (size_t)item * kC * kD;
    for (int e = tid; e < kC * kD; e += kThreads) {
        const int i = e / kD, c = e % kD;
        const float gm = sG[i][c], ea = __expf(gm), ed = __expf(sG[kC - 1][c] - gm);
        const float k0 = sK[i][c] * ea;
        A.Q0[tile + e] = sQ[i][c] * ea;
        A.K0[tile + e] = k0;
        A.Kd[tile + e] = sK[i][c] * ed;
        A.Gm[tile + e] = gm;
        sX[i][c] = sBeta[i] * k0;                      // beta K0, the right factor of W
    }
    {
        // B = strict_lower, Aqk = lower of the decayed products, each term with its own exponential
        // e^{Gamma_ic - Gamma_jc} <= 1 (j <= i): the loop on the lower triangle's threads only
        int i, j;
        tri_pair(tid, i, j);
        float b1 = 0.f, b2 = 0.f;
        if (tid < kLow) {
#pragma unroll 4
            for (int c = 0; c < kD; ++c) {
                const float t = sK[j][c] * __expf(sG[i][c] - sG[j][c]);
                b1 = fmaf(sK[i][c], t, b1);
                b2 = fmaf(sQ[i][c], t, b2);
            }
        }
        const float bv = j < i ? b1 : 0.f, av = j <= i ? b2 : 0.f;
        sB[i][j] = bv;
        A.Bm[(size_t)item * kC * kC + i * kC + j] = bv;
        A.Aqk[(size_t)item * kC * kC + i * kC + j] = av;
    }
    __syncthreads();
    {
        // Tm = (I + diag(beta) B)^-1 by forward substitution, x_i = -beta_i sum_{j<i} B_ij x_j down
        // column col (x_col = 1, zero above): thread (col, r) holds x_r, and the sum for row i runs
        // over the column's 16 threads (a half-warp) by shuffles
        static_assert(kC * kC == kThreads && kC == 16, "one thread per element, a column per half-warp");
        const int col = tid >> 4, r = tid & 15;
        float xr = r == col ? 1.f : 0.f;
#pragma unroll
        for (int i = 1; i < kC; ++i) {
            float p = r < i ? sB[i][r] * xr : 0.f;
#pragma unroll
            for (int o = 1; o < 16; o <<= 1) p += __shfl_xor_sync(0xffffffffu, p, o, 16);
            if (r == i && i > col) xr = -sBeta[i] * p;
        }
        sT[r][col] = xr;
    }
    __syncthreads();
    A.Tm[(size_t)item * kC * kC + tid] = sT[tid / kC][tid % kC];
    // W = Tm diag(beta) K0, U = Tm diag(beta) V (beta V into sG, whose Gamma is no longer needed)
    {
        float vv[8];
        ld_x8(A.v, src8, A.bf16, i8 < L, vv);
#pragma unroll
        for (int x = 0; x < 8; ++x) sG[i8][c8 + x] = sBeta[i8] * vv[x];
    }
    __syncthreads();
    {
        // row i of W and U over columns tn + 16 x: Tm is lower triangular, so the sums stop at kk = i
        const int i = tid / (kD / 8), tn = tid % (kD / 8);
        float w[1][8], u[1][8];
        zero(w); zero(u);
        for (int kk = 0; kk <= i; ++kk) {
            const float t = sT[i][kk];
#pragma unroll
            for (int x = 0; x < 8; ++x) {
                w[0][x] = fmaf(t, sX[kk][tn + (kD / 8) * x], w[0][x]);
                u[0][x] = fmaf(t, sG[kk][tn + (kD / 8) * x], u[0][x]);
            }
        }
#pragma unroll
        for (int x = 0; x < 8; ++x) {
            const int c = tn + (kD / 8) * x;
            A.W[tile + i * kD + c] = w[0][x];
            A.U[tile + i * kD + c] = u[0][x];
        }
    }
}

// ---- staging: 16-byte cp.async pieces, one commit group per chunk ------------------------------------

__device__ __forceinline__ void cp16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)), "l"(src)
                 : "memory");
}
// copies `bytes` (0 or 16) and zero-fills the rest of the 16 bytes
__device__ __forceinline__ void cp16z(void *dst, const void *src, int bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)), "l"(src),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// a [kC][kD] fp32 tile (rows of 512 B) into a [kC][ld] shared tile
__device__ __forceinline__ void stage_tile(float *dst, int ld, const float *src) {
    for (int e = threadIdx.x; e < kC * (kD / 4); e += kThreads) {
        const int i = e / (kD / 4), p = e % (kD / 4);
        cp16(dst + i * ld + p * 4, src + (size_t)i * kD + p * 4);
    }
}
__device__ __forceinline__ void stage_vec(float *dst, const float *src, int n) {
    for (int e = threadIdx.x; e < n / 4; e += kThreads) cp16(dst + e * 4, src + e * 4);
}

// ---- 2 + 3. the chains, on the tensor cores ----------------------------------------------------
// One CTA per (sequence, head) for each chain.  The forward chain carries the state S over the
// chunks (writing the state at every chunk start and Delta); the backward chain, chunks in
// reverse, carries Dout, the gradient reaching a chunk's S_next (writing Dout and dR, and dS0 at the
// sequence start); it needs no forward state, so the two run side by side in one launch.  The
// carried matrix stays in tensor memory transposed (lane j = dv channel, column c = dk channel)
// and every product runs as tcgen05 kind::tf32 MMAs on split operands x = hi + lo (hi rounded to
// tf32, lo the fp32 remainder) summed as hi.hi + hi.lo + lo.hi, which keeps fp32 accuracy:
//   forward   Delta^T = U^T - S^T W^T            (A = S^T from TMEM, K = dk)
//             S^T <- e^{Gamma_L} S^T + Delta^T Kd (A = Delta^T from shared memory, K = the chunk's tokens)
//   backward  dDelta^T = Dout^T Kd^T + dOs^T Aqk (A = Dout^T from TMEM, then dOs^T from shared memory)
//             dR^T = dDelta^T Tm                 (CUDA cores: 16 x 16 per dv channel)
//             Dout^T <- e^{Gamma_L} Dout^T + [dOs | -beta dR]^T [Q0; K0]   (A from shared memory)
// The B operands are built per chunk from the prep's fp32 tiles into 128-byte-swizzled K-major
// shared tiles, one chunk ahead, while the MMAs run; the A operands over the chunk's tokens are
// written by the threads that own their rows.

constexpr int kTcData = 512;                           // threads that own TMEM rows (16 warps)
constexpr int kTcThreads = kTcData + 32;               // and a warp whose lane 0 issues the MMAs
constexpr int kIssuer = kTcData;
constexpr uint32_t kTcCols = 512;
// tensor-memory columns: the carried matrix (fp32), its hi and lo parts (the A operand of the
// product over dk), and four 32-column accumulators that the product over dk cycles through (a
// chain of small MMAs into one accumulator waits on each one's write-back)
constexpr uint32_t TC_S = 0, TC_SH = 128, TC_SL = 256, TC_D = 384;
constexpr int kAcc = 4;
constexpr uint32_t kTcWait = 1u << 26;                 // polls of an MMA completion wait

// shared memory (bytes from the 1024-aligned base)
// forward: per stage, [W_hi; W_lo] (32 rows x 128 K, 4 atoms of 4 KB), Kd^T hi and lo (128 rows x
// 16 K, one atom each), e^{Gamma_L}; raw fp32 W and Kd tiles and Gamma_L as copied; the A operand
// over the chunk's tokens, Delta^T hi and lo (128 rows x 16 K)
constexpr uint32_t F_XW = 0, F_KH = 32768, F_GL = 98304, F_RAW = 99328, F_RAW_BYTES = 16896, F_AT = 133120,
                   F_MISC = 165888;
// backward: per stage, [Kd_hi; Kd_lo] (32 x 128 K) then [Aqk_hi; Aqk_lo] as B(m, t) = Aqk[m][t]
// (32 rows x 16 K), [Q0^T | K0^T] hi and lo (128 rows x 32 K); e^{Gamma_L}, beta, Tm; raw fp32 Kd,
// Q0, K0, Aqk, Tm tiles, Gamma_L and beta as copied; the A operand over the chunk's tokens,
// [dOs | -beta dR]^T hi and lo (128 rows x 32 K)
constexpr uint32_t B_X1 = 0, B_X4 = 40960, B_SMALL = 106496, B_SMALL_BYTES = 1664, B_RAW = 109824,
                   B_RAW_BYTES = 27200, B_AT = 164864, B_MISC = 197632;
constexpr size_t kTcSmem = 1024 + 197632 + 64;
static_assert(F_MISC <= B_MISC, "the backward layout is the larger one");
static_assert(F_AT % 1024 == 0 && B_AT % 1024 == 0, "swizzled tiles start on 1024-byte boundaries");
static_assert(F_RAW + 2 * F_RAW_BYTES <= F_AT && B_RAW + 2 * B_RAW_BYTES <= B_AT, "raw stages fit");

// byte offsets inside a raw backward stage
constexpr uint32_t BR_KD = 0, BR_Q0 = 8192, BR_K0 = 16384, BR_AQK = 24576, BR_TM = 25600, BR_GL = 26624,
                   BR_BETA = 27136;
// inside a small backward stage: e^{Gamma_L} [128], beta [16], Tm [16][16]
constexpr uint32_t BS_EGL = 0, BS_BETA = 512, BS_TM = 576;

// n_floats of fp32 at src into raw shared memory (16-byte pieces, this thread's commit group),
// by the data threads
__device__ __forceinline__ void tc_stage(uint8_t *dst, const float *src, int n_floats) {
    for (int e = threadIdx.x; e < n_floats / 4; e += kTcData) cp16(dst + e * 16, src + e * 4);
}
// four fp32 values split into hi and lo, stored as one 16-byte chunk each at byte offset o of the
// hi and lo tiles
__device__ __forceinline__ void put_split4(uint8_t *hi_tile, uint8_t *lo_tile, uint32_t o, float a, float b, float c,
                                           float d) {
    uint4 h, l;
    tc::split_tf32(a, h.x, l.x);
    tc::split_tf32(b, h.y, l.y);
    tc::split_tf32(c, h.z, l.z);
    tc::split_tf32(d, h.w, l.w);
    *reinterpret_cast<uint4 *>(hi_tile + o) = h;
    *reinterpret_cast<uint4 *>(lo_tile + o) = l;
}

// One thread marks an item's rows as written by this chain (release: every thread's stores came
// before the barrier that precedes the call).
__device__ __forceinline__ void publish_item(int *ready) {
    __threadfence();
    asm volatile("red.release.gpu.global.add.s32 [%0], 1;" ::"l"(ready) : "memory");
}

__global__ void __launch_bounds__(kTcThreads, 1) cb_tc_chains_kernel(const __grid_constant__ CbArgs A) {
    using namespace tc;
    // the grads (a programmatic dependent launch) may start on the SMs this grid leaves free
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    extern __shared__ uint8_t smraw[];
    uint8_t *sm = smem_align1024(smraw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool data = tid < kTcData, iss = tid == kIssuer;
    const int lq = warp & 3, cg = warp >> 2;           // TMEM lane quarter; column / token group
    const int j = 32 * lq + lane;                      // this thread's dv channel (TMEM lane)
    const int NH = A.N * A.H, H = A.H;
    const bool fwd = (int)blockIdx.x < NH;
    const int nh = fwd ? blockIdx.x : blockIdx.x - NH, n = nh / H, h = nh % H;
    const uint32_t misc = fwd ? F_MISC : B_MISC;
    uint64_t *mbar = reinterpret_cast<uint64_t *>(sm + misc);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + misc + 8);
    volatile uint32_t *sflag = reinterpret_cast<volatile uint32_t *>(sm + misc + 12);
    const uint32_t sbase = smem_u32(sm), mb = smem_u32(mbar);
    if (warp == 0) { tmem_alloc(smem_u32(tslot), kTcCols); tmem_relinquish(); }
    if (tid == 0) { mbar_init(mb, 1); fence_mbar_init(); *sflag = 0; }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tslot;
    const uint32_t tl = tbase + ((uint32_t)(32 * lq) << 16);
    uint32_t ph = 0;
    bool pend = false, failed = false;
    // test hook: the first forward chain issues no MMA for its first chunk and gives up that wait
    // after the armed number of tries
    bool starve = A.test_limit != 0 && blockIdx.x == 0;
    // the issuer waits for the MMAs it committed; everyone learns whether the wait ran out
    auto mma_wait = [&]() -> bool {
        if (iss && pend) {
            if (mbar_wait_bounded(mb, ph, starve ? A.test_limit : kTcWait)) {
                ph ^= 1u;
                pend = false;
            } else {
                *sflag = 1;
                atomicOr(A.status, 1u);
                atomicExch(A.abort, 1);                // the grads waiting for this chain's items stop
                if (starve) pend = false;              // nothing was issued for it
            }
            starve = false;
        }
        __syncthreads();
        tc_fence_after();
        return *sflag == 0;
    };
    // the carried matrix's row j, columns [32 cg, 32 cg + 32): into TMEM with its hi and lo parts
    auto put_carried = [&](const float (&x)[32], bool with_fp32) {
#pragma unroll
        for (int b = 0; b < 2; ++b) {
            uint32_t r[16], hi[16], lo[16];
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                r[u] = __float_as_uint(x[16 * b + u]);
                split_tf32(x[16 * b + u], hi[u], lo[u]);
            }
            if (with_fp32) tmem_st16(tl + TC_S + 32 * cg + 16 * b, r);
            tmem_st16(tl + TC_SH + 32 * cg + 16 * b, hi);
            tmem_st16(tl + TC_SL + 32 * cg + 16 * b, lo);
        }
    };
    auto get_carried = [&](float (&x)[32]) {
        uint32_t r[2][16];
        tmem_ld16(tl + TC_S + 32 * cg, r[0]);
        tmem_ld16(tl + TC_S + 32 * cg + 16, r[1]);
        tmem_wait_ld();
#pragma unroll
        for (int u = 0; u < 32; ++u) x[u] = __uint_as_float(r[u >> 4][u & 15]);
    };
    // x written out, then x -> e^{Gamma_L} x (row j's columns) into the fp32 columns
    auto scale_carried = [&](float (&x)[32], const float *egl, float *out) {
#pragma unroll
        for (int u = 0; u < 32; u += 4) {
            const float4 e4 = *reinterpret_cast<const float4 *>(egl + 32 * cg + u);
            out[(size_t)(32 * cg + u) * kD] = x[u];
            out[(size_t)(32 * cg + u + 1) * kD] = x[u + 1];
            out[(size_t)(32 * cg + u + 2) * kD] = x[u + 2];
            out[(size_t)(32 * cg + u + 3) * kD] = x[u + 3];
            x[u] *= e4.x; x[u + 1] *= e4.y; x[u + 2] *= e4.z; x[u + 3] *= e4.w;
        }
        uint32_t r[16];
#pragma unroll
        for (int b = 0; b < 2; ++b) {
#pragma unroll
            for (int u = 0; u < 16; ++u) r[u] = __float_as_uint(x[16 * b + u]);
            tmem_st16(tl + TC_S + 32 * cg + 16 * b, r);
        }
    };
    // e^{Gamma_L} x (row j's columns) into the fp32 columns, x left as it is
    auto scale_into_tmem = [&](const float (&x)[32], const float *egl) {
        uint32_t r[16];
#pragma unroll
        for (int b = 0; b < 2; ++b) {
#pragma unroll
            for (int u = 0; u < 16; u += 4) {
                const float4 e4 = *reinterpret_cast<const float4 *>(egl + 32 * cg + 16 * b + u);
                r[u] = __float_as_uint(x[16 * b + u] * e4.x);
                r[u + 1] = __float_as_uint(x[16 * b + u + 1] * e4.y);
                r[u + 2] = __float_as_uint(x[16 * b + u + 2] * e4.z);
                r[u + 3] = __float_as_uint(x[16 * b + u + 3] * e4.w);
            }
            tmem_st16(tl + TC_S + 32 * cg + 16 * b, r);
        }
    };
    // half b of row j's columns of x out to [dk][dv] (the stores are spread over two MMA windows)
    auto store_half = [&](const float (&x)[32], int b, float *out) {
#pragma unroll
        for (int u = 0; u < 16; ++u) out[(size_t)(32 * cg + 16 * b + u) * kD] = x[16 * b + u];
    };
    // the accumulators' sum over this thread's four tokens [4 cg, 4 cg + 4) (and + 16: the lo rows)
    auto sum_acc4 = [&](float (&d)[4]) {
        uint32_t r[2 * kAcc][4];
#pragma unroll
        for (int a = 0; a < kAcc; ++a) {
            tmem_ld4(tl + TC_D + 32 * a + 4 * cg, r[2 * a]);
            tmem_ld4(tl + TC_D + 32 * a + 16 + 4 * cg, r[2 * a + 1]);
        }
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float acc = 0.f;
#pragma unroll
            for (int a = 0; a < 2 * kAcc; ++a) acc += __uint_as_float(r[a][i]);
            d[i] = acc;
        }
    };
    const int q0 = A.chunk_off[n], nq = A.chunk_off[n + 1] - q0;
    int tb, te;                                        // the sequence's tokens: chunk c starts at tb + 16 c
    seq_bounds(A.cu, n, A.T, tb, te);
    float X[32];                                       // the carried matrix, row j, this thread's columns
    const uint32_t idN32 = idesc_tf32_f32(128, 32), idN16 = idesc_tf32_f32(128, 16), idN128 = idesc_tf32_f32(128, 128);
    // MMAs over dk: A = the carried matrix's hi / lo columns, B = a 32-row tile (hi rows 0-15, lo
    // rows 16-31) of 4 K atoms; K step kk goes to accumulator kk mod kAcc
    auto issue_over_dk = [&](uint32_t btile) {
        const uint64_t dB = sdesc_kmajor_sw128(sbase + btile);
#pragma unroll
        for (int kk = 0; kk < 16; ++kk)
            mma_tf32_ta(tbase + TC_D + 32 * (kk % kAcc), tbase + TC_SH + 8 * kk, dadd(dB, (kk >> 2) * 4096 + (kk & 3) * 32),
                        idN32, kk >= kAcc);
#pragma unroll
        for (int kk = 0; kk < 16; ++kk)
            mma_tf32_ta(tbase + TC_D + 32 * (kk % kAcc), tbase + TC_SL + 8 * kk, dadd(dB, (kk >> 2) * 4096 + (kk & 3) * 32),
                        idN16, 1);
    };

    if (fwd) {
        // ================= forward chain: S at every chunk start, Delta =================
        uint8_t *ath = sm + F_AT, *atl = sm + F_AT + 16384;
        auto raw = [&](int s) { return sm + F_RAW + s * F_RAW_BYTES; };
        auto stage_raw = [&](int c) {                // chunk c's W and Kd tiles into raw stage c & 1
            const size_t tile = ((size_t)(q0 + c) * H + h) * kC * kD;
            tc_stage(raw(c & 1), A.W + tile, kC * kD);
            tc_stage(raw(c & 1) + 8192, A.Kd + tile, kC * kD);
            tc_stage(raw(c & 1) + 16384, A.gl + ((size_t)(q0 + c) * H + h) * kD, kD);
            cp_commit();
        };
        auto build = [&](int c) {                    // raw stage c & 1 -> operand stage c & 1
            const int s = c & 1;
            const float *rw = reinterpret_cast<const float *>(raw(s)), *rk = rw + kC * kD;
            uint8_t *xw = sm + F_XW + s * 16384;
            uint8_t *kh = sm + F_KH + s * 32768, *kl = kh + 16384;
            {   // B(c, t) = W[t][c]: row t (hi), 16 + t (lo), four c per thread
                const int t = tid >> 5, c4 = (tid & 31) * 4;
                const float4 w = *reinterpret_cast<const float4 *>(rw + t * kD + c4);
                uint4 hv, lv;
                split_tf32(w.x, hv.x, lv.x); split_tf32(w.y, hv.y, lv.y);
                split_tf32(w.z, hv.z, lv.z); split_tf32(w.w, hv.w, lv.w);
                *reinterpret_cast<uint4 *>(xw + sw128_offset_f32(t, c4, 4096)) = hv;
                *reinterpret_cast<uint4 *>(xw + sw128_offset_f32(16 + t, c4, 4096)) = lv;
            }
            {   // B(t, c) = Kd[t][c]: row c, four t per thread
                const int c2 = tid & 127, t4 = (tid >> 7) * 4;
                put_split4(kh, kl, sw128_offset_f32(c2, t4, 16384), rk[t4 * kD + c2], rk[(t4 + 1) * kD + c2],
                           rk[(t4 + 2) * kD + c2], rk[(t4 + 3) * kD + c2]);
            }
            if (tid < kD) reinterpret_cast<float *>(sm + F_GL + s * 512)[tid] = expf(rw[2 * kC * kD + tid]);
        };
        if (data) {
#pragma unroll
            for (int u = 0; u < 32; ++u) X[u] = A.S0 ? A.S0[((size_t)nh * kD + 32 * cg + u) * kD + j] : 0.f;
            put_carried(X, true);
            tmem_wait_st();
            if (nq > 0) stage_raw(0);
            if (nq > 1) stage_raw(1);
            cp_wait<0>();
            named_bar(1, kTcData);
            if (nq > 0) build(0);
            fence_async_smem();
        }
        tc_fence_before();
        __syncthreads();
        for (int c = 0; c < nq; ++c) {
            const int s = c & 1;
            const size_t tile = ((size_t)(q0 + c) * H + h) * kC * kD;
            // ---- MMA: D = S^T [W_hi; W_lo]^T (N = 32) + S_lo^T W_hi^T (N = 16), over four accumulators ----
            if (iss) {
                tc_fence_after();
                if (!starve) {
                    issue_over_dk(F_XW + s * 16384);
                    mma_commit(mb);
                }
                pend = true;
            }
            // while it runs: U of this chunk, S_c out, S <- e^{Gamma_L} S, the next chunk's operands
            float u4[4];
            if (data) {
#pragma unroll
                for (int i = 0; i < 4; ++i) u4[i] = A.U[tile + (size_t)(4 * cg + i) * kD + j];
                scale_carried(X, reinterpret_cast<const float *>(sm + F_GL + s * 512),
                              A.St + ((size_t)(q0 + c + n) * H + h) * kD * kD + j);
                cp_wait<0>();
                named_bar(1, kTcData);
                if (c + 1 < nq) build(c + 1);
                fence_async_smem();
                if (c + 2 < nq) stage_raw(c + 2);
                tmem_wait_st();
            }
            if (!mma_wait()) { failed = true; break; }
            // ---- Delta^T = U^T - D, four tokens per thread: out, and split for the next MMA ----
            if (data) {
                float d[4];
                sum_acc4(d);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    d[i] = u4[i] - d[i];
                    A.Dl[tile + (size_t)(4 * cg + i) * kD + j] = d[i];
                }
                put_split4(ath, atl, sw128_offset_f32(j, 4 * cg, 16384), d[0], d[1], d[2], d[3]);
                fence_async_smem();
            }
            tc_fence_before();
            __syncthreads();
            // ---- MMA: S^T += Delta^T Kd  (hi.hi + hi.lo + lo.hi, K = 16 tokens) ----
            if (iss) {
                tc_fence_after();
                const uint64_t dAh = sdesc_kmajor_sw128(sbase + F_AT), dAl = sdesc_kmajor_sw128(sbase + F_AT + 16384);
                const uint64_t dKh = sdesc_kmajor_sw128(sbase + F_KH + s * 32768),
                               dKl = sdesc_kmajor_sw128(sbase + F_KH + s * 32768 + 16384);
#pragma unroll
                for (int sp = 0; sp < 3; ++sp)
#pragma unroll
                    for (int kk = 0; kk < 2; ++kk)
                        mma_tf32(tbase + TC_S, dadd(sp == 2 ? dAl : dAh, kk * 32), dadd(sp == 1 ? dKl : dKh, kk * 32), idN128, 1);
                mma_commit(mb);
                pend = true;
            }
            if (!mma_wait()) { failed = true; break; }
            if (data) {
                get_carried(X);
                put_carried(X, false);
                tmem_wait_st();
            }
            tc_fence_before();
            __syncthreads();
            // chunk c - 1's rows are all written (its state, its Delta, and the state after it)
            if (tid == 0 && c >= 1) publish_item(A.ready + (tile / (kC * kD) - H));
        }
        if (!failed && data) {
            float *st = A.St + ((size_t)(q0 + nq + n) * H + h) * kD * kD + j;
#pragma unroll
            for (int u = 0; u < 32; ++u) st[(size_t)(32 * cg + u) * kD] = X[u];
        }
        __syncthreads();
        if (tid == 0 && !failed && nq >= 1) publish_item(A.ready + (size_t)(q0 + nq - 1) * H + h);
    } else {
        // ================= backward chain: Dout, dR; dS0 =================
        const float scale = A.scale;
        uint8_t *ath = sm + B_AT, *atl = sm + B_AT + 16384;
        auto raw = [&](int s) { return sm + B_RAW + s * B_RAW_BYTES; };
        auto small = [&](int s) { return sm + B_SMALL + s * B_SMALL_BYTES; };
        // iteration it handles chunk c = nq - 1 - it in stage it & 1 (the raw stage likewise)
        auto stage_raw = [&](int c, int s) {
            const size_t item = (size_t)(q0 + c) * H + h, tile = item * kC * kD, sml = item * kC * kC;
            tc_stage(raw(s) + BR_KD, A.Kd + tile, kC * kD);
            tc_stage(raw(s) + BR_Q0, A.Q0 + tile, kC * kD);
            tc_stage(raw(s) + BR_K0, A.K0 + tile, kC * kD);
            tc_stage(raw(s) + BR_AQK, A.Aqk + sml, kC * kC);
            tc_stage(raw(s) + BR_TM, A.Tm + sml, kC * kC);
            tc_stage(raw(s) + BR_GL, A.gl + item * kD, kD);
            if (threadIdx.x < kC) {                      // beta is strided by H: 4-byte pieces, zero past the end
                const int t = tb + c * kC + (int)threadIdx.x;
                const float *src = A.beta + (size_t)(t < te ? t : tb + c * kC) * H + h;
                asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_u32(raw(s) + BR_BETA + 4 * threadIdx.x)),
                             "l"(src), "r"(t < te ? 4 : 0)
                             : "memory");
            }
            cp_commit();
        };
        auto build = [&](int c, int s) {
            const uint8_t *r = raw(s);
            const float *rkd = reinterpret_cast<const float *>(r + BR_KD), *rq = reinterpret_cast<const float *>(r + BR_Q0),
                        *rk = reinterpret_cast<const float *>(r + BR_K0);
            uint8_t *x1 = sm + B_X1 + s * 20480, *xa = x1 + 16384;
            uint8_t *x4h = sm + B_X4 + s * 32768, *x4l = x4h + 16384;
            {   // B(c, t) = Kd[t][c]: row t (hi), 16 + t (lo), four c per thread
                const int t = tid >> 5, c4 = (tid & 31) * 4;
                const float4 w = *reinterpret_cast<const float4 *>(rkd + t * kD + c4);
                uint4 hv, lv;
                split_tf32(w.x, hv.x, lv.x); split_tf32(w.y, hv.y, lv.y);
                split_tf32(w.z, hv.z, lv.z); split_tf32(w.w, hv.w, lv.w);
                *reinterpret_cast<uint4 *>(x1 + sw128_offset_f32(t, c4, 4096)) = hv;
                *reinterpret_cast<uint4 *>(x1 + sw128_offset_f32(16 + t, c4, 4096)) = lv;
            }
            {   // B(t, c) = Q0[t][c] and B(16 + t, c) = K0[t][c]: row c, four t per thread
                const int c2 = tid & 127, t4 = (tid >> 7) * 4;
                put_split4(x4h, x4l, sw128_offset_f32(c2, t4, 16384), rq[t4 * kD + c2], rq[(t4 + 1) * kD + c2],
                           rq[(t4 + 2) * kD + c2], rq[(t4 + 3) * kD + c2]);
                put_split4(x4h, x4l, sw128_offset_f32(c2, 16 + t4, 16384), rk[t4 * kD + c2], rk[(t4 + 1) * kD + c2],
                           rk[(t4 + 2) * kD + c2], rk[(t4 + 3) * kD + c2]);
            }
            if (tid < kC * kC / 4) {                     // B(m, t) = Aqk[m][t]: row t, four m per thread
                const int t = tid & 15, m4 = (tid >> 4) * 4;
                const float *ra = reinterpret_cast<const float *>(r + BR_AQK);
                uint4 hv, lv;
                split_tf32(ra[m4 * kC + t], hv.x, lv.x);
                split_tf32(ra[(m4 + 1) * kC + t], hv.y, lv.y);
                split_tf32(ra[(m4 + 2) * kC + t], hv.z, lv.z);
                split_tf32(ra[(m4 + 3) * kC + t], hv.w, lv.w);
                *reinterpret_cast<uint4 *>(xa + sw128_offset_f32(t, m4, 4096)) = hv;
                *reinterpret_cast<uint4 *>(xa + sw128_offset_f32(16 + t, m4, 4096)) = lv;
            }
            if (tid < kC * kC) reinterpret_cast<float *>(small(s) + BS_TM)[tid] = reinterpret_cast<const float *>(r + BR_TM)[tid];
            if (tid < kD)
                reinterpret_cast<float *>(small(s) + BS_EGL)[tid] = expf(reinterpret_cast<const float *>(r + BR_GL)[tid]);
            if (tid < kC) reinterpret_cast<float *>(small(s) + BS_BETA)[tid] = reinterpret_cast<const float *>(r + BR_BETA)[tid];
        };
        // dO of chunk c at tokens [4 cg, 4 cg + 4) of channel j (zero past the sequence's end)
        auto load_do = [&](int c, float (&o)[4]) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int t = tb + c * kC + 4 * cg + i;
                o[i] = t < te ? A.dO[((size_t)t * H + h) * kD + j] : 0.f;
            }
        };
        auto put_dos = [&](const float (&o)[4]) {
            put_split4(ath, atl, sw128_offset_f32(j, 4 * cg, 16384), scale * o[0], scale * o[1], scale * o[2], scale * o[3]);
        };
        float dov[4];
        if (data) {
#pragma unroll
            for (int u = 0; u < 32; ++u) X[u] = A.dSfin ? A.dSfin[((size_t)nh * kD + 32 * cg + u) * kD + j] : 0.f;
            put_carried(X, true);
            if (nq > 0) {
                load_do(nq - 1, dov);
                put_dos(dov);
            }
            tmem_wait_st();
            if (nq > 0) stage_raw(nq - 1, 0);
            if (nq > 1) stage_raw(nq - 2, 1);
            cp_wait<0>();
            named_bar(1, kTcData);
            if (nq > 0) build(nq - 1, 0);
            fence_async_smem();
        }
        tc_fence_before();
        __syncthreads();
        for (int it = 0; it < nq; ++it) {
            const int c = nq - 1 - it, s = it & 1;
            const size_t item = (size_t)(q0 + c) * H + h, tile = item * kC * kD;
            // ---- MMA: D = Dout^T [Kd_hi; Kd_lo]^T + dOs^T [Aqk_hi; Aqk_lo] (N = 32), then the lo
            // parts of the A operands against the hi rows (N = 16), over four accumulators ----
            if (iss) {
                tc_fence_after();
                issue_over_dk(B_X1 + s * 20480);
                const uint64_t dAh = sdesc_kmajor_sw128(sbase + B_AT), dAl = sdesc_kmajor_sw128(sbase + B_AT + 16384);
                const uint64_t dQ = sdesc_kmajor_sw128(sbase + B_X1 + s * 20480 + 16384);
#pragma unroll
                for (int kk = 0; kk < 2; ++kk) mma_tf32(tbase + TC_D + 32 * kk, dadd(dAh, kk * 32), dadd(dQ, kk * 32), idN32, 1);
#pragma unroll
                for (int kk = 0; kk < 2; ++kk) mma_tf32(tbase + TC_D + 32 * (2 + kk), dadd(dAl, kk * 32), dadd(dQ, kk * 32), idN16, 1);
                mma_commit(mb);
                pend = true;
            }
            // while it runs: Dout of this chunk out, Dout <- e^{Gamma_L} Dout, dO of the next
            // chunk, the next chunk's operands
            if (data) {
                scale_into_tmem(X, reinterpret_cast<const float *>(small(s) + BS_EGL));
                store_half(X, 0, A.Dn + item * kD * kD + j);
                if (c >= 1) load_do(c - 1, dov);
                cp_wait<0>();
                named_bar(1, kTcData);
                if (c >= 1) build(c - 1, s ^ 1);
                fence_async_smem();
                if (c >= 2) stage_raw(c - 2, s);
                tmem_wait_st();
            }
            if (!mma_wait()) { failed = true; break; }
            // ---- dDelta (all 16 tokens of channel j), dR = Tm^T dDelta for this thread's four ----
            if (data) {
                float dd[kC];                            // dDelta[m][j], summed over the accumulators
#pragma unroll
                for (int m = 0; m < kC; ++m) dd[m] = 0.f;
#pragma unroll
                for (int a = 0; a < kAcc; ++a) {
                    uint32_t r0[16], r1[16];
                    tmem_ld16(tl + TC_D + 32 * a, r0);
                    tmem_ld16(tl + TC_D + 32 * a + 16, r1);
                    tmem_wait_ld();
#pragma unroll
                    for (int m = 0; m < kC; ++m) dd[m] += __uint_as_float(r0[m]) + __uint_as_float(r1[m]);
                }
                const float *tm = reinterpret_cast<const float *>(small(s) + BS_TM);
                const float4 be = *reinterpret_cast<const float4 *>(small(s) + BS_BETA + 16 * cg);
                float dr[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int m = 0; m < kC; ++m) {
                    const float4 t4 = *reinterpret_cast<const float4 *>(tm + m * kC + 4 * cg);
                    dr[0] = fmaf(t4.x, dd[m], dr[0]); dr[1] = fmaf(t4.y, dd[m], dr[1]);
                    dr[2] = fmaf(t4.z, dd[m], dr[2]); dr[3] = fmaf(t4.w, dd[m], dr[3]);
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) A.dR[tile + (size_t)(4 * cg + i) * kD + j] = dr[i];
                put_split4(ath, atl, sw128_offset_f32(j, 16 + 4 * cg, 16384), -be.x * dr[0], -be.y * dr[1], -be.z * dr[2],
                           -be.w * dr[3]);
                fence_async_smem();
            }
            tc_fence_before();
            __syncthreads();
            // ---- MMA: Dout^T += [dOs | -beta dR]^T [Q0; K0]  (hi.hi + hi.lo + lo.hi, K = 32) ----
            if (iss) {
                tc_fence_after();
                const uint64_t dAh = sdesc_kmajor_sw128(sbase + B_AT), dAl = sdesc_kmajor_sw128(sbase + B_AT + 16384);
                const uint64_t dH = sdesc_kmajor_sw128(sbase + B_X4 + s * 32768),
                               dL = sdesc_kmajor_sw128(sbase + B_X4 + s * 32768 + 16384);
#pragma unroll
                for (int sp = 0; sp < 3; ++sp)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_tf32(tbase + TC_S, dadd(sp == 2 ? dAl : dAh, kk * 32), dadd(sp == 1 ? dL : dH, kk * 32), idN128, 1);
                mma_commit(mb);
                pend = true;
            }
            if (data) store_half(X, 1, A.Dn + item * kD * kD + j);   // while it runs
            if (!mma_wait()) { failed = true; break; }
            if (data) {
                get_carried(X);
                put_carried(X, false);
                if (c >= 1) {
                    put_dos(dov);
                    fence_async_smem();
                }
                tmem_wait_st();
            }
            tc_fence_before();
            __syncthreads();
            if (tid == 0) publish_item(A.ready + item);    // chunk c's Dout and dR rows are written
        }
        if (!failed && data) {
            float *d0 = A.dS0 + (size_t)nh * kD * kD + j;
#pragma unroll
            for (int u = 0; u < 32; ++u) d0[(size_t)(32 * cg + u) * kD] = X[u];
        }
    }
    // after a failure, let the MMAs in flight land (bounded) before the columns are freed
    if (iss && pend) mbar_wait_bounded(mb, ph, kTcWait);
    cp_wait<0>();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tbase, kTcCols);
}

// ---- 4. grads: two CTAs per (chunk, head), one per half of the dk columns --------------------------
// Every product below that runs over dk (dq, dkt, dkh and so dk, dg) needs, for output column c,
// only row c of S and of Dout, so a CTA holds half of each and two CTAs share an SM.
// dbeta sums over dk: each half adds its share into the zeroed output.

constexpr int kHC = kD / 2;        // dk columns of one grads CTA
constexpr int L4 = kD + 4;         // 16-byte aligned padded rows for float4 reads
constexpr int LH = kHC + 4;

struct GradSmem {
    float S[kHC][L4], Dn[kHC][L4];                 // rows c of this half: the chunk-start state and Dout
    float Dl[kC][L4], dR[kC][L4], dO[kC][L4];
    float q[kC][LH], k[kC][LH], Gm[kC][LH];        // this half's columns
    float dA[kC][LC], dAq[kC][LC], Bm[kC][kC];
    float beta[kC], gl[kHC];
    float glrow[kHC];                              // rowsum(S_next o Dout) per column of the half
};
constexpr size_t kGradSmem = sizeof(GradSmem);
constexpr uint32_t kGradWait = 1u << 22;          // polls (each >= 0.25 us) of an item's readiness

__global__ void __launch_bounds__(kThreads, 2) cb_grad_kernel(const __grid_constant__ CbArgs A) {
    extern __shared__ __align__(16) uint8_t dyn[];
    GradSmem &s = *reinterpret_cast<GradSmem *>(dyn);
    const int tid = threadIdx.x;
    const int half = blockIdx.x & 1, H = A.H, nq = A.chunk_off[A.N];
    // CTA pairs take the chunks outwards from where the two chains meet (rank r: that chunk, then one
    // below, one above, ...), so the items become ready in about this order.  A forward-chain step
    // is the shorter (about 0.77 of a backward one), so they meet past the middle, near 9/16 of the
    // chunks; ranks past either end continue on the other side.
    const int m = blockIdx.x >> 1, r = m / H, h = m % H;
    if (r >= nq) return;
    const int mid = (int)(((long long)nq * 9) >> 4);
    int qc = (r & 1) ? mid - ((r + 1) >> 1) : mid + (r >> 1);
    {
        // the two sides hold mid (below) and nq - mid (above) chunks: once one side is used up the
        // remaining ranks go to the other, in order
        const int lo_n = mid, hi_n = nq - mid;
        const int two = 2 * (lo_n < hi_n ? lo_n : hi_n);        // ranks that alternate
        if (r >= two) qc = lo_n < hi_n ? mid + (r - lo_n) : mid - 1 - (r - hi_n);
    }
    const int item = qc * H + h;
    // n is the chunk's sequence: its chunk-start state slot is qc + n
    const int t0 = A.ck_t0[qc], L = A.ck_len[qc], n = A.ck_seq[qc];
    const int cbase = half * kHC;
    {
        // both chains have written the item's rows (bounded wait; a chain that gave up raises abort)
        __shared__ int go;
        if (tid == 0) {
            int ok = 0;
            for (uint32_t k = 0; k < kGradWait; ++k) {
                int v;
                asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(A.ready + item) : "memory");
                if (v >= 2) { ok = 1; break; }
                if (*reinterpret_cast<volatile const int *>(A.abort) != 0) break;
                __nanosleep(256);
            }
            if (!ok) atomicOr(A.status, 1u);
            go = ok;
        }
        __syncthreads();
        if (!go) return;
    }
    const size_t tile = (size_t)item * kC * kD, small = (size_t)item * kC * kC;
    // this half's columns of q and k, as given (bf16 or fp32), 4 channels a thread: loaded first, so
    // that they do not queue behind the staging copies below, and stored once those are issued
    static_assert(kC * kHC == 4 * kThreads, "one 4-channel piece of q and of k per thread");
    const int iq = tid >> 4, cq = (tid & 15) * 4;
    float qv[4], kv[4];
    {
        const size_t src = ((size_t)(t0 + iq) * H + h) * kD + cbase + cq;
        if (iq >= L) {
#pragma unroll
            for (int x = 0; x < 4; ++x) qv[x] = kv[x] = 0.f;
        } else if (A.bf16) {
            const uint2 rq = __ldg(reinterpret_cast<const uint2 *>(reinterpret_cast<const __nv_bfloat16 *>(A.q) + src));
            const uint2 rk = __ldg(reinterpret_cast<const uint2 *>(reinterpret_cast<const __nv_bfloat16 *>(A.k) + src));
            const float2 q0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&rq.x));
            const float2 q1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&rq.y));
            const float2 k0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&rk.x));
            const float2 k1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&rk.y));
            qv[0] = q0.x; qv[1] = q0.y; qv[2] = q1.x; qv[3] = q1.y;
            kv[0] = k0.x; kv[1] = k0.y; kv[2] = k1.x; kv[3] = k1.y;
        } else {
            const float4 q4 = __ldg(reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(A.q) + src));
            const float4 k4 = __ldg(reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(A.k) + src));
            qv[0] = q4.x; qv[1] = q4.y; qv[2] = q4.z; qv[3] = q4.w;
            kv[0] = k4.x; kv[1] = k4.y; kv[2] = k4.z; kv[3] = k4.w;
        }
    }
    const float bv = tid < kC && tid < L ? A.beta[(size_t)(t0 + tid) * H + h] : 0.f;
    const float *St = A.St + ((size_t)(qc + n) * H + h) * kD * kD + (size_t)cbase * kD;
    const float *Dng = A.Dn + (size_t)item * kD * kD + (size_t)cbase * kD;
    stage_tile(&s.Dl[0][0], L4, A.Dl + tile);
    stage_tile(&s.dR[0][0], L4, A.dR + tile);
    for (int e = tid; e < kC * (kHC / 4); e += kThreads) {
        const int i = e / (kHC / 4), p = e % (kHC / 4);
        cp16(&s.Gm[i][p * 4], A.Gm + tile + (size_t)i * kD + cbase + p * 4);
    }
    for (int e = tid; e < kC * (kD / 4); e += kThreads) {
        const int i = e / (kD / 4), p = e % (kD / 4);
        const int ti = i < L ? t0 + i : t0;
        cp16z(&s.dO[i][p * 4], A.dO + ((size_t)ti * H + h) * kD + p * 4, i < L ? 16 : 0);
    }
    stage_vec(&s.Bm[0][0], A.Bm + small, kC * kC);
    stage_vec(s.gl, A.gl + (size_t)item * kD + cbase, kHC);
    cp_commit();
    // the half's rows of S and Dout in a second group, landing while dA and dAqk are formed
    for (int e = tid; e < kHC * (kD / 4); e += kThreads) {
        const int a = e / (kD / 4), p = e % (kD / 4);
        cp16(&s.S[a][p * 4], St + (size_t)a * kD + p * 4);
        cp16(&s.Dn[a][p * 4], Dng + (size_t)a * kD + p * 4);
    }
    cp_commit();
    {
        // the rows of the state after the chunk that the epilogue reads, into L2 meanwhile
        const float *sn = A.St + ((size_t)(qc + 1 + n) * H + h) * kD * kD + (size_t)cbase * kD;
        for (int e = tid; e < kHC * kD / 32; e += kThreads)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(sn + (size_t)e * 32));
    }
    *reinterpret_cast<float4 *>(&s.q[iq][cq]) = make_float4(qv[0], qv[1], qv[2], qv[3]);
    *reinterpret_cast<float4 *>(&s.k[iq][cq]) = make_float4(kv[0], kv[1], kv[2], kv[3]);
    if (tid < kC) s.beta[tid] = bv;
    cp_wait<1>();
    __syncthreads();
    const float scale = A.scale;
    {
        // dA = -strict_lower(dR Delta^T), dAqk = lower(dOs Delta^T): one element per thread, the
        // products on the lower triangle's threads only
        int i, j;
        tri_pair(tid, i, j);
        float a1 = 0.f, a2 = 0.f;
#pragma unroll 4
        for (int k = 0; k < (tid < kLow ? kD : 0); k += 4) {
            const float4 d4 = *reinterpret_cast<const float4 *>(&s.Dl[j][k]);
            const float4 r4 = *reinterpret_cast<const float4 *>(&s.dR[i][k]);
            const float4 o4 = *reinterpret_cast<const float4 *>(&s.dO[i][k]);
            a1 = fmaf(r4.x, d4.x, fmaf(r4.y, d4.y, fmaf(r4.z, d4.z, fmaf(r4.w, d4.w, a1))));
            a2 = fmaf(o4.x, d4.x, fmaf(o4.y, d4.y, fmaf(o4.z, d4.z, fmaf(o4.w, d4.w, a2))));
        }
        s.dA[i][j] = j < i ? -a1 : 0.f;
        s.dAq[i][j] = j <= i ? scale * a2 : 0.f;
    }
    cp_wait<0>();
    __syncthreads();
    const int i = tid / 16, tn = tid % 16;            // row i, local columns tn + 16 x (x < 4)
    const float bi = s.beta[i];
    float y[4], dos[4], dd[4];
    {
        // Y = dR S^T, dO S^T and Delta Dout^T over dv (rows c of S and Dout).  Each thread takes two
        // rows (ig, ig + 8) and half of dv, so that every S and Dout element it loads feeds two
        // rows; the two halves of dv meet through shared memory.
        const int ig = (tid >> 4) & 7, kh = tid >> 7, i0 = ig, i1 = ig + 8;
        float a[3][2][4];                              // [Y, dO S^T, Delta Dout^T][row][x]
#pragma unroll
        for (int t = 0; t < 3; ++t)
#pragma unroll
            for (int r = 0; r < 2; ++r)
#pragma unroll
                for (int x = 0; x < 4; ++x) a[t][r][x] = 0.f;
#pragma unroll 2
        for (int k = kh * (kD / 2); k < (kh + 1) * (kD / 2); k += 4) {
            const float4 r0 = *reinterpret_cast<const float4 *>(&s.dR[i0][k]), r1 = *reinterpret_cast<const float4 *>(&s.dR[i1][k]);
            const float4 o0 = *reinterpret_cast<const float4 *>(&s.dO[i0][k]), o1 = *reinterpret_cast<const float4 *>(&s.dO[i1][k]);
            const float4 l0 = *reinterpret_cast<const float4 *>(&s.Dl[i0][k]), l1 = *reinterpret_cast<const float4 *>(&s.Dl[i1][k]);
#pragma unroll
            for (int x = 0; x < 4; ++x) {
                const float4 sv = *reinterpret_cast<const float4 *>(&s.S[tn + 16 * x][k]);
                const float4 nv = *reinterpret_cast<const float4 *>(&s.Dn[tn + 16 * x][k]);
                a[0][0][x] = fmaf(r0.x, sv.x, fmaf(r0.y, sv.y, fmaf(r0.z, sv.z, fmaf(r0.w, sv.w, a[0][0][x]))));
                a[0][1][x] = fmaf(r1.x, sv.x, fmaf(r1.y, sv.y, fmaf(r1.z, sv.z, fmaf(r1.w, sv.w, a[0][1][x]))));
                a[1][0][x] = fmaf(o0.x, sv.x, fmaf(o0.y, sv.y, fmaf(o0.z, sv.z, fmaf(o0.w, sv.w, a[1][0][x]))));
                a[1][1][x] = fmaf(o1.x, sv.x, fmaf(o1.y, sv.y, fmaf(o1.z, sv.z, fmaf(o1.w, sv.w, a[1][1][x]))));
                a[2][0][x] = fmaf(l0.x, nv.x, fmaf(l0.y, nv.y, fmaf(l0.z, nv.z, fmaf(l0.w, nv.w, a[2][0][x]))));
                a[2][1][x] = fmaf(l1.x, nv.x, fmaf(l1.y, nv.y, fmaf(l1.z, nv.z, fmaf(l1.w, nv.w, a[2][1][x]))));
            }
        }
        __syncthreads();                               // S is read: its rows take the sums
        float (*acc)[kC][kHC] = reinterpret_cast<float (*)[kC][kHC]>(&s.S[0][0]);   // [3][row][column]
        static_assert(3 * kC * kHC <= kHC * L4, "the sums fit in S");
        if (kh == 1)
#pragma unroll
            for (int t = 0; t < 3; ++t)
#pragma unroll
                for (int r = 0; r < 2; ++r)
#pragma unroll
                    for (int x = 0; x < 4; ++x) acc[t][ig + 8 * r][tn + 16 * x] = a[t][r][x];
        __syncthreads();
        if (kh == 0)
#pragma unroll
            for (int t = 0; t < 3; ++t)
#pragma unroll
                for (int r = 0; r < 2; ++r)
#pragma unroll
                    for (int x = 0; x < 4; ++x) acc[t][ig + 8 * r][tn + 16 * x] += a[t][r][x];
        __syncthreads();
#pragma unroll
        for (int x = 0; x < 4; ++x) {
            y[x] = acc[0][i][tn + 16 * x];
            dos[x] = acc[1][i][tn + 16 * x];
            dd[x] = acc[2][i][tn + 16 * x];
        }
    }
    // the epilogue's v values, in flight during the pairwise sums
    const size_t row = ((size_t)(t0 + i) * H + h) * kD;
    float vv[4];
#pragma unroll
    for (int x = 0; x < 4; ++x) vv[x] = i < L ? ld_x(A.v, row + cbase + tn + 16 * x, A.bf16) : 0.f;
    // the pairwise decayed sums P1 .. P4 (K = kC): for m <= i the factor is e^{Gamma_i - Gamma_m},
    // for m >= i it is e^{Gamma_m - Gamma_i}; both are e^{-|Gamma_i - Gamma_m|}
    float gi[4], p1[4], p2[4], p34[4];
#pragma unroll
    for (int x = 0; x < 4; ++x) {
        gi[x] = s.Gm[i][tn + 16 * x];
        p1[x] = p2[x] = p34[x] = 0.f;
    }
    // dAqk is lower and dA strictly lower, so m < i feeds P1 and P2 only, m > i P3 and P4 only, and
    // m = i (factor 1) P1 and P3 through dAqk[i][i]
#pragma unroll 2
    for (int m = 0; m < i; ++m) {
        const float aq = s.dAq[i][m], ad = s.dA[i][m];
#pragma unroll
        for (int x = 0; x < 4; ++x) {
            const int c = tn + 16 * x;
            const float km = s.k[m][c] * __expf(gi[x] - s.Gm[m][c]);     // Gamma_i <= Gamma_m: <= 0
            p1[x] = fmaf(aq, km, p1[x]);
            p2[x] = fmaf(ad, km, p2[x]);
        }
    }
    {
        const float aii = s.dAq[i][i];
#pragma unroll
        for (int x = 0; x < 4; ++x) {
            const int c = tn + 16 * x;
            p1[x] = fmaf(aii, s.k[i][c], p1[x]);
            p34[x] = fmaf(aii, s.q[i][c], p34[x]);
        }
    }
#pragma unroll 2
    for (int m = i + 1; m < kC; ++m) {
        const float aqt = s.dAq[m][i], adt = s.dA[m][i] * s.beta[m];
#pragma unroll
        for (int x = 0; x < 4; ++x) {
            const int c = tn + 16 * x;
            const float e = __expf(s.Gm[m][c] - gi[x]);                  // Gamma_m <= Gamma_i: <= 0
            p34[x] = fmaf(aqt, s.q[m][c] * e, fmaf(adt, s.k[m][c] * e, p34[x]));
        }
    }
    // the chunk's last row also moves the state it hands on: rowsum(S_next o Dout), thread (column
    // cr, quarter pr of dv) taking 32 products, its rows of S_next loaded here and used after the
    // epilogue; the quarters start at rotated pieces so that the four threads of a column read
    // different banks of Dout
    const int cr = tid >> 2, pr = tid & 3;
    float4 snv[8];
    {
        const float *sn = A.St + ((size_t)(qc + 1 + n) * H + h) * kD * kD + (size_t)(cbase + cr) * kD + 32 * pr;
#pragma unroll
        for (int u = 0; u < 8; ++u) snv[u] = reinterpret_cast<const float4 *>(sn)[(u + pr) & 7];   // written by the chains: plain loads
    }
    // dbeta share: rowsum(v o dR) - rowsum(K0 o Y) over this half (+ rowsum(dA o B) once); dv = beta dR
    float pb = 0.f;
    float dgm[4];
#pragma unroll
    for (int x = 0; x < 4; ++x) {
        const int c = tn + 16 * x, cg = cbase + c;
        const float ea = __expf(gi[x]), ed = __expf(s.gl[c] - gi[x]);
        const float dr = s.dR[i][cg], kv = s.k[i][c], qv = s.q[i][c];
        pb += vv[x] * dr - kv * ea * y[x];
        const float dq = fmaf(scale * dos[x], ea, p1[x]);
        const float dkt = bi * (p2[x] - y[x] * ea);
        const float dkh = fmaf(dd[x], ed, p34[x]);
        if (i < L) {
            A.dv[row + cg] = bi * dr;
            A.dq[row + cg] = dq;
            A.dk[row + cg] = dkt + dkh;
        }
        dgm[x] = qv * dq + kv * (dkt - dkh);
    }
    // sum pb over the row's 16 threads (consecutive lanes of one half-warp)
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) pb += __shfl_xor_sync(0xffffffffu, pb, o);
    {
        float gsum = 0.f;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const float4 x4 = *reinterpret_cast<const float4 *>(&s.Dn[cr][32 * pr + 4 * ((u + pr) & 7)]);
            gsum = fmaf(snv[u].x, x4.x, fmaf(snv[u].y, x4.y, fmaf(snv[u].z, x4.z, fmaf(snv[u].w, x4.w, gsum))));
        }
        gsum += __shfl_xor_sync(0xffffffffu, gsum, 1);
        gsum += __shfl_xor_sync(0xffffffffu, gsum, 2);
        if (pr == 0) s.glrow[cr] = gsum;
    }
    __syncthreads();                                   // S free: dGamma goes there
    float (*dG)[L4] = s.S;
#pragma unroll
    for (int x = 0; x < 4; ++x) dG[i][tn + 16 * x] = dgm[x];
    if (tn == 0 && i < L) {
        float ab = 0.f;
        if (half == 0)
            for (int j = 0; j < i; ++j) ab = fmaf(s.dA[i][j], s.Bm[i][j], ab);
        atomicAdd(A.dbeta + (size_t)(t0 + i) * H + h, pb + ab);
    }
    __syncthreads();
    if (tid < kHC) {
        const int cg = cbase + tid;
        dG[L - 1][tid] += s.glrow[tid];
        float run = 0.f;
        for (int ii = L - 1; ii >= 0; --ii) {
            run += dG[ii][tid];
            A.dg[((size_t)(t0 + ii) * H + h) * kD + cg] = run;
        }
    }
}

size_t r256(size_t b) { return (b + 255) & ~size_t(255); }

struct Layout {
    size_t off_chunk, ck_t0, ck_len, ck_seq, ready, Q0, K0, Kd, Gm, W, U, Tm, Aqk, Bm, gl, Dl, dR, Dn, St, total;
};

Layout layout(int N, int T, int H) {
    const size_t Q = ((size_t)T + (size_t)(kC - 1) * (size_t)N) / kC + 1;
    const size_t NI = Q * (size_t)H;
    Layout l;
    size_t o = 0;
    auto take = [&](size_t bytes) { const size_t at = o; o += r256(bytes); return at; };
    l.off_chunk = take((size_t)(N + 1) * 4);
    l.ck_t0 = take(Q * 4);
    l.ck_len = take(Q * 4);
    l.ck_seq = take(Q * 4);
    l.ready = take((NI + 1) * 4);                      // per item, then the abort word
    const size_t tb = NI * kC * kD * 4, sb = NI * kC * kC * 4, vb = NI * kD * 4;
    l.Q0 = take(tb); l.K0 = take(tb); l.Kd = take(tb); l.Gm = take(tb); l.W = take(tb); l.U = take(tb);
    l.Tm = take(sb); l.Aqk = take(sb); l.Bm = take(sb);
    l.gl = take(vb);
    l.Dl = take(tb); l.dR = take(tb);
    l.Dn = take(NI * kD * kD * 4);
    l.St = take((Q + N) * (size_t)H * kD * kD * 4);
    l.total = o;
    return l;
}

std::atomic<uint64_t> g_grad_attr{0}, g_chains_attr{0};

}  // namespace

size_t backward_chunked_workspace(int N, int T, int H) { return layout(N, T, H).total; }

cudaError_t launch_backward_chunked(const void *q, const void *k, const void *v, int bf16, const float *g,
                                    const float *beta, const float *S0, const int32_t *cu, int N, int T, int H,
                                    float scale, const float *dO, const float *dSfin, float *dq, float *dk, float *dv,
                                    float *dg, float *dbeta, float *dS0, unsigned *status, void *ws, cudaStream_t s) {
    cudaError_t e;
    if (T == 0) {
        // no tokens: dS0 = dS_final (or zero)
        const size_t sb = (size_t)N * H * kD * kD * sizeof(float);
        if (dSfin) return cudaMemcpyAsync(dS0, dSfin, sb, cudaMemcpyDeviceToDevice, s);
        return cudaMemsetAsync(dS0, 0, sb, s);
    }
    const Layout l = layout(N, T, H);
    char *w = static_cast<char *>(ws);
    CbArgs A;
    A.q = q; A.k = k; A.v = v; A.bf16 = bf16; A.g = g; A.beta = beta; A.S0 = S0; A.dO = dO; A.dSfin = dSfin;
    A.cu = cu; A.N = N; A.T = T; A.H = H; A.scale = scale;
    A.Q = (int)(((size_t)T + (size_t)(kC - 1) * (size_t)N) / kC);
    A.chunk_off = reinterpret_cast<int32_t *>(w + l.off_chunk);
    A.ck_t0 = reinterpret_cast<int32_t *>(w + l.ck_t0);
    A.ck_len = reinterpret_cast<int32_t *>(w + l.ck_len);
    A.ck_seq = reinterpret_cast<int32_t *>(w + l.ck_seq);
    A.ready = reinterpret_cast<int *>(w + l.ready);
    A.abort = A.ready + (size_t)A.Q * H + H;           // past every item of the chunk bound
    auto f = [&](size_t off) { return reinterpret_cast<float *>(w + off); };
    A.Q0 = f(l.Q0); A.K0 = f(l.K0); A.Kd = f(l.Kd); A.Gm = f(l.Gm); A.W = f(l.W); A.U = f(l.U);
    A.Tm = f(l.Tm); A.Aqk = f(l.Aqk); A.Bm = f(l.Bm); A.gl = f(l.gl);
    A.Dl = f(l.Dl); A.dR = f(l.dR); A.Dn = f(l.Dn); A.St = f(l.St);
    A.dq = dq; A.dk = dk; A.dv = dv; A.dg = dg; A.dbeta = dbeta; A.dS0 = dS0; A.status = status;
    A.test_limit = take_test_timeout(kTestBackward);
    // chunk enumeration from the device cu_seqlens; the item grids cover the upper bound A.Q of
    // the chunk count and CTAs past the real chunks return at once
    cb_offsets_kernel<<<1, 32, 0, s>>>(A);
    count_launch();
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    cb_chunks_kernel<<<(unsigned)((A.Q + 255) / 256), 256, 0, s>>>(A);
    count_launch();
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const unsigned items = (unsigned)((size_t)A.Q * H), chains = (unsigned)((size_t)N * H);
    cb_prep_kernel<<<items, kThreads, 0, s>>>(A);
    count_launch();
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // the readiness flags, the abort word and dbeta (accumulated by the grads) start at zero
    if ((e = cudaMemsetAsync(A.ready, 0, ((size_t)A.Q * H + H + 1) * sizeof(int), s)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(dbeta, 0, (size_t)T * H * sizeof(float), s)) != cudaSuccess) return e;
    if (chains) {
        if ((e = smem_attr_once((const void *)cb_tc_chains_kernel, (int)kTcSmem, g_chains_attr)) != cudaSuccess)
            return e;
        cb_tc_chains_kernel<<<2 * chains, kTcThreads, kTcSmem, s>>>(A);
        count_launch();
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if ((e = smem_attr_once((const void *)cb_grad_kernel, (int)kGradSmem, g_grad_attr)) != cudaSuccess) return e;
    // a programmatic dependent launch: the grads start on the SMs the chains leave free and take
    // each item as soon as both chains have published it (their flags, not the launch order, carry
    // the dependency)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * items);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kGradSmem;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = chains ? 1 : 0;
    e = cudaLaunchKernelEx(&cfg, cb_grad_kernel, A);
    count_launch();
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace k3kda
