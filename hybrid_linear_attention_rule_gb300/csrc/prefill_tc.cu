// prefill_tc.cu -- chunked KDA prefill on the 5th-generation tensor cores
// (tcgen05 MMA, TMEM accumulators), bf16 inputs, dk = dv = 128, chunk 64, with
// the q/k/v short conv (+SiLU), q/k L2 norm and sigmoid output gate fused.
//
// The recurrence ("recurrent KDA state", HF discussion #187 feature list; FP32
// KdaState, metrale kimi_k3 docs) in its chunked (WY/UT) form.  For a chunk of
// 64 tokens with chunk-local cumulative log-decay G (per channel) and a
// per-channel reference r = (G_first + G_last) / 2:
//   Kh = k E, Qh = q E, Kb = k / E          with E = exp(G - r)
//   Akk = diag(beta) tril(Kh Kb^T, -1),  Aqk = tril(Qh Kb^T)
//   T  = (I + Akk)^-1,  Tb = T diag(beta)
//   S' = diag(exp(r)) S                        (state in the chunk's basis)
//   U  = Tb v,  Y = Kh S',  V' = U - Tb Y
//   O  = scale (Qh S' + Aqk V')  [* sigmoid(gate)]
//   S_next = diag(exp(G_last - r)) (S' + Kb^T V')
// (V' = U - W S with W = Tb Kh written as U - Tb (Kh S') so that no transposed
// copy of Kh or W is ever materialised.)  All exponents are of |G - r| <= half
// the chunk's total decay, so nothing overflows for per-chunk decays below
// ~170 nats per channel.
//
// Precision: every MMA operand that is not exactly bf16 is split into a bf16
// high part and a bf16 low part (x = hi + lo to ~2^-17 relative) and each
// product is hi*hi + hi*lo + lo*hi with fp32 accumulation in TMEM (only v,
// exact in bf16 without a conv, stays single).  Plain bf16 operands miss a
// 5e-3-of-RMS bar by 5-20x because the state and outputs are heavy tailed;
// the split keeps them near 1e-4 of RMS.
//
// Work layout: one CTA (16 warps) per (sequence, head); the CTA walks its
// chunks in order.  CUDA cores build the operands in 128B-swizzled K-major
// shared-memory tiles and invert the 64x64 unit-triangular matrix in fp32; a
// single elected thread issues the tcgen05.mma chains; the fp32 state lives in
// TMEM for the whole sequence.  TMEM columns: [0,64) Akk|Aqk then O^T,
// [64,128) Y^T, [128,192) U^T then V'^T, [192,320) S'^T.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace k3kda {
namespace {

using namespace tc;

constexpr int kC = 64;
constexpr int kD = 128;
constexpr int kWarps = 16;
constexpr int kThreads = 32 * kWarps;
constexpr int kTok = kC / kWarps;                // tokens per thread in the prep phase (4)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColA = 0, kColY = 64, kColU = 128, kColS = 192;
constexpr uint32_t kWaitLimit = 1u << 26;

// shared-memory plan (byte offsets from a 1024-aligned base).  Regions A and B
// are reused phase by phase within a chunk; the input rows of the next chunk are
// staged into them by bulk copies while this chunk's last MMAs run.
constexpr uint32_t OFF_X = 0;                    // [128 rows][128 K] hi: Kh rows 0-63, Qh rows 64-127
constexpr uint32_t OFF_XL = OFF_X + 32768;       // same, low parts
constexpr uint32_t OFF_GST = 65536;              // A: g rows fp32 [64][128]       (staged .. prep)
constexpr uint32_t OFF_V_HI = 65536;             // A: v rows [64 j][128 j']        (prep .. MMA U, MN-major A)
constexpr uint32_t OFF_V_LO = 81920;
constexpr uint32_t OFF_ST_HI = 65536;            // A: S'^T [128 rows j][128 K c]   (S' .. MMA Y/O)
constexpr uint32_t OFF_YT_HI = 65536;            // A: Y^T [128 rows j][64 K i]     (Y .. MMA V)
constexpr uint32_t OFF_YT_LO = 81920;
constexpr uint32_t OFF_QST = 98304;              // B: q rows bf16 [64][128]        (staged .. prep)
constexpr uint32_t OFF_KST = 114688;             // B: k rows bf16 [64][128]
constexpr uint32_t OFF_SCR_A = 98304;            // B: fp32 64x64                   (T solve)
constexpr uint32_t OFF_SCR_T = 114688;
constexpr uint32_t OFF_ST_LO = 98304;            // B: S'^T low parts
constexpr uint32_t OFF_VPT_HI = 98304;           // B: V'^T [128 rows j][64 K i]    (V' .. MMA O/S)
constexpr uint32_t OFF_VPT_LO = 114688;
constexpr uint32_t OFF_KB_HI = 131072;           // Kb [64 rows i][128 K c]: K-major B of MMA A, MN-major B of MMA S
constexpr uint32_t OFF_KB_LO = 147456;
constexpr uint32_t OFF_AQK_HI = 163840;          // [64 rows i][64 K i']      (extract .. MMA O)
constexpr uint32_t OFF_AQK_LO = 172032;
constexpr uint32_t OFF_SCAN = OFF_AQK_HI;        // fp32 [16 warps][128] partial sums, prep only
constexpr uint32_t OFF_TB_HI = 180224;           // [64 rows i][64 K j]       (T solve .. MMA V)
constexpr uint32_t OFF_TB_LO = 188416;
constexpr uint32_t OFF_VST = 196608;             // v rows bf16 [64][128] (staged .. prep)
constexpr uint32_t OFF_CONVW = 212992;           // fp32 [4 taps][384 channels]
constexpr uint32_t OFF_HIST = OFF_CONVW + 384 * 4 * 4;   // fp32 [3 tensors][3 rows][128]: pre-conv rows before the chunk
constexpr uint32_t OFF_BETA = OFF_HIST + 3 * 3 * 128 * 4;
constexpr uint32_t OFF_REF = OFF_BETA + 256;          // r per channel
constexpr uint32_t OFF_GL = OFF_REF + 512;            // G_last per channel
constexpr uint32_t OFF_G0 = OFF_GL + 512;             // G_first per channel
constexpr uint32_t OFF_FCOL = OFF_G0 + 512;           // state column factor for this chunk
constexpr uint32_t OFF_LOGF = OFF_FCOL + 512;         // log of the basis factor carried in TMEM
constexpr uint32_t OFF_MISC = OFF_LOGF + 512;         // mbarriers (2 x 8 B), tmem slot, flag
constexpr uint32_t kSmemUsed = OFF_MISC + 64;
constexpr uint32_t kSmemBytes = kSmemUsed + 1024;     // + alignment slack
static_assert(kSmemBytes <= 232448, "shared memory plan exceeds the per-CTA limit");

struct TcArgs {
    CUtensorMap tm_q, tm_k, tm_v, tm_g;   // [T, H, 128] bf16 (q, k, v) and fp32 (g); box 64 tokens x 1 head x 128
    CUtensorMap tm_gate;                  // [T, H, 128] bf16 gate logits (when gated)
    PrefillArgs p;
    const float *conv_w;     // [2*H*128 + H*128, W] or null
    float *conv_state;       // [N, W-1, 3*H*128] or null
    int W;
    int box_rows;            // tokens per staged tile: min(64, T)
};

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&v);
}
__device__ __forceinline__ void split_bf16(float x, float &hi, float &lo) {
    hi = __bfloat162float(__float2bfloat16_rn(x));
    lo = x - hi;
}
__device__ __forceinline__ int sidx(int r, int c) { return r * 64 + (c ^ (r & 31)); }   // fp32 64x64 scratch
// z * sigmoid(z) and sigmoid(z) with the fast (2 ulp) divide; the limits are exact (0 and 1)
__device__ __forceinline__ float silu_fast(float z) { return __fdividef(z, 1.0f + __expf(-z)); }
__device__ __forceinline__ float sigmoid_fast(float z) { return __fdividef(1.0f, 1.0f + __expf(-z)); }

// Advance a shared-memory descriptor's start address by `bytes` (a multiple of 16, no carry
// out of the 14-bit field for addresses below 256 KB).
__device__ __forceinline__ uint64_t dadd(uint64_t desc, uint32_t bytes) { return desc + (bytes >> 4); }

// Element (row, c) of a K-major tile whose K extent is 128 (two 64-wide atoms of rows*128 B each).
__device__ __forceinline__ uint32_t kmaj128(uint32_t rows, uint32_t row, uint32_t c) {
    return (c >> 6) * rows * 128u + sw128_offset(row, c & 63u);
}

// 16 TMEM columns of one lane -> split bf16 into row `row` of a K=64 tile at column col0
__device__ __forceinline__ void tile64_put16(uint8_t *sm, uint32_t off_hi, uint32_t off_lo, int row, int col0,
                                             const float (&v)[16]) {
    uint32_t hw[8], lw[8];
#pragma unroll
    for (int u = 0; u < 16; u += 2) {
        float h0, l0, h1, l1;
        split_bf16(v[u], h0, l0);
        split_bf16(v[u + 1], h1, l1);
        hw[u >> 1] = pack_bf16(h0, h1);
        lw[u >> 1] = pack_bf16(l0, l1);
    }
    const uint32_t o0 = sw128_offset(row, col0), o1 = sw128_offset(row, col0 + 8);
    *reinterpret_cast<uint4 *>(sm + off_hi + o0) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
    *reinterpret_cast<uint4 *>(sm + off_hi + o1) = make_uint4(hw[4], hw[5], hw[6], hw[7]);
    *reinterpret_cast<uint4 *>(sm + off_lo + o0) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
    *reinterpret_cast<uint4 *>(sm + off_lo + o1) = make_uint4(lw[4], lw[5], lw[6], lw[7]);
}

__global__ void __launch_bounds__(kThreads, 1) kda_prefill_tc_kernel(const __grid_constant__ TcArgs A) {
    extern __shared__ uint8_t smraw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
    const PrefillArgs &a = A.p;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nh = blockIdx.x, n = nh / a.H, h = nh % a.H;
    const int H = a.H;
    const uint32_t sbase = smem_u32(sm);
    float *sBeta = reinterpret_cast<float *>(sm + OFF_BETA);
    float *sRef = reinterpret_cast<float *>(sm + OFF_REF);
    float *sGL = reinterpret_cast<float *>(sm + OFF_GL);
    float *sG0 = reinterpret_cast<float *>(sm + OFF_G0);
    float *sFcol = reinterpret_cast<float *>(sm + OFF_FCOL);
    float *sLogf = reinterpret_cast<float *>(sm + OFF_LOGF);
    float *sScan = reinterpret_cast<float *>(sm + OFF_SCAN);
    float *sConvW = reinterpret_cast<float *>(sm + OFF_CONVW);
    float *scrA = reinterpret_cast<float *>(sm + OFF_SCR_A);
    float *scrT = reinterpret_cast<float *>(sm + OFF_SCR_T);
    float *sHist = reinterpret_cast<float *>(sm + OFF_HIST);
    uint64_t *mbar = reinterpret_cast<uint64_t *>(sm + OFF_MISC);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + OFF_MISC + 24);
    volatile uint32_t *sflag = reinterpret_cast<volatile uint32_t *>(sm + OFF_MISC + 28);
    const uint32_t mbar_a = smem_u32(mbar);          // MMA completion
    const uint32_t mbar_s = smem_u32(mbar + 1);      // staged input rows landed
    const uint32_t mbar_g = smem_u32(mbar + 2);      // staged gate tile landed

    int tb, te;
    seq_bounds(a.cu, n, a.T, tb, te);
    const int W = A.conv_w ? A.W : 0;
    const int Dall = 3 * H * kD;

    // ---- set-up: TMEM, barrier, conv weights, initial state ----
    if (warp == 0) { tmem_alloc(smem_u32(tslot), kTmemCols); tmem_relinquish(); }
    if (tid == 0) { mbar_init(mbar_a, 1); mbar_init(mbar_s, 1); mbar_init(mbar_g, 1); fence_mbar_init(); *sflag = 0; }
    // conv history of the first chunk: the conv-state rows (right-aligned), else zeros
    for (int e = tid; e < 3 * 3 * 128; e += kThreads) {
        const int which = e / 384, r = (e / 128) % 3, c = e & 127;
        const int row = W - 4 + r;                   // conv-state row holding token r - 3
        float x = 0.f;
        if (W > 1 && A.conv_state != nullptr && row >= 0)
            x = A.conv_state[((size_t)n * (W - 1) + row) * Dall + which * H * kD + h * kD + c];
        sHist[e] = x;
    }
    if (W > 0)
        for (int e = tid; e < 384 * 4; e += kThreads) {
            // tap-major, taps right-aligned in a 4-wide window: tap t multiplies token i - 3 + t
            const int t = e / 384, ch = e - t * 384;
            const int gch = (ch >> 7) * H * kD + h * kD + (ch & 127);
            sConvW[e] = t >= 4 - W ? A.conv_w[(size_t)gch * W + (t - (4 - W))] : 0.f;
        }
    if (tid < kD) sLogf[tid] = 0.f;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tslot;
    const uint32_t lrow = 32u * (warp & 3);             // first TMEM lane of this warp
    const uint32_t tl = tbase + (lrow << 16);
    const int quarter = warp >> 2;                       // which column quarter this warp handles
    {   // S'^T <- S0^T (true state; basis factor 1)
        const int j = lrow + lane;
        for (int cb = 0; cb < 32; cb += 16) {
            uint32_t r[16];
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                const int c = quarter * 32 + cb + u;
                r[u] = __float_as_uint(a.S0 ? a.S0[((size_t)nh * kD + c) * kD + j] : 0.f);
            }
            tmem_st16(tl + kColS + quarter * 32 + cb, r);
        }
        tmem_wait_st();
    }
    uint32_t phase = 0, sphase = 0, gphase = 0;
    bool failed = false;

    // A chunk's input rows are brought into shared memory by tiled TMA loads (one per
    // tensor, issued by one thread): g and v first (their regions free up earlier), then q
    // and k, all completing one phase of mbar_s.  Rows past T arrive as zeros; rows past the
    // sequence end are loaded but never used.
    const uint32_t kStageBytes = (uint32_t)A.box_rows * (kD * 4 + 3 * kD * 2);
    auto stage_gv = [&](int cs2) {
        if (tid != 0) return;
        fence_async_smem();
        mbar_arrive_expect_tx(mbar_s, kStageBytes);
        tma_load_3d(sbase + OFF_GST, &A.tm_g, 0, h, cs2, mbar_s);
        tma_load_3d(sbase + OFF_VST, &A.tm_v, 0, h, cs2, mbar_s);
    };
    auto stage_qk = [&](int cs2) {
        if (tid != 0) return;
        fence_async_smem();
        tma_load_3d(sbase + OFF_QST, &A.tm_q, 0, h, cs2, mbar_s);
        tma_load_3d(sbase + OFF_KST, &A.tm_k, 0, h, cs2, mbar_s);
    };
    if (tb < te) { stage_gv(tb); stage_qk(tb); }

    auto mma_wait = [&]() -> bool {
        if (tid == 0) {
            if (!mbar_wait_bounded(mbar_a, phase, kWaitLimit)) {
                *sflag = 1;
                atomicOr(a.status, 1u);
            }
        }
        phase ^= 1u;
        __syncthreads();
        const bool bad = *sflag != 0;
        tc_fence_after();
        return !bad;
    };

#ifdef K3KDA_PHASE_TIMERS
    // optional per-phase cycle counters (thread 0), written after the status word
    unsigned long long ph[10] = {0, 0, 0, 0, 0, 0, 0, 0, 0, 0};
    long long tlast = clock64();
#define PHASE(i)                                                   \
    if (tid == 0) {                                                \
        const long long now = clock64();                           \
        ph[i] += (unsigned long long)(now - tlast);                \
        tlast = now;                                               \
    }
#else
#define PHASE(i)
#endif
    for (int cs = tb; cs < te; cs += kC) {
        const int Lc = min(kC, te - cs);
        // ================= prep: conv, norm, decay, operands =================
        // thread owns tokens i0..i0+3 (i0 = 4*warp) and channels c0..c0+3 (c0 = 4*lane);
        // the chunk's input rows were staged into shared memory by bulk copies
        const int i0 = warp * kTok, c0 = lane * 4;
        if (tid == 0 && !mbar_wait_bounded(mbar_s, sphase, kWaitLimit)) {
            *sflag = 1;
            atomicOr(a.status, 1u);
        }
        sphase ^= 1u;
        __syncthreads();
        if (*sflag) { failed = true; break; }
        float G[kTok][4];
        {
            float run[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int ii = 0; ii < kTok; ++ii) {
                const int i = i0 + ii;
                float4 gv = make_float4(0.f, 0.f, 0.f, 0.f);
                if (i < Lc) gv = *reinterpret_cast<const float4 *>(sm + OFF_GST + i * (kD * 4) + c0 * 4);
                run[0] += gv.x; run[1] += gv.y; run[2] += gv.z; run[3] += gv.w;
#pragma unroll
                for (int m = 0; m < 4; ++m) G[ii][m] = run[m];
            }
            *reinterpret_cast<float4 *>(sScan + warp * kD + c0) = make_float4(run[0], run[1], run[2], run[3]);
        }
        if (tid < kC) sBeta[tid] = tid < Lc ? a.beta[(size_t)(cs + tid) * H + h] : 0.f;
        __syncthreads();
        {
            float off[4] = {0.f, 0.f, 0.f, 0.f};
            for (int w2 = 0; w2 < warp; ++w2) {
                const float4 s4 = *reinterpret_cast<const float4 *>(sScan + w2 * kD + c0);
                off[0] += s4.x; off[1] += s4.y; off[2] += s4.z; off[3] += s4.w;
            }
#pragma unroll
            for (int ii = 0; ii < kTok; ++ii)
#pragma unroll
                for (int m = 0; m < 4; ++m) G[ii][m] += off[m];
            if (warp == 0)
                *reinterpret_cast<float4 *>(sG0 + c0) = make_float4(G[0][0], G[0][1], G[0][2], G[0][3]);
            if (warp == kWarps - 1)
                *reinterpret_cast<float4 *>(sGL + c0) =
                    make_float4(G[kTok - 1][0], G[kTok - 1][1], G[kTok - 1][2], G[kTok - 1][3]);
        }
        __syncthreads();
        if (tid < kD) {
            const float r = 0.5f * (sG0[tid] + sGL[tid]);
            sRef[tid] = r;
            sFcol[tid] = expf(sLogf[tid] + r);     // TMEM basis -> this chunk's S' = exp(r) S
        }
        __syncthreads();
        float E[kTok][4], Eb[kTok][4];
        {
            const float4 r4 = *reinterpret_cast<const float4 *>(sRef + c0);
            const float rr[4] = {r4.x, r4.y, r4.z, r4.w};
#pragma unroll
            for (int m = 0; m < 4; ++m)
#pragma unroll
                for (int ii = 0; ii < kTok; ++ii) {
                    const float x = fminf(fmaxf(G[ii][m] - rr[m], -87.f), 87.f);
                    E[ii][m] = __expf(x);
                    Eb[ii][m] = __expf(-x);
                }
        }
        // conv (+SiLU) and norm of q (which 0), k (1) or v (2) for this thread's 4 tokens x 4 channels
        auto finish = [&](int which, float (&y)[kTok][4]) {
            const uint32_t st = which == 0 ? OFF_QST : (which == 1 ? OFF_KST : OFF_VST);
            float x[kTok + 3][4];
#pragma unroll
            for (int t = 0; t < kTok + 3; ++t) {
                const int i = i0 - 3 + t;               // chunk-local token
                if (i < 0) {
                    const float4 hv = *reinterpret_cast<const float4 *>(sHist + (which * 3 + 3 + i) * 128 + c0);
                    x[t][0] = hv.x; x[t][1] = hv.y; x[t][2] = hv.z; x[t][3] = hv.w;
                } else if (i < Lc) {
                    const uint2 raw = *reinterpret_cast<const uint2 *>(sm + st + i * (kD * 2) + c0 * 2);
                    const __nv_bfloat162 p0 = *reinterpret_cast<const __nv_bfloat162 *>(&raw.x);
                    const __nv_bfloat162 p1 = *reinterpret_cast<const __nv_bfloat162 *>(&raw.y);
                    x[t][0] = __low2float(p0); x[t][1] = __high2float(p0);
                    x[t][2] = __low2float(p1); x[t][3] = __high2float(p1);
                } else {
                    x[t][0] = x[t][1] = x[t][2] = x[t][3] = 0.f;
                }
            }
            if (W > 0) {
                float4 w4[4];
#pragma unroll
                for (int t = 0; t < 4; ++t)
                    w4[t] = *reinterpret_cast<const float4 *>(sConvW + t * 384 + which * kD + c0);
#pragma unroll
                for (int ii = 0; ii < kTok; ++ii) {
                    float acc[4];
                    acc[0] = w4[0].x * x[ii][0]; acc[1] = w4[0].y * x[ii][1];
                    acc[2] = w4[0].z * x[ii][2]; acc[3] = w4[0].w * x[ii][3];
#pragma unroll
                    for (int t = 1; t < 4; ++t) {
                        acc[0] = fmaf(w4[t].x, x[ii + t][0], acc[0]); acc[1] = fmaf(w4[t].y, x[ii + t][1], acc[1]);
                        acc[2] = fmaf(w4[t].z, x[ii + t][2], acc[2]); acc[3] = fmaf(w4[t].w, x[ii + t][3], acc[3]);
                    }
#pragma unroll
                    for (int m = 0; m < 4; ++m) y[ii][m] = (i0 + ii < Lc) ? silu_fast(acc[m]) : 0.f;
                }
            } else {
#pragma unroll
                for (int ii = 0; ii < kTok; ++ii)
#pragma unroll
                    for (int m = 0; m < 4; ++m) y[ii][m] = x[ii + 3][m];
            }
            if (a.l2 && which < 2) {
#pragma unroll
                for (int ii = 0; ii < kTok; ++ii) {
                    float ss = y[ii][0] * y[ii][0] + y[ii][1] * y[ii][1] + y[ii][2] * y[ii][2] + y[ii][3] * y[ii][3];
                    ss = warp_sum(ss);
                    const float inv = rsqrtf(ss + K3KDA_L2_EPS);
#pragma unroll
                    for (int m = 0; m < 4; ++m) y[ii][m] *= inv;
                }
            }
        };
        // one token's 4 channels, split, into row `row` of a K=128 tile (hi and lo tiles)
        auto put_row_split = [&](uint32_t off_hi, uint32_t off_lo, uint32_t rows, int row, const float (&v)[4]) {
            float hv[4], lv[4];
#pragma unroll
            for (int m = 0; m < 4; ++m) split_bf16(v[m], hv[m], lv[m]);
            const uint32_t o = kmaj128(rows, row, c0);
            *reinterpret_cast<uint2 *>(sm + off_hi + o) = make_uint2(pack_bf16(hv[0], hv[1]), pack_bf16(hv[2], hv[3]));
            *reinterpret_cast<uint2 *>(sm + off_lo + o) = make_uint2(pack_bf16(lv[0], lv[1]), pack_bf16(lv[2], lv[3]));
        };
        {
            float y[kTok][4];
            // q -> Qh = q E  (rows 64..127 of X / XL)
            finish(0, y);
#pragma unroll
            for (int ii = 0; ii < kTok; ++ii) {
                float t4[4];
#pragma unroll
                for (int m = 0; m < 4; ++m) t4[m] = y[ii][m] * E[ii][m];
                put_row_split(OFF_X, OFF_XL, 128, 64 + i0 + ii, t4);
            }
            // k -> Kh = k E (rows 0..63 of X / XL), Kb = k / E (rows; the state update reads them MN-major)
            finish(1, y);
#pragma unroll
            for (int ii = 0; ii < kTok; ++ii) {
                float t4[4], u4[4];
#pragma unroll
                for (int m = 0; m < 4; ++m) { t4[m] = y[ii][m] * E[ii][m]; u4[m] = y[ii][m] * Eb[ii][m]; }
                put_row_split(OFF_X, OFF_XL, 128, i0 + ii, t4);
                put_row_split(OFF_KB_HI, OFF_KB_LO, 64, i0 + ii, u4);
            }
            // v -> v rows (hi/lo; lo is zero unless the conv made v inexact), read MN-major by MMA U
            finish(2, y);
#pragma unroll
            for (int ii = 0; ii < kTok; ++ii) put_row_split(OFF_V_HI, OFF_V_LO, 64, i0 + ii, y[ii]);
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        PHASE(0);
        // pre-conv rows 61..63 of this chunk are the conv history of the next one
        if (W > 0 && cs + kC < te)
            for (int e = tid; e < 3 * 3 * 128; e += kThreads) {
                const int which = e / 384, r = (e / 128) % 3, c = e & 127;
                const uint32_t st = which == 0 ? OFF_QST : (which == 1 ? OFF_KST : OFF_VST);
                sHist[e] = __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(sm + st + (kC - 3 + r) * (kD * 2) + c * 2));
            }
        // ================= MMA: [Kh; Qh] Kb^T  -> Akk | Aqk =================
        if (tid == 0) {
            tc_fence_after();
            const uint32_t id = idesc_bf16_f32(128, 64);
            const uint64_t dX = sdesc_kmajor_sw128(sbase + OFF_X), dXL = sdesc_kmajor_sw128(sbase + OFF_XL);
            const uint64_t dKh = sdesc_kmajor_sw128(sbase + OFF_KB_HI), dKl = sdesc_kmajor_sw128(sbase + OFF_KB_LO);
#pragma unroll
            for (int sp = 0; sp < 3; ++sp)
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_bf16(tbase + kColA, dadd(sp == 2 ? dXL : dX, (kk >> 2) * 16384 + (kk & 3) * 32),
                             dadd(sp == 1 ? dKl : dKh, (kk >> 2) * 8192 + (kk & 3) * 32), id, (sp | kk) != 0);
            mma_commit(mbar_a);
        }
        if (!mma_wait()) { failed = true; break; }
        PHASE(1);
        // ================= Akk -> fp32 scratch, Aqk -> split tile =================
        {
            const int colbase = quarter * 16;
            uint32_t r0[16];
            tmem_ld16(tl + kColA + colbase, r0);
            tmem_wait_ld();
            const int row = lrow + lane;
            if (row < 64) {
                const float b = sBeta[row];
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    const int j = colbase + u;
                    scrA[sidx(row, j)] = j < row ? b * __uint_as_float(r0[u]) : 0.f;
                }
            } else {
                const int i = row - 64;
                float v[16];
#pragma unroll
                for (int u = 0; u < 16; ++u) v[u] = colbase + u > i ? 0.f : __uint_as_float(r0[u]);
                tile64_put16(sm, OFF_AQK_HI, OFF_AQK_LO, i, colbase, v);
            }
        }
        __syncthreads();
        PHASE(2);
        // ================= T = (I + Akk)^-1 in fp32, Tb = T diag(beta) (hi/lo) =================
        // diagonal 16x16 blocks by substitution (one column per thread); the upper blocks
        // (0,1) and (2,3) that the block products read are zeroed at the same time
        if (warp < 4 && lane < 16) {
            const int b = warp, col = lane, ib = b * 16;
            float x[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) x[i] = (i == col) ? 1.f : 0.f;
#pragma unroll
            for (int i = 1; i < 16; ++i) {
                float s0 = 0.f, s1 = 0.f;
#pragma unroll
                for (int j = 0; j < i; j += 2) {
                    s0 = fmaf(scrA[sidx(ib + i, ib + j)], x[j], s0);
                    if (j + 1 < i) s1 = fmaf(scrA[sidx(ib + i, ib + j + 1)], x[j + 1], s1);
                }
                if (i > col) x[i] = -(s0 + s1);
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) scrT[sidx(ib + i, ib + col)] = x[i];
        } else if (warp >= 4) {
            for (int e = tid - 128; e < 512; e += kThreads - 128) {
                const int blk = e >> 8, r = (e >> 4) & 15, c = e & 15;
                scrT[sidx(blk * 32 + r, blk * 32 + 16 + c)] = 0.f;
            }
        }
        __syncthreads();
        // level 1: T[b+1,b] = -T[b+1,b+1] (A[b+1,b] T[b,b]) for b = 0, 2; P parked in block (0, 2 + b/2)
        {
            const int e = tid;                               // 512 elements, one per thread
            const int pb = e >> 8, r = (e >> 4) & 15, c = e & 15, b = 2 * pb;
            float s0 = 0.f, s1 = 0.f;
#pragma unroll
            for (int m = 0; m < 16; m += 2) {
                s0 = fmaf(scrA[sidx((b + 1) * 16 + r, b * 16 + m)], scrT[sidx(b * 16 + m, b * 16 + c)], s0);
                s1 = fmaf(scrA[sidx((b + 1) * 16 + r, b * 16 + m + 1)], scrT[sidx(b * 16 + m + 1, b * 16 + c)], s1);
            }
            scrT[sidx(r, (2 + pb) * 16 + c)] = s0 + s1;
            __syncthreads();
            s0 = 0.f; s1 = 0.f;
#pragma unroll
            for (int m = 0; m < 16; m += 2) {
                s0 = fmaf(scrT[sidx((b + 1) * 16 + r, (b + 1) * 16 + m)], scrT[sidx(m, (2 + pb) * 16 + c)], s0);
                s1 = fmaf(scrT[sidx((b + 1) * 16 + r, (b + 1) * 16 + m + 1)], scrT[sidx(m + 1, (2 + pb) * 16 + c)], s1);
            }
            scrT[sidx((b + 1) * 16 + r, b * 16 + c)] = -(s0 + s1);
            __syncthreads();
        }
        // level 2: T[32:64, 0:32] = -T2 (A[32:64, 0:32] T1); P (32x32) parked in T[0:32, 32:64].
        // 256 threads, each a 2x2 output tile (rows r0, r0+1; columns cc, cc+1; r0, cc even).  With
        // the XOR swizzle, (row even, columns 2k, 2k+1) and (row m, columns cc, cc+1) are adjacent
        // words, so every operand pair is one 8-byte load (for odd m the pair is stored swapped).
        {
            const int r0 = ((tid >> 4) & 15) * 2, cc = (tid & 15) * 2;
            auto block_prod = [&](const float *Lm, int lrow, int lcol, int rcol, float (&p)[4]) {
                p[0] = p[1] = p[2] = p[3] = 0.f;
#pragma unroll
                for (int m = 0; m < 32; m += 2) {
                    const float2 a0 = *reinterpret_cast<const float2 *>(Lm + sidx(lrow + r0, lcol + m));
                    const float2 a1 = *reinterpret_cast<const float2 *>(Lm + sidx(lrow + r0 + 1, lcol + m) - 1);
                    const float2 be = *reinterpret_cast<const float2 *>(scrT + sidx(m, rcol + cc));
                    const float2 bo = *reinterpret_cast<const float2 *>(scrT + sidx(m + 1, rcol + cc) - 1);
                    // row r0 + 1 is odd: its pair (m, m+1) sits swapped, like the odd-m row of the right factor
                    p[0] = fmaf(a0.x, be.x, p[0]); p[1] = fmaf(a0.x, be.y, p[1]);
                    p[2] = fmaf(a1.y, be.x, p[2]); p[3] = fmaf(a1.y, be.y, p[3]);
                    p[0] = fmaf(a0.y, bo.y, p[0]); p[1] = fmaf(a0.y, bo.x, p[1]);
                    p[2] = fmaf(a1.x, bo.y, p[2]); p[3] = fmaf(a1.x, bo.x, p[3]);
                }
            };
            float p[4];
            if (tid < 256) {
                block_prod(scrA, 32, 0, 0, p);
                // the park area is read by nobody in this pass
                *reinterpret_cast<float2 *>(scrT + sidx(r0, 32 + cc)) = make_float2(p[0], p[1]);
                *reinterpret_cast<float2 *>(scrT + sidx(r0 + 1, 32 + cc) - 1) = make_float2(p[3], p[2]);
            }
            __syncthreads();
            if (tid < 256) {
                block_prod(scrT, 32, 32, 32, p);
                // T21 lives in rows 32..63, columns 0..31: not read by this pass
                *reinterpret_cast<float2 *>(scrT + sidx(32 + r0, cc)) = make_float2(-p[0], -p[1]);
                *reinterpret_cast<float2 *>(scrT + sidx(33 + r0, cc) - 1) = make_float2(-p[3], -p[2]);
            }
        }
        __syncthreads();
        {
            const int i = tid >> 3, jq = (tid & 7) * 8;
            uint32_t hw[4], lw[4];
#pragma unroll
            for (int u = 0; u < 8; u += 2) {
                const int j = jq + u;
                const float t0 = j <= i ? scrT[sidx(i, j)] * sBeta[j] : 0.f;
                const float t1 = j + 1 <= i ? scrT[sidx(i, j + 1)] * sBeta[j + 1] : 0.f;
                float h0, l0, h1, l1;
                split_bf16(t0, h0, l0);
                split_bf16(t1, h1, l1);
                hw[u >> 1] = pack_bf16(h0, h1);
                lw[u >> 1] = pack_bf16(l0, l1);
            }
            const uint32_t o0 = sw128_offset(i, jq);
            *reinterpret_cast<uint4 *>(sm + OFF_TB_HI + o0) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
            *reinterpret_cast<uint4 *>(sm + OFF_TB_LO + o0) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        PHASE(3);
        // ================= MMA: U^T = v^T Tb^T =================
        if (tid == 0) {
            tc_fence_after();
            const uint32_t id = idesc_bf16_f32(128, 64, false, /*a_mn=*/true);
            const uint64_t dVh = sdesc_mnmajor_sw128(sbase + OFF_V_HI, 8192), dVl = sdesc_mnmajor_sw128(sbase + OFF_V_LO, 8192);
            const uint64_t dTh = sdesc_kmajor_sw128(sbase + OFF_TB_HI), dTl = sdesc_kmajor_sw128(sbase + OFF_TB_LO);
            const int nsplit = W > 0 ? 3 : 2;           // v is exact bf16 without a conv
#pragma unroll
            for (int sp = 0; sp < 3; ++sp)
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    if (sp < nsplit)
                        mma_bf16(tbase + kColU, dadd(sp == 2 ? dVl : dVh, kk * 2048), dadd(sp == 1 ? dTl : dTh, kk * 32),
                                 id, (sp | kk) != 0);
            mma_commit(mbar_a);
        }
        if (!mma_wait()) { failed = true; break; }
        PHASE(4);
        // ================= S'^T = S^T diag(fcol) -> TMEM and split A tile =================
        {
            const int j = lrow + lane;
            for (int cb = 0; cb < 32; cb += 16) {
                const int col = quarter * 32 + cb;              // state column (channel c) of u = 0
                uint32_t r[16];
                tmem_ld16(tl + kColS + col, r);
                tmem_wait_ld();
                float v[16];
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    v[u] = __uint_as_float(r[u]) * sFcol[col + u];
                    r[u] = __float_as_uint(v[u]);
                }
                tmem_st16(tl + kColS + col, r);
                tile64_put16(sm, OFF_ST_HI + (col >> 6) * 16384, OFF_ST_LO + (col >> 6) * 16384, j, col & 63, v);
            }
            tmem_wait_st();
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        PHASE(5);
        // ================= MMA: Y^T = S'^T Kh^T,  O^T = S'^T Qh^T =================
        if (tid == 0) {
            tc_fence_after();
            const uint32_t id = idesc_bf16_f32(128, 64);
            const uint64_t dSh = sdesc_kmajor_sw128(sbase + OFF_ST_HI), dSl = sdesc_kmajor_sw128(sbase + OFF_ST_LO);
            const uint64_t dX = sdesc_kmajor_sw128(sbase + OFF_X), dXL = sdesc_kmajor_sw128(sbase + OFF_XL);
#pragma unroll
            for (int rowoff = 0; rowoff < 2; ++rowoff) {        // 0: Kh rows -> Y^T, 1: Qh rows -> O^T
                const uint32_t dcol = rowoff ? kColA : kColY;
#pragma unroll
                for (int sp = 0; sp < 3; ++sp)
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        mma_bf16(tbase + dcol, dadd(sp == 2 ? dSl : dSh, (kk >> 2) * 16384 + (kk & 3) * 32),
                                 dadd(sp == 1 ? dXL : dX, (kk >> 2) * 16384 + rowoff * 8192 + (kk & 3) * 32), id,
                                 (sp | kk) != 0);
            }
            mma_commit(mbar_a);
        }
        if (!mma_wait()) { failed = true; break; }
        PHASE(6);
        // 16 TMEM columns of this warp -> split [128 rows][64 K] tile
        auto tmem_to_tile64 = [&](uint32_t col, uint32_t off_hi, uint32_t off_lo) {
            uint32_t r0[16];
            tmem_ld16(tl + col + quarter * 16, r0);
            tmem_wait_ld();
            float v[16];
#pragma unroll
            for (int u = 0; u < 16; ++u) v[u] = __uint_as_float(r0[u]);
            tile64_put16(sm, off_hi, off_lo, lrow + lane, quarter * 16, v);
        };
        // ================= Y^T -> split tile;  MMA: V'^T = U^T - Y^T Tb^T =================
        tmem_to_tile64(kColY, OFF_YT_HI, OFF_YT_LO);
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            const uint32_t idn = idesc_bf16_f32(128, 64, true);
            const uint64_t dYh = sdesc_kmajor_sw128(sbase + OFF_YT_HI), dYl = sdesc_kmajor_sw128(sbase + OFF_YT_LO);
            const uint64_t dTh = sdesc_kmajor_sw128(sbase + OFF_TB_HI), dTl = sdesc_kmajor_sw128(sbase + OFF_TB_LO);
#pragma unroll
            for (int sp = 0; sp < 3; ++sp)
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16(tbase + kColU, dadd(sp == 2 ? dYl : dYh, kk * 32), dadd(sp == 1 ? dTl : dTh, kk * 32), idn, 1);
            mma_commit(mbar_a);
        }
        if (!mma_wait()) { failed = true; break; }
        if (cs + kC < te) stage_gv(cs + kC);          // Y^T region and the v staging rows are free now
        if (a.gate && tid == 0) {                     // this chunk's gate tile into the (now dead) Tb region
            fence_async_smem();
            mbar_arrive_expect_tx(mbar_g, (uint32_t)A.box_rows * kD * 2);
            tma_load_3d(sbase + OFF_TB_HI, &A.tm_gate, 0, h, cs, mbar_g);
        }
        PHASE(7);
        // ================= V'^T -> split tile;  MMA: O^T += V'^T Aqk^T,  S'^T += V'^T Kb =================
        tmem_to_tile64(kColU, OFF_VPT_HI, OFF_VPT_LO);
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            const uint32_t id64 = idesc_bf16_f32(128, 64);
            const uint32_t id128 = idesc_bf16_f32(128, 128, false, false, /*b_mn=*/true);
            const uint64_t dVh = sdesc_kmajor_sw128(sbase + OFF_VPT_HI), dVl = sdesc_kmajor_sw128(sbase + OFF_VPT_LO);
            const uint64_t dAh = sdesc_kmajor_sw128(sbase + OFF_AQK_HI), dAl = sdesc_kmajor_sw128(sbase + OFF_AQK_LO);
            const uint64_t dKh = sdesc_mnmajor_sw128(sbase + OFF_KB_HI, 8192), dKl = sdesc_mnmajor_sw128(sbase + OFF_KB_LO, 8192);
#pragma unroll
            for (int sp = 0; sp < 3; ++sp)
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16(tbase + kColA, dadd(sp == 2 ? dVl : dVh, kk * 32), dadd(sp == 1 ? dAl : dAh, kk * 32), id64, 1);
#pragma unroll
            for (int sp = 0; sp < 3; ++sp)
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16(tbase + kColS, dadd(sp == 2 ? dVl : dVh, kk * 32), dadd(sp == 1 ? dKl : dKh, kk * 2048), id128, 1);
            mma_commit(mbar_a);
        }
        if (a.gate && tid == 0 && !mbar_wait_bounded(mbar_g, gphase, kWaitLimit)) {
            *sflag = 1;
            atomicOr(a.status, 1u);
        }
        gphase ^= 1u;
        if (!mma_wait()) { failed = true; break; }   // its barrier also publishes the gate tile
        if (cs + kC < te) stage_qk(cs + kC);          // V'^T region is free now
        PHASE(8);
        // ================= epilogue: O^T -> gate -> out; carry the basis factor =================
        {
            const int j = lrow + lane;
            uint32_t r0[16];
            tmem_ld16(tl + kColA + quarter * 16, r0);
            tmem_wait_ld();
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                const int i = quarter * 16 + u;
                if (i < Lc) {
                    float o = a.scale * __uint_as_float(r0[u]);
                    if (a.gate)
                        o *= sigmoid_fast(__bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(
                            sm + OFF_TB_HI + i * (kD * 2) + j * 2)));
                    store_elt(a.out, ((size_t)(cs + i) * H + h) * kD + j, o, a.out_bf16);
                }
            }
        }
        PHASE(9);
        if (tid < kD) sLogf[tid] = sGL[tid] - sRef[tid];
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    }
#ifdef K3KDA_PHASE_TIMERS
    if (tid == 0 && blockIdx.x == 0) {
        unsigned long long *dst = reinterpret_cast<unsigned long long *>(a.status) + 8;
        for (int i = 0; i < 10; ++i) dst[i] = ph[i];
    }
#endif
#undef PHASE
    if (!failed) {
        // ---- final state: S = S'^T diag(exp(logf)) ----
        if (a.Sfin) {
            const int j = lrow + lane;
            for (int cb = 0; cb < 32; cb += 16) {
                uint32_t r[16];
                tmem_ld16(tl + kColS + quarter * 32 + cb, r);
                tmem_wait_ld();
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    const int c = quarter * 32 + cb + u;
                    a.Sfin[((size_t)nh * kD + c) * kD + j] = __uint_as_float(r[u]) * expf(sLogf[c]);
                }
            }
        }
        // ---- conv state: the last W-1 pre-conv inputs of this head's q, k, v channels ----
        if (A.conv_state != nullptr && W > 1) {
            const int L = te - tb;
            float keep[3] = {0.f, 0.f, 0.f};
            const int e = tid;
            const int which = e >> 7, c = e & 127;
            const int gch = which * H * kD + h * kD + c;
            if (e < 384) {
                const void *src = which == 0 ? a.q : (which == 1 ? a.k : a.v);
#pragma unroll
                for (int r = 0; r < 3; ++r)
                    if (r < W - 1) {
                        const int p = L - (W - 1) + r;
                        keep[r] = p >= 0
                            ? __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(src)[((size_t)(tb + p) * H + h) * kD + c])
                            : A.conv_state[((size_t)n * (W - 1) + (L + r)) * Dall + gch];
                    }
            }
            __syncthreads();
            if (e < 384)
#pragma unroll
                for (int r = 0; r < 3; ++r)
                    if (r < W - 1) A.conv_state[((size_t)n * (W - 1) + r) * Dall + gch] = keep[r];
        }
    } else if (tid == 0) {
        mbar_wait_bounded(mbar_a, phase ^ 1u, kWaitLimit);   // let an in-flight MMA drain before freeing TMEM
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tbase, kTmemCols);
}

}  // namespace

bool tc_prefill_supported(int in_bf16, int dk, int dv, int chunk) {
    return in_bf16 && dk == kD && dv == kD && chunk == kC;
}

size_t tc_prefill_workspace(int N, int H) { (void)N; (void)H; return 0; }

namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

// [T, H, 128] row-major tensor as a 3-D map (128 channels, H heads, T tokens); box = one
// head's 128 channels for 64 consecutive tokens, no swizzle (plain row-major staging).
cudaError_t make_map(CUtensorMap *m, const void *base, CUtensorMapDataType dt, int esz, int T, int H) {
    const cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)H, (cuuint64_t)T};
    const cuuint64_t strides[2] = {(cuuint64_t)kD * esz, (cuuint64_t)H * kD * esz};
    const cuuint32_t box[3] = {(cuuint32_t)kD, 1u, (cuuint32_t)(T < kC ? T : kC)};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    const CUresult r = g_encode(m, dt, 3, const_cast<void *>(base), dims, strides, box, estr,
                                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_prefill_tc_fused(const PrefillArgs &p, const float *conv_w, float *conv_state, int W,
                                    cudaStream_t s) {
    if ((long long)p.N * p.H == 0) return cudaSuccess;
    if (g_encode == nullptr) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || fn == nullptr)
            return e != cudaSuccess ? e : cudaErrorSymbolNotFound;
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    TcArgs A{};
    if (p.T > 0) {
        cudaError_t e;
        if ((e = make_map(&A.tm_q, p.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.T, p.H)) != cudaSuccess ||
            (e = make_map(&A.tm_k, p.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.T, p.H)) != cudaSuccess ||
            (e = make_map(&A.tm_v, p.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.T, p.H)) != cudaSuccess ||
            (e = make_map(&A.tm_g, p.g, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, p.T, p.H)) != cudaSuccess ||
            (p.gate && (e = make_map(&A.tm_gate, p.gate, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.T, p.H)) != cudaSuccess))
            return e;
    }
    static bool attr_done = false;
    if (!attr_done) {
        cudaError_t e = cudaFuncSetAttribute(kda_prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_done = true;
    }
    A.p = p;
    A.conv_w = conv_w;
    A.conv_state = conv_state;
    A.W = conv_w ? W : 0;
    A.box_rows = p.T < kC ? p.T : kC;
    kda_prefill_tc_kernel<<<(unsigned)(p.N * p.H), kThreads, kSmemBytes, s>>>(A);
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_prefill_tc(const PrefillArgs &a, const int32_t *order, cudaStream_t s) {
    (void)order;
    return launch_prefill_tc_fused(a, nullptr, nullptr, 0, s);
}

}  // namespace k3kda
