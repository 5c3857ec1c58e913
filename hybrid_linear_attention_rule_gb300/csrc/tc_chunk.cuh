// tc_chunk.cuh -- the state-independent part of one 64-token KDA chunk on the
// tensor-core path (bf16 inputs, dk = dv = 128), shared by the single-pass
// prefill kernel and the chunk-prep kernel of the two-pass prefill.
//
// From a chunk's staged input rows it builds, in shared memory: the decayed
// operands Kh = k E, Qh = q E, Kb = k / E (E = exp(G - r), r the per-channel
// mid-point of the chunk-local cumulative log-decay G) as split-bf16 K-major
// tiles, the v rows, Akk = diag(beta) tril(Kh Kb^T, -1) (fp32) and Aqk =
// tril(Qh Kb^T) (split-bf16) from one tcgen05 MMA chain, and Tb = (I + Akk)^-1
// diag(beta) (split-bf16) by a block-recursive fp32 triangular inverse.  The
// WY/UT form of the delta rule this serves is the one of "recurrent KDA
// state" (HF discussion #187 feature list; KdaState in the metrale kimi_k3
// docs).  Every function but issue_mma_a is called by all threads of the CTA
// (16 warps) and ends with a CTA barrier.
#pragma once

#include <cuda.h>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace k3kda {
namespace tcc {

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
constexpr uint32_t OFF_AQK_HI = 163840;          // Aqk^T [64 rows i'][64 i]  (extract .. MMA O; MN-major B)
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

// The stage functions take the offsets of their tiles from a plan.  The single-pass kernel uses
// the plan above (regions A and B reused by its state chain).  The chunk-prep kernel of the
// two-pass path uses one in which the next chunk's q, k, v rows land during this chunk's MMA A
// and its g rows during MMA U/W: region R holds the staged g rows, then Kb (until MMA A), then
// the solve's scratch.
struct PlanFused {
    static constexpr uint32_t GST = OFF_GST, QST = OFF_QST, KST = OFF_KST, VST = OFF_VST;
    static constexpr uint32_t V_HI = OFF_V_HI, V_LO = OFF_V_LO, KB_HI = OFF_KB_HI, KB_LO = OFF_KB_LO;
    static constexpr uint32_t SCR_A = OFF_SCR_A, SCR_T = OFF_SCR_T, AQK_HI = OFF_AQK_HI, AQK_LO = OFF_AQK_LO;
    static constexpr uint32_t TB_HI = OFF_TB_HI, TB_LO = OFF_TB_LO, SCAN = OFF_SCAN;
    static constexpr uint32_t X_HI = OFF_X, X_LO = OFF_XL, X_ATOM = 16384;   // [Kh; Qh]: hi atoms, then lo atoms
    static constexpr bool KB_STACKED = false;    // Kb hi and lo as two 64-row tiles
    static constexpr bool CALLER_STAGES = false; // prep_qk loads beta and owns every tile it writes
};
struct PlanPrep {
    static constexpr uint32_t V_HI = 65536, V_LO = 81920;                  // v rows      (prep_v .. MMA U)
    static constexpr uint32_t QST = 98304, KST = 114688, VST = 131072;     // staged rows (MMA A .. next prep)
    static constexpr uint32_t GST = 147456;                                // R: staged g (solve .. next prep_qk)
    static constexpr uint32_t KB_HI = 147456, KB_LO = 163840;              // R: Kb       (prep_qk .. MMA A)
    static constexpr uint32_t SCR_A = 147456, SCR_T = 163840;              // R: scratch  (extract .. solve)
    static constexpr uint32_t AQK_HI = 180224, AQK_LO = 188416;            // Aqk^T       (extract .. its store)
    static constexpr uint32_t SCAN = AQK_HI;                               // g partial sums (prep_qk)
    static constexpr uint32_t TB_HI = 196608, TB_LO = 204800;              // Tb          (solve .. MMA U/W)
    // [Kh; Qh] with the hi and lo tiles of each K atom adjacent ([hi 0 | lo 0 | hi 1 | lo 1], 16 KB
    // each): per K atom the 256 rows [Kh_hi; Qh_hi; Kh_lo; Qh_lo] are then one N = 256 operand
    static constexpr uint32_t X_HI = 0, X_LO = 16384, X_ATOM = 32768;
    // Kb hi in rows 0-63 and lo in rows 64-127 of one 128-row tile: MMA A then reads [Kb_hi; Kb_lo]
    // as one N = 128 operand (hi*hi and hi*lo in one chain) and adds lo*hi with N = 64
    static constexpr bool KB_STACKED = true;
    // the caller writes BETA before prep_qk, and the bulk stores still reading X rows 0-63 (issued
    // by thread 0) are waited for inside prep_qk, before those rows are rewritten
    static constexpr bool CALLER_STAGES = true;
};
static_assert(PlanPrep::TB_LO + 8192 <= OFF_CONVW, "prep plan runs into the small arrays");

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

// ---- stage 1: staged rows + conv history -> operand tiles ----
// Thread (warp, lane) owns tokens 4*warp .. +3 and channels 4*lane .. +3 of the chunk.

// Conv (+SiLU) and, for q and k with the L2 norm on, the norm of tensor `which` (0 q, 1 k, 2 v)
// for this thread's 4 tokens x 4 channels: reads the staged rows at `st` and the pre-conv rows
// before the chunk in HIST (tensor-major, three rows each).
__device__ __forceinline__ void conv_rows(const uint8_t *sm, const PrefillArgs &a, int which, uint32_t st,
                                          int Lc, int W, float (&y)[kTok][4]) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int i0 = warp * kTok, c0 = lane * 4;
    const float *sConvW = reinterpret_cast<const float *>(sm + OFF_CONVW);
    const float *sHist = reinterpret_cast<const float *>(sm + OFF_HIST);
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
        for (int t = 0; t < 4; ++t) w4[t] = *reinterpret_cast<const float4 *>(sConvW + t * 384 + which * kD + c0);
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
}

// One token's 4 channels, split, into row `row` of a K=128 tile (hi and lo tiles) whose two
// 64-wide K atoms lie `atom` bytes apart.
__device__ __forceinline__ void put_row_split(uint8_t *sm, uint32_t off_hi, uint32_t off_lo, uint32_t atom, int row,
                                              int c0, const float (&v)[4]) {
    float hv[4], lv[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) split_bf16(v[m], hv[m], lv[m]);
    const uint32_t o = (c0 >> 6) * atom + sw128_offset(row, c0 & 63);
    *reinterpret_cast<uint2 *>(sm + off_hi + o) = make_uint2(pack_bf16(hv[0], hv[1]), pack_bf16(hv[2], hv[3]));
    *reinterpret_cast<uint2 *>(sm + off_lo + o) = make_uint2(pack_bf16(lv[0], lv[1]), pack_bf16(lv[2], lv[3]));
}

// q and k: reads GST, QST, KST and the q, k rows of HIST; writes X/XL ([Kh; Qh] rows), KB, BETA,
// G0, GL, REF, and FCOL = exp(LOGF + r) when fcol is given.  Reads of GST all precede the first
// barrier, so GST may share its region with KB.
template <class P>
__device__ __forceinline__ void prep_qk(uint8_t *sm, const PrefillArgs &a, int cs, int Lc, int h, int W,
                                        const float *logf, float *fcol) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = a.H;
    const int i0 = warp * kTok, c0 = lane * 4;
    float *sBeta = reinterpret_cast<float *>(sm + OFF_BETA);
    float *sRef = reinterpret_cast<float *>(sm + OFF_REF);
    float *sGL = reinterpret_cast<float *>(sm + OFF_GL);
    float *sG0 = reinterpret_cast<float *>(sm + OFF_G0);
    float *sScan = reinterpret_cast<float *>(sm + P::SCAN);
    float G[kTok][4];
    {
        float run[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int ii = 0; ii < kTok; ++ii) {
            const int i = i0 + ii;
            float4 gv = make_float4(0.f, 0.f, 0.f, 0.f);
            if (i < Lc) gv = *reinterpret_cast<const float4 *>(sm + P::GST + i * (kD * 4) + c0 * 4);
            run[0] += gv.x; run[1] += gv.y; run[2] += gv.z; run[3] += gv.w;
#pragma unroll
            for (int m = 0; m < 4; ++m) G[ii][m] = run[m];
        }
        *reinterpret_cast<float4 *>(sScan + warp * kD + c0) = make_float4(run[0], run[1], run[2], run[3]);
    }
    if (!P::CALLER_STAGES && tid < kC) sBeta[tid] = tid < Lc ? a.beta[(size_t)(cs + tid) * H + h] : 0.f;
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
        if (fcol) fcol[tid] = expf(logf[tid] + r);     // TMEM basis -> this chunk's S' = exp(r) S
    }
    if (P::CALLER_STAGES && tid == 0) bulk_wait_read_all();   // X rows are rewritten below
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
    float y[kTok][4];
    // q -> Qh = q E  (rows 64..127 of X / XL)
    conv_rows(sm, a, 0, P::QST, Lc, W, y);
#pragma unroll
    for (int ii = 0; ii < kTok; ++ii) {
        float t4[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) t4[m] = y[ii][m] * E[ii][m];
        put_row_split(sm, P::X_HI, P::X_LO, P::X_ATOM, 64 + i0 + ii, c0, t4);
    }
    // k -> Kh = k E (rows 0..63 of X / XL), Kb = k / E (rows; the state update reads them MN-major)
    conv_rows(sm, a, 1, P::KST, Lc, W, y);
#pragma unroll
    for (int ii = 0; ii < kTok; ++ii) {
        float t4[4], u4[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) { t4[m] = y[ii][m] * E[ii][m]; u4[m] = y[ii][m] * Eb[ii][m]; }
        put_row_split(sm, P::X_HI, P::X_LO, P::X_ATOM, i0 + ii, c0, t4);
        if (P::KB_STACKED) put_row_split(sm, P::KB_HI, P::KB_HI + 8192, 16384, i0 + ii, c0, u4);
        else put_row_split(sm, P::KB_HI, P::KB_LO, 8192, i0 + ii, c0, u4);
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
}

// v: reads VST and the v rows of HIST; writes V_HI/LO (v rows, hi/lo; lo is zero unless the conv
// made v inexact), read MN-major by MMA U.
template <class P>
__device__ __forceinline__ void prep_v(uint8_t *sm, const PrefillArgs &a, int Lc, int W) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int i0 = warp * kTok, c0 = lane * 4;
    float y[kTok][4];
    conv_rows(sm, a, 2, P::VST, Lc, W, y);
#pragma unroll
    for (int ii = 0; ii < kTok; ++ii) put_row_split(sm, P::V_HI, P::V_LO, 8192, i0 + ii, c0, y[ii]);
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
}

template <class P>
__device__ __forceinline__ void prep_chunk(uint8_t *sm, const PrefillArgs &a, int cs, int Lc, int h, int W,
                                           const float *logf, float *fcol) {
    prep_qk<P>(sm, a, cs, Lc, h, W, logf, fcol);
    prep_v<P>(sm, a, Lc, W);
}

// ---- stage 2 (one thread): [Kh; Qh] Kb^T -> TMEM columns [col, col + 64) (with a stacked Kb tile:
// [col, col + 128), the sum of the two halves), commit to mbar ----
template <class P>
__device__ __forceinline__ void issue_mma_a(uint32_t sbase, uint32_t tmem_col_addr, uint32_t mbar) {
    tc_fence_after();
    const uint64_t dX = sdesc_kmajor_sw128(sbase + P::X_HI), dXL = sdesc_kmajor_sw128(sbase + P::X_LO);
    if (P::KB_STACKED) {
        // X_hi [Kb_hi; Kb_lo]^T (N = 128), then X_lo Kb_hi^T into the first 64 columns
        const uint64_t dK = sdesc_kmajor_sw128(sbase + P::KB_HI);
        const uint32_t id128 = idesc_bf16_f32(128, 128), id64 = idesc_bf16_f32(128, 64);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
            mma_bf16(tmem_col_addr, dadd(dX, (kk >> 2) * P::X_ATOM + (kk & 3) * 32),
                     dadd(dK, (kk >> 2) * 16384 + (kk & 3) * 32), id128, kk != 0);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
            mma_bf16(tmem_col_addr, dadd(dXL, (kk >> 2) * P::X_ATOM + (kk & 3) * 32),
                     dadd(dK, (kk >> 2) * 16384 + (kk & 3) * 32), id64, 1);
    } else {
        const uint32_t id = idesc_bf16_f32(128, 64);
        const uint64_t dKh = sdesc_kmajor_sw128(sbase + P::KB_HI), dKl = sdesc_kmajor_sw128(sbase + P::KB_LO);
#pragma unroll
        for (int sp = 0; sp < 3; ++sp)
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                mma_bf16(tmem_col_addr, dadd(sp == 2 ? dXL : dX, (kk >> 2) * P::X_ATOM + (kk & 3) * 32),
                         dadd(sp == 1 ? dKl : dKh, (kk >> 2) * 8192 + (kk & 3) * 32), id, (sp | kk) != 0);
    }
    mma_commit(mbar);
}

// ---- stage 3: Akk (times beta, strictly lower) -> fp32 scratch A, Aqk (lower) -> split tile (transposed) ----
// tl is this warp's TMEM lane base, col the first column of the MMA A result.
template <class P>
__device__ __forceinline__ void extract_a(uint8_t *sm, uint32_t tl, uint32_t col) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quarter = warp >> 2, lrow = 32 * (warp & 3);
    const float *sBeta = reinterpret_cast<const float *>(sm + OFF_BETA);
    float *scrA = reinterpret_cast<float *>(sm + P::SCR_A);
    // ================= Akk -> fp32 scratch, Aqk -> split tile =================
    {
        const int colbase = quarter * 16;
        uint32_t r0[16];
        tmem_ld16(tl + col + colbase, r0);
        if (P::KB_STACKED) {
            uint32_t r1[16];
            tmem_ld16(tl + col + 64 + colbase, r1);
            tmem_wait_ld();
#pragma unroll
            for (int u = 0; u < 16; ++u) r0[u] = __float_as_uint(__uint_as_float(r0[u]) + __uint_as_float(r1[u]));
        } else {
            tmem_wait_ld();
        }
        const int row = lrow + lane;
        if (row < 64) {
            const float b = sBeta[row];
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                const int j = colbase + u;
                scrA[sidx(row, j)] = j < row ? b * __uint_as_float(r0[u]) : 0.f;
            }
        } else {
            // Aqk stored transposed, [i'][i]: the MMAs read it as an MN-major B operand, so that
            // it can sit beside the Kb rows in one N = 192 operand; a warp's 32 lanes (32
            // consecutive i) fill 64 contiguous bytes of one row i'
            const int i = row - 64;
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                const int ip = colbase + u;
                float hv, lv;
                split_bf16(ip > i ? 0.f : __uint_as_float(r0[u]), hv, lv);
                const uint32_t o = sw128_offset(ip, i);
                *reinterpret_cast<__nv_bfloat16 *>(sm + P::AQK_HI + o) = __float2bfloat16_rn(hv);
                *reinterpret_cast<__nv_bfloat16 *>(sm + P::AQK_LO + o) = __float2bfloat16_rn(lv);
            }
        }
    }
    __syncthreads();
}

// ---- stage 4: T = (I + Akk)^-1 (fp32, block recursive), Tb = T diag(beta) -> split tile ----
template <class P>
__device__ __forceinline__ void solve_tb(uint8_t *sm) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const float *sBeta = reinterpret_cast<const float *>(sm + OFF_BETA);
    const float *scrA = reinterpret_cast<const float *>(sm + P::SCR_A);
    float *scrT = reinterpret_cast<float *>(sm + P::SCR_T);
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
        *reinterpret_cast<uint4 *>(sm + P::TB_HI + o0) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
        *reinterpret_cast<uint4 *>(sm + P::TB_LO + o0) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
}

// ---- optional per-phase cycle counters (compile with -DK3KDA_PHASE_TIMERS) ----
// Thread 0 accumulates clock64() deltas per phase; flush() adds them to a device array.
struct PhaseClock {
#ifdef K3KDA_PHASE_TIMERS
    unsigned long long ph[8];
    long long last;
    __device__ PhaseClock() {
        for (int i = 0; i < 8; ++i) ph[i] = 0;
        last = clock64();
    }
    __device__ __forceinline__ void tick(int i) {
        if (threadIdx.x == 0) {
            const long long now = clock64();
            ph[i] += (unsigned long long)(now - last);
            last = now;
        }
    }
    __device__ __forceinline__ void flush(unsigned long long *dst) {
        if (threadIdx.x == 0 && blockIdx.x == 0)
            for (int i = 0; i < 8; ++i) dst[i] = ph[i];
    }
#else
    __device__ __forceinline__ void tick(int) {}
    __device__ __forceinline__ void flush(unsigned long long *) {}
#endif
};

// ---- host side ----
// [T, H, 128] row-major tensor as a 3-D TMA map (128 channels, H heads, T tokens); box =
// one head's 128 channels for min(64, T) consecutive tokens, no swizzle.
cudaError_t make_row_map(CUtensorMap *m, const void *base, CUtensorMapDataType dt, int esz, int T, int H);

}  // namespace tcc
}  // namespace k3kda
