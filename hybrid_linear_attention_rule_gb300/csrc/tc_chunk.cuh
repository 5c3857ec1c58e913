// tc_chunk.cuh -- the state-independent part of one 64-token KDA chunk on the
// tensor-core path (bf16 inputs, dk = dv = 128), shared by the single-pass
// prefill kernel and the chunk-prep kernel of the two-pass prefill.
//
// From a chunk's staged input rows it builds, in shared memory: the decayed
// operands Kh = k E, Qh = q E, Kb = k / E (E = exp(G - rho), G the chunk-local
// cumulative log-decay and rho a per-channel reference) as split-bf16 K-major
// tiles, the v rows, Akk = diag(beta) tril(Kh Kb^T, -1) (fp32) and Aqk =
// tril(Qh Kb^T) (split-bf16) from one tcgen05 MMA chain, and Tb = (I + Akk)^-1
// diag(beta) (split-bf16) by a block-recursive fp32 triangular inverse; and, in
// registers, Kd = k exp(G_last - G), the operand of the state update.  The
// WY/UT form of the delta rule this serves is the one of "recurrent KDA state"
// (HF discussion #187 feature list; KdaState in the metrale kimi_k3 docs).
//
// Range.  The recurrence puts no bound on the decay, so no exponent here may
// exceed the fp32 range whatever g is.  For a channel whose decay across the
// chunk (G_first - G_last) is at most kStrongDecay nats, rho is the mid-point
// of G and every factor E, 1/E lies within exp(+-kStrongDecay / 2).  A channel
// that decays more ("strong") takes rho = G_first, so that E <= 1, and is left
// out of the factorised product (its Kb column is zero); its share of Akk and
// Aqk, sum_c x_ic k_jc exp(G_ic - G_jc) over the strong channels c, is formed
// exactly on the CUDA cores and written into the MMA's TMEM accumulator before
// the chain runs.  The state side never divides by a decay: the scan uses
// exp(rho) <= 1, exp(G_last) <= 1 and Kd.
//
// Every function but issue_mma_a is called by all threads of the CTA (16 warps)
// and ends with a CTA barrier.
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
// In-chunk decay (nats, G_first - G_last of one channel) above which a channel's share of Akk and
// Aqk is computed exactly instead of through E and 1/E: below it every factor stays within
// exp(+-80), far inside the fp32 range.
constexpr float kStrongDecay = 160.f;

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
constexpr uint32_t OFF_REF = OFF_BETA + 256;          // rho per channel
constexpr uint32_t OFF_GL = OFF_REF + 512;            // G_last per channel
constexpr uint32_t OFF_G0 = OFF_GL + 512;             // G_first per channel
constexpr uint32_t OFF_FCOL = OFF_G0 + 512;           // exp(rho) per channel (single-pass state pass)
constexpr uint32_t OFF_LOGF = OFF_FCOL + 512;         // exp(G_last) per channel (single-pass state pass)
constexpr uint32_t OFF_SMASK = 32;                    // (from OFF_MISC) 4 words: strong channels of the chunk
constexpr uint32_t OFF_MISC = OFF_LOGF + 512;         // mbarriers (3 x 8 B), tmem slot, flag, strong masks
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
    // strong-channel correction: staged rows (GST/V region, free once G is in registers) and the
    // fp32 correction (the Aqk and Tb tiles, free until the extract)
    static constexpr uint32_t STRONG_STAGE = OFF_V_HI, STRONG_ACC = OFF_AQK_HI;
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
    // strong-channel correction: staged rows (the v tiles, written by prep_v afterwards) and the
    // fp32 correction (the Aqk and Tb tiles, free until the extract)
    static constexpr uint32_t STRONG_STAGE = V_HI, STRONG_ACC = AQK_HI;
};
static_assert(PlanPrep::TB_LO + 8192 <= OFF_CONVW, "prep plan runs into the small arrays");
static_assert(PlanPrep::STRONG_ACC + 32768 == PlanPrep::TB_LO + 8192 && PlanFused::STRONG_ACC + 32768 == OFF_TB_LO + 8192,
              "the strong-channel correction (32 KB) must span the Aqk and Tb tiles exactly");
static_assert(PlanPrep::STRONG_STAGE + 24576 <= PlanPrep::QST && PlanFused::STRONG_STAGE + 24576 <= OFF_QST,
              "the strong-channel staging (24 KB) must fit the v tiles");

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
// for NT tokens from i0 x this lane's 4 channels: reads the staged rows at `st` and the pre-conv
// rows before the chunk in HIST (tensor-major, three rows each).
template <int NT>
__device__ __forceinline__ void conv_rows(const uint8_t *sm, const PrefillArgs &a, int which, uint32_t st,
                                          int Lc, int W, int i0, float (&y)[NT][4]) {
    const int c0 = (threadIdx.x & 31) * 4;
    const float *sConvW = reinterpret_cast<const float *>(sm + OFF_CONVW);
    const float *sHist = reinterpret_cast<const float *>(sm + OFF_HIST);
    float x[NT + 3][4];
#pragma unroll
    for (int t = 0; t < NT + 3; ++t) {
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
        for (int ii = 0; ii < NT; ++ii) {
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
        for (int ii = 0; ii < NT; ++ii)
#pragma unroll
            for (int m = 0; m < 4; ++m) y[ii][m] = x[ii + 3][m];
    }
    if (a.l2 && which < 2) {
#pragma unroll
        for (int ii = 0; ii < NT; ++ii) {
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

// ---- strong channels (in-chunk decay above kStrongDecay) ----
__device__ __forceinline__ const uint32_t *strong_mask(const uint8_t *sm) {
    return reinterpret_cast<const uint32_t *>(sm + OFF_MISC + OFF_SMASK);
}
// 4 bits: whether channels c0 .. c0 + 3 (c0 a multiple of 4) are strong
__device__ __forceinline__ uint32_t strong_bits4(const uint32_t *mask, int c0) { return (mask[c0 >> 5] >> (c0 & 31)) & 15u; }
// rank of strong channel c among the strong channels
__device__ __forceinline__ int strong_rank(const uint32_t *mask, int c) {
    int p = __popc(mask[c >> 5] & ((1u << (c & 31)) - 1u));
    for (int w = 0; w < (c >> 5); ++w) p += __popc(mask[w]);
    return p;
}

// The strong channels' share of the MMA A result, exactly: for row i and column j of the chunk
//   D[i][j] = sum_c k_ic k_jc exp(G_ic - G_jc),   D[64 + i][j] = sum_c q_ic k_jc exp(G_ic - G_jc)
// over the strong channels c (j <= i; the extract masks the rest and applies beta), written into
// TMEM columns [col, col + 64) of the MMA A accumulator (and zeros into [col + 64, col + 128) for a
// stacked Kb, whose N = 128 chain accumulates there too).  The strong channels go in groups of 32
// through a staging area ([k | q | G log2 e][32 channels][64 tokens] fp32); each of 272 threads
// holds a block of 4 rows i x 2 columns j of the lower triangle, so that every exponential
// serves both the k row and the q row; the blocks meet in an fp32 [128][64] array whose 16-byte
// slots are swizzled by row.
template <class P>
__device__ __forceinline__ void strong_correction(uint8_t *sm, const float (&yq)[kTok][4], const float (&yk)[kTok][4],
                                                  const float (&G)[kTok][4], uint32_t tl, uint32_t col) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int i0 = warp * kTok, c0 = lane * 4;
    const uint32_t *mask = strong_mask(sm);
    float *stK = reinterpret_cast<float *>(sm + P::STRONG_STAGE);
    float *stQ = stK + 32 * kC, *stG = stQ + 32 * kC;
    float *acc = reinterpret_cast<float *>(sm + P::STRONG_ACC);
    const int ns = __popc(mask[0]) + __popc(mask[1]) + __popc(mask[2]) + __popc(mask[3]);
    const uint32_t mine = strong_bits4(mask, c0);
    const int rank0 = mine ? strong_rank(mask, c0) : 0;
    // this thread's block: rows 4 bi .. + 3, columns 2 bj .. + 1 (row block bi holds 2 bi + 2 blocks)
    const bool unit = tid < 272;
    int bi = 0;
    while ((bi + 1) * (bi + 2) <= tid) ++bi;
    const int bj = tid - bi * (bi + 1);
    float akk[4][2], aqk[4][2];
#pragma unroll
    for (int u = 0; u < 4; ++u) akk[u][0] = akk[u][1] = aqk[u][0] = aqk[u][1] = 0.f;
    constexpr float kLog2e = 1.4426950408889634f;
    for (int g0 = 0; g0 < ns; g0 += 32) {
        int p = rank0;
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            if ((mine >> m) & 1u) {
                if (p >= g0 && p < g0 + 32) {
                    const int s = p - g0;
                    *reinterpret_cast<float4 *>(stK + s * kC + i0) = make_float4(yk[0][m], yk[1][m], yk[2][m], yk[3][m]);
                    *reinterpret_cast<float4 *>(stQ + s * kC + i0) = make_float4(yq[0][m], yq[1][m], yq[2][m], yq[3][m]);
                    *reinterpret_cast<float4 *>(stG + s * kC + i0) =
                        make_float4(G[0][m] * kLog2e, G[1][m] * kLog2e, G[2][m] * kLog2e, G[3][m] * kLog2e);
                }
                ++p;
            }
        }
        __syncthreads();
        if (unit) {
            const int ng = min(32, ns - g0);
            for (int s = 0; s < ng; ++s) {
                const float4 ki = *reinterpret_cast<const float4 *>(stK + s * kC + 4 * bi);
                const float4 qi = *reinterpret_cast<const float4 *>(stQ + s * kC + 4 * bi);
                const float4 gi = *reinterpret_cast<const float4 *>(stG + s * kC + 4 * bi);
                const float2 kj = *reinterpret_cast<const float2 *>(stK + s * kC + 2 * bj);
                const float2 gj = *reinterpret_cast<const float2 *>(stG + s * kC + 2 * bj);
                const float kiv[4] = {ki.x, ki.y, ki.z, ki.w}, qiv[4] = {qi.x, qi.y, qi.z, qi.w};
                const float giv[4] = {gi.x, gi.y, gi.z, gi.w};
                const float kjv[2] = {kj.x, kj.y}, gjv[2] = {gj.x, gj.y};
#pragma unroll
                for (int u = 0; u < 4; ++u)
#pragma unroll
                    for (int v = 0; v < 2; ++v) {
                        // G is non-increasing, so the exponent is <= 0 wherever j <= i; above the
                        // diagonal (masked by the extract) it is capped at 0
                        const float t = kjv[v] * exp2f(fminf(giv[u] - gjv[v], 0.f));
                        akk[u][v] = fmaf(kiv[u], t, akk[u][v]);
                        aqk[u][v] = fmaf(qiv[u], t, aqk[u][v]);
                    }
            }
        }
        __syncthreads();                                 // the staging area is rewritten by the next group
    }
    if (unit) {
        const int slot = bj >> 1, half = (bj & 1) * 2;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int r = 4 * bi + u;
            *reinterpret_cast<float2 *>(acc + r * 64 + ((slot ^ (r & 15)) << 2) + half) = make_float2(akk[u][0], akk[u][1]);
            *reinterpret_cast<float2 *>(acc + (64 + r) * 64 + ((slot ^ (r & 15)) << 2) + half) =
                make_float2(aqk[u][0], aqk[u][1]);
        }
    }
    __syncthreads();
    {
        // TMEM lane row = this warp's lane base + lane; columns 16 * quarter .. + 15
        const int row = 32 * (warp & 3) + lane, quarter = warp >> 2, rb = (row & 63) >> 2;
        uint32_t v[16];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const int slot = quarter * 4 + t;
            const float4 x = slot <= rb ? *reinterpret_cast<const float4 *>(acc + row * 64 + ((slot ^ (row & 15)) << 2))
                                        : make_float4(0.f, 0.f, 0.f, 0.f);
            v[4 * t] = __float_as_uint(x.x); v[4 * t + 1] = __float_as_uint(x.y);
            v[4 * t + 2] = __float_as_uint(x.z); v[4 * t + 3] = __float_as_uint(x.w);
        }
        tmem_st16(tl + col + quarter * 16, v);
        if (P::KB_STACKED) {
#pragma unroll
            for (int t = 0; t < 16; ++t) v[t] = 0u;
            tmem_st16(tl + col + 64 + quarter * 16, v);
        }
        tmem_wait_st();
    }
}

// q and k: reads GST, QST, KST and the q, k rows of HIST; writes X/XL ([Kh; Qh] rows), KB, BETA
// (unless the caller stages it), G0, GL, REF (rho) and the strong-channel masks; returns Kd =
// k exp(G_last - G) for this thread's 4 tokens x 4 channels in kd, and whether the chunk has a
// strong channel, whose exact share of MMA A is then already in TMEM columns [col, col + 64) (the
// chain must accumulate onto it).  Reads of GST all precede the first barrier, so GST may share
// its region with KB and the strong-channel staging.
template <class P>
__device__ __forceinline__ bool prep_qk(uint8_t *sm, const PrefillArgs &a, int cs, int Lc, int h, int W, uint32_t tl,
                                        uint32_t col, float (&kd)[kTok][4]) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = a.H;
    const int i0 = warp * kTok, c0 = lane * 4;
    float *sBeta = reinterpret_cast<float *>(sm + OFF_BETA);
    float *sRef = reinterpret_cast<float *>(sm + OFF_REF);
    float *sGL = reinterpret_cast<float *>(sm + OFF_GL);
    float *sG0 = reinterpret_cast<float *>(sm + OFF_G0);
    float *sScan = reinterpret_cast<float *>(sm + P::SCAN);
    uint32_t *sMask = reinterpret_cast<uint32_t *>(sm + OFF_MISC + OFF_SMASK);
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
    bool strong = false;
    if (tid < kD) {
        const float g0 = sG0[tid], gl = sGL[tid];
        strong = g0 - gl > kStrongDecay;
        sRef[tid] = strong ? g0 : 0.5f * (g0 + gl);
    }
    {
        const uint32_t m = __ballot_sync(0xffffffffu, strong);
        if (warp < 4 && lane == 0) sMask[warp] = m;
    }
    if (P::CALLER_STAGES && tid == 0) bulk_wait_read_all();   // X rows are rewritten below
    const bool any_strong = __syncthreads_or(strong) != 0;
    float yq[kTok][4], yk[kTok][4];
    conv_rows<kTok>(sm, a, 0, P::QST, Lc, W, i0, yq);
    conv_rows<kTok>(sm, a, 1, P::KST, Lc, W, i0, yk);
    if (any_strong) strong_correction<P>(sm, yq, yk, G, tl, col);
    {
        const float4 r4 = *reinterpret_cast<const float4 *>(sRef + c0);
        const float4 l4 = *reinterpret_cast<const float4 *>(sGL + c0);
        const float rr[4] = {r4.x, r4.y, r4.z, r4.w}, gl[4] = {l4.x, l4.y, l4.z, l4.w};
        const uint32_t sb = strong_bits4(sMask, c0);
        // exp(G_last - G) = exp(G_last - rho) exp(rho - G): two factors within exp(+-80) for the
        // other channels; a strong channel (no 1/E) takes its own exponential
        float cgl[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) cgl[m] = __expf(gl[m] - rr[m]);
#pragma unroll
        for (int ii = 0; ii < kTok; ++ii) {
            float qh[4], kh[4], kb[4];
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                // |G - rho| <= kStrongDecay / 2 for the other channels; G - rho <= 0 for strong ones,
                // whose factorised product is left out (Kb column zero)
                const float x = G[ii][m] - rr[m];
                const float e = __expf(x);
                const float eb = ((sb >> m) & 1u) ? 0.f : __expf(-x);
                qh[m] = yq[ii][m] * e;
                kh[m] = yk[ii][m] * e;
                kb[m] = yk[ii][m] * eb;
                kd[ii][m] = kb[m] * cgl[m];
            }
            if (sb != 0u) {
#pragma unroll
                for (int m = 0; m < 4; ++m)
                    if ((sb >> m) & 1u) kd[ii][m] = yk[ii][m] * __expf(gl[m] - G[ii][m]);
            }
            put_row_split(sm, P::X_HI, P::X_LO, P::X_ATOM, 64 + i0 + ii, c0, qh);   // Qh rows 64..127
            put_row_split(sm, P::X_HI, P::X_LO, P::X_ATOM, i0 + ii, c0, kh);        // Kh rows 0..63
            if (P::KB_STACKED) put_row_split(sm, P::KB_HI, P::KB_HI + 8192, 16384, i0 + ii, c0, kb);
            else put_row_split(sm, P::KB_HI, P::KB_LO, 8192, i0 + ii, c0, kb);
        }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    return any_strong;
}

// v: reads VST and the v rows of HIST; writes V_HI/LO (v rows, hi/lo; lo is zero unless the conv
// made v inexact), read MN-major by MMA U.
template <class P>
__device__ __forceinline__ void prep_v(uint8_t *sm, const PrefillArgs &a, int Lc, int W) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int i0 = warp * kTok, c0 = lane * 4;
    float y[kTok][4];
    conv_rows<kTok>(sm, a, 2, P::VST, Lc, W, i0, y);
#pragma unroll
    for (int ii = 0; ii < kTok; ++ii) put_row_split(sm, P::V_HI, P::V_LO, 8192, i0 + ii, c0, y[ii]);
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
}

// Kd (4 tokens x 4 channels of this thread) as split-bf16 rows of a K = 128 tile whose two 64-wide
// K atoms lie 16 KB apart, each the hi 64-row tile then the lo one: the layout of a stacked Kb tile
// and of the record's Kd part, read MN-major by the state update.  dst is a shared or a global
// (generic) address.
__device__ __forceinline__ void put_kd(uint8_t *dst, const float (&kd)[kTok][4]) {
    const int warp = threadIdx.x >> 5, c0 = (threadIdx.x & 31) * 4;
#pragma unroll
    for (int ii = 0; ii < kTok; ++ii) {
        float hv[4], lv[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) split_bf16(kd[ii][m], hv[m], lv[m]);
        const uint32_t o = (c0 >> 6) * 16384u + sw128_offset(warp * kTok + ii, c0 & 63);
        *reinterpret_cast<uint2 *>(dst + o) = make_uint2(pack_bf16(hv[0], hv[1]), pack_bf16(hv[2], hv[3]));
        *reinterpret_cast<uint2 *>(dst + o + 8192) = make_uint2(pack_bf16(lv[0], lv[1]), pack_bf16(lv[2], lv[3]));
    }
}

// ---- stage 2 (one thread): [Kh; Qh] Kb^T -> TMEM columns [col, col + 64) (with a stacked Kb tile:
// [col, col + 128), the sum of the two halves), commit to mbar; with acc the chain adds onto what
// the columns hold (the strong channels' share) ----
template <class P>
__device__ __forceinline__ void issue_mma_a(uint32_t sbase, uint32_t tmem_col_addr, uint32_t mbar, bool acc) {
    tc_fence_after();
    const uint64_t dX = sdesc_kmajor_sw128(sbase + P::X_HI), dXL = sdesc_kmajor_sw128(sbase + P::X_LO);
    if (P::KB_STACKED) {
        // X_hi [Kb_hi; Kb_lo]^T (N = 128), then X_lo Kb_hi^T into the first 64 columns
        const uint64_t dK = sdesc_kmajor_sw128(sbase + P::KB_HI);
        const uint32_t id128 = idesc_bf16_f32(128, 128), id64 = idesc_bf16_f32(128, 64);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
            mma_bf16(tmem_col_addr, dadd(dX, (kk >> 2) * P::X_ATOM + (kk & 3) * 32),
                     dadd(dK, (kk >> 2) * 16384 + (kk & 3) * 32), id128, acc || kk != 0);
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
                         dadd(sp == 1 ? dKl : dKh, (kk >> 2) * 8192 + (kk & 3) * 32), id, acc || (sp | kk) != 0);
    }
    mma_commit(mbar);
}

// ---- stages 3 and 4: T = (I + Akk)^-1 (fp32, block recursive), Tb = T diag(beta) -> split tile,
// and Aqk (lower) -> split tile (transposed), from the MMA A result in TMEM columns [col, col + 64)
// (plus [col + 64, col + 128) for a stacked Kb).  The warps on TMEM lanes 0-63 (warp & 3 < 2) take
// Akk and the substitution, those on lanes 64-127 take Aqk meanwhile.  tl is this warp's TMEM lane
// base.
template <class P>
__device__ __forceinline__ void mma_a_row16(uint32_t tl, uint32_t col, uint32_t (&r0)[16]) {
    tmem_ld16(tl + col, r0);
    if (P::KB_STACKED) {
        uint32_t r1[16];
        tmem_ld16(tl + col + 64, r1);
        tmem_wait_ld();
#pragma unroll
        for (int u = 0; u < 16; ++u) r0[u] = __float_as_uint(__uint_as_float(r0[u]) + __uint_as_float(r1[u]));
    } else {
        tmem_wait_ld();
    }
}

// Akk (times beta, strictly lower) -> fp32 scratch A, by the warps on lanes 0-63; they also zero
// the upper blocks (0,1) and (2,3) of T that the block products read.
template <class P>
__device__ __forceinline__ void extract_akk(uint8_t *sm, uint32_t tl, uint32_t col) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if ((warp & 3) < 2) {
        const int quarter = warp >> 2, row = 32 * (warp & 3) + lane, colbase = quarter * 16;
        const float b = reinterpret_cast<const float *>(sm + OFF_BETA)[row];
        float *scrA = reinterpret_cast<float *>(sm + P::SCR_A);
        float *scrT = reinterpret_cast<float *>(sm + P::SCR_T);
        uint32_t r0[16];
        mma_a_row16<P>(tl, col + colbase, r0);
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            const int j = colbase + u;
            scrA[sidx(row, j)] = j < row ? b * __uint_as_float(r0[u]) : 0.f;
        }
        const int e = (warp >> 2) * 64 + (warp & 1) * 32 + lane;    // 0 .. 255
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int f = e + 256 * k, blk = f >> 8, r = (f >> 4) & 15, c = f & 15;
            scrT[sidx(blk * 32 + r, blk * 32 + 16 + c)] = 0.f;
        }
    }
    __syncthreads();
}

template <class P>
__device__ __forceinline__ void solve_tb(uint8_t *sm, uint32_t tl, uint32_t col) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const float *sBeta = reinterpret_cast<const float *>(sm + OFF_BETA);
    const float *scrA = reinterpret_cast<const float *>(sm + P::SCR_A);
    float *scrT = reinterpret_cast<float *>(sm + P::SCR_T);
    // ================= T = (I + Akk)^-1 in fp32, Tb = T diag(beta) (hi/lo) =================
    // Rows of the fp32 scratch are stored with their 16-byte slots permuted by the row (sidx): the
    // four words from column c (a multiple of 4) of row r are the slot at r*64 + (c ^ (r & 28)),
    // word w holding column c + (w ^ (r & 3)).
    //
    // Diagonal 16x16 blocks by substitution, x_i = -sum_{j<i} A_ij x_j down each column of the
    // block inverse: warps 4b and 4b+1 take block b, four threads per column, each holding rows
    // 4p .. 4p+3 of the column and summing over its own four of them (A is zero on and above the
    // diagonal, so entries not yet final contribute nothing).  Meanwhile the warps on lanes 64-127
    // store Aqk^T as split bf16 [i'][i]: the MMAs read it as an MN-major B operand, so that it can
    // sit beside the Kd rows in one N = 192 operand; a warp's 32 lanes (32 consecutive i) fill 64
    // contiguous bytes of one row i'.
    if ((warp & 3) < 2) {
        const int ib = (warp >> 2) * 16;
        const int t = (warp & 1) * 32 + lane, col = t >> 2, p = t & 3;
        float xr[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) xr[u] = (4 * p + u == col) ? 1.f : 0.f;
#pragma unroll
        for (int i = 1; i < 16; ++i) {
            const int r = ib + i;
            const float4 a4 = *reinterpret_cast<const float4 *>(scrA + r * 64 + ((ib + 4 * p) ^ (r & 28)));
            const float av[4] = {a4.x, a4.y, a4.z, a4.w};
            float s = fmaf(av[0 ^ (i & 3)], xr[0], av[1 ^ (i & 3)] * xr[1]);
            s = fmaf(av[2 ^ (i & 3)], xr[2], s);
            s = fmaf(av[3 ^ (i & 3)], xr[3], s);
            s += __shfl_xor_sync(0xffffffffu, s, 1);
            s += __shfl_xor_sync(0xffffffffu, s, 2);
            if (i > col && p == (i >> 2)) xr[i & 3] = -s;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) scrT[sidx(ib + 4 * p + u, ib + col)] = xr[u];
    } else {
        const int colbase = (warp >> 2) * 16, i = 32 * (warp & 3) + lane - 64;
        uint32_t r0[16];
        mma_a_row16<P>(tl, col + colbase, r0);
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
    __syncthreads();
    // sum_{m<16} L[R][c0 + m] R[r0 + m][rc] with L's row read as four 16-byte slots (c0 a multiple of 16)
    auto dot16 = [&](const float *L, int R, int c0, int r0, int rc) {
        const int xh = R & 28, xl = R & 3;
        float s0 = 0.f, s1 = 0.f;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float4 a4 = *reinterpret_cast<const float4 *>(L + R * 64 + ((c0 + 4 * q) ^ xh));
            s0 = fmaf(a4.x, scrT[sidx(r0 + 4 * q + (0 ^ xl), rc)], s0);
            s1 = fmaf(a4.y, scrT[sidx(r0 + 4 * q + (1 ^ xl), rc)], s1);
            s0 = fmaf(a4.z, scrT[sidx(r0 + 4 * q + (2 ^ xl), rc)], s0);
            s1 = fmaf(a4.w, scrT[sidx(r0 + 4 * q + (3 ^ xl), rc)], s1);
        }
        return s0 + s1;
    };
    // level 1: T[b+1,b] = -T[b+1,b+1] (A[b+1,b] T[b,b]) for b = 0, 2; P parked in block (0, 2 + b/2).
    // One element per thread; the two half-warps take rows r and r + 4, so that both read the
    // right factor's rows in the same order (one row of 16 words per step).
    {
        const int w = warp, pb = w >> 3, b = 2 * pb, c = lane & 15;
        const int r = (w & 3) + 4 * ((lane >> 4) & 1) + 8 * ((w >> 2) & 1);
        const float s = dot16(scrA, (b + 1) * 16 + r, b * 16, b * 16, b * 16 + c);
        scrT[sidx(r, (2 + pb) * 16 + c)] = s;
        __syncthreads();
        const float s2 = dot16(scrT, (b + 1) * 16 + r, (b + 1) * 16, 0, (2 + pb) * 16 + c);
        scrT[sidx((b + 1) * 16 + r, b * 16 + c)] = -s2;
        __syncthreads();
    }
    // level 2: T[32:64, 0:32] = -T2 (A[32:64, 0:32] T1); P (32x32) parked in T[0:32, 32:64].
    // Warps 0-7: 64 tiles of 4 x 4 outputs, four threads per tile each summing a quarter of the 32
    // terms, so that every 16-byte load serves four products; both factors are read a slot at a
    // time (rows r0 + rr with r0 a multiple of 4, so the word order within a slot is fixed).
    {
        const int hq = tid & 3, tile = (tid >> 2) & 63, tr = tile >> 3, tc = tile & 7;
        auto block_prod = [&](const float *Lm, int lrow, int lcol, int rcol, float (&acc)[4][4]) {
#pragma unroll
            for (int rr = 0; rr < 4; ++rr)
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) acc[rr][cc] = 0.f;
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const int m0 = 8 * hq + 4 * q;               // four consecutive terms
                float av[4][4];
#pragma unroll
                for (int rr = 0; rr < 4; ++rr) {
                    const int R = lrow + 4 * tr + rr;
                    const float4 v = *reinterpret_cast<const float4 *>(Lm + R * 64 + ((lcol + m0) ^ (R & 28)));
                    av[rr][0] = v.x; av[rr][1] = v.y; av[rr][2] = v.z; av[rr][3] = v.w;
                }
#pragma unroll
                for (int mm = 0; mm < 4; ++mm) {
                    const int M = m0 + mm;
                    const float4 v = *reinterpret_cast<const float4 *>(scrT + M * 64 + ((rcol + 4 * tc) ^ (M & 28)));
                    const float bv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int rr = 0; rr < 4; ++rr)
#pragma unroll
                        for (int cc = 0; cc < 4; ++cc)
                            acc[rr][cc] = fmaf(av[rr][mm ^ rr], bv[cc ^ mm], acc[rr][cc]);
                }
            }
#pragma unroll
            for (int rr = 0; rr < 4; ++rr)
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    acc[rr][cc] += __shfl_xor_sync(0xffffffffu, acc[rr][cc], 1);
                    acc[rr][cc] += __shfl_xor_sync(0xffffffffu, acc[rr][cc], 2);
                }
        };
        // thread hq of a tile writes row hq of it (negated if neg) at rows orow.., columns ocol..
        auto put_row = [&](const float (&acc)[4][4], int orow, int ocol, float sgn) {
#pragma unroll
            for (int rr = 0; rr < 4; ++rr)
                if (rr == hq) {
                    const int R = orow + 4 * tr + rr;
                    *reinterpret_cast<float4 *>(scrT + R * 64 + ((ocol + 4 * tc) ^ (R & 28))) =
                        make_float4(sgn * acc[rr][0 ^ rr], sgn * acc[rr][1 ^ rr], sgn * acc[rr][2 ^ rr], sgn * acc[rr][3 ^ rr]);
                }
        };
        float acc[4][4];
        if (warp < 8) {
            block_prod(scrA, 32, 0, 0, acc);
            put_row(acc, 0, 32, 1.f);                    // the park area is read by nobody in this pass
        }
        __syncthreads();
        if (warp < 8) {
            block_prod(scrT, 32, 32, 32, acc);
            put_row(acc, 32, 0, -1.f);                   // T21: not read by this pass
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
