// prefill_split.cu -- two-pass chunked KDA prefill on the tensor cores (bf16
// inputs, dk = dv = 128, chunk 64, conv / L2 norm / gate fused), for the case
// where a few long sequences leave most SMs idle under one CTA per
// (sequence, head).
//
// The WY/UT chunk form ("recurrent KDA state", HF discussion #187 feature
// list; KdaState in the metrale kimi_k3 docs) splits every chunk into a part
// that needs only the chunk's own inputs and a short part that needs the state
// carried in from the previous chunk:
//
//   pass 1, chunk prep (one work item per (chunk, head), all SMs, persistent):
//       conv, norm, decay -> Kh, Qh, Kb, v;  Akk, Aqk;  Tb = (I + Akk)^-1 diag(beta)
//       W = Tb Kh,  U = Tb v                                   -> one record per item
//   pass 2, chunk scan (one CTA per (sequence, head), chunks in order):
//       S' = diag(exp(r)) S;  V' = U - W S';  O = scale (Qh S' + Aqk V') [* sigmoid(gate)]
//       S_next = diag(exp(G_last - r)) (S' + Kb^T V')
//
// The record of an item (148,480 bytes, in the caller's workspace) holds the
// split-bf16 tiles [W; Qh], Kb and Aqk in the exact 128B-swizzled shared-memory
// layout in which the scan kernel's MMAs read them, U^T in fp32 and the
// per-channel r and G_last, so the scan kernel fetches it with three plain bulk
// copies that overlap its own MMAs.  The scan keeps the fp32 state in TMEM for
// the whole sequence, like the single-pass kernel; per chunk it runs two MMA
// chains (N = 128 against [W; Qh], then O += V'^T Aqk^T and S += V'^T Kb).
#include <cuda.h>

#include "tc_chunk.cuh"

namespace k3kda {
namespace {

using namespace tc;
using namespace tcc;

// ---- one chunk record (byte offsets; identical to the scan kernel's smem layout) ----
constexpr uint32_t REC_X = 0;            // [W rows 0-63; Qh rows 64-127] x 128 K, split: hi 32 KB, lo 32 KB
constexpr uint32_t REC_KB = 65536;       // Kb rows [64][128 K], split: hi 16 KB, lo 16 KB
constexpr uint32_t REC_AQK = 98304;      // Aqk [64][64 K], split: hi 8 KB, lo 8 KB
constexpr uint32_t REC_U = 114688;       // U^T fp32 [128 dv][64 tok]; 16-byte units XOR-swizzled by (dv & 15)
constexpr uint32_t REC_VEC = 147456;     // r[128], G_last[128] fp32
constexpr uint32_t REC_BYTES = 148480;
static_assert(OFF_XL == OFF_X + 32768, "the [Kh; Qh] tile pair must be contiguous (one bulk store)");
static_assert(OFF_KB_LO == OFF_KB_HI + 16384 && OFF_AQK_HI == OFF_KB_HI + 32768 && OFF_AQK_LO == OFF_AQK_HI + 8192,
              "Kb and Aqk tiles must be contiguous in the prep kernel's layout (one bulk store)");
static_assert(OFF_GL == OFF_REF + 512, "r and G_last must be adjacent (one bulk store)");

// byte offset of U^T element (dv j, token i) inside the U block
__device__ __forceinline__ uint32_t u_off(uint32_t j, uint32_t i) {
    return j * 256u + ((((i >> 2) ^ (j & 15u)) << 4) | ((i & 3u) << 2));
}

// ============================ chunk offsets ============================
// off[n] = number of 64-token chunks in sequences 0 .. n-1 (off[0] = 0, off[N] = total), capped
// at qmax, the number of records the workspace holds: a malformed device cu_seqlens (overlapping
// sequences) then loses chunks instead of sending either pass past the workspace.
__global__ void __launch_bounds__(1024) kda_chunk_offsets_kernel(const int32_t *cu, int N, int T, int qmax,
                                                                 int32_t *off) {
    __shared__ int32_t part[32];
    __shared__ int32_t carry;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) { carry = 0; off[0] = 0; }
    __syncthreads();
    for (int base = 0; base < N; base += 1024) {
        const int n = base + tid;
        int x = 0;
        if (n < N) {
            int tb, te;
            seq_bounds(cu, n, T, tb, te);
            x = (te - tb + kC - 1) / kC;
        }
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, d);
            if (lane >= d) x += y;
        }
        if (lane == 31) part[warp] = x;
        __syncthreads();
        if (warp == 0) {
            int w = part[lane];
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, w, d);
                if (lane >= d) w += y;
            }
            part[lane] = w;
        }
        __syncthreads();
        const int incl = carry + x + (warp > 0 ? part[warp - 1] : 0);
        if (n < N) off[n + 1] = min(incl, qmax);
        __syncthreads();
        if (tid == 1023) carry = incl;
        __syncthreads();
    }
}

// ============================ pass 1: chunk prep ============================
struct PrepArgs {
    CUtensorMap tm_q, tm_k, tm_v, tm_g;   // [T, H, 128] (bf16 q, k, v; fp32 g), box min(64, T) tokens of one head
    PrefillArgs p;
    const float *conv_w;      // [3*H*128, W] or null
    const float *conv_state;  // [N, W-1, 3*H*128] initial conv state or null (read only here)
    int W;
    int box_rows;
    const int32_t *chunk_off; // [N + 1]
    uint8_t *rec;             // [total chunks * H] records
};

constexpr uint32_t kPrepTmemCols = 256;
constexpr uint32_t kColWp = 64, kColUp = 128;    // W^T and U^T results ([0, 64): Akk | Aqk)

__global__ void __launch_bounds__(kThreads, 1) kda_chunk_prep_kernel(const __grid_constant__ PrepArgs A) {
    extern __shared__ uint8_t smraw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
    const PrefillArgs &a = A.p;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = a.H, N = a.N;
    const uint32_t sbase = smem_u32(sm);
    float *sConvW = reinterpret_cast<float *>(sm + OFF_CONVW);
    float *sHist = reinterpret_cast<float *>(sm + OFF_HIST);
    uint64_t *mbar = reinterpret_cast<uint64_t *>(sm + OFF_MISC);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + OFF_MISC + 24);
    volatile uint32_t *sflag = reinterpret_cast<volatile uint32_t *>(sm + OFF_MISC + 28);
    const uint32_t mbar_a = smem_u32(mbar);          // MMA completion
    const uint32_t mbar_s = smem_u32(mbar + 1);      // staged input rows landed
    const int W = A.conv_w ? A.W : 0;
    const int Dall = 3 * H * kD;

    if (warp == 0) { tmem_alloc(smem_u32(tslot), kPrepTmemCols); tmem_relinquish(); }
    if (tid == 0) { mbar_init(mbar_a, 1); mbar_init(mbar_s, 1); fence_mbar_init(); *sflag = 0; }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tslot;
    const uint32_t lrow = 32u * (warp & 3);
    const uint32_t tl = tbase + (lrow << 16);
    const int quarter = warp >> 2;
    const int total = A.chunk_off[N] * H;
    const uint32_t kStageBytes = (uint32_t)A.box_rows * (kD * 4 + 3 * kD * 2);

    // thread 0's view of the outstanding asynchronous operations
    uint32_t aph = 0, sph = 0;
    bool pend_a = false, pend_s = false;
    auto wait_on = [&](uint32_t bar, uint32_t &ph, bool &pend) {
        if (!pend) return;
        if (!mbar_wait_bounded(bar, ph, kWaitLimit)) {
            *sflag = 1;
            atomicOr(a.status, 1u);
            return;
        }
        ph ^= 1u;
        pend = false;
    };
    auto mma_wait = [&]() -> bool {
        if (tid == 0 && !*sflag) wait_on(mbar_a, aph, pend_a);
        __syncthreads();
        const bool bad = *sflag != 0;
        tc_fence_after();
        return !bad;
    };

    int cur_h = -1;
    for (int it = blockIdx.x; it < total; it += gridDim.x) {
        const int qc = it / H, h = it - qc * H;
        int lo = 0, hi = N;                              // sequence n with off[n] <= qc < off[n + 1]
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (A.chunk_off[mid] <= qc) lo = mid; else hi = mid;
        }
        const int n = lo;
        int tb, te;
        seq_bounds(a.cu, n, a.T, tb, te);
        const int cs = tb + (qc - A.chunk_off[n]) * kC;
        const int Lc = min(kC, te - cs);

        // stage this chunk's rows once the previous record has been read out of shared memory
        if (tid == 0) {
            bulk_wait_read_all();
            mbar_arrive_expect_tx(mbar_s, kStageBytes);
            tma_load_3d(sbase + OFF_GST, &A.tm_g, 0, h, cs, mbar_s);
            tma_load_3d(sbase + OFF_VST, &A.tm_v, 0, h, cs, mbar_s);
            tma_load_3d(sbase + OFF_QST, &A.tm_q, 0, h, cs, mbar_s);
            tma_load_3d(sbase + OFF_KST, &A.tm_k, 0, h, cs, mbar_s);
            pend_s = true;
        }
        if (W > 0) {
            if (h != cur_h) {
                for (int e = tid; e < 384 * 4; e += kThreads) {
                    // tap-major, taps right-aligned in a 4-wide window: tap t multiplies token i - 3 + t
                    const int t = e / 384, ch = e - t * 384;
                    const int gch = (ch >> 7) * H * kD + h * kD + (ch & 127);
                    sConvW[e] = t >= 4 - W ? A.conv_w[(size_t)gch * W + (t - (4 - W))] : 0.f;
                }
                cur_h = h;
            }
            // conv history: pre-conv q, k, v rows of tokens cs-3 .. cs-1 of this sequence, from the
            // inputs, or from the initial conv state (right-aligned) before the sequence start
            for (int e = tid; e < 3 * 3 * 128; e += kThreads) {
                const int which = e / 384, r = (e / 128) % 3, c = e & 127;
                const int t = cs - 3 + r;
                float x = 0.f;
                if (t >= tb) {
                    const void *src = which == 0 ? a.q : (which == 1 ? a.k : a.v);
                    x = __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(src)[((size_t)t * H + h) * kD + c]);
                } else {
                    const int row = W - 1 + (t - tb);
                    if (W > 1 && A.conv_state != nullptr && row >= 0)
                        x = A.conv_state[((size_t)n * (W - 1) + row) * Dall + which * H * kD + h * kD + c];
                }
                sHist[e] = x;
            }
        }
        if (tid == 0) wait_on(mbar_s, sph, pend_s);
        __syncthreads();
        if (*sflag) break;

        prep_chunk(sm, a, cs, Lc, h, W, nullptr, nullptr);
        if (tid == 0) { issue_mma_a(sbase, tbase + kColA, mbar_a); pend_a = true; }
        if (!mma_wait()) break;
        extract_a(sm, tl, kColA);
        solve_tb(sm);

        // ---- MMA: U^T = v^T Tb^T and W^T = Kh^T Tb^T (Kh rows 0-63 of X read MN-major) ----
        if (tid == 0) {
            tc_fence_after();
            const uint32_t id = idesc_bf16_f32(128, 64, false, /*a_mn=*/true);
            const uint64_t dVh = sdesc_mnmajor_sw128(sbase + OFF_V_HI, 8192), dVl = sdesc_mnmajor_sw128(sbase + OFF_V_LO, 8192);
            const uint64_t dKh = sdesc_mnmajor_sw128(sbase + OFF_X, 16384), dKl = sdesc_mnmajor_sw128(sbase + OFF_XL, 16384);
            const uint64_t dTh = sdesc_kmajor_sw128(sbase + OFF_TB_HI), dTl = sdesc_kmajor_sw128(sbase + OFF_TB_LO);
            const int nsplit = W > 0 ? 3 : 2;           // v is exact bf16 without a conv
#pragma unroll
            for (int sp = 0; sp < 3; ++sp)
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    if (sp < nsplit)
                        mma_bf16(tbase + kColUp, dadd(sp == 2 ? dVl : dVh, kk * 2048), dadd(sp == 1 ? dTl : dTh, kk * 32),
                                 id, (sp | kk) != 0);
#pragma unroll
            for (int sp = 0; sp < 3; ++sp)
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16(tbase + kColWp, dadd(sp == 2 ? dKl : dKh, kk * 2048), dadd(sp == 1 ? dTl : dTh, kk * 32),
                             id, (sp | kk) != 0);
            mma_commit(mbar_a);
            pend_a = true;
        }
        if (!mma_wait()) break;

        // ---- U^T -> fp32 block (region A: the v rows are dead), W -> X/XL rows 0-63 ----
        {
            const int j = lrow + lane;                  // dv channel for U^T, dk channel for W^T
            uint32_t r[16];
            tmem_ld16(tl + kColUp + quarter * 16, r);
            tmem_wait_ld();
#pragma unroll
            for (int t = 0; t < 4; ++t)
                *reinterpret_cast<uint4 *>(sm + OFF_GST + u_off(j, quarter * 16 + 4 * t)) =
                    make_uint4(r[4 * t], r[4 * t + 1], r[4 * t + 2], r[4 * t + 3]);
            tmem_ld16(tl + kColWp + quarter * 16, r);
            tmem_wait_ld();
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                float hv, lv;
                split_bf16(__uint_as_float(r[u]), hv, lv);
                const uint32_t o = kmaj128(128, quarter * 16 + u, j);
                *reinterpret_cast<__nv_bfloat16 *>(sm + OFF_X + o) = __float2bfloat16_rn(hv);
                *reinterpret_cast<__nv_bfloat16 *>(sm + OFF_XL + o) = __float2bfloat16_rn(lv);
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            uint8_t *rec = A.rec + (size_t)it * REC_BYTES;
            bulk_s2g(rec + REC_X, sbase + OFF_X, 65536);
            bulk_s2g(rec + REC_KB, sbase + OFF_KB_HI, 49152);   // Kb hi, Kb lo, Aqk hi, Aqk lo
            bulk_s2g(rec + REC_U, sbase + OFF_GST, 32768);
            bulk_s2g(rec + REC_VEC, sbase + OFF_REF, 1024);     // r, G_last
            bulk_commit();
        }
        tc_fence_after();
    }
    if (tid == 0) {
        bulk_wait_all();
        // after a timed-out wait, let what is still in flight land before the CTA exits
        if (pend_a) mbar_wait_bounded(mbar_a, aph, kWaitLimit);
        if (pend_s) mbar_wait_bounded(mbar_s, sph, kWaitLimit);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tbase, kPrepTmemCols);
}

// ============================ pass 2: chunk scan ============================
struct ScanArgs {
    CUtensorMap tm_gate;      // [T, H, 128] bf16 gate logits (when gated)
    PrefillArgs p;
    float *conv_state;        // [N, W-1, 3*H*128] advanced at the end, or null
    int W;
    int box_rows;
    const int32_t *chunk_off;
    const uint8_t *rec;
};

// scan kernel shared memory: the record image [0, REC_BYTES), then
constexpr uint32_t Q_ST_HI = REC_BYTES;             // S'^T [128 rows j][128 K c] hi   (S' .. MMA W/O)
constexpr uint32_t Q_ST_LO = Q_ST_HI + 32768;       //                           lo
constexpr uint32_t Q_VPT_HI = Q_ST_HI;              // V'^T [128 rows j][64 K i] hi   (V' .. MMA O/S)
constexpr uint32_t Q_VPT_LO = Q_ST_HI + 16384;      //                           lo
constexpr uint32_t Q_GATE = Q_ST_LO;                // gate logits bf16 [64 tok][128] (MMA W/O .. epilogue)
constexpr uint32_t Q_LOGF = Q_ST_LO + 32768;        // log of the basis factor carried in TMEM
constexpr uint32_t Q_FCOL = Q_LOGF + 512;           // state column factor of this chunk
constexpr uint32_t Q_MISC = Q_FCOL + 512;           // 5 mbarriers, tmem slot, flag
constexpr uint32_t kScanSmemBytes = Q_MISC + 64 + 1024;
static_assert(Q_ST_HI % 1024 == 0 && Q_ST_LO % 1024 == 0 && Q_VPT_LO % 1024 == 0, "tile alignment");
static_assert(kScanSmemBytes <= 232448, "scan kernel shared memory exceeds the per-CTA limit");

constexpr uint32_t kScanTmemCols = 256;
constexpr uint32_t kColD = 0;      // [0, 64): (W S')^T, then [64, 128): O^T
constexpr uint32_t kColSs = 128;   // S'^T, 128 columns

__global__ void __launch_bounds__(kThreads, 1) kda_chunk_scan_kernel(const __grid_constant__ ScanArgs A) {
    extern __shared__ uint8_t smraw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
    const PrefillArgs &a = A.p;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nh = blockIdx.x, n = nh / a.H, h = nh % a.H;
    const int H = a.H;
    const uint32_t sbase = smem_u32(sm);
    float *sLogf = reinterpret_cast<float *>(sm + Q_LOGF);
    float *sFcol = reinterpret_cast<float *>(sm + Q_FCOL);
    const float *sVec = reinterpret_cast<const float *>(sm + REC_VEC);
    uint64_t *mbar = reinterpret_cast<uint64_t *>(sm + Q_MISC);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + Q_MISC + 40);
    volatile uint32_t *sflag = reinterpret_cast<volatile uint32_t *>(sm + Q_MISC + 44);
    const uint32_t mb_a = smem_u32(mbar), mb_x = smem_u32(mbar + 1), mb_k = smem_u32(mbar + 2),
                   mb_u = smem_u32(mbar + 3), mb_g = smem_u32(mbar + 4);

    int tb, te;
    seq_bounds(a.cu, n, a.T, tb, te);
    const int q0 = A.chunk_off[n];
    const int nq = A.chunk_off[n + 1] - q0;
    const int W = A.W;
    const int Dall = 3 * H * kD;

    if (warp == 0) { tmem_alloc(smem_u32(tslot), kScanTmemCols); tmem_relinquish(); }
    if (tid == 0) {
        mbar_init(mb_a, 1); mbar_init(mb_x, 1); mbar_init(mb_k, 1); mbar_init(mb_u, 1); mbar_init(mb_g, 1);
        fence_mbar_init();
        *sflag = 0;
    }
    if (tid < kD) sLogf[tid] = 0.f;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tslot;
    const uint32_t lrow = 32u * (warp & 3);
    const uint32_t tl = tbase + (lrow << 16);
    const int quarter = warp >> 2;
    {   // S'^T <- S0^T (true state; basis factor 1)
        const int j = lrow + lane;
        for (int cb = 0; cb < 32; cb += 16) {
            uint32_t r[16];
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                const int c = quarter * 32 + cb + u;
                r[u] = __float_as_uint(a.S0 ? a.S0[((size_t)nh * kD + c) * kD + j] : 0.f);
            }
            tmem_st16(tl + kColSs + quarter * 32 + cb, r);
        }
        tmem_wait_st();
    }

    auto rec_of = [&](int c) { return A.rec + ((size_t)(q0 + c) * H + h) * REC_BYTES; };
    // thread 0's view of the outstanding asynchronous operations
    uint32_t aph = 0, xph = 0, kph = 0, uph = 0, gph = 0;
    bool pend_a = false, pend_x = false, pend_k = false, pend_u = false, pend_g = false;
    auto wait_on = [&](uint32_t bar, uint32_t &ph, bool &pend) -> bool {
        if (!pend) return true;
        if (!mbar_wait_bounded(bar, ph, kWaitLimit)) {
            *sflag = 1;
            atomicOr(a.status, 1u);
            return false;
        }
        ph ^= 1u;
        pend = false;
        return true;
    };
    auto load = [&](uint32_t bar, uint32_t off, int c, uint32_t bytes, bool &pend) {
        mbar_arrive_expect_tx(bar, bytes);
        bulk_g2s(sbase + off, rec_of(c) + off, bytes, bar);
        pend = true;
    };
    auto mma_wait = [&]() -> bool {
        if (tid == 0 && !*sflag) wait_on(mb_a, aph, pend_a);
        __syncthreads();
        const bool bad = *sflag != 0;
        tc_fence_after();
        return !bad;
    };
    if (tid == 0 && nq > 0) {
        load(mb_x, REC_X, 0, 65536, pend_x);
        load(mb_k, REC_KB, 0, 49152, pend_k);
        load(mb_u, REC_U, 0, 33792, pend_u);             // U^T, r, G_last
    }

    bool failed = false;
    for (int c = 0; c < nq; ++c) {
        const int cs = tb + c * kC;
        const int Lc = min(kC, te - cs);
        const bool more = c + 1 < nq;
        // ---- basis change: fcol = exp(logf_prev + r), logf = G_last - r ----
        if (tid == 0) wait_on(mb_u, uph, pend_u);
        __syncthreads();
        if (*sflag) { failed = true; break; }
        if (tid < kD) {
            const float r = sVec[tid];
            sFcol[tid] = expf(sLogf[tid] + r);
            sLogf[tid] = sVec[kD + tid] - r;
        }
        __syncthreads();
        // ---- S'^T = S^T diag(fcol) -> TMEM and split A tile ----
        {
            const int j = lrow + lane;
            for (int cb = 0; cb < 32; cb += 16) {
                const int col = quarter * 32 + cb;
                uint32_t r[16];
                tmem_ld16(tl + kColSs + col, r);
                tmem_wait_ld();
                float v[16];
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    v[u] = __uint_as_float(r[u]) * sFcol[col + u];
                    r[u] = __float_as_uint(v[u]);
                }
                tmem_st16(tl + kColSs + col, r);
                tile64_put16(sm, Q_ST_HI + (col >> 6) * 16384, Q_ST_LO + (col >> 6) * 16384, j, col & 63, v);
            }
            tmem_wait_st();
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        // ---- MMA: D^T = S'^T [W; Qh]^T  ((W S')^T in columns 0-63, (Qh S')^T in 64-127) ----
        if (tid == 0 && wait_on(mb_x, xph, pend_x)) {
            tc_fence_after();
            const uint32_t id = idesc_bf16_f32(128, 128);
            const uint64_t dSh = sdesc_kmajor_sw128(sbase + Q_ST_HI), dSl = sdesc_kmajor_sw128(sbase + Q_ST_LO);
            const uint64_t dX = sdesc_kmajor_sw128(sbase + REC_X), dXL = sdesc_kmajor_sw128(sbase + REC_X + 32768);
#pragma unroll
            for (int sp = 0; sp < 3; ++sp)
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_bf16(tbase + kColD, dadd(sp == 2 ? dSl : dSh, (kk >> 2) * 16384 + (kk & 3) * 32),
                             dadd(sp == 1 ? dXL : dX, (kk >> 2) * 16384 + (kk & 3) * 32), id, (sp | kk) != 0);
            mma_commit(mb_a);
            pend_a = true;
        }
        if (!mma_wait()) { failed = true; break; }
        if (tid == 0) {
            if (more) load(mb_x, REC_X, c + 1, 65536, pend_x);    // [W; Qh] of the next chunk
            if (a.gate) {                                          // this chunk's gate rows (S' tile is dead)
                mbar_arrive_expect_tx(mb_g, (uint32_t)A.box_rows * kD * 2);
                tma_load_3d(sbase + Q_GATE, &A.tm_gate, 0, h, cs, mb_g);
                pend_g = true;
            }
        }
        // ---- V'^T = U^T - (W S')^T -> split tile ----
        {
            const int j = lrow + lane;
            uint32_t r[16];
            tmem_ld16(tl + kColD + quarter * 16, r);
            tmem_wait_ld();
            float v[16];
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const float4 u4 = *reinterpret_cast<const float4 *>(sm + REC_U + u_off(j, quarter * 16 + 4 * t));
                v[4 * t + 0] = u4.x - __uint_as_float(r[4 * t + 0]);
                v[4 * t + 1] = u4.y - __uint_as_float(r[4 * t + 1]);
                v[4 * t + 2] = u4.z - __uint_as_float(r[4 * t + 2]);
                v[4 * t + 3] = u4.w - __uint_as_float(r[4 * t + 3]);
            }
            tile64_put16(sm, Q_VPT_HI, Q_VPT_LO, j, quarter * 16, v);
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        // ---- MMA: O^T += V'^T Aqk^T,  S'^T += V'^T Kb ----
        if (tid == 0) {
            if (more) load(mb_u, REC_U, c + 1, 33792, pend_u);    // U^T, r, G_last of the next chunk
            if (wait_on(mb_k, kph, pend_k)) {
                tc_fence_after();
                const uint32_t id64 = idesc_bf16_f32(128, 64);
                const uint32_t id128 = idesc_bf16_f32(128, 128, false, false, /*b_mn=*/true);
                const uint64_t dVh = sdesc_kmajor_sw128(sbase + Q_VPT_HI), dVl = sdesc_kmajor_sw128(sbase + Q_VPT_LO);
                const uint64_t dAh = sdesc_kmajor_sw128(sbase + REC_AQK), dAl = sdesc_kmajor_sw128(sbase + REC_AQK + 8192);
                const uint64_t dKh = sdesc_mnmajor_sw128(sbase + REC_KB, 8192),
                               dKl = sdesc_mnmajor_sw128(sbase + REC_KB + 16384, 8192);
#pragma unroll
                for (int sp = 0; sp < 3; ++sp)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_bf16(tbase + kColD + 64, dadd(sp == 2 ? dVl : dVh, kk * 32), dadd(sp == 1 ? dAl : dAh, kk * 32),
                                 id64, 1);
#pragma unroll
                for (int sp = 0; sp < 3; ++sp)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_bf16(tbase + kColSs, dadd(sp == 2 ? dVl : dVh, kk * 32), dadd(sp == 1 ? dKl : dKh, kk * 2048),
                                 id128, 1);
                mma_commit(mb_a);
                pend_a = true;
            }
            if (!*sflag) wait_on(mb_g, gph, pend_g);
        }
        if (!mma_wait()) { failed = true; break; }       // its barrier also publishes the gate rows
        if (tid == 0 && more) load(mb_k, REC_KB, c + 1, 49152, pend_k);   // Kb, Aqk of the next chunk
        // ---- epilogue: O^T -> scale, gate -> out ----
        {
            const int j = lrow + lane;
            uint32_t r0[16];
            tmem_ld16(tl + kColD + 64 + quarter * 16, r0);
            tmem_wait_ld();
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                const int i = quarter * 16 + u;
                if (i < Lc) {
                    float o = a.scale * __uint_as_float(r0[u]);
                    if (a.gate)
                        o *= sigmoid_fast(__bfloat162float(
                            *reinterpret_cast<const __nv_bfloat16 *>(sm + Q_GATE + i * (kD * 2) + j * 2)));
                    store_elt(a.out, ((size_t)(cs + i) * H + h) * kD + j, o, a.out_bf16);
                }
            }
        }
        tc_fence_before();
    }
    if (!failed) {
        // ---- final state: S = S'^T diag(exp(logf)) ----
        if (a.Sfin) {
            const int j = lrow + lane;
            for (int cb = 0; cb < 32; cb += 16) {
                uint32_t r[16];
                tmem_ld16(tl + kColSs + quarter * 32 + cb, r);
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
    }
    if (tid == 0) {
        // after a failure, let what is still in flight land before the CTA exits
        if (pend_a) mbar_wait_bounded(mb_a, aph, kWaitLimit);
        if (pend_x) mbar_wait_bounded(mb_x, xph, kWaitLimit);
        if (pend_k) mbar_wait_bounded(mb_k, kph, kWaitLimit);
        if (pend_u) mbar_wait_bounded(mb_u, uph, kWaitLimit);
        if (pend_g) mbar_wait_bounded(mb_g, gph, kWaitLimit);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tbase, kScanTmemCols);
}

size_t max_chunks(int N, int T) { return ((size_t)T + 63u * (size_t)N) / kC; }
size_t round256_(size_t b) { return (b + 255) & ~size_t(255); }

}  // namespace

// Workspace of the two-pass path (after the status word): chunk offsets, then the records.
size_t tc_split_workspace(int N, int T, int H) {
    return round256_((size_t)(N + 1) * sizeof(int32_t)) + max_chunks(N, T) * (size_t)H * REC_BYTES;
}

cudaError_t launch_prefill_tc_split(const PrefillArgs &p, const float *conv_w, float *conv_state, int W,
                                    void *ws, cudaStream_t s) {
    if ((long long)p.N * p.H == 0) return cudaSuccess;
    int32_t *chunk_off = static_cast<int32_t *>(ws);
    uint8_t *rec = static_cast<uint8_t *>(ws) + round256_((size_t)(p.N + 1) * sizeof(int32_t));
    const int box_rows = p.T < kC ? p.T : kC;
    cudaError_t e;
    static bool attr_done = false;
    if (!attr_done) {
        if ((e = cudaFuncSetAttribute(kda_chunk_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)kSmemBytes)) != cudaSuccess ||
            (e = cudaFuncSetAttribute(kda_chunk_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)kScanSmemBytes)) != cudaSuccess)
            return e;
        attr_done = true;
    }
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return e;

    kda_chunk_offsets_kernel<<<1, 1024, 0, s>>>(p.cu, p.N, p.T, (int)max_chunks(p.N, p.T), chunk_off);
    count_launch();
    if ((e = cudaGetLastError()) != cudaSuccess) return e;

    const size_t items = max_chunks(p.N, p.T) * (size_t)p.H;
    if (items > 0) {
        PrepArgs P{};
        if ((e = make_row_map(&P.tm_q, p.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.T, p.H)) != cudaSuccess ||
            (e = make_row_map(&P.tm_k, p.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.T, p.H)) != cudaSuccess ||
            (e = make_row_map(&P.tm_v, p.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.T, p.H)) != cudaSuccess ||
            (e = make_row_map(&P.tm_g, p.g, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, p.T, p.H)) != cudaSuccess)
            return e;
        P.p = p;
        P.conv_w = conv_w;
        P.conv_state = conv_state;
        P.W = conv_w ? W : 0;
        P.box_rows = box_rows;
        P.chunk_off = chunk_off;
        P.rec = rec;
        const unsigned grid = (unsigned)(items < (size_t)sms ? items : (size_t)sms);
        kda_chunk_prep_kernel<<<grid, kThreads, kSmemBytes, s>>>(P);
        count_launch();
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }

    ScanArgs S{};
    if (p.gate && p.T > 0 &&
        (e = make_row_map(&S.tm_gate, p.gate, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.T, p.H)) != cudaSuccess)
        return e;
    S.p = p;
    S.conv_state = conv_w ? conv_state : nullptr;
    S.W = conv_w ? W : 0;
    S.box_rows = box_rows;
    S.chunk_off = chunk_off;
    S.rec = rec;
    kda_chunk_scan_kernel<<<(unsigned)(p.N * p.H), kThreads, kScanSmemBytes, s>>>(S);
    count_launch();
    return cudaGetLastError();
}

}  // namespace k3kda
