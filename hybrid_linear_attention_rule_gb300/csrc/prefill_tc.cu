// prefill_tc.cu -- chunked KDA prefill on the 5th-generation tensor cores
// (tcgen05 MMA, TMEM accumulators), bf16 inputs, dk = dv = 128, chunk 64, with
// the q/k/v short conv (+SiLU), q/k L2 norm and sigmoid output gate fused.
//
// The recurrence ("recurrent KDA state", HF discussion #187 feature list; FP32
// KdaState, metrale kimi_k3 docs) in its chunked (WY/UT) form.  For a chunk of
// 64 tokens with chunk-local cumulative log-decay G (per channel) and a
// per-channel reference rho (the mid-point of G, or G_first for a channel that
// decays by more than kStrongDecay nats within the chunk):
//   Kh = k E, Qh = q E, Kb = k / E, Kd = k exp(G_last - G),   E = exp(G - rho)
//   Akk = diag(beta) tril(Kh Kb^T, -1),  Aqk = tril(Qh Kb^T)
//       (a strong channel's share of both is formed exactly in tc_chunk.cuh)
//   T  = (I + Akk)^-1,  Tb = T diag(beta)
//   S' = diag(exp(rho)) S
//   U  = Tb v,  Y = Kh S',  V' = U - Tb Y
//   O  = scale (Qh S' + Aqk V')  [* sigmoid(gate)]
//   S_next = diag(exp(G_last)) S + Kd^T V'
// (V' = U - W S with W = Tb Kh written as U - Tb (Kh S') so that no transposed
// copy of Kh or W is ever materialised.)  Every factor applied to the state is
// at most 1 and every E, 1/E stays within exp(+-kStrongDecay / 2), so nothing
// overflows whatever the decay.
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
// [64,128) Y^T, [128,192) U^T then V'^T, [192,320) S^T (the state).
#include <cuda.h>
#include <cudaTypedefs.h>

#include "tc_chunk.cuh"

namespace k3kda {
namespace {

using namespace tc;
using namespace tcc;



struct TcArgs {
    CUtensorMap tm_q, tm_k, tm_v, tm_g;   // [T, H, 128] bf16 (q, k, v) and fp32 (g); box 64 tokens x 1 head x 128
    CUtensorMap tm_gate;                  // [T, H, 128] bf16 gate logits (when gated)
    PrefillArgs p;
    const float *conv_w;     // [2*H*128 + H*128, W] or null
    float *conv_state;       // [N, W-1, 3*H*128] or null
    int W;
    int box_rows;            // tokens per staged tile: min(64, T)
};

__global__ void __launch_bounds__(kThreads, 1) kda_prefill_tc_kernel(const __grid_constant__ TcArgs A) {
    extern __shared__ uint8_t smraw[];
    uint8_t *sm = smem_align1024(smraw);
    const PrefillArgs &a = A.p;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nh = blockIdx.x, n = nh / a.H, h = nh % a.H;
    const int sn = seq_slot(a.slot, a.num_slots, n);           // state / conv-state row (-1: none)
    const size_t snh = (size_t)(sn < 0 ? 0 : sn) * a.H + h;
    const int H = a.H;
    const uint32_t sbase = smem_u32(sm);
    float *sRef = reinterpret_cast<float *>(sm + OFF_REF);
    float *sGL = reinterpret_cast<float *>(sm + OFF_GL);
    float *sFA = reinterpret_cast<float *>(sm + OFF_FCOL);     // exp(rho) of the current chunk
    float *sFS = reinterpret_cast<float *>(sm + OFF_LOGF);     // exp(G_last) of the current chunk
    float *sConvW = reinterpret_cast<float *>(sm + OFF_CONVW);
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
        if (W > 1 && A.conv_state != nullptr && row >= 0 && sn >= 0)
            x = A.conv_state[((size_t)sn * (W - 1) + row) * Dall + which * H * kD + h * kD + c];
        sHist[e] = x;
    }
    if (W > 0)
        for (int e = tid; e < 384 * 4; e += kThreads) {
            // tap-major, taps right-aligned in a 4-wide window: tap t multiplies token i - 3 + t
            const int t = e / 384, ch = e - t * 384;
            const int gch = (ch >> 7) * H * kD + h * kD + (ch & 127);
            sConvW[e] = t >= 4 - W ? A.conv_w[(size_t)gch * W + (t - (4 - W))] : 0.f;
        }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tslot;
    const uint32_t lrow = 32u * (warp & 3);             // first TMEM lane of this warp
    const uint32_t tl = tbase + (lrow << 16);
    const int quarter = warp >> 2;                       // which column quarter this warp handles
    {   // S^T <- S0^T
        const int j = lrow + lane;
        for (int cb = 0; cb < 32; cb += 16) {
            uint32_t r[16];
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                const int c = quarter * 32 + cb + u;
                r[u] = __float_as_uint((a.S0 && sn >= 0) ? a.S0[(snh * kD + c) * kD + j] : 0.f);
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
    // test hook: CTA 0 stages nothing and gives up its first wait early (nothing is then in flight)
    const bool tskip = a.test_limit != 0 && blockIdx.x == 0;
    if (tb < te && !tskip) { stage_gv(tb); stage_qk(tb); }

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
        // ================= prep: conv, norm, decay, operands (staged rows -> tiles) =================
        if (tid == 0 && !mbar_wait_bounded(mbar_s, sphase, tskip && cs == tb ? a.test_limit : kWaitLimit)) {
            *sflag = 1;
            atomicOr(a.status, 1u);
        }
        sphase ^= 1u;
        __syncthreads();
        if (*sflag) { failed = true; break; }
        float kd[kTok][4];
        const bool strong = prep_qk<PlanFused>(sm, a, cs, Lc, h, W, tl, kColA, kd);
        if (tid < kD) {
            sFA[tid] = expf(sRef[tid]);
            sFS[tid] = expf(sGL[tid]);
        }
        prep_v<PlanFused>(sm, a, Lc, W);
        PHASE(0);
        // pre-conv rows 61..63 of this chunk are the conv history of the next one
        if (W > 0 && cs + kC < te)
            for (int e = tid; e < 3 * 3 * 128; e += kThreads) {
                const int which = e / 384, r = (e / 128) % 3, c = e & 127;
                const uint32_t st = which == 0 ? OFF_QST : (which == 1 ? OFF_KST : OFF_VST);
                sHist[e] = __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(sm + st + (kC - 3 + r) * (kD * 2) + c * 2));
            }
        // ================= MMA: [Kh; Qh] Kb^T  -> Akk | Aqk =================
        if (tid == 0) issue_mma_a<PlanFused>(sbase, tbase + kColA, mbar_a, strong);
        if (!mma_wait()) { failed = true; break; }
        // MMA A has read Kb: the Kb region takes Kd (stacked hi / lo tiles), the B operand of MMA S
        put_kd(sm + OFF_KB_HI, kd);
        fence_async_smem();
        PHASE(1);
        extract_akk<PlanFused>(sm, tl, kColA);
        PHASE(2);
        solve_tb<PlanFused>(sm, tl, kColA);
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
        // ================= state pass: S'^T = S^T diag(exp(rho)) -> split A tile;
        //                   S^T <- S^T diag(exp(G_last)) in TMEM (MMA S adds V'^T Kd) =================
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
                    const float x = __uint_as_float(r[u]);
                    v[u] = x * sFA[col + u];
                    r[u] = __float_as_uint(x * sFS[col + u]);
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
        // ================= V'^T -> split tile;  MMA: O^T += V'^T Aqk^T,  S^T += V'^T Kd =================
        tmem_to_tile64(kColU, OFF_VPT_HI, OFF_VPT_LO);
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            const uint32_t id64b = idesc_bf16_f32(128, 64, false, false, /*b_mn=*/true);
            const uint32_t id128 = idesc_bf16_f32(128, 128, false, false, /*b_mn=*/true);
            const uint64_t dVh = sdesc_kmajor_sw128(sbase + OFF_VPT_HI), dVl = sdesc_kmajor_sw128(sbase + OFF_VPT_LO);
            const uint64_t dAh = sdesc_mnmajor_sw128(sbase + OFF_AQK_HI, 8192), dAl = sdesc_mnmajor_sw128(sbase + OFF_AQK_LO, 8192);
            // Kd: per 64-wide K atom (16 KB apart) the hi tile, then the lo tile 8 KB after it
            const uint64_t dKh = sdesc_mnmajor_sw128(sbase + OFF_KB_HI, 16384),
                           dKl = sdesc_mnmajor_sw128(sbase + OFF_KB_HI + 8192, 16384);
#pragma unroll
            for (int sp = 0; sp < 3; ++sp)
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16(tbase + kColA, dadd(sp == 2 ? dVl : dVh, kk * 32), dadd(sp == 1 ? dAl : dAh, kk * 2048), id64b, 1);
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
        // ================= epilogue: O^T -> gate -> out =================
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
        // ---- final state ----
        if (a.Sfin && sn >= 0) {
            const int j = lrow + lane;
            for (int cb = 0; cb < 32; cb += 16) {
                uint32_t r[16];
                tmem_ld16(tl + kColS + quarter * 32 + cb, r);
                tmem_wait_ld();
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    const int c = quarter * 32 + cb + u;
                    a.Sfin[(snh * kD + c) * kD + j] = __uint_as_float(r[u]);
                }
            }
        }
        // ---- conv state: the last W-1 pre-conv inputs of this head's q, k, v channels ----
        if (A.conv_state != nullptr && W > 1 && sn >= 0) {
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
                            : A.conv_state[((size_t)sn * (W - 1) + (L + r)) * Dall + gch];
                    }
            }
            __syncthreads();
            if (e < 384)
#pragma unroll
                for (int r = 0; r < 3; ++r)
                    if (r < W - 1) A.conv_state[((size_t)sn * (W - 1) + r) * Dall + gch] = keep[r];
        }
    } else if (tid == 0 && !tskip) {                   // (a starved first wait issued no MMA)
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

}  // namespace

namespace tcc {
namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
}  // namespace

cudaError_t make_row_map(CUtensorMap *m, const void *base, CUtensorMapDataType dt, int esz, int T, int H) {
    if (g_encode == nullptr) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || fn == nullptr)
            return e != cudaSuccess ? e : cudaErrorSymbolNotFound;
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    const cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)H, (cuuint64_t)T};
    const cuuint64_t strides[2] = {(cuuint64_t)kD * esz, (cuuint64_t)H * kD * esz};
    const cuuint32_t box[3] = {(cuuint32_t)kD, 1u, (cuuint32_t)(T < kC ? T : kC)};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    const CUresult r = g_encode(m, dt, 3, const_cast<void *>(base), dims, strides, box, estr,
                                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}
}  // namespace tcc

cudaError_t launch_prefill_tc_fused(const PrefillArgs &p, const float *conv_w, float *conv_state, int W,
                                    cudaStream_t s) {
    if ((long long)p.N * p.H == 0) return cudaSuccess;
    TcArgs A{};
    if (p.T > 0) {
        cudaError_t e;
        if ((e = make_row_map(&A.tm_q, p.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.T, p.H)) != cudaSuccess ||
            (e = make_row_map(&A.tm_k, p.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.T, p.H)) != cudaSuccess ||
            (e = make_row_map(&A.tm_v, p.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.T, p.H)) != cudaSuccess ||
            (e = make_row_map(&A.tm_g, p.g, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, p.T, p.H)) != cudaSuccess ||
            (p.gate && (e = make_row_map(&A.tm_gate, p.gate, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.T, p.H)) != cudaSuccess))
            return e;
    }
    static std::atomic<uint64_t> attr_done{0};
    if (cudaError_t e = smem_attr_once((const void *)kda_prefill_tc_kernel, (int)kSmemBytes, attr_done))
        return e;
    A.p = p;
    A.conv_w = conv_w;
    A.conv_state = conv_state;
    A.W = conv_w ? W : 0;
    A.box_rows = p.T < kC ? p.T : kC;
    A.p.test_limit = take_test_timeout(kTestSinglePass);
    kda_prefill_tc_kernel<<<(unsigned)(p.N * p.H), kThreads, kSmemBytes, s>>>(A);
    count_launch();
    return cudaGetLastError();
}

}  // namespace k3kda
