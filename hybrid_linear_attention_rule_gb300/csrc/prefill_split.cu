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
//       conv, norm, decay -> Kh, Qh, Kb, Kd, v;  Akk, Aqk;  Tb = (I + Akk)^-1 diag(beta)
//       W = Tb Kh,  U = Tb v                                   -> one record per item
//   pass 2, chunk scan (one CTA per (sequence, head), chunks in order):
//       S' = diag(exp(rho)) S;  V' = U - W S';  O = scale (Qh S' + Aqk V') [* sigmoid(gate)]
//       S_next = diag(exp(G_last)) S + Kd^T V'
// (Kh = k exp(G - rho), Qh = q exp(G - rho) with rho a per-channel reference,
// Kd = k exp(G_last - G): W S' and Qh S' carry exp(G) from the chunk start to
// each token, Kd the decay from each token to the chunk end; every factor the
// scan applies is <= 1, so the state needs no rescaling whatever the decay.)
//
// The record of an item (148,480 bytes, in the caller's workspace) holds the
// split-bf16 tiles [W; Qh], Kd and Aqk^T in the exact 128B-swizzled shared-memory
// layout in which the scan kernel's MMAs read them, U^T in fp32 and the
// per-channel rho and G_last; the scan kernel fetches the tiles with bulk copies
// that overlap its own MMAs.  It keeps the fp32 state in TMEM for the whole
// sequence, like the single-pass kernel; per chunk it runs two MMA chains, both
// with the A operand in TMEM: N = 128 against [W; Qh], then N = 192 against
// [Aqk^T | Kd] (O += V'^T Aqk^T beside S += V'^T Kd in adjacent TMEM columns).
// The time of a tcgen05 MMA here is set by the instruction count far more than
// by N, hence the wide chains.
#include <cuda.h>

#include <algorithm>
#include <cstdlib>
#include <mutex>

#include "tc_chunk.cuh"

namespace k3kda {
namespace {

using namespace tc;
using namespace tcc;

// ---- one chunk record (byte offsets; identical to the scan kernel's smem layout) ----
constexpr uint32_t REC_X = 0;            // [W rows 0-63; Qh rows 64-127] x 128 K, per 64-wide K atom hi then lo (16 KB each)
constexpr uint32_t REC_B = 65536;        // MN-major B of MMA O/S: 8 KB N-blocks Aqk^T hi, lo, then Kd hi, lo per K atom
constexpr uint32_t REC_U = 114688;       // U^T fp32 as 16 blocks of 4 tokens: [tok / 4][128 dv][4 tok]
constexpr uint32_t REC_VEC = 147456;     // rho[128], G_last[128] fp32
constexpr uint32_t REC_BYTES = 148480;
static_assert(PlanPrep::X_LO == PlanPrep::X_HI + 16384 && PlanPrep::X_ATOM == 32768,
              "the record's [W; Qh] part is the prep plan's X tile: [hi 0 | lo 0 | hi 1 | lo 1]");
static_assert(OFF_GL == OFF_REF + 512, "rho and G_last are adjacent");

// byte offset of U^T element (dv j, token i) inside the U block: a warp's 32 consecutive dv
// channels with the same 4 tokens fill 512 contiguous bytes (coalesced stores, conflict-free loads)
__device__ __forceinline__ uint32_t u_off(uint32_t j, uint32_t i) {
    return (i >> 2) * 2048u + j * 16u + (i & 3u) * 4u;
}

// ============================ segment offsets ============================
// A call runs in segments: segment k covers the local chunks [k per, (k + 1) per) of every
// sequence (one segment of unbounded length when the call is not segmented).  Block k writes the
// record table of segment k, off = tables + k (N + 1): off[n] = number of records (chunks) of
// sequences 0 .. n-1 in the segment (off[0] = 0, off[N] = the segment's total), capped at qmax,
// the number of records a segment's buffer holds: a malformed device cu_seqlens (overlapping
// sequences) then loses chunks instead of sending either pass past the workspace.
__global__ void __launch_bounds__(1024) kda_segment_offsets_kernel(const int32_t *cu, int N, int T, int per, int qmax,
                                                                   int32_t *tables) {
    __shared__ int32_t part[32];
    __shared__ int32_t carry;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const long long lo = (long long)blockIdx.x * per;
    int32_t *off = tables + (size_t)blockIdx.x * (N + 1);
    if (tid == 0) { carry = 0; off[0] = 0; }
    __syncthreads();
    for (int base = 0; base < N; base += 1024) {
        const int n = base + tid;
        int x = 0;
        if (n < N) {
            int tb, te;
            seq_bounds(cu, n, T, tb, te);
            const long long nq = (te - tb + kC - 1) / kC;
            x = (int)(nq <= lo ? 0 : (nq - lo < per ? nq - lo : per));
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

// ============================ one launch for every segment ============================
// In the overlap shape one cooperative launch runs every segment: n_scan of its CTAs are the scan
// chains, the rest the prep, all resident at once (the first segment is prepared beforehand by a
// launch of the prep kernel on every SM, so that the chains start at once).  They meet through counters in the workspace:
// a chain starts segment k once prep_done[k] = n_prep (every record of the segment written), and
// the prep writes segment k's records into its ring buffer once scan_done[k - ring] = n_scan (the
// previous reader of that buffer is through).  A CTA that gives up a wait, or whose own bounded
// waits run out, raises abort, and every other CTA stops at its next wait.
struct SegPlan {
    const int32_t *tables;   // [nseg][N + 1] record tables
    uint8_t *rec;            // record buffers
    int nseg, per, ring, linear;
    size_t slot_records;     // records one ring buffer holds
    int *prep_done, *scan_done;   // [nseg]
    int *abort;
    int n_scan, n_prep;
    int first_seg;           // segments before it were prepared by an earlier launch on all SMs
};
constexpr uint32_t kSpinLimit = 1u << 23;              // polls of a cross-CTA wait (each >= 0.2 us)

__device__ __forceinline__ int ld_acquire_gpu(const int *p) {
    int v;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void red_release_add_gpu(int *p, int v) {
    asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// Orders this thread's generic-proxy accesses to global memory with its async-proxy (bulk copy)
// accesses on either side of the fence.
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}
// One thread waits until *ctr >= target; false (abort raised) when the wait runs out or another
// CTA has aborted.
__device__ __forceinline__ bool wait_counter(const SegPlan *pl, const int *ctr, int target) {
    for (uint32_t i = 0; i < kSpinLimit; ++i) {
        if (ld_acquire_gpu(ctr) >= target) return true;
        if (*reinterpret_cast<volatile const int *>(pl->abort) != 0) return false;
        __nanosleep(200);
    }
    atomicExch(pl->abort, 1);
    return false;
}
// record buffer of segment k
__device__ __forceinline__ uint8_t *seg_records(const SegPlan *pl, int k, int H) {
    return pl->rec + (pl->linear ? (size_t)k * pl->per * H : (size_t)(k % pl->ring) * pl->slot_records) * REC_BYTES;
}

// ============================ pass 1: chunk prep ============================
struct PrepArgs {
    CUtensorMap tm_q, tm_k, tm_v, tm_g;   // [T, H, 128] (bf16 q, k, v; fp32 g), box min(64, T) tokens of one head
    PrefillArgs p;
    const float *conv_w;      // [3*H*128, W] or null
    const float *conv_state;  // [N, W-1, 3*H*128] initial conv state or null (read only here)
    int W;
    int box_rows;
    const int32_t *seg_off;   // [N + 1] this segment's record table (record r of sequence n: seg_off[n] + r)
    int seg_lo;               // first local chunk of the segment
    uint8_t *rec;             // the segment's records: [record * H + h]
};

constexpr uint32_t kPrepTmemCols = 512;
// MMA A result in [0, 128) (two halves summed: hi*hi + lo*hi | hi*lo), U^T and W^T likewise
constexpr uint32_t kColUp = 128, kColWp = 256;

// The prep of one segment (pl null: A's segment, CTA cta of ncta) or of every segment of the plan.
template <bool kPersist>
__device__ __forceinline__ void prep_body(const PrepArgs &A, const SegPlan *pl, int cta, int ncta) {
    extern __shared__ uint8_t smraw[];
    uint8_t *sm = smem_align1024(smraw);
    const PrefillArgs &a = A.p;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = a.H, N = a.N;
    const uint32_t sbase = smem_u32(sm);
    float *sConvW = reinterpret_cast<float *>(sm + OFF_CONVW);
    float *sHist = reinterpret_cast<float *>(sm + OFF_HIST);
    float *sBeta = reinterpret_cast<float *>(sm + OFF_BETA);
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

    // the segment in hand: its record table, first local chunk and record buffer
    const int32_t *seg_off = A.seg_off;
    int seg_lo = A.seg_lo;
    uint8_t *seg_rec = A.rec;
    int nq = 0;
    int cur_h = -1;                                      // head whose conv weights are loaded
    PhaseClock clk;   // phases: 0 staging wait, 1 prep q/k, 2 prep v (MMA A), 3 history + MMA A wait, 4 extract, 5 solve, 6 MMA U/W, 7 records out
    const int nseg = kPersist ? pl->nseg : 1;
    for (int k = kPersist ? pl->first_seg : 0; k < nseg; ++k) {
    if (kPersist) {
        seg_off = pl->tables + (size_t)k * (N + 1);
        seg_lo = k * pl->per;
        seg_rec = seg_records(pl, k, H);
        // the buffer's previous reader, the scan of segment k - ring, must be through
        if (!pl->linear && k >= pl->ring) {
            if (tid == 0) {
                if (!wait_counter(pl, pl->scan_done + (k - pl->ring), pl->n_scan)) {
                    *sflag = 1;
                    atomicOr(a.status, 1u);
                }
                fence_proxy_async_global();              // the bulk stores below follow the reads
            }
            __syncthreads();
            if (*sflag) break;
        }
    }
    // Items in head-major order (head, chunk), each CTA taking a contiguous run of them: a CTA's
    // consecutive items are then mostly consecutive chunks of one head, whose conv history is the
    // previous chunk's last staged rows and whose conv weights are already loaded.
    nq = seg_off[N];                                     // records (chunks) of this segment
    const long long total = (long long)nq * H;
    const int m_lo = (int)(total * cta / ncta);
    const int m_hi = (int)(total * (cta + 1) / ncta);
    struct Item { int h, qc, n, tb, te, cs, qend; };   // qc: record; qend: one past the sequence's last record
    auto locate = [&](int m) {
        Item x;
        x.h = m / nq;
        x.qc = m - x.h * nq;
        int lo = 0, hi = N;                              // sequence n with off[n] <= qc < off[n + 1]
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (seg_off[mid] <= x.qc) lo = mid; else hi = mid;
        }
        x.n = lo;
        seq_bounds(a.cu, x.n, a.T, x.tb, x.te);
        x.cs = x.tb + (seg_lo + x.qc - seg_off[x.n]) * kC;
        x.qend = seg_off[x.n + 1];
        return x;
    };
    // item m + 1 after item x = item m: the next chunk of the same sequence and head without
    // touching global memory, else a fresh lookup
    auto advance = [&](const Item &x, int m) {
        if ((m + 1) % nq != 0 && x.qc + 1 < x.qend) {
            Item y = x;
            y.qc += 1;
            y.cs += kC;
            return y;
        }
        return locate(m + 1);
    };
    auto rec_of = [&](const Item &x) { return seg_rec + ((size_t)x.qc * H + x.h) * REC_BYTES; };
    // conv weights of the item's head and its conv history (pre-conv q, k, v rows of tokens
    // cs-3 .. cs-1 from the inputs, or from the right-aligned initial conv state before the
    // sequence start), by all threads; the prep stages are their only readers
    auto load_history = [&](const Item &x) {
        if (W == 0) return;
        if (x.h != cur_h) {
            for (int e = tid; e < 384 * 4; e += kThreads) {
                // tap-major, taps right-aligned in a 4-wide window: tap t multiplies token i - 3 + t
                const int t = e / 384, ch = e - t * 384;
                const int gch = (ch >> 7) * H * kD + x.h * kD + (ch & 127);
                sConvW[e] = t >= 4 - W ? A.conv_w[(size_t)gch * W + (t - (4 - W))] : 0.f;
            }
            cur_h = x.h;
        }
        for (int e = tid; e < 3 * 3 * 128; e += kThreads) {
            const int which = e / 384, r = (e / 128) % 3, c = e & 127;
            const int t = x.cs - 3 + r;
            float v = 0.f;
            if (t >= x.tb) {
                const void *src = which == 0 ? a.q : (which == 1 ? a.k : a.v);
                v = __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(src)[((size_t)t * H + x.h) * kD + c]);
            } else {
                const int row = W - 1 + (t - x.tb);
                const int sn = seq_slot(a.slot, a.num_slots, x.n);
                if (W > 1 && A.conv_state != nullptr && row >= 0 && sn >= 0)
                    v = A.conv_state[((size_t)sn * (W - 1) + row) * Dall + which * H * kD + x.h * kD + c];
            }
            sHist[e] = v;
        }
    };
    // the conv history of the chunk after a whole chunk: its last three staged rows
    auto copy_history = [&]() {
        if (W == 0) return;
        for (int e = tid; e < 3 * 3 * 128; e += kThreads) {
            const int which = e / 384, r = (e / 128) % 3, c = e & 127;
            const uint32_t st = which == 0 ? PlanPrep::QST : (which == 1 ? PlanPrep::KST : PlanPrep::VST);
            sHist[e] = __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(sm + st + (kC - 3 + r) * (kD * 2) + c * 2));
        }
    };
    // An item's rows land on one phase of mbar_s in two pieces (thread 0): q, k, v while the
    // previous item's MMA A runs, g once the previous item's triangular solve has freed region R.
    auto stage_qkv = [&](const Item &x) {
        mbar_arrive_expect_tx(mbar_s, kStageBytes);
        tma_load_3d(sbase + PlanPrep::QST, &A.tm_q, 0, x.h, x.cs, mbar_s);
        tma_load_3d(sbase + PlanPrep::KST, &A.tm_k, 0, x.h, x.cs, mbar_s);
        tma_load_3d(sbase + PlanPrep::VST, &A.tm_v, 0, x.h, x.cs, mbar_s);
        pend_s = true;
    };
    auto stage_g = [&](const Item &x) { tma_load_3d(sbase + PlanPrep::GST, &A.tm_g, 0, x.h, x.cs, mbar_s); };
    // the g rows into L2 ahead of their staging copy, which is issued late (after the previous
    // item's solve); q, k and v are staged a whole item ahead and need no prefetch
    auto prefetch_rows = [&](const Item &x) { tma_prefetch_3d(&A.tm_g, 0, x.h, x.cs); };

    Item x, y;                                           // this item and the next
    if (m_lo < m_hi) {
        x = locate(m_lo);
        y = m_lo + 1 < m_hi ? advance(x, m_lo) : x;
        if (tid == 0) {
            stage_qkv(x);
            stage_g(x);
            if (m_lo + 1 < m_hi) prefetch_rows(y);
        }
        load_history(x);
        if (tid < kC) sBeta[tid] = tid < x.te - x.cs ? a.beta[(size_t)(x.cs + tid) * H + x.h] : 0.f;
    }
    for (int m = m_lo; m < m_hi; ++m, x = y, y = m + 1 < m_hi ? advance(y, m) : y) {
        const bool has_next = m + 1 < m_hi;
        const bool cont = has_next && y.h == x.h && y.n == x.n && y.cs == x.cs + kC;
        const int Lc = min(kC, x.te - x.cs);
        uint8_t *rec = rec_of(x);
        if (tid == 0) {
            bulk_wait_read_but_last();                   // all but W have left shared memory (prep_qk waits for W)
            wait_on(mbar_s, sph, pend_s);
        }
        __syncthreads();
        if (*sflag) break;
        clk.tick(0);

        float kd[kTok][4];
        const bool strong = prep_qk<PlanPrep>(sm, a, x.cs, Lc, x.h, W, tl, kColA, kd);
        clk.tick(1);
        if (tid == 0) {
            issue_mma_a<PlanPrep>(sbase, tbase + kColA, mbar_a, strong);
            pend_a = true;
            // Qh (rows 64..127 of each K atom, hi and lo) is final: out now
#pragma unroll
            for (int p = 0; p < 4; ++p)
                bulk_s2g(rec + REC_X + p * 16384 + 8192, sbase + PlanPrep::X_HI + p * 16384 + 8192, 8192);
            bulk_commit();
        }
        put_kd(rec + REC_B + 16384, kd);                 // Kd straight from registers, in the record's layout
        if (tid < kD) {                                  // rho, G_last
            reinterpret_cast<float *>(rec + REC_VEC)[tid] = reinterpret_cast<const float *>(sm + OFF_REF)[tid];
            reinterpret_cast<float *>(rec + REC_VEC)[kD + tid] = reinterpret_cast<const float *>(sm + OFF_GL)[tid];
        }
        prep_v<PlanPrep>(sm, a, Lc, W);                  // overlaps MMA A
        clk.tick(2);
        if (has_next) {
            if (cont) copy_history(); else load_history(y);
        }
        __syncthreads();                                 // this item's staged rows are consumed
        if (tid == 0) {
            if (has_next) stage_qkv(y);
            bulk_wait_read_all();                        // the Qh rows have left (X is rewritten by the next prep)
        }
        if (!mma_wait()) break;
        clk.tick(3);
        extract_akk<PlanPrep>(sm, tl, kColA);
        clk.tick(4);
        solve_tb<PlanPrep>(sm, tl, kColA);
        float beta_next = 0.f;                           // the next item's beta, written after MMA U/W
        if (has_next && tid < kC && tid < y.te - y.cs) beta_next = a.beta[(size_t)(y.cs + tid) * H + y.h];
        if (tid == 0) {
            static_assert(PlanPrep::AQK_LO == PlanPrep::AQK_HI + 8192, "Aqk^T hi and lo must be adjacent");
            bulk_s2g(rec + REC_B, sbase + PlanPrep::AQK_HI, 16384);
            bulk_commit();
            if (has_next) stage_g(y);                    // region R is free
        }
        clk.tick(5);

        // ---- MMA: U^T = v^T Tb^T and W^T = Kh^T Tb^T (Kh rows 0-63 of X read MN-major).  Tb_hi and
        // Tb_lo are adjacent 64-row tiles, one N = 128 operand: x_hi [Tb_hi; Tb_lo]^T, then x_lo Tb_hi^T
        // into the first 64 columns; the result is the sum of the two halves ----
        if (tid == 0) {
            tc_fence_after();
            const uint32_t id128 = idesc_bf16_f32(128, 128, false, /*a_mn=*/true),
                           id64 = idesc_bf16_f32(128, 64, false, /*a_mn=*/true);
            const uint64_t dVh = sdesc_mnmajor_sw128(sbase + PlanPrep::V_HI, 8192),
                           dVl = sdesc_mnmajor_sw128(sbase + PlanPrep::V_LO, 8192);
            const uint64_t dKh = sdesc_mnmajor_sw128(sbase + PlanPrep::X_HI, PlanPrep::X_ATOM),
                           dKl = sdesc_mnmajor_sw128(sbase + PlanPrep::X_LO, PlanPrep::X_ATOM);
            const uint64_t dT = sdesc_kmajor_sw128(sbase + PlanPrep::TB_HI);
            static_assert(PlanPrep::TB_LO == PlanPrep::TB_HI + 8192, "Tb hi and lo must form one 128-row tile");
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_bf16(tbase + kColUp, dadd(dVh, kk * 2048), dadd(dT, kk * 32), id128, kk != 0);
            if (W > 0)                                   // v is exact bf16 without a conv
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16(tbase + kColUp, dadd(dVl, kk * 2048), dadd(dT, kk * 32), id64, 1);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_bf16(tbase + kColWp, dadd(dKh, kk * 2048), dadd(dT, kk * 32), id128, kk != 0);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_bf16(tbase + kColWp, dadd(dKl, kk * 2048), dadd(dT, kk * 32), id64, 1);
            mma_commit(mbar_a);
            pend_a = true;
            // the g rows of the item after next into L2, while the MMAs run (the issue may wait
            // on the copy engine)
            if (m + 2 < m_hi) prefetch_rows(advance(y, m + 1));
        }
        if (!mma_wait()) break;
        clk.tick(6);

        // ---- U^T -> the record (straight from registers), W -> X/XL rows 0-63 -> the record ----
        {
            const int j = lrow + lane;                  // dv channel for U^T, dk channel for W^T
            uint32_t r[16], r2[16];
            auto ld_sum = [&](uint32_t col) {
                tmem_ld16(tl + col + quarter * 16, r);
                tmem_ld16(tl + col + 64 + quarter * 16, r2);
                tmem_wait_ld();
#pragma unroll
                for (int u = 0; u < 16; ++u) r[u] = __float_as_uint(__uint_as_float(r[u]) + __uint_as_float(r2[u]));
            };
            ld_sum(kColUp);
#pragma unroll
            for (int t = 0; t < 4; ++t)
                *reinterpret_cast<uint4 *>(rec + REC_U + u_off(j, quarter * 16 + 4 * t)) =
                    make_uint4(r[4 * t], r[4 * t + 1], r[4 * t + 2], r[4 * t + 3]);
            ld_sum(kColWp);
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                float hv, lv;
                split_bf16(__uint_as_float(r[u]), hv, lv);
                const uint32_t o = (j >> 6) * PlanPrep::X_ATOM + sw128_offset(quarter * 16 + u, j & 63);
                *reinterpret_cast<__nv_bfloat16 *>(sm + PlanPrep::X_HI + o) = __float2bfloat16_rn(hv);
                *reinterpret_cast<__nv_bfloat16 *>(sm + PlanPrep::X_LO + o) = __float2bfloat16_rn(lv);
            }
        }
        if (has_next && tid < kC) sBeta[tid] = beta_next;
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
#pragma unroll
            for (int p = 0; p < 4; ++p) bulk_s2g(rec + REC_X + p * 16384, sbase + PlanPrep::X_HI + p * 16384, 8192);
            bulk_commit();
        }
        tc_fence_after();
        clk.tick(7);
    }
    if (kPersist) {
        // the segment's records are written (the bulk stores complete, everyone's stores before
        // the barrier): publish them
        __syncthreads();
        if (tid == 0) {
            bulk_wait_all();
            fence_proxy_async_global();
            __threadfence();
            if (*sflag) atomicExch(pl->abort, 1);
            else red_release_add_gpu(pl->prep_done + k, 1);
        }
    }
    if (*sflag) break;
    }   // segments
    clk.flush(reinterpret_cast<unsigned long long *>(a.status) + 16);
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

__global__ void __launch_bounds__(kThreads, 1) kda_chunk_prep_kernel(const __grid_constant__ PrepArgs A) {
    prep_body<false>(A, nullptr, blockIdx.x, gridDim.x);
}

// ============================ pass 2: chunk scan ============================
struct ScanArgs {
    CUtensorMap tm_gate;      // [T, H, 128] bf16 gate logits (when gated), box min(64, T) tokens of one head
    CUtensorMap tm_out;       // [T, H, 128] bf16 outputs (when stored as bf16), same box
    PrefillArgs p;
    int box_rows;
    float *conv_state;        // [N, W-1, 3*H*128] advanced at the end, or null
    int W;
    const int32_t *seg_off;   // [N + 1] this segment's record table
    int seg_lo;               // first local chunk of the segment
    const uint8_t *rec;       // the segment's records: [record * H + h]
    float *carry_S;           // [N*H][128 dv][128 dk] state handed between launches
};

// scan kernel shared memory: [W; Qh] of even chunks and [Aqk^T | Kb] at their record offsets, then
// [W; Qh] of odd chunks (the next chunk's tile lands while this chunk's MMAs read the other)
constexpr uint32_t Q_X1 = REC_U;                    // [W; Qh] tile of odd chunks (64 KB)
constexpr uint32_t Q_G0 = Q_X1 + 65536;             // gate logits bf16 [64 tok][128] of even / odd chunks
constexpr uint32_t Q_G1 = Q_G0 + 16384;
constexpr uint32_t Q_OST = Q_G1 + 16384;            // bf16 outputs [64 tok][128] of one chunk, stored by TMA
constexpr uint32_t Q_FA = Q_OST + 16384;            // exp(rho) per channel of the chunk whose state pass is next
constexpr uint32_t Q_FS = Q_FA + 512;               // exp(G_last) per channel, same chunk
constexpr uint32_t Q_MISC = Q_FS + 512;             // 6 mbarriers, tmem slot, flag
constexpr uint32_t kScanSmemBytes = Q_MISC + 64 + 1024;
static_assert(Q_X1 % 1024 == 0, "tile alignment");
static_assert(kScanSmemBytes <= 232448, "scan kernel shared memory exceeds the per-CTA limit");

// Tensor memory: the MMA A operands S'^T and V'^T live here as split bf16 (two values per
// 32-bit column, the even K index in the low half), so shared memory only feeds the B operands.
// MMA W writes D = S'^T [W_hi; Qh_hi; W_lo; Qh_lo]^T into columns [0, 256) (S'_lo adds into the
// first 128): (W S')^T = D[0, 64) + D[128, 192), (Qh S')^T = D[64, 128) + D[192, 256).  The V'
// phase then puts each thread's V'^T K-step (hi 8 | lo 8) over the columns of D[0, 64) it has
// read, and O^T = (Qh S')^T into D[192, 256), next to the state.
constexpr uint32_t kScanTmemCols = 512;
constexpr uint32_t kColD = 0;       // D, 256 columns; V'^T split in [0, 64)
constexpr uint32_t kColO = 192;     // O^T (fp32)
constexpr uint32_t kColSs = 256;    // S^T fp32 (the state), 128 columns
static_assert(kColO + 64 == kColSs, "O^T and S^T must be adjacent: one N = 192 chain accumulates into both");
constexpr uint32_t kColSh = 384;    // S'^T hi / lo, bf16 pairs: 64 columns each
constexpr uint32_t kColSl = 448;

// 16 consecutive K values of one TMEM lane -> split bf16 pairs at columns col_hi, col_lo (8 each)
__device__ __forceinline__ void tmem_put_split16(uint32_t col_hi, uint32_t col_lo, const float (&v)[16]) {
    uint32_t hw[8], lw[8];
#pragma unroll
    for (int u = 0; u < 16; u += 2) {
        float h0, l0, h1, l1;
        split_bf16(v[u], h0, l0);
        split_bf16(v[u + 1], h1, l1);
        hw[u >> 1] = pack_bf16(h0, h1);
        lw[u >> 1] = pack_bf16(l0, l1);
    }
    tmem_st8(col_hi, hw);
    tmem_st8(col_lo, lw);
}

// spare issuing lanes of the scan: lane 0 of warps 15 and 14
constexpr int kIssueX = kThreads - 32, kIssueK = kThreads - 64;

// Per chunk: MMA [(W S')^T | (Qh S')^T], while the gate's sigmoid is taken; V'^T = U^T - (W S')^T;
// MMA [O^T | S^T] += V'^T [Aqk^T | Kd]; then one phase writes this chunk's outputs and runs the next
// chunk's state pass.  [W; Qh] and the gate rows (both double-buffered, two chunks ahead) and
// [Aqk^T | Kd] arrive by bulk copies issued as soon as their buffers are free; U^T, rho and
// G_last are read by the threads that use them, one chunk ahead, into registers.
// The scan of one segment (pl null: A's segment, with the state carried in and out through
// A.carry_S) or of every segment of the plan (the state staying in TMEM), for chain nh.
template <bool kPersist>
__device__ __forceinline__ void scan_body(const ScanArgs &A, const SegPlan *pl, int nh) {
    extern __shared__ uint8_t smraw[];
    uint8_t *sm = smem_align1024(smraw);
    const PrefillArgs &a = A.p;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n = nh / a.H, h = nh % a.H;
    const int H = a.H;
    const uint32_t sbase = smem_u32(sm);
    float *sFA = reinterpret_cast<float *>(sm + Q_FA);
    float *sFS = reinterpret_cast<float *>(sm + Q_FS);
    uint64_t *mbar = reinterpret_cast<uint64_t *>(sm + Q_MISC);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + Q_MISC + 48);
    volatile uint32_t *sflag = reinterpret_cast<volatile uint32_t *>(sm + Q_MISC + 52);
    const uint32_t mb_a = smem_u32(mbar), mb_x0 = smem_u32(mbar + 1), mb_x1 = smem_u32(mbar + 2),
                   mb_k = smem_u32(mbar + 3), mb_g0 = smem_u32(mbar + 4), mb_g1 = smem_u32(mbar + 5);

    int tb, te;
    seq_bounds(a.cu, n, a.T, tb, te);
    const int nq = (te - tb + kC - 1) / kC;
    // the segment in hand: its record table, first local chunk and record buffer; this sequence's
    // chunks in it are [c_begin, c_end) (local indices; records seg_off[n] ..)
    const int32_t *seg_off = kPersist ? pl->tables : A.seg_off;
    int seg_lo = kPersist ? 0 : A.seg_lo;
    const uint8_t *seg_rec = kPersist ? seg_records(pl, 0, a.H) : A.rec;
    int q0 = seg_off[n], c_begin = seg_lo, c_end = seg_lo + (seg_off[n + 1] - q0);
    const int c_begin0 = c_begin;                         // the first segment's
    // one launch per segment: an empty sequence belongs to the first segment, and a chain with no
    // chunks in the segment has nothing to do
    if (!kPersist && c_begin >= c_end && !(nq == 0 && seg_lo == 0)) return;
    const bool first = kPersist || c_begin == 0, last = kPersist || c_end == nq;
    const int sn = seq_slot(a.slot, a.num_slots, n);           // state / conv-state row (-1: none)
    const size_t snh = (size_t)(sn < 0 ? 0 : sn) * a.H + h;
    const int W = A.W;
    const int Dall = 3 * H * kD;
    const bool gated = a.gate != nullptr;

    if (warp == 0) { tmem_alloc(smem_u32(tslot), kScanTmemCols); tmem_relinquish(); }
    if (tid == 0) {
        mbar_init(mb_a, 1); mbar_init(mb_x0, 1); mbar_init(mb_x1, 1); mbar_init(mb_k, 1);
        mbar_init(mb_g0, 1); mbar_init(mb_g1, 1);
        fence_mbar_init();
        *sflag = 0;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tslot;
    const uint32_t lrow = 32u * (warp & 3);
    const uint32_t tl = tbase + (lrow << 16);
    const int quarter = warp >> 2;
    const int j = lrow + lane;                          // this thread's TMEM lane: dv channel
    // S^T <- S0^T at the sequence start, else the carried state.  The per-channel factors of the
    // next state pass are formed by the last four warps (vt >= 0), which have no copies or MMAs to
    // issue, so that the issuing warp does not trail the others
    const int vt = tid - (kThreads - kD);
    {
        for (int cb = 0; cb < 32; cb += 16) {
            uint32_t r[16];
            if (first) {
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    const int c = quarter * 32 + cb + u;
                    r[u] = __float_as_uint((a.S0 && sn >= 0) ? a.S0[(snh * kD + c) * kD + j] : 0.f);
                }
            } else {
                const float *carry = A.carry_S + ((size_t)nh * kD + j) * kD + quarter * 32 + cb;
#pragma unroll
                for (int u = 0; u < 16; u += 4) {
                    const uint4 v = *reinterpret_cast<const uint4 *>(carry + u);
                    r[u] = v.x; r[u + 1] = v.y; r[u + 2] = v.z; r[u + 3] = v.w;
                }
            }
            tmem_st16(tl + kColSs + quarter * 32 + cb, r);
        }
        tmem_wait_st();
    }

    // record of local chunk c: chain_rec + c H REC_BYTES, chain_rec set per segment
    const uint8_t *chain_rec = seg_rec + ((ptrdiff_t)(q0 - seg_lo) * H + h) * (ptrdiff_t)REC_BYTES;
    auto rec_of = [&](int c) { return chain_rec + (ptrdiff_t)c * H * (ptrdiff_t)REC_BYTES; };
    // thread 0's view of the outstanding asynchronous operations
    uint32_t aph = 0, kph = 0, xph0 = 0, xph1 = 0, gph0 = 0, gph1 = 0;
    bool pend_a = false, pend_k = false, pend_x0 = false, pend_x1 = false, pend_g0 = false, pend_g1 = false;
    // test hook: CTA 0 issues no copy of its first [W; Qh] tile and gives up that wait early
    const bool tskip = a.test_limit != 0 && nh == 0 && c_begin < c_end;
    uint32_t xlim = tskip ? a.test_limit : kWaitLimit;
    auto wait_on = [&](uint32_t bar, uint32_t &ph, bool &pend, uint32_t lim = kWaitLimit) -> bool {
        if (!pend) return true;
        if (!mbar_wait_bounded(bar, ph, lim)) {
            *sflag = 1;
            atomicOr(a.status, 1u);
            return false;
        }
        ph ^= 1u;
        pend = false;
        return true;
    };
    // Copies are issued by thread 0 before the loop and by the spare lanes kIssueX / kIssueK inside
    // it (their warps have slack where they issue); thread 0 alone waits on every copy and keeps
    // the pending flags and phases, setting a flag at the point where the copy is issued.
    auto issue = [&](uint32_t bar, uint32_t dst, uint32_t off, int c, uint32_t bytes) {
        mbar_arrive_expect_tx(bar, bytes);
        bulk_g2s(sbase + dst, rec_of(c) + off, bytes, bar);
    };
    auto load = [&](uint32_t bar, uint32_t dst, uint32_t off, int c, uint32_t bytes, bool &pend) {
        issue(bar, dst, off, c, bytes);
        pend = true;
    };
    auto issue_x = [&](int c) {
        if (c & 1) issue(mb_x1, Q_X1, REC_X, c, 65536);
        else issue(mb_x0, REC_X, REC_X, c, 65536);
    };
    auto mark_x = [&](int c) { if (c & 1) pend_x1 = true; else pend_x0 = true; };
    auto load_x = [&](int c) {
        issue_x(c);
        mark_x(c);
    };
    auto wait_x = [&](int c) {
        const uint32_t lim = xlim;
        xlim = kWaitLimit;
        return (c & 1) ? wait_on(mb_x1, xph1, pend_x1, lim) : wait_on(mb_x0, xph0, pend_x0, lim);
    };
    auto issue_gate = [&](int c) {                   // chunk c's gate rows -> buffer c & 1
        const uint32_t bar = (c & 1) ? mb_g1 : mb_g0;
        mbar_arrive_expect_tx(bar, (uint32_t)A.box_rows * kD * 2);
        tma_load_3d(sbase + ((c & 1) ? Q_G1 : Q_G0), &A.tm_gate, 0, h, tb + c * kC, bar);
    };
    auto mark_gate = [&](int c) { if (c & 1) pend_g1 = true; else pend_g0 = true; };
    auto load_gate = [&](int c) {
        issue_gate(c);
        mark_gate(c);
    };
    auto wait_gate = [&](int c) { return (c & 1) ? wait_on(mb_g1, gph1, pend_g1) : wait_on(mb_g0, gph0, pend_g0); };
    // the other threads wait for chunk c's gate rows themselves (no CTA barrier): the phase of
    // buffer c & 1 is the number of earlier loads into it, mod 2
    auto gate_ready = [&](int c) {
        const int b = c & 1;
        // every chunk from the first one of the launch loads its rows into buffer c & 1, in order
        const int c0 = kPersist ? 0 : c_begin;
        const int first_b = c0 + ((b - c0) & 1);
        mbar_wait_bounded(b ? mb_g1 : mb_g0, (uint32_t)(((c - first_b) >> 1) & 1), kWaitLimit);
    };
    auto mma_wait = [&]() -> bool {
        if (tid == 0 && !*sflag) wait_on(mb_a, aph, pend_a);
        __syncthreads();
        const bool bad = *sflag != 0;
        tc_fence_after();
        return !bad;
    };

    // register-resident operands, one chunk ahead
    float uR[16];                 // U^T row j, tokens 16*quarter .. +15
    float rN = 0.f, glN = 0.f;    // vt >= 0: rho and G_last of the chunk after the current one
    auto load_u = [&](int c) {
        const uint8_t *p = rec_of(c) + REC_U;
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const float4 v = __ldcg(reinterpret_cast<const float4 *>(p + u_off(j, quarter * 16 + 4 * t)));
            uR[4 * t] = v.x; uR[4 * t + 1] = v.y; uR[4 * t + 2] = v.z; uR[4 * t + 3] = v.w;
        }
    };
    auto load_vec = [&](int c) {
        const float *p = reinterpret_cast<const float *>(rec_of(c) + REC_VEC);
        rN = __ldcg(p + vt);
        glN = __ldcg(p + kD + vt);
    };
    // the state pass of a chunk: S'^T = S^T diag(exp(rho)) as split bf16 (the A operand of MMA W/Qh),
    // and the fp32 accumulator S^T <- S^T diag(exp(G_last)), onto which MMA O/S adds V'^T Kd
    auto state_pass = [&]() {
        uint32_t r[2][16];
        tmem_ld16(tl + kColSs + quarter * 32, r[0]);
        tmem_ld16(tl + kColSs + quarter * 32 + 16, r[1]);
        tmem_wait_ld();
#pragma unroll
        for (int b = 0; b < 2; ++b) {
            const int col = quarter * 32 + 16 * b;
            float v[16], fa[16], fs[16];
#pragma unroll
            for (int u = 0; u < 16; u += 4) {
                *reinterpret_cast<float4 *>(fa + u) = *reinterpret_cast<const float4 *>(sFA + col + u);
                *reinterpret_cast<float4 *>(fs + u) = *reinterpret_cast<const float4 *>(sFS + col + u);
            }
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                const float x = __uint_as_float(r[b][u]);
                v[u] = x * fa[u];
                r[b][u] = __float_as_uint(x * fs[u]);
            }
            tmem_st16(tl + kColSs + col, r[b]);
            tmem_put_split16(tl + kColSh + col / 2, tl + kColSl + col / 2, v);
        }
        tmem_wait_st();
    };

    // a chunk's record and gate rows into L2 ahead of their copies into shared memory (one thread)
    auto prefetch_chunk = [&](int c) {
        prefetch_l2(rec_of(c), REC_BYTES);
        if (gated) tma_prefetch_3d(&A.tm_gate, 0, h, tb + c * kC);
    };

    bool failed = false;
    PhaseClock clk;   // phases: 0 MMA W, 1 V' tile, 2 MMA O/S, 3 epilogue + next state pass
    const int nseg = kPersist ? pl->nseg : 1;
    for (int k = 0; k < nseg; ++k) {
    if (kPersist) {
        if (k > 0) {
            const int32_t *off = pl->tables + (size_t)k * (a.N + 1);
            c_begin = k * pl->per;
            c_end = c_begin + (off[n + 1] - off[n]);
            chain_rec = seg_records(pl, k, H) + ((ptrdiff_t)(off[n] - c_begin) * H + h) * (ptrdiff_t)REC_BYTES;
        }
        // every record of the segment is written (by this launch's prep CTAs, or before it); the
        // bulk copies below read them
        if (tid == 0) {
            if (k >= pl->first_seg && !wait_counter(pl, pl->prep_done + k, pl->n_prep)) {
                *sflag = 1;
                atomicOr(a.status, 1u);
            }
            fence_proxy_async_global();
        }
        __syncthreads();
        if (*sflag) {
            failed = true;
            break;
        }
    }
    if (c_begin < c_end) {
        const int c = c_begin;
        if (tid == 0) {
            if (!(tskip && k == 0)) load_x(c);
            else if (c & 1) pend_x1 = true;
            else pend_x0 = true;
            load(mb_k, REC_B, REC_B, c, 49152, pend_k);     // [Aqk^T | Kb] hi, lo
            for (int d = 1; d <= 2 && c + d < c_end; ++d) prefetch_chunk(c + d);
            if (gated) load_gate(c);
            if (c + 1 < c_end) {
                load_x(c + 1);
                if (gated) load_gate(c + 1);
            }
        }
        load_u(c);
        if (vt >= 0) {
            load_vec(c);
            sFA[vt] = expf(rN);
            sFS[vt] = expf(glN);
            if (c + 1 < c_end) load_vec(c + 1);
        }
        __syncthreads();
        state_pass();
        tc_fence_before();
        __syncthreads();
    }
    for (int c = c_begin; c < c_end; ++c) {
        const int cs = tb + c * kC;
        const int Lc = min(kC, te - cs);
        const bool more = c + 1 < c_end;
        // ---- MMA: D = S'^T [W; Qh]^T, hi and lo parts in separate columns ----
        if (tid == 0 && wait_x(c)) {
            tc_fence_after();
            // per K atom the tile's 256 rows are [W_hi; Qh_hi; W_lo; Qh_lo]: S'_hi against all of
            // them (N = 256), then S'_lo against the hi rows (N = 128)
            const uint32_t id256 = idesc_bf16_f32(128, 256), id128 = idesc_bf16_f32(128, 128);
            const uint32_t xoff = (c & 1) ? Q_X1 : REC_X;
            const uint64_t dX = sdesc_kmajor_sw128(sbase + xoff);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                mma_bf16_ta(tbase + kColD, tbase + kColSh + kk * 8, dadd(dX, (kk >> 2) * 32768 + (kk & 3) * 32), id256,
                            kk != 0);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                mma_bf16_ta(tbase + kColD, tbase + kColSl + kk * 8, dadd(dX, (kk >> 2) * 32768 + (kk & 3) * 32), id128, 1);
            mma_commit(mb_a);
            pend_a = true;
        }
        // the sigmoid of this chunk's gate logits, while MMA W runs
        float sg[16];
        if (gated) {
            if (tid == 0) {
                if (!*sflag) wait_gate(c);
            } else {
                gate_ready(c);
            }
            const uint8_t *gt = sm + ((c & 1) ? Q_G1 : Q_G0);
#pragma unroll
            for (int u = 0; u < 16; ++u)
                sg[u] = sigmoid_fast(__bfloat162float(
                    *reinterpret_cast<const __nv_bfloat16 *>(gt + (quarter * 16 + u) * (kD * 2) + j * 2)));
        } else {
#pragma unroll
            for (int u = 0; u < 16; ++u) sg[u] = 1.f;
        }
        // the next chunk's state-pass factors, while the MMAs run (this chunk's pass has read them)
        if (vt >= 0 && more) {
            sFA[vt] = expf(rN);
            sFS[vt] = expf(glN);
            if (c + 2 < c_end) load_vec(c + 2);
        }
        if (!mma_wait()) { failed = true; break; }
        clk.tick(0);
        // ---- V'^T = U^T - (W S')^T -> split, over the columns just read; O^T = (Qh S')^T ----
        {
            uint32_t r[16], r2[16];
            tmem_ld16(tl + kColD + quarter * 16, r);
            tmem_ld16(tl + kColD + 128 + quarter * 16, r2);
            tmem_wait_ld();
            // (Qh S')^T's two parts go out at once, read while V' is formed (other columns)
            uint32_t r3[16], r4[16];
            tmem_ld16(tl + kColD + 64 + quarter * 16, r3);
            tmem_ld16(tl + kColO + quarter * 16, r4);
            float v[16];
#pragma unroll
            for (int u = 0; u < 16; ++u) v[u] = uR[u] - (__uint_as_float(r[u]) + __uint_as_float(r2[u]));
            tmem_put_split16(tl + kColD + quarter * 16, tl + kColD + quarter * 16 + 8, v);
            tmem_wait_ld();
#pragma unroll
            for (int u = 0; u < 16; ++u) r3[u] = __float_as_uint(__uint_as_float(r3[u]) + __uint_as_float(r4[u]));
            tmem_st16(tl + kColO + quarter * 16, r3);
            tmem_wait_st();
        }
        if (more) load_u(c + 1);
        if (tid == 0) bulk_wait_read_all();              // the previous chunk's output tile has been read
        tc_fence_before();
        __syncthreads();
        clk.tick(1);
        // ---- MMA: [O^T | S^T] += V'^T [Aqk^T | Kd]  (N = 192: columns kColO .. kColSs + 127) ----
        if (tid == 0 && wait_on(mb_k, kph, pend_k)) {
            tc_fence_after();
            const uint32_t id = idesc_bf16_f32(128, 192, false, false, /*b_mn=*/true);
            // N-blocks (Aqk^T, Kb atom 0, Kb atom 1) 16 KB apart, the lo blocks 8 KB after the hi ones
            const uint64_t dBh = sdesc_mnmajor_sw128(sbase + REC_B, 16384),
                           dBl = sdesc_mnmajor_sw128(sbase + REC_B + 8192, 16384);
#pragma unroll
            for (int sp = 0; sp < 3; ++sp)
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16_ta(tbase + kColO, tbase + kColD + kk * 16 + (sp == 2 ? 8 : 0),
                                dadd(sp == 1 ? dBl : dBh, kk * 2048), id, 1);
            mma_commit(mb_a);
            pend_a = true;
        }
        // this chunk's [W; Qh] buffer is free since MMA W: the tile two chunks ahead, and the record
        // three chunks ahead into L2, while MMA O/S runs
        if (c + 2 < c_end) {
            if (tid == kIssueX) issue_x(c + 2);
            if (tid == 0) mark_x(c + 2);
        }
        if (tid == kIssueX && c + 3 < c_end) prefetch_chunk(c + 3);
        if (!mma_wait()) { failed = true; break; }
        // the buffers read by MMA O/S and by the gate's sigmoid are free
        if (more) {                                      // [Aqk^T | Kd] of the next chunk
            if (tid == kIssueK) issue(mb_k, REC_B, REC_B, c + 1, 49152);
            if (tid == 0) pend_k = true;
        }
        if (gated && c + 2 < c_end) {
            if (tid == kIssueX) issue_gate(c + 2);
            if (tid == 0) mark_gate(c + 2);
        }
        clk.tick(2);
        // ---- this chunk's outputs, then the next chunk's state pass ----
        // bf16 outputs go through a shared tile and one TMA store that runs behind the next chunk,
        // unless the chunk is a ragged sequence end inside the tensor (the box would cross into
        // the next sequence's rows; TMA clips only at the tensor's end)
        const bool tma_out = a.out_bf16 && (Lc == kC || te == a.T);
        {
            uint32_t r0[16];
            tmem_ld16(tl + kColO + quarter * 16, r0);
            tmem_wait_ld();
            if (tma_out) {
                __nv_bfloat16 *ot = reinterpret_cast<__nv_bfloat16 *>(sm + Q_OST);
#pragma unroll
                for (int u = 0; u < 16; ++u)
                    ot[(quarter * 16 + u) * kD + j] = __float2bfloat16_rn(a.scale * __uint_as_float(r0[u]) * sg[u]);
            } else {
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    const int i = quarter * 16 + u;
                    if (i < Lc) store_elt(a.out, ((size_t)(cs + i) * H + h) * kD + j, a.scale * __uint_as_float(r0[u]) * sg[u],
                                          a.out_bf16);
                }
            }
        }
        if (more) state_pass();
        if (tma_out) fence_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0 && tma_out) {
            tma_store_3d(&A.tm_out, sbase + Q_OST, 0, h, cs);
            bulk_commit();
        }
        clk.tick(3);
    }
    if (kPersist && tid == 0) {
        // the segment's records have all been read (copies landed, U rows in registers and used)
        if (failed) atomicExch(pl->abort, 1);
        else red_release_add_gpu(pl->scan_done + k, 1);
    }
    if (failed) break;
    }   // segments
    clk.flush(reinterpret_cast<unsigned long long *>(a.status) + 8);
    if (!failed && !last) {
        tc_fence_after();
        // ---- hand the state to the launch that continues the sequence ----
        float *carry = A.carry_S + ((size_t)nh * kD + j) * kD;
        for (int cb = 0; cb < 32; cb += 16) {
            uint32_t r[16];
            tmem_ld16(tl + kColSs + quarter * 32 + cb, r);
            tmem_wait_ld();
#pragma unroll
            for (int u = 0; u < 16; u += 4)
                *reinterpret_cast<uint4 *>(carry + quarter * 32 + cb + u) = make_uint4(r[u], r[u + 1], r[u + 2], r[u + 3]);
        }
    }
    if (!failed && last) {
        tc_fence_after();
        // ---- final state ----
        if (a.Sfin && sn >= 0) {
            for (int cb = 0; cb < 32; cb += 16) {
                uint32_t r[16];
                tmem_ld16(tl + kColSs + quarter * 32 + cb, r);
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
    }
    if (tid == 0) {
        bulk_wait_all();                                 // output tiles written
        if (tskip) {                                     // the starved tile was never requested
            if (c_begin0 & 1) pend_x1 = false;
            else pend_x0 = false;
        }
        // after a failure, let what is still in flight land before the CTA exits
        if (pend_a) mbar_wait_bounded(mb_a, aph, kWaitLimit);
        if (pend_x0) mbar_wait_bounded(mb_x0, xph0, kWaitLimit);
        if (pend_x1) mbar_wait_bounded(mb_x1, xph1, kWaitLimit);
        if (pend_k) mbar_wait_bounded(mb_k, kph, kWaitLimit);
        if (pend_g0) mbar_wait_bounded(mb_g0, gph0, kWaitLimit);
        if (pend_g1) mbar_wait_bounded(mb_g1, gph1, kWaitLimit);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tbase, kScanTmemCols);
}

__global__ void __launch_bounds__(kThreads, 1) kda_chunk_scan_kernel(const __grid_constant__ ScanArgs A) {
    // the prep of the next segment, launched as a programmatic dependent, may start beside this
    // scan: it reads only inputs and writes the ring buffer that the scan before this one read
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    scan_body<false>(A, nullptr, blockIdx.x);
}

// The segments of an overlap-shape call in one cooperative launch: n_scan CTAs run the scan chains,
// the rest the prep of segments first_seg.. (see SegPlan).
struct SegmentsArgs {
    PrepArgs P;
    ScanArgs S;
    SegPlan plan;
};
__global__ void __launch_bounds__(kThreads, 1) kda_prefill_segments_kernel(const __grid_constant__ SegmentsArgs A) {
    // the chains are the last n_scan CTAs: with one CTA per SM these fill whole TPCs (SM pairs), so
    // that no chain shares its TPC with a prep CTA (a chain beside a prep CTA slows both)
    const int b = blockIdx.x;
    if (b >= A.plan.n_prep) scan_body<true>(A.S, &A.plan, b - A.plan.n_prep);
    else prep_body<true>(A.P, &A.plan, b, A.plan.n_prep);
}

size_t max_chunks(int N, int T) { return ((size_t)T + 63u * (size_t)N) / kC; }
size_t round256_(size_t b) { return (b + 255) & ~size_t(255); }

// Segmented calls.  A call runs in segments of `per` local chunks of every sequence, whose records
// go to a ring of buffers, so the workspace does not grow with T.  Three shapes:
//   one segment  few chunks in all: every record has its own place, prep then scan;
//   overlap      few (sequence, head) chains (<= 64) with >= 128 chunks: one cooperative launch in
//                which the chains run beside the prep of the following segments (kda_prefill_
//                segments_kernel), segments of ~64 chunks whose items fill whole waves of the prep
//                CTAs, a ring of three, the chains' states staying in TMEM;
//   bounded      many chains whose records would exceed kRecordBudget: segments as long as a ring
//                of two within the budget allows, all sequences advancing together (the longest
//                sets the number of segments; with a host copy of cu_seqlens it is exact, else the
//                bound ceil(T / 64) is used and the segments past the longest sequence are empty),
//                prep then scan per segment on the caller's stream, each prep a programmatic
//                dependent of the scan before it so that the two overlap, the chains' states
//                handed from one scan launch to the next through the carry buffer.
// Everything runs on the caller's stream; the library keeps no stream or event of its own.
constexpr int kSegChunks = 64;
constexpr int kMaxSegsOverlap = 64;
constexpr size_t kRecordBudget = size_t(5) << 28;       // 1.25 GiB of records in the bounded shape
size_t carry_bytes(int N, int H) { return (size_t)N * H * kD * kD * sizeof(float); }

struct SegShape {
    int mode;            // 0 one segment, 1 overlap, 2 bounded
    int per_min, per_max;
    int ring;
    size_t slot_records; // records (chunk, head) one ring buffer holds
    long long nseg_max;  // segments at most (record tables in the workspace)
    bool linear;         // one sequence whose records all fit: segment k's records at chunk k * per
};

SegShape seg_shape(int N, int T, int H) {
    const size_t maxq = max_chunks(N, T);
    const long long longest = ((long long)T + kC - 1) / kC;
    SegShape sh{0, 1 << 30, 1 << 30, 1, maxq * (size_t)H, 1, false};
    if ((long long)N * H <= 64 && longest >= 2 * kSegChunks) {
        sh.mode = 1;
        sh.ring = 3;
        sh.per_max = std::max(kSegChunks * 5 / 4, (int)((longest + kMaxSegsOverlap - 1) / kMaxSegsOverlap));
        sh.per_min = std::min(kSegChunks * 3 / 4, sh.per_max);
    } else if (maxq * H * REC_BYTES > kRecordBudget) {
        sh.mode = 2;
        sh.ring = 2;
        sh.per_max = sh.per_min =
            (int)std::max<size_t>(1, kRecordBudget / ((size_t)sh.ring * N * H * REC_BYTES));
    }
    if (sh.mode) {
        sh.slot_records = std::min((size_t)N * sh.per_max, maxq) * H;
        sh.nseg_max = (longest + sh.per_min - 1) / sh.per_min;
        if (N == 1 && maxq <= (size_t)sh.ring * sh.per_max) {
            // one sequence whose records take no more room than the ring: each at its own place
            sh.linear = true;
            sh.ring = 1;
            sh.slot_records = maxq * H;
        }
    }
    return sh;
}
size_t tables_bytes(const SegShape &sh, int N) { return round256_((size_t)sh.nseg_max * (N + 1) * sizeof(int32_t)); }
// prep_done[nseg_max], scan_done[nseg_max], abort
size_t counters_bytes(const SegShape &sh) { return round256_(((size_t)2 * sh.nseg_max + 1) * sizeof(int)); }

}  // namespace

// Workspace of the two-pass path (after the status word): the segments' record tables, then for a
// segmented call the segment counters and the scan's state carry, then the ring of record buffers
// (one buffer holding every record when the call is one segment).
size_t tc_split_workspace(int N, int T, int H) {
    const SegShape sh = seg_shape(N, T, H);
    return tables_bytes(sh, N) + (sh.mode ? counters_bytes(sh) + round256_(carry_bytes(N, H)) : 0) +
           (size_t)sh.ring * sh.slot_records * REC_BYTES;
}

cudaError_t launch_prefill_tc_split(const PrefillArgs &p, const float *conv_w, float *conv_state, int W,
                                    void *ws, cudaStream_t s) {
    if ((long long)p.N * p.H == 0) return cudaSuccess;
    const SegShape sh = seg_shape(p.N, p.T, p.H);
    uint8_t *w = static_cast<uint8_t *>(ws);
    int32_t *tables = reinterpret_cast<int32_t *>(w);
    w += tables_bytes(sh, p.N);
    float *carry_S = nullptr;
    int *counters = nullptr;
    if (sh.mode) {
        counters = reinterpret_cast<int *>(w);
        w += counters_bytes(sh);
        carry_S = reinterpret_cast<float *>(w);
        w += round256_(carry_bytes(p.N, p.H));
    }
    uint8_t *rec = w;
    const int box_rows = p.T < kC ? p.T : kC;
    cudaError_t e;
    static std::atomic<uint64_t> prep_attr{0}, scan_attr{0}, seg_attr{0};
    constexpr size_t kSegmentsSmem = kSmemBytes > kScanSmemBytes ? kSmemBytes : kScanSmemBytes;
    if ((e = smem_attr_once((const void *)kda_chunk_prep_kernel, (int)kSmemBytes, prep_attr)) != cudaSuccess ||
        (e = smem_attr_once((const void *)kda_chunk_scan_kernel, (int)kScanSmemBytes, scan_attr)) != cudaSuccess ||
        (e = smem_attr_once((const void *)kda_prefill_segments_kernel, (int)kSegmentsSmem, seg_attr)) != cudaSuccess)
        return e;
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return e;

    // segment length and count: the longest sequence from the host copy when there is one
    long long longest = ((long long)p.T + kC - 1) / kC;
    if (p.cu_host) {
        longest = 0;
        for (int n = 0; n < p.N; ++n)
            longest = std::max<long long>(longest, ((long long)p.cu_host[n + 1] - p.cu_host[n] + kC - 1) / kC);
    }
    const int reserve = (int)std::min<long long>((long long)p.N * p.H, sms);   // SMs left to a concurrent scan
    const int prep_ctas = sh.mode == 1 ? std::max(1, sms - reserve) : sms;
    int per = sh.per_max;
    if (sh.mode == 1) {
        // segment length near kSegChunks whose (chunk, head) items fill whole waves of the prep grid
        const int n_chains = std::max(1, p.N);
        per = kSegChunks;
        double best = 0.0;
        for (int c = sh.per_min; c <= kSegChunks * 5 / 4; ++c) {
            const long long items = (long long)c * n_chains * p.H, waves = (items + prep_ctas - 1) / prep_ctas;
            const double eff = (double)items / (double)(waves * prep_ctas);
            if (eff > best + 1e-9 || (eff > best - 1e-9 && std::abs(c - kSegChunks) < std::abs(per - kSegChunks))) {
                best = eff;
                per = c;
            }
        }
        per = std::max(per, (int)((longest + kMaxSegsOverlap - 1) / kMaxSegsOverlap));
        per = std::min(per, sh.per_max);
    }
    const int nseg = sh.mode ? (int)std::max<long long>(1, (longest + per - 1) / per) : 1;
    if (nseg > sh.nseg_max) return cudaErrorInvalidValue;        // cannot happen: per >= per_min
    const int qcap = (int)(sh.slot_records / p.H);                  // records one buffer holds

    kda_segment_offsets_kernel<<<nseg, 1024, 0, s>>>(p.cu, p.N, p.T, sh.mode ? per : (1 << 30), qcap, tables);
    count_launch();
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const size_t qmax = max_chunks(p.N, p.T);

    PrepArgs P{};
    if (qmax > 0 &&
        ((e = make_row_map(&P.tm_q, p.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.T, p.H)) != cudaSuccess ||
         (e = make_row_map(&P.tm_k, p.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.T, p.H)) != cudaSuccess ||
         (e = make_row_map(&P.tm_v, p.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.T, p.H)) != cudaSuccess ||
         (e = make_row_map(&P.tm_g, p.g, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, p.T, p.H)) != cudaSuccess))
        return e;
    P.p = p;
    P.conv_w = conv_w;
    P.conv_state = conv_state;
    P.W = conv_w ? W : 0;
    P.box_rows = box_rows;
    P.rec = rec;

    ScanArgs S{};
    if (p.gate && p.T > 0 &&
        (e = make_row_map(&S.tm_gate, p.gate, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.T, p.H)) != cudaSuccess)
        return e;
    if (p.out_bf16 && p.T > 0 &&
        (e = make_row_map(&S.tm_out, p.out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.T, p.H)) != cudaSuccess)
        return e;
    S.box_rows = box_rows;
    S.p = p;
    S.conv_state = conv_w ? conv_state : nullptr;
    S.W = conv_w ? W : 0;
    S.rec = rec;
    S.carry_S = carry_S;
    const unsigned scan_grid = (unsigned)(p.N * p.H);

    // segment k: its record table, first local chunk and ring buffer
    auto set_segment = [&](int k) {
        P.seg_off = S.seg_off = tables + (size_t)k * (p.N + 1);
        P.seg_lo = S.seg_lo = k * per;
        P.rec = rec + (sh.linear ? (size_t)k * per * p.H : (size_t)(k % sh.ring) * sh.slot_records) * REC_BYTES;
        S.rec = P.rec;
    };
    // overlap: launch as a programmatic dependent of the scan launched before it on the stream
    auto prep = [&](int max_ctas, cudaStream_t st, bool overlap = false) -> cudaError_t {
        const unsigned grid = (unsigned)std::min<size_t>(sh.slot_records, (size_t)max_ctas);
        if (grid == 0) return cudaSuccess;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(grid);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = kSmemBytes;
        cfg.stream = st;
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        at[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = at;
        cfg.numAttrs = overlap ? 1 : 0;
        cudaError_t err = cudaLaunchKernelEx(&cfg, kda_chunk_prep_kernel, P);
        count_launch();
        return err != cudaSuccess ? err : cudaGetLastError();
    };
    auto scan = [&](int k, cudaStream_t st) -> cudaError_t {
        S.p.test_limit = k == 0 ? take_test_timeout(kTestScan) : 0u;
        kda_chunk_scan_kernel<<<scan_grid, kThreads, kScanSmemBytes, st>>>(S);
        count_launch();
        return cudaGetLastError();
    };
    if (sh.mode == 0) {
        set_segment(0);
        if (qmax > 0 && (e = prep(sms, s)) != cudaSuccess) return e;
        return scan(0, s);
    }
    if (sh.mode == 1) {
        // one cooperative launch, when every CTA of it can be resident at once
        int coop = 0, per_sm = 0;
        const int n_scan = p.N * p.H;
        if ((e = cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev)) != cudaSuccess ||
            (e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kda_prefill_segments_kernel, kThreads,
                                                               kSegmentsSmem)) != cudaSuccess)
            return e;
        if (coop && per_sm >= 1 && n_scan < sms) {
            if ((e = cudaMemsetAsync(counters, 0, counters_bytes(sh), s)) != cudaSuccess) return e;
            set_segment(0);
            if ((e = prep(sms, s)) != cudaSuccess) return e;
            SegmentsArgs X;
            X.P = P;
            X.S = S;
            X.S.p.test_limit = take_test_timeout(kTestScan);
            X.plan.tables = tables;
            X.plan.rec = rec;
            X.plan.nseg = nseg;
            X.plan.per = per;
            X.plan.ring = sh.ring;
            X.plan.linear = sh.linear ? 1 : 0;
            X.plan.slot_records = sh.slot_records;
            X.plan.prep_done = counters;
            X.plan.scan_done = counters + sh.nseg_max;
            X.plan.abort = counters + 2 * sh.nseg_max;
            X.plan.n_scan = n_scan;
            X.plan.n_prep = sms - n_scan;
            X.plan.first_seg = 1;
            void *args[] = {&X};
            e = cudaLaunchCooperativeKernel((const void *)kda_prefill_segments_kernel, dim3((unsigned)sms),
                                            dim3(kThreads), args, kSegmentsSmem, s);
            count_launch();
            return e;
        }
    }
    // segment by segment on the caller's stream, the prep of segment k + 1 beside the scan of segment
    // k: it is a programmatic dependent of that scan, and stream order still puts every scan after
    // its own prep and after the scan before it, so a ring buffer (two or three) is rewritten only
    // once the scan that read it has finished
    for (int k = 0; k < nseg; ++k) {
        set_segment(k);
        if ((e = prep(sms, s, k > 0)) != cudaSuccess || (e = scan(k, s)) != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace k3kda
