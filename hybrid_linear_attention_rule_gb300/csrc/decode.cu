// decode.cu -- one KDA decode token for N independent sequences.
//
// metrale kimi_k3 docs, Functions: kda_decode_token ("One decode token: conv
// update then recurrent step"); Structs: KdaState (both buffers FP32,
// read-modify-write).  Per (sequence n, head h):
//   conv (+SiLU) of the new q, k, v channels against the conv window, window
//   shifted in place; q, k L2-normalised; then with alpha = exp(g):
//     a = k^T (Diag(alpha) S),  b = q^T (Diag(alpha) S)
//     d = beta (v - a)
//     S' = Diag(alpha) S + k d^T          (= (I - beta k k^T) Diag(alpha) S + beta k v^T)
//     o  = scale (b + (q . k) d)  [* sigmoid(gate)]   (= scale S'^T q)
// so one read pass and one write pass over S suffice.
//
// Roofline: HBM.  Per (n, h) the fp32 state is 4*dk*dv bytes read and the
// same written; everything else is < 10 % of that.  Persistent CTAs (one per
// SM) walk the (n, h) items with a two-stage shared-memory ring: a producer
// warp streams each item's state and its small inputs (q, k, v, g, gate, the
// conv window and weights) with cp.async.bulk copies that complete on an
// mbarrier, while 16 consumer warps work on the previous item.  Consumers pull
// the state into registers (warp w: rows w, w+16, ...; lane l: columns
// 4l..4l+3), hand the stage back at once, reduce the column sums across warps
// through shared memory, and write the new state straight to HBM with
// streaming 128-bit stores, so loads of the next items overlap compute and
// stores of this one.
#include "common.cuh"
#include "tc_ptx.cuh"

namespace k3kda {
namespace {

using namespace tc;

constexpr int kConsumerWarps = 16;
constexpr int kConsumers = 32 * kConsumerWarps;
constexpr int kDecThreads = kConsumers + 32;      // + one producer warp
constexpr int kMaxD = 128;
constexpr int kRowsPerWarp = kMaxD / kConsumerWarps;   // 8
constexpr int kStages = 2;
constexpr uint32_t kWaitLimit = 1u << 26;

// stage layout (bytes)
constexpr uint32_t ST_S = 0;                       // fp32 [dk][dv] (<= 64 KB)
constexpr uint32_t ST_Q = 65536;                   // <= 128 x 4 B each
constexpr uint32_t ST_K = ST_Q + 512;
constexpr uint32_t ST_V = ST_K + 512;
constexpr uint32_t ST_GATE = ST_V + 512;
constexpr uint32_t ST_G = ST_GATE + 512;
constexpr uint32_t ST_CS = ST_G + 512;             // fp32 [W-1 <= 3][2dk + dv <= 384]
constexpr uint32_t ST_CW = ST_CS + 3 * 384 * 4;    // fp32 [2dk + dv][W <= 4]
constexpr uint32_t kStageBytes = ST_CW + 384 * 4 * 4;          // 78848 = 77 KiB
constexpr uint32_t OFF_RED = kStages * kStageBytes;            // fp32 [2][8][128]
constexpr uint32_t OFF_VEC = OFF_RED + 2 * kConsumerWarps * kMaxD * 4;   // sq, sk, sv, salpha, sd, sgate
constexpr uint32_t OFF_MISC = OFF_VEC + 6 * kMaxD * 4;
constexpr uint32_t kSmemBytes = OFF_MISC + 64 + 1024;

struct DecodeArgs {
    const void *q, *k, *v;
    int bf16;
    const float *g, *beta;
    const void *gate;
    const float *conv_w;
    float *conv_state;
    float *state;
    int N, H, dk, dv, W;
    float scale;
    int l2;
    void *out;
    int out_bf16;
    const int32_t *slot;    // [N] state / conv-state row of each sequence, or null (row n)
    int num_slots;
    unsigned test_limit;    // 0; else the armed test hook's tries (see TestTimeout)
};

// This device's decode status word: a decode kernel that gives up a bounded wait ORs 2 into it
// (its outputs are then invalid); k3kda_decode_status reads and clears it.
__device__ unsigned int g_decode_status;

__global__ void __launch_bounds__(kDecThreads, 1) decode_kernel(DecodeArgs a) {
    extern __shared__ uint8_t smraw[];
    uint8_t *sm = smem_align1024(smraw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int dk = a.dk, dv = a.dv, H = a.H, W = a.W;
    const int NH = a.N * a.H;
    const int esz = a.bf16 ? 2 : 4;
    const int nch = 2 * dk + dv;                          // this head's conv channels
    const int D = 2 * H * dk + H * dv;
    float *red = reinterpret_cast<float *>(sm + OFF_RED);
    float *sq = reinterpret_cast<float *>(sm + OFF_VEC), *sk = sq + kMaxD, *sv = sk + kMaxD;
    float *salpha = sv + kMaxD, *sd = salpha + kMaxD, *sgate = sd + kMaxD;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + OFF_MISC);   // full[2], empty[2]
    float *sred = reinterpret_cast<float *>(sm + OFF_MISC + 32);
    volatile uint32_t *sflag = reinterpret_cast<volatile uint32_t *>(sm + OFF_MISC + 48);
    const uint32_t full0 = smem_u32(&bars[0]), empty0 = smem_u32(&bars[2]);

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, kConsumerWarps);
        }
        fence_mbar_init();
        *sflag = 0;
    }
    __syncthreads();

    if (warp == kConsumerWarps) {
        // ---------------- producer ----------------
        // test hook: CTA 0 stages nothing, so its consumers' first wait runs out
        if (lane == 0 && !(a.test_limit != 0 && blockIdx.x == 0)) {
            // m counts the items actually staged: an item whose slot is out of range is skipped by
            // the producer and the consumers alike, so both sides agree on stages and parities
            for (int kk = 0, m = 0;; ++kk) {
                const int it = blockIdx.x + kk * gridDim.x;
                if (it >= NH) break;
                const int n = it / H, h = it - (it / H) * H;
                const int sn = seq_slot(a.slot, a.num_slots, n);
                if (sn < 0) continue;
                const int s = m & 1;
                const uint32_t P = smem_u32(sm + s * kStageBytes);
                if (m >= kStages && !mbar_wait_bounded(empty0 + 8 * s, ((m - kStages) >> 1) & 1, kWaitLimit)) {
                    atomicOr(&g_decode_status, 2u);
                    break;
                }
                ++m;
                const size_t sit = (size_t)sn * H + h;      // the state this item reads and writes
                uint32_t bytes = (uint32_t)(dk * dv * 4 + 2 * dk * esz + dv * esz + dk * 4);
                if (a.gate) bytes += dv * esz;
                if (a.conv_w) bytes += (uint32_t)(nch * 4 * (W - 1) + nch * 4 * W);
                mbar_arrive_expect_tx(full0 + 8 * s, bytes);
                const uint32_t fb = full0 + 8 * s;
                bulk_g2s(P + ST_S, a.state + sit * dk * dv, dk * dv * 4, fb);
                bulk_g2s(P + ST_Q, (const char *)a.q + (size_t)it * dk * esz, dk * esz, fb);
                bulk_g2s(P + ST_K, (const char *)a.k + (size_t)it * dk * esz, dk * esz, fb);
                bulk_g2s(P + ST_V, (const char *)a.v + (size_t)it * dv * esz, dv * esz, fb);
                if (a.gate) bulk_g2s(P + ST_GATE, (const char *)a.gate + (size_t)it * dv * esz, dv * esz, fb);
                bulk_g2s(P + ST_G, a.g + (size_t)it * dk, dk * 4, fb);
                if (a.conv_w) {
                    const size_t seg[3] = {(size_t)h * dk, (size_t)H * dk + (size_t)h * dk,
                                           2 * (size_t)H * dk + (size_t)h * dv};
                    const uint32_t len[3] = {(uint32_t)dk, (uint32_t)dk, (uint32_t)dv};
                    const uint32_t loc[3] = {0, (uint32_t)dk, (uint32_t)(2 * dk)};
                    for (int r = 0; r < W - 1; ++r)
                        for (int u = 0; u < 3; ++u)
                            bulk_g2s(P + ST_CS + (r * nch + loc[u]) * 4,
                                     a.conv_state + ((size_t)sn * (W - 1) + r) * D + seg[u], len[u] * 4, fb);
                    for (int u = 0; u < 3; ++u)
                        bulk_g2s(P + ST_CW + loc[u] * W * 4, a.conv_w + seg[u] * W, len[u] * W * 4, fb);
                }
            }
        }
        return;
    }

    // ---------------- consumers (256 threads, named barrier 1) ----------------
    const bool colok = 4 * lane < dv;
    uint32_t tlim = a.test_limit != 0 && blockIdx.x == 0 ? a.test_limit : kWaitLimit;
    for (int kk = 0, m = 0;; ++kk) {
        const int it = blockIdx.x + kk * gridDim.x;
        if (it >= NH) break;
        const int n = it / H, h = it - (it / H) * H;
        const int sn = seq_slot(a.slot, a.num_slots, n);
        if (sn < 0) {                                  // no state to update: the output row is zero
            if (tid < dv) store_elt(a.out, (size_t)it * dv + tid, 0.f, a.out_bf16);
            continue;
        }
        const int s = m & 1;
        uint8_t *P = sm + s * kStageBytes;
        const size_t sit = (size_t)sn * H + h;
        const float bval = tid < dv ? __ldg(a.beta + it) : 0.f;   // in flight while the stage lands
        if (tid == 0 && !mbar_wait_bounded(full0 + 8 * s, (m >> 1) & 1, tlim)) {
            *sflag = 1;
            atomicOr(&g_decode_status, 2u);
        }
        tlim = kWaitLimit;
        ++m;
        named_bar(1, kConsumers);
        if (*sflag) break;

        // 1. conv update + SiLU for this head's q, k, v channels (window from the stage)
        const float *cs = reinterpret_cast<const float *>(P + ST_CS);
        const float *cw = reinterpret_cast<const float *>(P + ST_CW);
        for (int i = tid; i < nch; i += kConsumers) {
            const int which = i < dk ? 0 : (i < 2 * dk ? 1 : 2);
            const int li = which == 0 ? i : (which == 1 ? i - dk : i - 2 * dk);
            const uint8_t *src = P + (which == 0 ? ST_Q : (which == 1 ? ST_K : ST_V));
            const float x = a.bf16 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(src)[li])
                                   : reinterpret_cast<const float *>(src)[li];
            float y = x;
            if (a.conv_w != nullptr) {
                const float *w = cw + (size_t)i * W;
                float acc = w[W - 1] * x;
                float prev[3] = {0.f, 0.f, 0.f};
#pragma unroll
                for (int r = 0; r < 3; ++r)
                    if (r < W - 1) { prev[r] = cs[r * nch + i]; acc = fmaf(w[r], prev[r], acc); }
                const int ch = which == 0 ? h * dk + li : (which == 1 ? H * dk + h * dk + li : 2 * H * dk + h * dv + li);
                float *gcs = a.conv_state + (size_t)sn * (W - 1) * D + ch;
#pragma unroll
                for (int r = 0; r < 2; ++r)
                    if (r < W - 2) gcs[(size_t)r * D] = prev[r + 1];
                if (W > 1) gcs[(size_t)(W - 2) * D] = x;
                y = acc / (1.0f + expf(-acc));
            }
            if (which == 0) sq[li] = y;
            else if (which == 1) sk[li] = y;
            else sv[li] = y;
        }
        const float *gg = reinterpret_cast<const float *>(P + ST_G);
        for (int c = tid; c < dk; c += kConsumers) salpha[c] = expf(gg[c]);
        if (a.gate)
            for (int j = tid; j < dv; j += kConsumers)
                sgate[j] = a.bf16 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(P + ST_GATE)[j])
                                  : reinterpret_cast<const float *>(P + ST_GATE)[j];
        // 2. state rows -> registers; then the stage goes back to the producer
        const float *Ss = reinterpret_cast<const float *>(P + ST_S);
        float4 sr[kRowsPerWarp];
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r) {
            const int c = warp + kConsumerWarps * r;
            sr[r] = (c < dk && colok) ? *reinterpret_cast<const float4 *>(Ss + (size_t)c * dv + 4 * lane)
                                      : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        named_bar(1, kConsumers);          // every read of the stage is done
        if (lane == 0) mbar_arrive(empty0 + 8 * s);

        // 3. |q|^2, |k|^2, q.k
        if (warp < 3) {
            float acc = 0.f;
            for (int c = lane; c < dk; c += 32) {
                const float x = warp == 1 ? sk[c] : sq[c];
                const float y = warp == 0 ? sq[c] : sk[c];
                acc = fmaf(x, y, acc);
            }
            acc = warp_sum(acc);
            if (lane == 0) sred[warp] = acc;
        }
        named_bar(1, kConsumers);
        float rq = 1.f, rk = 1.f;
        if (a.l2) {
            rq = 1.0f / sqrtf(sred[0] + K3KDA_L2_EPS);
            rk = 1.0f / sqrtf(sred[1] + K3KDA_L2_EPS);
        }
        const float qk = sred[2] * rq * rk;

        // 4. decay in registers; partial column sums of k^T S and q^T S
        float pa[4] = {0.f, 0.f, 0.f, 0.f}, pb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r) {
            const int c = warp + kConsumerWarps * r;
            if (c < dk) {
                const float al = salpha[c], kc = sk[c] * rk, qc = sq[c] * rq;
                sr[r].x *= al; sr[r].y *= al; sr[r].z *= al; sr[r].w *= al;
                pa[0] = fmaf(kc, sr[r].x, pa[0]); pa[1] = fmaf(kc, sr[r].y, pa[1]);
                pa[2] = fmaf(kc, sr[r].z, pa[2]); pa[3] = fmaf(kc, sr[r].w, pa[3]);
                pb[0] = fmaf(qc, sr[r].x, pb[0]); pb[1] = fmaf(qc, sr[r].y, pb[1]);
                pb[2] = fmaf(qc, sr[r].z, pb[2]); pb[3] = fmaf(qc, sr[r].w, pb[3]);
            }
        }
        if (colok) {
            *reinterpret_cast<float4 *>(&red[(0 * kConsumerWarps + warp) * kMaxD + 4 * lane]) = make_float4(pa[0], pa[1], pa[2], pa[3]);
            *reinterpret_cast<float4 *>(&red[(1 * kConsumerWarps + warp) * kMaxD + 4 * lane]) = make_float4(pb[0], pb[1], pb[2], pb[3]);
        }
        named_bar(1, kConsumers);

        // 5. per column: d = beta (v - a), o = scale (b + qk d) [* sigmoid(gate)]
        if (tid < dv) {
            float av = 0.f, bv = 0.f;
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) {
                av += red[w * kMaxD + tid];
                bv += red[(kConsumerWarps + w) * kMaxD + tid];
            }
            const float d = bval * (sv[tid] - av);
            sd[tid] = d;
            float o = a.scale * fmaf(qk, d, bv);
            if (a.gate) o = o / (1.0f + expf(-sgate[tid]));
            store_elt(a.out, (size_t)it * dv + tid, o, a.out_bf16);
        }
        named_bar(1, kConsumers);

        // 6. rank-1 update, streamed straight to HBM
        if (colok) {
            float *Sg = a.state + sit * dk * dv;
            const float4 dd = *reinterpret_cast<const float4 *>(&sd[4 * lane]);
#pragma unroll
            for (int r = 0; r < kRowsPerWarp; ++r) {
                const int c = warp + kConsumerWarps * r;
                if (c < dk) {
                    const float kc = sk[c] * rk;
                    float4 x = sr[r];
                    x.x = fmaf(kc, dd.x, x.x); x.y = fmaf(kc, dd.y, x.y);
                    x.z = fmaf(kc, dd.z, x.z); x.w = fmaf(kc, dd.w, x.w);
                    __stcs(reinterpret_cast<float4 *>(Sg + (size_t)c * dv + 4 * lane), x);
                }
            }
        }
        named_bar(1, kConsumers);          // sq/sk/sd are rewritten by the next item
    }
}

std::atomic<uint64_t> g_decode_attr{0};

}  // namespace

cudaError_t launch_decode(const void *q, const void *k, const void *v, int in_bf16, const float *g,
                          const float *beta, const void *gate, const float *conv_w, float *conv_state,
                          float *state, int N, int H, int dk, int dv, int W, float scale, int l2,
                          void *out, int out_bf16, cudaStream_t s, const int32_t *slot, int num_slots) {
    if (N == 0) return cudaSuccess;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = smem_attr_once((const void *)decode_kernel, (int)kSmemBytes, g_decode_attr);
    if (e != cudaSuccess) return e;
    DecodeArgs a{q, k, v, in_bf16, g, beta, gate, conv_w, conv_state, state, N, H, dk, dv, conv_w ? W : 0, scale,
                 l2, out, out_bf16, slot, num_slots, take_test_timeout(kTestDecode)};
    const long long items = (long long)N * H;
    const int grid = (int)(items < sms ? items : sms);
    decode_kernel<<<grid, kDecThreads, kSmemBytes, s>>>(a);
    count_launch();
    return cudaGetLastError();
}

cudaError_t decode_status(cudaStream_t s, unsigned *word) {
    cudaError_t e = cudaMemcpyFromSymbolAsync(word, g_decode_status, sizeof(unsigned), 0, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess || *word == 0) return e;
    const unsigned zero = 0;
    e = cudaMemcpyToSymbolAsync(g_decode_status, &zero, sizeof(unsigned), 0, cudaMemcpyHostToDevice, s);
    return e == cudaSuccess ? cudaStreamSynchronize(s) : e;
}

}  // namespace k3kda
