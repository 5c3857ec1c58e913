// short_conv.cu -- causal depthwise short convolution (+SiLU) over packed
// variable-length sequences, and the conv-state update.
//
// "independent Q/K/V short convolutions" (HF discussion #187, "Experimental
// Native Vulkan Backend for Kimi K3", feature list); width 4 in production
// (metrale kimi_k3 docs, Structs: KdaConfig "production is 128/4"); the conv
// state is one of the two FP32 read-modify-write buffers of KdaState.
//
// y[t, c] = act(sum_i w[c, i] * x[t - (W-1) + i, c]); history before a
// sequence start comes from the conv state rows (oldest first) or is zero.
// This is an HBM-streaming kernel (8 flop per element): each thread owns one
// channel and walks TT consecutive tokens with a register window, so every
// input element is read once and every warp access is a contiguous run of
// channels.
#include "common.cuh"

namespace k3kda {
namespace {

constexpr int kConvThreads = 128;
constexpr int kConvTokens = 32;   // tokens per thread (one register window walk)

__device__ __forceinline__ int find_seq(const int32_t *cu, int N, int T, int t) {
    if (cu == nullptr) return 0;
    int lo = 0, hi = N - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        int b, e;
        seq_bounds(cu, mid, T, b, e);
        if (b <= t) lo = mid; else hi = mid - 1;
    }
    return lo;
}

struct ConvIO {
    const void *x; int64_t x_stride; int x_bf16;
    const float *w;                     // [Dc, W] rows of the channels handled
    const float *cs; int64_t cs_stride; // conv state base (channel offset applied), row stride
    void *out; int64_t out_stride; int out_bf16;
    const int32_t *slot; int num_slots;  // conv-state row of each sequence (null: its index)
};

template <int W>
__global__ void __launch_bounds__(kConvThreads)
short_conv_kernel(ConvIO io, const int32_t *cu, int N, int T, int Dc, int silu) {
    const int c = blockIdx.x * kConvThreads + threadIdx.x;
    if (c >= Dc) return;
    const int t0 = blockIdx.y * kConvTokens;
    if (t0 >= T) return;
    const int t1 = min(t0 + kConvTokens, T);
    float w[W];
#pragma unroll
    for (int i = 0; i < W; ++i) w[i] = io.w[(size_t)c * W + i];

    int n = find_seq(cu, N, T, t0);
    int b, e;
    seq_bounds(cu, n, T, b, e);
    // Value at absolute position p of sequence n (p may be before its start b).
    auto hist = [&](int p) -> float {
        if (p >= b) return load_elt(io.x, (size_t)p * io.x_stride + c, io.x_bf16);
        if (io.cs == nullptr || W == 1) return 0.0f;
        const int row = (W - 1) + (p - b);      // 0 .. W-2 for a well-formed cu_seqlens
        const int sn = seq_slot(io.slot, io.num_slots, n);
        if (row < 0 || sn < 0) return 0.0f;
        return io.cs[((size_t)sn * (W - 1) + row) * io.cs_stride + c];
    };
    float win[W];
#pragma unroll
    for (int i = 0; i < W - 1; ++i) win[i] = hist(t0 - (W - 1) + i);
    for (int t = t0; t < t1; ++t) {
        if (t >= e) {                            // crossed into a later sequence
            while (t >= e && n < N - 1) { ++n; seq_bounds(cu, n, T, b, e); }
#pragma unroll
            for (int i = 0; i < W - 1; ++i) win[i] = hist(t - (W - 1) + i);
        }
        win[W - 1] = load_elt(io.x, (size_t)t * io.x_stride + c, io.x_bf16);
        float acc = 0.0f;
#pragma unroll
        for (int i = 0; i < W; ++i) acc = fmaf(w[i], win[i], acc);
        store_elt(io.out, (size_t)t * io.out_stride + c, silu ? siluf_(acc) : acc, io.out_bf16);
#pragma unroll
        for (int i = 0; i < W - 1; ++i) win[i] = win[i + 1];
    }
}

// New conv state: row r of sequence n <- input at position L - (W-1) + r, or
// the old row L + r when that position is before the start.  Rows are visited
// in increasing r, and row r only reads old rows > r, so the update is in place.
__global__ void conv_state_kernel(const void *x, int64_t x_stride, int x_bf16, float *cs,
                                  int64_t cs_stride, const int32_t *cu, int N, int T, int Dc, int W,
                                  const int32_t *slot, int num_slots) {
    const int c = blockIdx.x * blockDim.x + threadIdx.x;
    const int n = blockIdx.y;
    if (c >= Dc || n >= N) return;
    const int sn = seq_slot(slot, num_slots, n);
    if (sn < 0) return;
    int b, e;
    seq_bounds(cu, n, T, b, e);
    const int L = e - b;
    for (int r = 0; r < W - 1; ++r) {
        const int p = L - (W - 1) + r;
        float val;
        if (p >= 0) val = load_elt(x, (size_t)(b + p) * x_stride + c, x_bf16);
        else val = cs[((size_t)sn * (W - 1) + (L + r)) * cs_stride + c];
        cs[((size_t)sn * (W - 1) + r) * cs_stride + c] = val;
    }
}

}  // namespace

cudaError_t launch_short_conv_strided(const void *x, int64_t x_stride, int x_bf16, const float *w,
                                      const float *cs, int64_t cs_stride, const int32_t *cu, int N,
                                      int T, int Dc, int W, int silu, void *out, int64_t out_stride,
                                      int out_bf16, cudaStream_t s, const int32_t *slot, int num_slots) {
    if (T == 0 || Dc == 0) return cudaSuccess;
    ConvIO io{x, x_stride, x_bf16, w, cs, cs_stride, out, out_stride, out_bf16, slot, num_slots};
    dim3 grid((Dc + kConvThreads - 1) / kConvThreads, (T + kConvTokens - 1) / kConvTokens);
    switch (W) {
        case 1: short_conv_kernel<1><<<grid, kConvThreads, 0, s>>>(io, cu, N, T, Dc, silu); count_launch(); break;
        case 2: short_conv_kernel<2><<<grid, kConvThreads, 0, s>>>(io, cu, N, T, Dc, silu); count_launch(); break;
        case 3: short_conv_kernel<3><<<grid, kConvThreads, 0, s>>>(io, cu, N, T, Dc, silu); count_launch(); break;
        case 4: short_conv_kernel<4><<<grid, kConvThreads, 0, s>>>(io, cu, N, T, Dc, silu); count_launch(); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

cudaError_t launch_conv_state_update_strided(const void *x, int64_t x_stride, int x_bf16, float *cs,
                                             int64_t cs_stride, const int32_t *cu, int N, int T,
                                             int Dc, int W, cudaStream_t s, const int32_t *slot,
                                             int num_slots) {
    if (W <= 1 || N == 0 || Dc == 0) return cudaSuccess;
    dim3 grid((Dc + 255) / 256, N);
    conv_state_kernel<<<grid, 256, 0, s>>>(x, x_stride, x_bf16, cs, cs_stride, cu, N, T, Dc, W, slot, num_slots);
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_short_conv(const void *x, int x_bf16, const float *w, const float *cs_in,
                              const int32_t *cu, int N, int T, int D, int W, int silu,
                              void *out, int out_bf16, cudaStream_t s) {
    return launch_short_conv_strided(x, D, x_bf16, w, cs_in, D, cu, N, T, D, W, silu, out, D,
                                     out_bf16, s);
}

cudaError_t launch_conv_state_update(const void *x, int x_bf16, float *cs, const int32_t *cu,
                                     int N, int T, int D, int W, cudaStream_t s) {
    return launch_conv_state_update_strided(x, D, x_bf16, cs, D, cu, N, T, D, W, s);
}

}  // namespace k3kda
