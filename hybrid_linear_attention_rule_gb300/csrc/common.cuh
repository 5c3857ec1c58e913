// common.cuh -- device helpers and internal launcher declarations shared by the
// kernels of libk3kda (sm_103a).  Nothing here is part of the C ABI.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include <stddef.h>

#include <atomic>

#include "k3kda.h"

namespace k3kda {

// ---- element access ------------------------------------------------------

__device__ __forceinline__ float load_elt(const void *p, size_t i, int bf16) {
    if (bf16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(p)[i]);
    return reinterpret_cast<const float *>(p)[i];
}

__device__ __forceinline__ void store_elt(void *p, size_t i, float x, int bf16) {
    if (bf16) reinterpret_cast<__nv_bfloat16 *>(p)[i] = __float2bfloat16_rn(x);
    else reinterpret_cast<float *>(p)[i] = x;
}

__device__ __forceinline__ float sigmoidf_(float z) { return 1.0f / (1.0f + __expf(-z)); }
__device__ __forceinline__ float siluf_(float z) { return z / (1.0f + __expf(-z)); }

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// Sequence bounds for sequence n from a device cu_seqlens, clamped into
// [0, T] and made non-decreasing so that a malformed array can never send a
// kernel out of bounds (the host validates whenever it has a host copy).
__device__ __forceinline__ void seq_bounds(const int32_t *cu, int n, int T, int &b, int &e) {
    if (cu == nullptr) { b = 0; e = T; return; }
    int lo = cu[n], hi = cu[n + 1];
    lo = lo < 0 ? 0 : (lo > T ? T : lo);
    hi = hi < lo ? lo : (hi > T ? T : hi);
    b = lo; e = hi;
}

// Pool slot of sequence n when a call maps its sequences onto a slot-indexed state pool
// (continuous batching), n itself otherwise; -1 when the map's entry is outside [0, num_slots):
// such a sequence starts from zero state and conv history and writes neither back.
__device__ __forceinline__ int seq_slot(const int32_t *slot, int num_slots, int n) {
    if (slot == nullptr) return n;
    const int s = slot[n];
    return (s >= 0 && s < num_slots) ? s : -1;
}

// Raise a kernel's dynamic shared-memory limit on the current device, once per device (the
// attribute belongs to the device's context); safe to call from several host threads.
inline cudaError_t smem_attr_once(const void *func, int bytes, std::atomic<uint64_t> &done) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = dev >= 0 && dev < 64 ? uint64_t(1) << dev : 0;
    if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
    e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_release);
    return e;
}

// Counts every kernel this library launches (reported by k3kda_launch_count).
void count_launch();

// Test hook for the bounded in-kernel waits.  k3kda_test_arm_wait_timeout (exported for the tests,
// not part of the public header) arms one of these; the next launch of that kernel takes the armed
// count (and disarms it), and its CTA 0 then issues none of the copies its first bounded wait waits
// for and gives up that wait after the armed number of tries, so the kernel's timeout path runs
// (status recorded, nothing left in flight, TMEM freed) on a GPU that is working normally.
enum TestTimeout { kTestScan = 0, kTestSinglePass = 1, kTestDecode = 2, kTestBackward = 3, kTestKinds = 4 };
unsigned take_test_timeout(int which);

// ---- launchers (defined in the kernel files, called by the C ABI layer) ----

cudaError_t launch_short_conv(const void *x, int x_bf16, const float *w, const float *cs_in,
                              const int32_t *cu, int N, int T, int D, int W, int silu,
                              void *out, int out_bf16, cudaStream_t s);
cudaError_t launch_conv_state_update(const void *x, int x_bf16, float *cs, const int32_t *cu,
                                     int N, int T, int D, int W, cudaStream_t s);

cudaError_t launch_short_conv_strided(const void *x, int64_t x_stride, int x_bf16, const float *w,
                                      const float *cs, int64_t cs_stride, const int32_t *cu, int N,
                                      int T, int Dc, int W, int silu, void *out, int64_t out_stride,
                                      int out_bf16, cudaStream_t s, const int32_t *slot = nullptr,
                                      int num_slots = 0);
cudaError_t launch_conv_state_update_strided(const void *x, int64_t x_stride, int x_bf16, float *cs,
                                             int64_t cs_stride, const int32_t *cu, int N, int T,
                                             int Dc, int W, cudaStream_t s, const int32_t *slot = nullptr,
                                             int num_slots = 0);

// Read and clear this device's decode status word (0, or nonzero after a decode kernel gave up a
// bounded wait); synchronises s.
cudaError_t decode_status(cudaStream_t s, unsigned *word);
cudaError_t launch_decode(const void *q, const void *k, const void *v, int in_bf16, const float *g,
                          const float *beta, const void *gate, const float *conv_w, float *conv_state,
                          float *state, int N, int H, int dk, int dv, int W, float scale, int l2,
                          void *out, int out_bf16, cudaStream_t s, const int32_t *slot = nullptr,
                          int num_slots = 0);

struct PrefillArgs {
    const void *q, *k, *v;   // [T,H,dk] x2, [T,H,dv]; element type by in_bf16
    int64_t q_row, k_row, v_row;   // element stride between tokens (H*dk or D for fused-conv buffers)
    int in_bf16;
    const float *g, *beta, *S0;
    const int32_t *cu;
    int N, T, H, dk, dv, chunk;
    float scale;
    int l2;
    const void *gate;        // [T,H,dv] logits or null
    int gate_bf16;           // element type of gate (the q/k/v buffers may be fp32 after a conv stage)
    void *out;
    int out_bf16;
    float *Sfin;
    unsigned int *status;    // device status word (workspace offset 0)
    const int32_t *slot;     // [N] pool slot of each sequence for S0 / Sfin / conv state, or null (slot n)
    int num_slots;
    unsigned test_limit;     // 0; else the armed test hook's tries (see TestTimeout)
    const int32_t *cu_host;  // host copy of cu (validated), or null: read on the host only, to plan segments
};

cudaError_t launch_prefill_f32(const PrefillArgs &a, cudaStream_t s);
// reverse-mode gradients of the recurrence in chunked form (csrc/backward_chunked.cu); dk = dv = 128
size_t backward_chunked_workspace(int N, int T, int H);
cudaError_t launch_backward_chunked(const void *q, const void *k, const void *v, int bf16, const float *g,
                                    const float *beta, const float *S0, const int32_t *cu, int N, int T, int H,
                                    float scale, const float *dO, const float *dSfin, float *dq, float *dk, float *dv,
                                    float *dg, float *dbeta, float *dS0, unsigned *status, void *ws, cudaStream_t s);

// one decode token of the gated attention layers (csrc/mla_decode.cu); dq in {64, 128, 192, 256},
// dv in {64, 128, 256}
size_t mla_splits(int L_max);
size_t mla_workspace(int N, int H, int dq, int dv, int L_max);
cudaError_t launch_mla_decode(const void *q, const void *k_new, const void *v_new, int in_bf16, const void *gate,
                              void *k_cache, void *v_cache, int cache_bf16, int32_t *cache_len, int N, int H, int dq,
                              int dv, int L_max, int rope_dim, float theta, float scale, void *out, int out_bf16,
                              void *ws, cudaStream_t st, const int32_t *slot = nullptr, int num_slots = 0);

}  // namespace k3kda
