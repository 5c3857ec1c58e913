// noalloc.cu -- k3kda_prefill_noalloc: the chunked prefill without a caller
// workspace.
//
// Some callers cannot allocate device memory at the point where they run the
// mixer: code inside a custom allocator or memory pool, runtimes that forbid
// cudaMalloc after start-up, or plug-ins that only receive pre-allocated
// input and output buffers.  This entry point serves them.  Its scratch (the
// status word and, for the fp32 CUDA-core shapes with a fused conv, the fp32
// conv staging buffer) lives in a fixed-size array that the library itself
// reserves in device memory; every GPU that loads the library holds that
// array until the process exits.
#include "common.cuh"

namespace {

// 16 MiB of library-held device scratch, shared by every call on a device.
constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// The device address of the array on the current device.  In host code the array's name is only a
// host-side stand-in; the runtime resolves it per device and context.  Looked up on every call
// (cheap, allocates nothing), so that a device reset or a new context never leaves a stale address.
int scratch_address(void **out) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return K3KDA_ERR_CUDA;
    *out = p;
    return K3KDA_OK;
}

}  // namespace

extern "C" {

size_t k3kda_prefill_workspace_min(int N, int T, int H, int dk, int dv, int chunk, int in_dtype, int has_conv);
int k3kda_prefill(const void *q, const void *k, const void *v, int in_dtype, const float *g, const float *beta,
                  const float *initial_state, const int32_t *cu_seqlens, const int32_t *cu_seqlens_host, int N,
                  int T, int H, int dk, int dv, int chunk, float scale, int use_qk_l2norm,
                  const k3kda_conv_args *conv, const void *gate, void *out, int out_dtype, float *final_state,
                  void *workspace, size_t workspace_bytes, void *stream);

int k3kda_prefill_noalloc(const void *q, const void *k, const void *v, int in_dtype, const float *g,
                          const float *beta, const float *initial_state, const int32_t *cu_seqlens,
                          const int32_t *cu_seqlens_host, int N, int T, int H, int dk, int dv, int chunk,
                          float scale, int use_qk_l2norm, const k3kda_conv_args *conv, const void *gate,
                          void *out, int out_dtype, float *final_state, void *stream) {
    // Reject work whose scratch would not fit before touching the device.
    const size_t need = k3kda_prefill_workspace_min(N, T, H, dk, dv, chunk, in_dtype, conv != nullptr);
    if (need > kNoAllocScratchBytes) return K3KDA_ERR_WORKSPACE;
    void *scratch = nullptr;
    if (int st = scratch_address(&scratch)) return st;
    // The status word must start at zero; the rest is written before it is read.
    if (cudaMemsetAsync(scratch, 0, 256, static_cast<cudaStream_t>(stream)) != cudaSuccess) return K3KDA_ERR_CUDA;
    return k3kda_prefill(q, k, v, in_dtype, g, beta, initial_state, cu_seqlens, cu_seqlens_host, N, T, H, dk, dv,
                         chunk, scale, use_qk_l2norm, conv, gate, out, out_dtype, final_state, scratch,
                         kNoAllocScratchBytes, stream);
}

// The status word of the library-held scratch on the current device: synchronise `stream`, read
// and clear it (K3KDA_OK, or K3KDA_ERR_TIMEOUT when a kernel of the last k3kda_prefill_noalloc
// call on this device gave up a bounded wait).
int k3kda_workspace_status(void *workspace, void *stream);

int k3kda_prefill_noalloc_status(void *stream) {
    void *scratch = nullptr;
    if (int st = scratch_address(&scratch)) return st;
    return k3kda_workspace_status(scratch, stream);
}

}  // extern "C"
