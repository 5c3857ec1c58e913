// api.cu -- the C ABI of libk3kda (declared in include/k3kda.h): argument
// validation on the host, workspace accounting and kernel launches on the
// caller's stream.  No entry point allocates, synchronises (except
// k3kda_workspace_status, whose job it is), throws or prints.
#include <stdio.h>
#include <atomic>
#include <string.h>
#include <vector>

#include "common.cuh"

namespace k3kda {
size_t prefill_f32_smem_bytes(int chunk, int dk, int dv);
bool tc_prefill_supported(int in_bf16, int dk, int dv, int chunk);
size_t tc_prefill_workspace(int N, int H);
cudaError_t launch_prefill_tc_fused(const PrefillArgs &p, const float *conv_w, float *conv_state, int W,
                                    cudaStream_t s);
size_t tc_split_workspace(int N, int T, int H);
cudaError_t launch_prefill_tc_split(const PrefillArgs &p, const float *conv_w, float *conv_state, int W,
                                    void *ws, cudaStream_t s);
}  // namespace k3kda

using namespace k3kda;

namespace {

std::atomic<long long> g_launches{0};

thread_local char g_last_error[256] = "";

int cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return K3KDA_OK;
    snprintf(g_last_error, sizeof(g_last_error), "%s: %s", cudaGetErrorName(e), cudaGetErrorString(e));
    return K3KDA_ERR_CUDA;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }
bool head_dim_ok(int d) { return d >= 16 && d <= 128 && d % 16 == 0; }
bool dtype_ok(int t) { return t == K3KDA_F32 || t == K3KDA_BF16; }

// Host-side check of a host copy of cu_seqlens.
bool cu_ok(const int32_t *cu, int N, int T) {
    if (cu[0] != 0 || cu[N] != T) return false;
    for (int n = 0; n < N; ++n)
        if (cu[n + 1] < cu[n]) return false;
    return true;
}

// Host-side check of a host copy of a slot map: every entry in [0, num_slots), none repeated
// (two sequences updating one slot in the same call would race).
bool slots_ok(const int32_t *slot, int N, int num_slots) {
    if (num_slots < 1) return false;
    std::vector<unsigned char> seen((size_t)num_slots, 0);
    for (int n = 0; n < N; ++n) {
        const int32_t x = slot[n];
        if (x < 0 || x >= num_slots || seen[(size_t)x]) return false;
        seen[(size_t)x] = 1;
    }
    return true;
}
constexpr size_t kStatusBytes = 256;

size_t round256(size_t b) { return (b + 255) & ~size_t(255); }

size_t conv_buffer_bytes(int T, int H, int dk, int dv) {
    return round256((size_t)T * (2 * (size_t)H * dk + (size_t)H * dv) * sizeof(float));
}

}  // namespace

void k3kda::count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

namespace {
std::atomic<unsigned> g_test_timeout[kTestKinds];
}  // namespace

unsigned k3kda::take_test_timeout(int which) {
    return which >= 0 && which < kTestKinds ? g_test_timeout[which].exchange(0u) : 0u;
}

extern "C" {

long long k3kda_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

// Test hook (see TestTimeout in common.cuh): which = 0 the two-pass prefill's chunk scan, 1 the
// single-pass prefill, 2 the decode step, 3 the backward's chains (the forward chain of the first
// (sequence, head) issues no MMA for its first chunk); tries = how many times the starved wait
// polls (0 disarms).
// Only for tests on a working GPU: the armed call's outputs are invalid by design.
int k3kda_test_arm_wait_timeout(int which, unsigned tries) {
    if (which < 0 || which >= kTestKinds) return K3KDA_ERR_INVALID_ARG;
    g_test_timeout[which].store(tries);
    return K3KDA_OK;
}


const char *k3kda_status_string(int status) {
    switch (status) {
        case K3KDA_OK: return "K3KDA_OK";
        case K3KDA_ERR_INVALID_ARG: return "K3KDA_ERR_INVALID_ARG";
        case K3KDA_ERR_UNSUPPORTED: return "K3KDA_ERR_UNSUPPORTED";
        case K3KDA_ERR_ALIGNMENT: return "K3KDA_ERR_ALIGNMENT";
        case K3KDA_ERR_WORKSPACE: return "K3KDA_ERR_WORKSPACE";
        case K3KDA_ERR_CUDA: return "K3KDA_ERR_CUDA";
        case K3KDA_ERR_TIMEOUT: return "K3KDA_ERR_TIMEOUT";
        default: return "K3KDA_UNKNOWN_STATUS";
    }
}

int k3kda_version(void) { return K3KDA_VERSION; }

const char *k3kda_last_error(void) { return g_last_error; }

int k3kda_short_conv(const void *x, int x_dtype, const float *weight, float *conv_state,
                     const int32_t *cu_seqlens, int N, int T, int D, int W, int apply_silu,
                     void *out, int out_dtype, void *stream) {
    if (N < 1 || T < 0 || D < 1 || W < 1 || W > 4) return K3KDA_ERR_INVALID_ARG;
    if (!dtype_ok(x_dtype) || !dtype_ok(out_dtype)) return K3KDA_ERR_INVALID_ARG;
    if ((T > 0 && (!x || !out)) || !weight) return K3KDA_ERR_INVALID_ARG;
    if (cu_seqlens == nullptr && N != 1) return K3KDA_ERR_INVALID_ARG;
    if (x == out && x != nullptr) return K3KDA_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(out) || !aligned16(weight) || !aligned16(conv_state))
        return K3KDA_ERR_ALIGNMENT;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int st = cuda_status(launch_short_conv(x, x_dtype == K3KDA_BF16, weight, conv_state, cu_seqlens, N, T,
                                           D, W, apply_silu, out, out_dtype == K3KDA_BF16, s));
    if (st != K3KDA_OK || conv_state == nullptr) return st;
    return cuda_status(launch_conv_state_update(x, x_dtype == K3KDA_BF16, conv_state, cu_seqlens, N, T, D,
                                                W, s));
}

size_t k3kda_prefill_workspace_size(int N, int T, int H, int dk, int dv, int chunk, int in_dtype,
                                    int has_conv) {
    size_t b = kStatusBytes;
    if (N < 0 || T < 0 || H < 0 || dk < 0 || dv < 0) return b;
    if (tc_prefill_supported(in_dtype == K3KDA_BF16, dk, dv, chunk))
        return b + round256(tc_split_workspace(N, T, H));   // chunk records of the two-pass path
    if (has_conv) b += conv_buffer_bytes(T, H, dk, dv);
    return b;
}

size_t k3kda_prefill_workspace_min(int N, int T, int H, int dk, int dv, int chunk, int in_dtype,
                                   int has_conv) {
    if (N >= 0 && T >= 0 && H >= 0 && dk >= 0 && dv >= 0 &&
        tc_prefill_supported(in_dtype == K3KDA_BF16, dk, dv, chunk))
        return kStatusBytes + round256(tc_prefill_workspace(N, H));   // single-pass kernel
    return k3kda_prefill_workspace_size(N, T, H, dk, dv, chunk, in_dtype, has_conv);
}

static int prefill_impl(const void *q, const void *k, const void *v, int in_dtype, const float *g,
                        const float *beta, const float *initial_state, const int32_t *cu_seqlens,
                        const int32_t *cu_seqlens_host, int N, int T, int H, int dk, int dv, int chunk,
                        float scale, int use_qk_l2norm, const k3kda_conv_args *conv, const void *gate,
                        void *out, int out_dtype, float *final_state, void *workspace,
                        size_t workspace_bytes, void *stream, const int32_t *slot, int num_slots) {
    if (N < 1 || T < 0 || H < 1) return K3KDA_ERR_INVALID_ARG;
    if (!dtype_ok(in_dtype) || !dtype_ok(out_dtype)) return K3KDA_ERR_INVALID_ARG;
    if (!head_dim_ok(dk) || !head_dim_ok(dv)) return K3KDA_ERR_UNSUPPORTED;
    if (chunk != 16 && chunk != 32 && chunk != 64) return K3KDA_ERR_UNSUPPORTED;
    if (T > 0 && (!q || !k || !v || !g || !beta || !out)) return K3KDA_ERR_INVALID_ARG;
    if (cu_seqlens == nullptr && N != 1) return K3KDA_ERR_INVALID_ARG;
    if (cu_seqlens_host && !cu_ok(cu_seqlens_host, N, T)) return K3KDA_ERR_INVALID_ARG;
    if (conv && (!conv->weight || conv->W < 1 || conv->W > 4)) return K3KDA_ERR_INVALID_ARG;
    if ((long long)N * H * 4 > 0x7fffffffLL) return K3KDA_ERR_UNSUPPORTED;
    for (const void *p : {q, k, v, (const void *)g, (const void *)initial_state, gate, (const void *)out,
                          (const void *)final_state})
        if (!aligned16(p)) return K3KDA_ERR_ALIGNMENT;
    if (!aligned4(beta)) return K3KDA_ERR_ALIGNMENT;
    if (conv && (!aligned16(conv->weight) || !aligned16(conv->conv_state))) return K3KDA_ERR_ALIGNMENT;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return K3KDA_ERR_WORKSPACE;
    const size_t need = k3kda_prefill_workspace_min(N, T, H, dk, dv, chunk, in_dtype, conv != nullptr);
    if (workspace_bytes < need) return K3KDA_ERR_WORKSPACE;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    char *ws = static_cast<char *>(workspace);
    unsigned int *status = reinterpret_cast<unsigned int *>(ws);
    size_t off = kStatusBytes;

    PrefillArgs a{};
    a.q = q; a.k = k; a.v = v;
    a.q_row = (int64_t)H * dk; a.k_row = (int64_t)H * dk; a.v_row = (int64_t)H * dv;
    a.in_bf16 = in_dtype == K3KDA_BF16;
    a.g = g; a.beta = beta; a.S0 = initial_state; a.cu = cu_seqlens;
    a.N = N; a.T = T; a.H = H; a.dk = dk; a.dv = dv; a.chunk = chunk;
    a.scale = scale; a.l2 = use_qk_l2norm != 0;
    a.gate = gate; a.gate_bf16 = in_dtype == K3KDA_BF16; a.out = out; a.out_bf16 = out_dtype == K3KDA_BF16; a.Sfin = final_state;
    a.status = status;
    a.slot = slot;
    a.num_slots = num_slots;
    a.cu_host = cu_seqlens_host;

    if (tc_prefill_supported(a.in_bf16, dk, dv, chunk)) {
        const float *cw = conv ? conv->weight : nullptr;
        float *cst = conv ? conv->conv_state : nullptr;
        const int W = conv ? conv->W : 0;
        // two-pass path when the workspace holds the chunk records, else the single-pass kernel
        if (T > 0 && workspace_bytes - off >= tc_split_workspace(N, T, H))
            return cuda_status(launch_prefill_tc_split(a, cw, cst, W, ws + off, s));
        return cuda_status(launch_prefill_tc_fused(a, cw, cst, W, s));
    }
    if (conv) {
        // Conv stage: q, k, v channels convolved (+SiLU) into an fp32 [T, D] buffer in the
        // workspace, then the conv state is advanced; the chunked kernel reads that buffer.
        const int64_t Dq = (int64_t)H * dk, Dv = (int64_t)H * dv, D = 2 * Dq + Dv;
        float *buf = reinterpret_cast<float *>(ws + off);
        off += conv_buffer_bytes(T, H, dk, dv);
        const int W = conv->W;
        const void *src[3] = {q, k, v};
        const int64_t width[3] = {Dq, Dq, Dv}, choff[3] = {0, Dq, 2 * Dq};
        for (int i = 0; i < 3; ++i) {
            int st = cuda_status(launch_short_conv_strided(
                src[i], width[i], a.in_bf16, conv->weight + choff[i] * W,
                conv->conv_state ? conv->conv_state + choff[i] : nullptr, D, cu_seqlens, N, T, (int)width[i],
                W, 1, buf + choff[i], D, 0, s, slot, num_slots));
            if (st != K3KDA_OK) return st;
        }
        if (conv->conv_state)
            for (int i = 0; i < 3; ++i) {
                int st = cuda_status(launch_conv_state_update_strided(src[i], width[i], a.in_bf16,
                                                                      conv->conv_state + choff[i], D,
                                                                      cu_seqlens, N, T, (int)width[i], W, s,
                                                                      slot, num_slots));
                if (st != K3KDA_OK) return st;
            }
        a.q = buf; a.k = buf + Dq; a.v = buf + 2 * Dq;
        a.q_row = a.k_row = a.v_row = D;
        a.in_bf16 = 0;
    }
    if (T == 0 && final_state == nullptr) return K3KDA_OK;
    if (prefill_f32_smem_bytes(chunk, dk, dv) > 227 * 1024) return K3KDA_ERR_UNSUPPORTED;
    return cuda_status(launch_prefill_f32(a, s));
}

int k3kda_prefill(const void *q, const void *k, const void *v, int in_dtype, const float *g,
                  const float *beta, const float *initial_state, const int32_t *cu_seqlens,
                  const int32_t *cu_seqlens_host, int N, int T, int H, int dk, int dv, int chunk,
                  float scale, int use_qk_l2norm, const k3kda_conv_args *conv, const void *gate,
                  void *out, int out_dtype, float *final_state, void *workspace,
                  size_t workspace_bytes, void *stream) {
    return prefill_impl(q, k, v, in_dtype, g, beta, initial_state, cu_seqlens, cu_seqlens_host, N, T, H, dk, dv,
                        chunk, scale, use_qk_l2norm, conv, gate, out, out_dtype, final_state, workspace,
                        workspace_bytes, stream, nullptr, 0);
}

int k3kda_prefill_slots(const void *q, const void *k, const void *v, int in_dtype, const float *g,
                        const float *beta, float *state_pool, const int32_t *state_idx,
                        const int32_t *state_idx_host, int num_slots, const int32_t *cu_seqlens,
                        const int32_t *cu_seqlens_host, int N, int T, int H, int dk, int dv, int chunk,
                        float scale, int use_qk_l2norm, const k3kda_conv_args *conv, const void *gate,
                        void *out, int out_dtype, void *workspace, size_t workspace_bytes, void *stream) {
    if (N < 1 || num_slots < 1 || !state_pool || !state_idx) return K3KDA_ERR_INVALID_ARG;
    if ((long long)num_slots * H * 4 > 0x7fffffffLL) return K3KDA_ERR_UNSUPPORTED;
    if (!aligned4(state_idx)) return K3KDA_ERR_ALIGNMENT;
    if (state_idx_host && !slots_ok(state_idx_host, N, num_slots)) return K3KDA_ERR_INVALID_ARG;
    return prefill_impl(q, k, v, in_dtype, g, beta, state_pool, cu_seqlens, cu_seqlens_host, N, T, H, dk, dv,
                        chunk, scale, use_qk_l2norm, conv, gate, out, out_dtype, state_pool, workspace,
                        workspace_bytes, stream, state_idx, num_slots);
}

size_t k3kda_backward_workspace_size(int N, int T, int H, int dk, int dv) {
    if (N < 0 || T < 0 || H < 0 || dk != 128 || dv != 128) return kStatusBytes;
    return kStatusBytes + backward_chunked_workspace(N, T, H);
}

int k3kda_backward(const void *q, const void *k, const void *v, int in_dtype, const float *g, const float *beta,
                   const float *initial_state, const int32_t *cu_seqlens, const int32_t *cu_seqlens_host, int N,
                   int T, int H, int dk, int dv, float scale, const float *dO, const float *dS_final, float *dq,
                   float *dk_out, float *dv_out, float *dg, float *dbeta, float *dS0, void *workspace,
                   size_t workspace_bytes, void *stream) {
    if (N < 1 || T < 0 || H < 1) return K3KDA_ERR_INVALID_ARG;
    if (!dtype_ok(in_dtype)) return K3KDA_ERR_INVALID_ARG;
    if (dk != 128 || dv != 128) return K3KDA_ERR_UNSUPPORTED;
    if (T > 0 && (!q || !k || !v || !g || !beta || !dO || !dq || !dk_out || !dv_out || !dg || !dbeta))
        return K3KDA_ERR_INVALID_ARG;
    if (!dS0) return K3KDA_ERR_INVALID_ARG;
    if (cu_seqlens == nullptr && N != 1) return K3KDA_ERR_INVALID_ARG;
    if (cu_seqlens_host && !cu_ok(cu_seqlens_host, N, T)) return K3KDA_ERR_INVALID_ARG;
    // grids: 2 x (chunks of 16 tokens) x H items and N x H x 8 column blocks
    if ((long long)N * H * 8 > 0x7fffffffLL || 2 * ((long long)T / 16 + N + 1) * H > 0x7fffffffLL)
        return K3KDA_ERR_UNSUPPORTED;
    for (const void *p : {q, k, v, (const void *)g, (const void *)initial_state, (const void *)dO,
                          (const void *)dS_final, (const void *)dq, (const void *)dk_out, (const void *)dv_out,
                          (const void *)dg, (const void *)dS0})
        if (!aligned16(p)) return K3KDA_ERR_ALIGNMENT;
    if (!aligned4(beta) || !aligned4(dbeta)) return K3KDA_ERR_ALIGNMENT;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return K3KDA_ERR_WORKSPACE;
    if (workspace_bytes < k3kda_backward_workspace_size(N, T, H, dk, dv)) return K3KDA_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    char *ws = static_cast<char *>(workspace);
    return cuda_status(launch_backward_chunked(q, k, v, in_dtype == K3KDA_BF16, g, beta, initial_state, cu_seqlens, N, T, H,
                                       scale, dO, dS_final, dq, dk_out, dv_out, dg, dbeta, dS0,
                                       reinterpret_cast<unsigned *>(ws), ws + kStatusBytes, s));
}

int k3kda_workspace_status(void *workspace, void *stream) {
    if (!workspace) return K3KDA_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned int word = 0;
    int st = cuda_status(cudaMemcpyAsync(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost, s));
    if (st != K3KDA_OK) return st;
    st = cuda_status(cudaStreamSynchronize(s));
    if (st != K3KDA_OK) return st;
    if (word == 0) return K3KDA_OK;
    st = cuda_status(cudaMemsetAsync(workspace, 0, sizeof(word), s));
    if (st != K3KDA_OK) return st;
    st = cuda_status(cudaStreamSynchronize(s));
    return st != K3KDA_OK ? st : K3KDA_ERR_TIMEOUT;
}

int k3kda_decode_status(void *stream) {
    unsigned word = 0;
    const int st = cuda_status(decode_status(static_cast<cudaStream_t>(stream), &word));
    if (st != K3KDA_OK) return st;
    return word == 0 ? K3KDA_OK : K3KDA_ERR_TIMEOUT;
}

static int decode_impl(const void *q, const void *k, const void *v, int in_dtype, const float *g,
                       const float *beta, const void *gate, const float *conv_weight, float *conv_state,
                       float *state, int N, int H, int dk, int dv, int W, float scale, int use_qk_l2norm,
                       void *out, int out_dtype, void *stream, const int32_t *slot, int num_slots) {
    if (N < 0 || H < 1) return K3KDA_ERR_INVALID_ARG;
    if (!dtype_ok(in_dtype) || !dtype_ok(out_dtype)) return K3KDA_ERR_INVALID_ARG;
    if (!head_dim_ok(dk) || !head_dim_ok(dv)) return K3KDA_ERR_UNSUPPORTED;
    if (N > 0 && (!q || !k || !v || !g || !beta || !state || !out)) return K3KDA_ERR_INVALID_ARG;
    if (conv_weight && (W < 1 || W > 4 || (W > 1 && !conv_state))) return K3KDA_ERR_INVALID_ARG;
    if ((long long)N * H > 0x7fffffffLL) return K3KDA_ERR_UNSUPPORTED;
    for (const void *p : {q, k, v, (const void *)g, gate, (const void *)conv_weight, (const void *)conv_state,
                          (const void *)state, (const void *)out})
        if (!aligned16(p)) return K3KDA_ERR_ALIGNMENT;
    if (!aligned4(beta)) return K3KDA_ERR_ALIGNMENT;
    return cuda_status(launch_decode(q, k, v, in_dtype == K3KDA_BF16, g, beta, gate, conv_weight, conv_state,
                                     state, N, H, dk, dv, conv_weight ? W : 0, scale, use_qk_l2norm != 0, out,
                                     out_dtype == K3KDA_BF16, static_cast<cudaStream_t>(stream), slot, num_slots));
}

int k3kda_decode_step(const void *q, const void *k, const void *v, int in_dtype, const float *g,
                      const float *beta, const void *gate, const float *conv_weight, float *conv_state,
                      float *state, int N, int H, int dk, int dv, int W, float scale, int use_qk_l2norm,
                      void *out, int out_dtype, void *stream) {
    return decode_impl(q, k, v, in_dtype, g, beta, gate, conv_weight, conv_state, state, N, H, dk, dv, W, scale,
                       use_qk_l2norm, out, out_dtype, stream, nullptr, 0);
}

int k3kda_decode_step_slots(const void *q, const void *k, const void *v, int in_dtype, const float *g,
                            const float *beta, const void *gate, const float *conv_weight, float *conv_state_pool,
                            float *state_pool, const int32_t *state_idx, const int32_t *state_idx_host,
                            int num_slots, int N, int H, int dk, int dv, int W, float scale, int use_qk_l2norm,
                            void *out, int out_dtype, void *stream) {
    if (N < 0 || num_slots < 1 || (N > 0 && !state_idx)) return K3KDA_ERR_INVALID_ARG;
    if ((long long)num_slots * H > 0x7fffffffLL) return K3KDA_ERR_UNSUPPORTED;
    if (!aligned4(state_idx)) return K3KDA_ERR_ALIGNMENT;
    if (state_idx_host && !slots_ok(state_idx_host, N, num_slots)) return K3KDA_ERR_INVALID_ARG;
    return decode_impl(q, k, v, in_dtype, g, beta, gate, conv_weight, conv_state_pool, state_pool, N, H, dk, dv, W,
                       scale, use_qk_l2norm, out, out_dtype, stream, state_idx, num_slots);
}

size_t k3mla_decode_workspace_size(int N, int H, int dqk, int dv, int L_max) {
    if (N < 0 || H < 1 || dqk < 1 || dv < 1 || L_max < 1) return 0;
    return mla_workspace(N, H, dqk, dv, L_max);
}

static int mla_impl(const void *q, const void *k_new, const void *v_new, int in_dtype, const void *gate,
                    void *k_cache, void *v_cache, int cache_dtype, int32_t *cache_len, int N, int H, int dqk, int dv,
                    int L_max, int rope_dim, float rope_theta, float scale, void *out, int out_dtype, void *workspace,
                    size_t workspace_bytes, void *stream, const int32_t *slot, int num_slots) {
    if (N < 0 || H < 1 || L_max < 1) return K3KDA_ERR_INVALID_ARG;
    if (!dtype_ok(in_dtype) || !dtype_ok(cache_dtype) || !dtype_ok(out_dtype)) return K3KDA_ERR_INVALID_ARG;
    if (rope_dim < 0 || (rope_dim & 1) || rope_dim > dqk) return K3KDA_ERR_INVALID_ARG;
    if (rope_dim > 0 && !(rope_theta > 0.f)) return K3KDA_ERR_INVALID_ARG;
    if ((dqk != 64 && dqk != 128 && dqk != 192 && dqk != 256) || (dv != 64 && dv != 128 && dv != 256))
        return K3KDA_ERR_UNSUPPORTED;
    if ((long long)N * H * (long long)mla_splits(L_max) > 0x7fffffffLL) return K3KDA_ERR_UNSUPPORTED;
    if (N == 0) return K3KDA_OK;
    if (!q || !k_new || !v_new || !k_cache || !v_cache || !cache_len || !out) return K3KDA_ERR_INVALID_ARG;
    for (const void *p : {q, k_new, v_new, gate, (const void *)k_cache, (const void *)v_cache, (const void *)out})
        if (!aligned16(p)) return K3KDA_ERR_ALIGNMENT;
    if (!aligned4(cache_len)) return K3KDA_ERR_ALIGNMENT;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return K3KDA_ERR_WORKSPACE;
    if (workspace_bytes < mla_workspace(N, H, dqk, dv, L_max)) return K3KDA_ERR_WORKSPACE;
    return cuda_status(launch_mla_decode(q, k_new, v_new, in_dtype == K3KDA_BF16, gate, k_cache, v_cache,
                                         cache_dtype == K3KDA_BF16, cache_len, N, H, dqk, dv, L_max, rope_dim,
                                         rope_theta, scale, out, out_dtype == K3KDA_BF16, workspace,
                                         static_cast<cudaStream_t>(stream), slot, num_slots));
}

int k3mla_decode_step(const void *q, const void *k_new, const void *v_new, int in_dtype, const void *gate,
                      void *k_cache, void *v_cache, int cache_dtype, int32_t *cache_len, int N, int H, int dqk,
                      int dv, int L_max, int rope_dim, float rope_theta, float scale, void *out, int out_dtype,
                      void *workspace, size_t workspace_bytes, void *stream) {
    return mla_impl(q, k_new, v_new, in_dtype, gate, k_cache, v_cache, cache_dtype, cache_len, N, H, dqk, dv, L_max,
                    rope_dim, rope_theta, scale, out, out_dtype, workspace, workspace_bytes, stream, nullptr, 0);
}

int k3mla_decode_step_slots(const void *q, const void *k_new, const void *v_new, int in_dtype, const void *gate,
                            void *k_cache_pool, void *v_cache_pool, int cache_dtype, int32_t *cache_len_pool,
                            const int32_t *cache_idx, const int32_t *cache_idx_host, int num_slots, int N, int H,
                            int dqk, int dv, int L_max, int rope_dim, float rope_theta, float scale, void *out,
                            int out_dtype, void *workspace, size_t workspace_bytes, void *stream) {
    if (N < 0 || num_slots < 1 || (N > 0 && !cache_idx)) return K3KDA_ERR_INVALID_ARG;
    if ((long long)num_slots * H > 0x7fffffffLL) return K3KDA_ERR_UNSUPPORTED;
    if (!aligned4(cache_idx)) return K3KDA_ERR_ALIGNMENT;
    if (cache_idx_host && !slots_ok(cache_idx_host, N, num_slots)) return K3KDA_ERR_INVALID_ARG;
    return mla_impl(q, k_new, v_new, in_dtype, gate, k_cache_pool, v_cache_pool, cache_dtype, cache_len_pool, N, H,
                    dqk, dv, L_max, rope_dim, rope_theta, scale, out, out_dtype, workspace, workspace_bytes, stream,
                    cache_idx, num_slots);
}

}  // extern "C"

