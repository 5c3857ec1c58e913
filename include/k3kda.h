/*
 * k3kda.h -- C ABI of the GB300 (sm_103a) KDA mixer library (libk3kda.so).
 *
 * KDA (Kimi Delta Attention) is the linear-attention mixer of the Kimi K3 /
 * KimiLinear hybrid.  The pages this library follows name its pieces without
 * writing the equations out:
 *   - "Experimental Native Vulkan Backend for Kimi K3" (Hugging Face
 *     discussion #187), feature list: independent Q/K/V short convolutions,
 *     recurrent KDA state, KDA output gating;
 *   - metrale_model_arch::kimi_k3 docs: Structs KdaConfig (head dim 128, conv
 *     width 4 in production; tiny dims legal), KdaState (per-sequence state,
 *     both buffers FP32, read-modify-write); Constants KDA_L2_EPS (eps of the
 *     in-kernel q/k L2 norm); Functions kda_decode_token ("conv update then
 *     recurrent step"); Re-exports launch_k3_kda_decode_token (the decode
 *     launch over a caller-held device state);
 *   - mlite-k3 README ("What this repository is"): unsupported inputs fail
 *     explicitly rather than being approximated.
 * The recurrence itself is the gated delta rule, per sequence and head:
 *     S_t = (I - beta_t k_t k_t^T) Diag(exp(g_t)) S_{t-1} + beta_t k_t v_t^T
 *     o_t = scale * S_t^T q_t          (then o_t * sigmoid(gate_t) if gated)
 * with S in R^{dk x dv} kept in FP32.
 *
 * Entry points: the causal short conv, the chunked prefill (plain, slot-pooled, without a
 * workspace), the decode step (plain, slot-pooled), the gradients of the recurrence, and the
 * decode token of the hybrid's other layer kind, gated attention (k3mla_*), each described where
 * it is declared.
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers unless a name ends in _host.
 *     Every buffer is owned by the caller; the library allocates nothing and
 *     keeps no per-call state.  Layouts are dense row-major, last index
 *     fastest, with no padding.
 *   - Work is enqueued on `stream` (a cudaStream_t passed as void*; NULL =
 *     legacy default stream) and runs asynchronously; no entry point
 *     synchronises.  Inputs must stay alive until the stream reaches the work.
 *   - Every entry point returns a k3kda_status.  Arguments are checked on the
 *     host before anything is launched; an invalid call launches nothing and
 *     returns a negative status.  Nothing aborts, throws or prints.
 *   - Supported head dims: dk, dv in {16, 32, ..., 128} (multiples of 16),
 *     unless an entry point says otherwise (the backward takes 128, the
 *     attention calls their own widths).  Conv width W in {1, 2, 3, 4}.
 *     Chunk in {16, 32, 64}.
 *   - Element types: q, k, v and gate share one type (k3kda_dtype); g, beta,
 *     conv weights and all states are FP32.  Pointers must be 16-byte aligned,
 *     except beta, which needs 4-byte alignment (so token slices of it work).
 *   - The L2 norm is x * (sum_c x_c^2 + eps)^(-1/2) over dk with eps =
 *     K3KDA_L2_EPS; the pages name this constant but print no value (1e-6 is
 *     used, the default of the flash-linear-attention norm it is taken from).
 */
#ifndef K3KDA_H
#define K3KDA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define K3KDA_VERSION 1
#define K3KDA_L2_EPS 1e-6f

typedef enum {
    K3KDA_OK = 0,
    K3KDA_ERR_INVALID_ARG = -1,  /* null pointer, bad size, bad cu_seqlens        */
    K3KDA_ERR_UNSUPPORTED = -2,  /* legal but not implemented (e.g. dk = 200)     */
    K3KDA_ERR_ALIGNMENT = -3,    /* a pointer is not 16-byte aligned              */
    K3KDA_ERR_WORKSPACE = -4,    /* workspace missing or smaller than required    */
    K3KDA_ERR_CUDA = -5,         /* a CUDA launch or runtime call failed          */
    K3KDA_ERR_TIMEOUT = -6       /* a bounded in-kernel wait gave up (see below)  */
} k3kda_status;

typedef enum { K3KDA_F32 = 0, K3KDA_BF16 = 1 } k3kda_dtype;

/* Human-readable name of a status code (static string, never NULL). */
const char *k3kda_status_string(int status);

/* K3KDA_VERSION of the loaded library. */
int k3kda_version(void);

/* Number of CUDA kernels this library has launched in this process (all
 * entry points, all threads).  A diagnostic for launch accounting. */
long long k3kda_launch_count(void);

/* Text of the last CUDA error seen by this thread inside the library ("" if
 * none).  Valid until the next call from the same thread. */
const char *k3kda_last_error(void);

/*
 * k3kda_short_conv -- causal depthwise short convolution with SiLU
 * ("independent Q/K/V short convolutions", HF discussion #187 feature list;
 * width 4 in production, metrale KdaConfig).  For every packed sequence n
 * (tokens cu_seqlens[n] .. cu_seqlens[n+1]-1) and channel c:
 *     y[t, c] = act( sum_{i=0}^{W-1} weight[c, i] * x[t - (W-1) + i, c] )
 * where positions before the sequence start read conv_state[n, W-1+tau, c]
 * (tau < 0; rows are oldest first) or zero when conv_state is NULL, and act is
 * SiLU (z * sigmoid(z)) when apply_silu is nonzero, else the identity.  No bias.
 *
 *   x          [T, D]       x_dtype (F32 or BF16)
 *   weight     [D, W]       FP32; weight[c, W-1] multiplies the current token
 *   conv_state [N, W-1, D]  FP32, read-modify-write; NULL => zero history and
 *                           no state written.  On return row r holds the
 *                           pre-conv input at position L_n - (W-1) + r of
 *                           sequence n (older rows shift in when L_n < W-1).
 *   cu_seqlens [N+1]        int32 device; NULL allowed only when N == 1
 *   out        [T, D]       out_dtype; may not alias x
 * Errors: INVALID_ARG for N < 1, T < 0, D < 1, W outside 1..4, null x/weight/
 * out; ALIGNMENT when x/out/weight/conv_state are not 16-byte aligned.
 */
int k3kda_short_conv(const void *x, int x_dtype, const float *weight, float *conv_state,
                     const int32_t *cu_seqlens, int N, int T, int D, int W, int apply_silu,
                     void *out, int out_dtype, void *stream);

/* Optional fused short conv for k3kda_prefill: the q, k and v channels are
 * convolved (+SiLU) as one tensor of D = 2*H*dk + H*dv channels ordered
 * [q heads | k heads | v heads], with the k3kda_short_conv semantics above. */
typedef struct k3kda_conv_args {
    const float *weight;   /* [D, W] FP32, required                              */
    float *conv_state;     /* [N, W-1, D] FP32 read-modify-write, or NULL (zero) */
    int W;                 /* 1..4                                               */
} k3kda_conv_args;

/* Bytes of device workspace with which k3kda_prefill runs its fastest path for
 * these arguments (always a multiple of 256; at least 256, which holds the
 * device status word).  For the tensor-core shape (BF16, dk = dv = 128, chunk
 * 64) this is the two-pass path's chunk-record buffer, 148,480 bytes per
 * (64-token chunk, head) held at once: every chunk's record (about 2.3 KB per
 * token and head) when N*H > 64 or the sequences are short; with N*H <= 64 and
 * at least 128 chunks, at most three pipeline segments' worth (max(80,
 * chunks/64) chunks each), independent of T, plus 66 KB per sequence and head. */
size_t k3kda_prefill_workspace_size(int N, int T, int H, int dk, int dv, int chunk,
                                    int in_dtype, int has_conv);

/* The smallest workspace k3kda_prefill accepts for these arguments.  For the
 * tensor-core shape it is 256 bytes and selects the single-pass kernel (one
 * CTA per sequence and head); other shapes need what
 * k3kda_prefill_workspace_size returns. */
size_t k3kda_prefill_workspace_min(int N, int T, int H, int dk, int dv, int chunk,
                                   int in_dtype, int has_conv);

/*
 * k3kda_prefill -- chunked KDA prefill over packed variable-length sequences
 * (the "recurrent KDA state" of HF discussion #187, computed chunk by chunk;
 * the state is the FP32 KdaState of the metrale docs).  For each sequence n
 * and head h the recurrence above runs over the sequence's tokens starting
 * from initial_state[n, h] (zero if NULL), writing o for every token and the
 * last state to final_state[n, h].  State, conv history and chunking restart
 * at every cu_seqlens boundary; the last chunk of a sequence may be partial.
 *
 *   q, k           [T, H, dk]      in_dtype   (pre-conv when conv != NULL)
 *   v              [T, H, dv]      in_dtype
 *   g              [T, H, dk]      FP32 log-decay (alpha = exp(g); any g <= 0,
 *                                  however strong the decay: no exponent the
 *                                  kernels form can leave the fp32 range)
 *   beta           [T, H]          FP32
 *   initial_state  [N, H, dk, dv]  FP32 or NULL (zeros)
 *   cu_seqlens     [N+1]           int32 device, cu[0] = 0, non-decreasing,
 *                                  cu[N] = T; NULL allowed only when N == 1
 *   cu_seqlens_host[N+1]           optional host copy; when given it is
 *                                  validated (INVALID_ARG if malformed)
 *   chunk          16, 32 or 64 (the chunk length of the chunked form)
 *   scale          output scale (usually dk^-0.5)
 *   use_qk_l2norm  nonzero: L2-normalise q and k per (token, head) in kernel,
 *                  after the conv when there is one
 *   conv           NULL, or the fused q/k/v short conv + SiLU
 *   gate           [T, H, dv] in_dtype logits, or NULL (no output gate)
 *   out            [T, H, dv] out_dtype
 *   final_state    [N, H, dk, dv] FP32 or NULL; may alias initial_state
 *   workspace      device scratch of at least k3kda_prefill_workspace_min()
 *                  bytes (k3kda_prefill_workspace_size() for the fastest path),
 *                  256-byte aligned, its first 256 bytes zero on the first
 *                  use, exclusively owned by this call until it completes on
 *                  the stream
 * The fast paths (tensor cores, split-BF16 operands) run for in_dtype BF16,
 * dk = dv = 128, chunk 64: with the full workspace a two-pass scheme (a
 * chunk-prep kernel over every (chunk, head) on all SMs, then a scan kernel per
 * sequence and head that carries the state); with less, one single-pass kernel
 * per sequence and head.  Every other supported shape runs an FP32 CUDA-core
 * chunked kernel.  All compute the same chunked algebra.
 * Long inputs run the two passes as a pipeline of chunk segments whose records
 * go to a ring of buffers in the workspace.  With few (sequence, head) pairs
 * (N*H <= 64) and at least 128 chunks the whole pipeline is one cooperative
 * launch that takes every SM: N*H of its CTAs carry the states while the others
 * prepare the following segments, ordered by counters in the workspace (every
 * wait bounded); with many pairs each segment's prep is a programmatic
 * dependent of the previous segment's scan.  Everything runs on `stream`: the
 * library creates no stream or event, and calls on different streams are
 * independent (two cooperative launches run one after the other).
 * Errors: INVALID_ARG, UNSUPPORTED, ALIGNMENT, WORKSPACE, CUDA as above.
 * A bounded in-kernel wait that gives up records K3KDA_ERR_TIMEOUT in the
 * workspace status word (see k3kda_workspace_status) instead of hanging.
 */
int k3kda_prefill(const void *q, const void *k, const void *v, int in_dtype,
                  const float *g, const float *beta, const float *initial_state,
                  const int32_t *cu_seqlens, const int32_t *cu_seqlens_host,
                  int N, int T, int H, int dk, int dv, int chunk, float scale,
                  int use_qk_l2norm, const k3kda_conv_args *conv, const void *gate,
                  void *out, int out_dtype, float *final_state,
                  void *workspace, size_t workspace_bytes, void *stream);

/* Synchronise `stream`, read and clear the status word at the start of a
 * prefill workspace: K3KDA_OK, or K3KDA_ERR_TIMEOUT if a kernel that used this
 * workspace gave up a bounded wait (its outputs are then invalid). */
int k3kda_workspace_status(void *workspace, void *stream);

/*
 * Slot-indexed state pools (continuous batching).  A serving runtime keeps the
 * recurrent state of every live request in one FP32 pool and, per call, maps
 * the call's sequences onto pool slots ("HybridCache" slot identity; state
 * buffers FP32 and read-modify-write per the KdaState docs).  These two calls
 * are k3kda_prefill / k3kda_decode_step with that indirection:
 *   state_pool       [num_slots, H, dk, dv] FP32; sequence n starts from
 *                    state_pool[state_idx[n]] and its final state is written
 *                    back there (zero a slot before a new request's prefill)
 *   conv_state_pool  [num_slots, W-1, 2*H*dk + H*dv] FP32, likewise per slot
 *                    (for prefill: conv->conv_state is the pool)
 *   state_idx        [N] int32, device, 4-byte aligned
 *   state_idx_host   optional host copy: validated, INVALID_ARG when an entry
 *                    is outside [0, num_slots) or repeated
 * A device entry outside [0, num_slots) is never dereferenced: that sequence
 * runs from zero state and conv history, writes nothing to the pools, and a
 * decode writes a zero output row.  Repeated entries race (undefined result).
 * Other arguments, layouts, errors: as k3kda_prefill / k3kda_decode_step.
 */
int k3kda_prefill_slots(const void *q, const void *k, const void *v, int in_dtype,
                        const float *g, const float *beta, float *state_pool,
                        const int32_t *state_idx, const int32_t *state_idx_host, int num_slots,
                        const int32_t *cu_seqlens, const int32_t *cu_seqlens_host,
                        int N, int T, int H, int dk, int dv, int chunk, float scale,
                        int use_qk_l2norm, const k3kda_conv_args *conv, const void *gate,
                        void *out, int out_dtype, void *workspace, size_t workspace_bytes,
                        void *stream);

int k3kda_decode_step_slots(const void *q, const void *k, const void *v, int in_dtype,
                            const float *g, const float *beta, const void *gate,
                            const float *conv_weight, float *conv_state_pool, float *state_pool,
                            const int32_t *state_idx, const int32_t *state_idx_host, int num_slots,
                            int N, int H, int dk, int dv, int W, float scale, int use_qk_l2norm,
                            void *out, int out_dtype, void *stream);

/*
 * k3kda_prefill_noalloc -- k3kda_prefill for callers that cannot allocate
 * device memory where they call the mixer (inside an allocator or memory
 * pool, in runtimes that forbid cudaMalloc after start-up, in plug-ins that
 * are handed only their input and output buffers).  The pages have no
 * counterpart: this is a convenience of this library.
 *
 * Arguments and results are those of k3kda_prefill without the workspace:
 * the scratch comes from a 16 MiB device array that the library reserves
 * statically (K3KDA_NOALLOC_SCRATCH_BYTES); every GPU that loads the library
 * holds it until the process exits.  The call itself allocates nothing.
 *   - Work whose k3kda_prefill_workspace_min() exceeds the array (only the
 *     fp32 CUDA-core shapes with a fused conv need more than 256 bytes: their
 *     fp32 [T, 2*H*dk + H*dv] conv staging buffer) returns
 *     K3KDA_ERR_WORKSPACE before anything is enqueued.  Tensor-core shapes
 *     whose chunk records fit in the array run the two-pass path, larger ones
 *     the single-pass kernel.
 *   - Every call looks up the array's device address on the current device
 *     (the runtime resolves it per device and context; nothing is cached, so
 *     a device reset leaves no stale address).  Make the first call on a
 *     device before any stream capture.
 *   - All calls on a device share the one array and it keeps the last call's
 *     contents.  Each call clears the status word on `stream` before its
 *     kernels; calls whose work overlaps on the GPU (different streams, no
 *     ordering between them) race on the array.  A timed-out in-kernel wait is
 *     recorded in the array's status word: k3kda_prefill_noalloc_status reads it.
 */
#define K3KDA_NOALLOC_SCRATCH_BYTES (16u << 20)
int k3kda_prefill_noalloc(const void *q, const void *k, const void *v, int in_dtype,
                          const float *g, const float *beta, const float *initial_state,
                          const int32_t *cu_seqlens, const int32_t *cu_seqlens_host,
                          int N, int T, int H, int dk, int dv, int chunk, float scale,
                          int use_qk_l2norm, const k3kda_conv_args *conv, const void *gate,
                          void *out, int out_dtype, float *final_state, void *stream);

/* The status of the last k3kda_prefill_noalloc call on the current device:
 * synchronise `stream`, read and clear the status word of the library-held
 * array.  K3KDA_OK, or K3KDA_ERR_TIMEOUT if one of its kernels gave up a
 * bounded wait (its outputs are then invalid); K3KDA_ERR_CUDA on a runtime
 * error.  Allocates nothing.  The pages have no counterpart. */
int k3kda_prefill_noalloc_status(void *stream);

/*
 * k3kda_decode_step -- one new token for each of N independent sequences
 * ("One decode token: conv update then recurrent step", metrale kda_decode_token;
 * launch_k3_kda_decode_token over a KdaDeviceState).  Per sequence n and head h:
 *   1. conv: the token's pre-conv q, k, v channels are shifted into the conv
 *      window (conv_state rows are the previous W-1 inputs, oldest first),
 *      convolved with conv_weight and passed through SiLU; conv_state is
 *      updated in place to the newest W-1 inputs (skipped when conv_weight
 *      is NULL: q, k, v are used as given);
 *   2. q, k L2-normalised when use_qk_l2norm;
 *   3. S <- (I - beta k k^T) Diag(exp(g)) S + beta k v^T  in place (FP32);
 *   4. out = scale * S^T q, times sigmoid(gate) when gate != NULL.
 *
 *   q, k        [N, H, dk] in_dtype      v, gate [N, H, dv] in_dtype
 *   g           [N, H, dk] FP32           beta   [N, H] FP32
 *   conv_weight [2*H*dk + H*dv, W] FP32 or NULL;  conv_state [N, W-1, 2*H*dk + H*dv]
 *   state       [N, H, dk, dv] FP32, read-modify-write in place
 *   out         [N, H, dv] out_dtype
 * Errors: INVALID_ARG, UNSUPPORTED, ALIGNMENT, CUDA.  The decode takes no
 * workspace: a bounded in-kernel wait that gives up is recorded in a status
 * word the library keeps per device, which k3kda_decode_status reads.
 */
int k3kda_decode_step(const void *q, const void *k, const void *v, int in_dtype,
                      const float *g, const float *beta, const void *gate,
                      const float *conv_weight, float *conv_state, float *state,
                      int N, int H, int dk, int dv, int W, float scale, int use_qk_l2norm,
                      void *out, int out_dtype, void *stream);

/* Synchronise `stream`, read and clear the current device's decode status word:
 * K3KDA_OK, or K3KDA_ERR_TIMEOUT if a k3kda_decode_step / _slots kernel on
 * this device gave up a bounded wait since the last read (its outputs are then
 * invalid); K3KDA_ERR_CUDA on a runtime error.  Shared by every decode call on
 * the device (failure detection, no counterpart on the pages). */
int k3kda_decode_status(void *stream);

/* ---- backward of the recurrence ----
 * Reverse-mode gradients of the ungated KDA recurrence (the one k3kda_prefill runs, without
 * the conv, norm and gate around it; "native forward + backward" in the feature list of
 * "Experimental Native Vulkan Backend for Kimi K3", Hugging Face discussion #187):
 *     S_t = (I - beta_t k_t k_t^T) Diag(exp g_t) S_{t-1} + beta_t k_t v_t^T,   o_t = scale S_t^T q_t,
 * with S_0 = initial_state (zero when NULL) and state, chunking and everything else
 * restarting at every cu_seqlens boundary.  Given dO = dL/do [T, H, dv] and dS_final =
 * dL/dS_final [N, H, dk, dv] (zero when NULL) it writes dq, dk, dg [T, H, dk], dv [T, H, dv],
 * dbeta [T, H] and dS0 [N, H, dk, dv], all FP32.  q, k are used as given (apply the L2 norm's
 * and the conv's own derivatives around this call when they precede it).
 *
 *   q, k [T, H, dk], v [T, H, dv]  in_dtype;  g [T, H, dk], beta [T, H], dO [T, H, dv] FP32
 *   cu_seqlens: int32 [N+1] device, cu_seqlens_host: optional host copy (validated when given)
 * Only dk = dv = 128 (UNSUPPORTED otherwise).  FP32-accurate, in chunked form: the chunk algebra
 * of the recurrence (per 16-token chunk) differentiated, with one sequential pass over the chunks
 * for the states and one for the gradients reaching each chunk boundary (tensor-core MMAs on
 * operands split into two tf32 parts, three products each), and the per-token gradients of every
 * chunk computed in parallel on CUDA cores.  dbeta is zeroed and accumulated by the call.  A
 * bounded wait for the tensor cores that runs out sets the workspace's status word (see
 * k3kda_workspace_status).  Asynchronous on `stream`; the workspace
 * (k3kda_backward_workspace_size bytes, 256-byte aligned, caller-owned) is scratch only.
 * Errors: INVALID_ARG, UNSUPPORTED, ALIGNMENT (16 bytes for every array but beta, dbeta: 4),
 * WORKSPACE, CUDA. */
size_t k3kda_backward_workspace_size(int N, int T, int H, int dk, int dv);
int k3kda_backward(const void *q, const void *k, const void *v, int in_dtype,
                   const float *g, const float *beta, const float *initial_state,
                   const int32_t *cu_seqlens, const int32_t *cu_seqlens_host,
                   int N, int T, int H, int dk, int dv, float scale,
                   const float *dO, const float *dS_final,
                   float *dq, float *dk_out, float *dv_out, float *dg, float *dbeta, float *dS0,
                   void *workspace, size_t workspace_bytes, void *stream);

/* ---- Gated attention (MLA) layers: one decode token ------------------------------------------
 * The hybrid's other 24 layers (mlite-k3 README, "What this repository is": the 69 KDA +
 * 24 gated-MLA layer schedule) decode with metrale_model_arch::kimi_k3 docs, Functions:
 * mla_decode_token -- optional RoPE, append K/V, scaled dot-product attention, optional output
 * gate; the projections stay outside (Modules: mla, "gated NoPE MLA").  For every sequence n
 * and head h, with pos = cache_len[n] (tokens already cached):
 *   q' = RoPE(q, pos), k' = RoPE(k_new, pos)     (rotate-half on the first rope_dim dims; pair
 *        (i, i + rope_dim/2) turned by pos * rope_theta^(-2i/rope_dim); rope_dim = 0: NoPE)
 *   k_cache[n,h,pos] = k', v_cache[n,h,pos] = v_new  (stored in cache_dtype, bf16 rounded to
 *        nearest even)
 *   out[n,h] = softmax_j(scale * q' . k_cache[n,h,j], j = 0..pos) . v_cache[n,h,0..pos]
 *              (* sigmoid(gate[n,h]) when gate is given)
 *   cache_len[n] = pos + 1.
 * Layouts (row-major, contiguous): q, k_new [N, H, dqk]; v_new, gate, out [N, H, dv] (q, k_new,
 * v_new and gate in in_dtype, out in out_dtype); k_cache [N, H, L_max, dqk], v_cache
 * [N, H, L_max, dv] in cache_dtype (each (sequence, head) owns L_max contiguous rows); cache_len
 * int32 [N] in device memory, read and advanced by the call.  dqk in {64, 128, 192, 256}, dv in
 * {64, 128, 256} (UNSUPPORTED otherwise): keys may be wider than values, e.g. 128 rotation-free
 * dims and a 64-dim RoPE part.
 * A sequence whose cache is full (pos >= L_max) or whose length is negative gets NaN outputs;
 * its cache rows and length are left as they were (the length lives on the device, so this is
 * reported in the data, not in the status).
 * Ownership: every buffer is the caller's; the workspace (k3mla_decode_workspace_size bytes,
 * 256-byte aligned) is scratch.  Three kernel launches on `stream`, nothing synchronises.
 * Errors: INVALID_ARG (negative sizes, odd or too large rope_dim, rope_theta <= 0 with RoPE,
 * null pointers), UNSUPPORTED (dqk, dv, or N*H*ceil(L_max/512) above 2^31-1), ALIGNMENT (16 bytes for
 * every array but cache_len: 4), WORKSPACE, CUDA.  N = 0 returns OK without a launch. */
size_t k3mla_decode_workspace_size(int N, int H, int dqk, int dv, int L_max);
int k3mla_decode_step(const void *q, const void *k_new, const void *v_new, int in_dtype, const void *gate,
                      void *k_cache, void *v_cache, int cache_dtype, int32_t *cache_len,
                      int N, int H, int dqk, int dv, int L_max, int rope_dim, float rope_theta, float scale,
                      void *out, int out_dtype, void *workspace, size_t workspace_bytes, void *stream);

/* The same token step over a slot-indexed cache pool (continuous batching: the hybrid cache's
 * slot identity, as for the KDA state pools): sequence n reads and appends to slot cache_idx[n]
 * of k_cache_pool [num_slots, H, L_max, dqk], v_cache_pool [num_slots, H, L_max, dv] and
 * cache_len_pool int32 [num_slots]; q, k_new, v_new, gate and out stay indexed by n.  cache_idx is
 * int32 [N] in device memory; a sequence whose entry is outside [0, num_slots) gets NaN outputs
 * and writes nothing.  When cache_idx_host (a host copy) is given it is checked: every entry in
 * range and none repeated (two sequences appending to one slot would race), else INVALID_ARG.
 * The workspace is k3mla_decode_workspace_size(N, ...) bytes; errors as k3mla_decode_step. */
int k3mla_decode_step_slots(const void *q, const void *k_new, const void *v_new, int in_dtype, const void *gate,
                            void *k_cache_pool, void *v_cache_pool, int cache_dtype, int32_t *cache_len_pool,
                            const int32_t *cache_idx, const int32_t *cache_idx_host, int num_slots,
                            int N, int H, int dqk, int dv, int L_max, int rope_dim, float rope_theta, float scale,
                            void *out, int out_dtype, void *workspace, size_t workspace_bytes, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* K3KDA_H */
