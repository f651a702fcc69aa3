/*
 * gdn.h -- C ABI of the gated delta rule kernels (sm_103a).
 *
 * The gated delta rule is the recurrence inside the Gated DeltaNet mixer of
 * the Qwen3.5 and Qwen3-Next hybrid models (qwen3_5_text page, Notes -> "The
 * DeltaNet mixer"; qwen3_next page, Notes -> "The DeltaNet mixer fuses its
 * projections per key head").  Per value head h it keeps a state S of shape
 * [key_dim][value_dim] and, for every token t,
 *
 *     q~ = l2norm(q_t) * scale      k^ = l2norm(k_t)    (scale = key_dim^-1/2)
 *     S  <- exp(g_t) * S
 *     u   = beta_t * (v_t - S^T k^)
 *     S  <- S + k^ u^T
 *     o_t = S^T q~
 *
 * Value head h reads key head h / (HV / HK): queries and keys are
 * repeat_interleave'd up to the value heads, heads 2j and 2j+1 being copies of
 * key head j on a 2:1 model (same passages).  l2norm(x) = x / sqrt(sum x^2 +
 * 1e-6) (the pages give no epsilon; this is the reading taken).
 *
 * Argument names follow the pages' linear_attn value table (qwen3_5_text page,
 * "02 . support() -> Values, by host"): queries, keys, values, decays, beta,
 * initial state ("state_input ... or None at the start of a prompt (a copy of
 * the cache's buffer)"), outputs ("attention_head_outputs") and the final
 * state ("state_output"), with the layouts given there:
 *
 *     queries, keys  [batch, seq, key_heads,   key_dim]    (LinearQK)
 *     values, out    [batch, seq, value_heads, value_dim]  (LinearV)
 *     decays, beta   [batch, seq, value_heads]             (Gates, float32)
 *     state          [batch, value_heads, key_dim, value_dim]  float32
 *     states         [batch, seq, value_heads, key_dim, value_dim]  float32
 *
 * All tensors are dense, row-major (last index fastest) and on the device.
 * decays are natural-log decays (exp(g) of the state is kept), finite and
 * <= 0 (qwen3_next page: "float32, at most 0"); they are not validated.
 *
 * Conventions of every entry point:
 *   - Every pointer argument that names a tensor is a DEVICE pointer of the
 *     current CUDA device, 16-byte aligned.  The caller owns every buffer; the
 *     library allocates no device memory and keeps no state between calls
 *     (the one exception is gdn_prefill_noalloc's fixed scratch array, a
 *     static part of the library's device image, described there).
 *   - Work is enqueued on `cuda_stream` (a cudaStream_t; NULL = legacy default
 *     stream) and runs asynchronously; the call returns after enqueueing.
 *   - A negative return is an error detected before anything was enqueued
 *     (bad arguments), except GDN_ERR_CUDA, which reports a failed launch.
 *     Errors found in device data (a malformed cu_seqlens) are written to the
 *     status word at the start of the workspace; read it with
 *     gdn_workspace_status().  No entry point traps or aborts.
 *   - Supported shapes: key_dim = value_dim in {32, 64, 128} (every model on
 *     the pages has 128 x 128 heads); value_heads a multiple of key_heads;
 *     dtype GDN_BF16 or GDN_F32 for queries, keys, values and out (decays,
 *     beta and states are always float32).
 */
#ifndef GDN_H
#define GDN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GDN_OK = 0,
    GDN_ERR_INVALID_ARG = -1,   /* null pointer, negative size, HV % HK != 0, ... */
    GDN_ERR_UNSUPPORTED = -2,   /* key_dim / value_dim / dtype not supported       */
    GDN_ERR_MISALIGNED = -3,    /* a tensor pointer is not 16-byte aligned         */
    GDN_ERR_WORKSPACE = -4,     /* workspace NULL or smaller than required         */
    GDN_ERR_CUDA = -5,          /* a CUDA launch or runtime call failed            */
    GDN_ERR_TIMEOUT = -6,       /* a bounded device-side wait gave up (status word) */
    GDN_ERR_BAD_SEQLENS = -7    /* cu_seqlens not 0 = c0 <= c1 <= ... <= cN = T     */
} gdn_status;

typedef enum { GDN_BF16 = 0, GDN_F32 = 1 } gdn_dtype;

/* Layout of the projections feeding gdn_conv_gate_prologue */
typedef enum {
    GDN_LAYOUT_QKV = 0,   /* in_proj_qkv: the cat(q, k, v) channels; in_proj_b, in_proj_a */
    GDN_LAYOUT_QKVZ = 1   /* in_proj_qkvz / in_proj_ba grouped per key head (Qwen3-Next)  */
} gdn_proj_layout;

/*
 * Chunked prefill over a batch of equal-length sequences ("a prompt's chunked
 * one", linear_attn value table).  Runs the rule over every (batch row, value
 * head) from `initial_state` (NULL = zeros, the start of a prompt) and writes
 * the per-token outputs, the final state and, if `states` is not NULL, the
 * state after every token (the pages' `states`, num_v_heads x key_dim x
 * value_dim float32 per token; qwen3_5_text page, Notes -> "Loading").
 *
 *   queries, keys   [B, T, HK, Dk]   dtype
 *   values          [B, T, HV, Dv]   dtype
 *   decays, beta    [B, T, HV]       float32
 *   initial_state   [B, HV, Dk, Dv]  float32 or NULL
 *   out             [B, T, HV, Dv]   dtype
 *   final_state     [B, HV, Dk, Dv]  float32; may equal initial_state (the
 *                                    cache continued in place); other overlap
 *                                    is not allowed
 *   states          [B, T, HV, Dk, Dv] float32 or NULL (16-byte alignment
 *                   suffices; at 32 bytes the kernels write whole sectors)
 *   scale           multiplier of the normalised queries; <= 0 -> Dk^-1/2
 *   use_qk_l2norm   1: l2-normalise queries and keys in the kernel (the
 *                   model's convention); 0: use them as given
 *   workspace       device scratch of gdn_prefill_workspace_size(B*T, B, HV,
 *                   Dk, Dv) bytes, 256-byte aligned; owned by the caller; it
 *                   must not be used by another call still running.
 * B == 0 or T == 0 is allowed: the final state is then the initial state.
 */
int gdn_prefill(const void *queries, const void *keys, const void *values,
                const float *decays, const float *beta, const float *initial_state,
                void *out, float *final_state, float *states,
                int B, int T, int HK, int HV, int Dk, int Dv, gdn_dtype dtype,
                float scale, int use_qk_l2norm,
                void *workspace, size_t workspace_bytes, void *cuda_stream);

/*
 * Chunked prefill over N sequences packed back to back (batch 1, T_total
 * tokens), sequence i owning tokens [cu_seqlens[i], cu_seqlens[i+1]) -- the
 * cu_seqlens packing convention the pages use for per-image attention
 * (qwen3_5_text page, vision notes).  Chunks restart at every sequence start,
 * so the result equals N separate prefills.  Zero-length sequences are
 * allowed (their final state is their initial state).
 *
 *   queries, keys   [T_total, HK, Dk]    values, out  [T_total, HV, Dv]
 *   decays, beta    [T_total, HV]
 *   cu_seqlens      device int32 [N + 1]; must satisfy 0 = c0 <= ... <= cN =
 *                   T_total, checked on the device: a violation sets
 *                   GDN_ERR_BAD_SEQLENS in the workspace status word and the
 *                   kernels then write nothing
 *   initial_state   [N, HV, Dk, Dv] or NULL      final_state [N, HV, Dk, Dv]
 *   states          [T_total, HV, Dk, Dv] or NULL
 *   workspace       gdn_prefill_workspace_size(T_total, N, HV, Dk, Dv) bytes
 */
int gdn_prefill_varlen(const void *queries, const void *keys, const void *values,
                       const float *decays, const float *beta, const float *initial_state,
                       void *out, float *final_state, float *states,
                       const int32_t *cu_seqlens, int N, int T_total,
                       int HK, int HV, int Dk, int Dv, gdn_dtype dtype,
                       float scale, int use_qk_l2norm,
                       void *workspace, size_t workspace_bytes, void *cuda_stream);

/*
 * gdn_prefill / gdn_prefill_varlen followed by the gated RMS norm of the mixer output
 * (see gdn_gated_rmsnorm below for the definition), in one call on one stream: `out`
 * receives norm(y, gate=silu(gate_z)) * norm_weight.  The norm kernel runs over the
 * prefill's output in place (the faster of the designs measured: forming the norm inside
 * the prefill's sequential kernel made that kernel's output warps its bottleneck).
 *   gate_z       [B, T, HV, Dv] (packed: [1, T_total, HV, Dv]) dtype of values
 *   norm_weight  [Dv] float32;  norm_eps finite and >= 0
 * Everything else (arguments, states, workspace, errors) as gdn_prefill /
 * gdn_prefill_varlen; gate_z or norm_weight NULL, or a bad norm_eps, is
 * GDN_ERR_INVALID_ARG.
 */
int gdn_prefill_gated(const void *queries, const void *keys, const void *values,
                      const float *decays, const float *beta, const float *initial_state,
                      void *out, float *final_state, float *states,
                      const void *gate_z, const float *norm_weight, float norm_eps,
                      int B, int T, int HK, int HV, int Dk, int Dv, gdn_dtype dtype,
                      float scale, int use_qk_l2norm,
                      void *workspace, size_t workspace_bytes, void *cuda_stream);
int gdn_prefill_varlen_gated(const void *queries, const void *keys, const void *values,
                             const float *decays, const float *beta,
                             const float *initial_state, void *out, float *final_state,
                             float *states, const void *gate_z, const float *norm_weight,
                             float norm_eps, const int32_t *cu_seqlens, int N, int T_total,
                             int HK, int HV, int Dk, int Dv, gdn_dtype dtype, float scale,
                             int use_qk_l2norm, void *workspace, size_t workspace_bytes,
                             void *cuda_stream);

/*
 * One decode step ("a decode step's recurrent one", linear_attn value
 * table): one token per sequence, continuing the cache's state in place.
 *
 *   queries, keys   [B, HK, Dk]      dtype
 *   values          [B, HV, Dv]      dtype
 *   decays, beta    [B, HV]          float32
 *   state           [B, HV, Dk, Dv]  float32, read and overwritten in place
 *   out             [B, HV, Dv]      dtype
 * Needs no workspace.  B == 0 is allowed (nothing is done).
 */
int gdn_decode_step(const void *queries, const void *keys, const void *values,
                    const float *decays, const float *beta,
                    float *state, void *out,
                    int B, int HK, int HV, int Dk, int Dv, gdn_dtype dtype,
                    float scale, int use_qk_l2norm, void *cuda_stream);

/*
 * The step before the rule in the mixer (qwen3_5_text page, Notes -> "The DeltaNet
 * mixer"; qwen3_next page, Notes -> "The DeltaNet mixer fuses its projections per key
 * head"), writing the rule's inputs:
 *
 *     queries, keys, values = split(silu(conv1d(cat(q, k, v))))   causal, width 4
 *     beta   = sigmoid(b)
 *     decays = -exp(A_log) * softplus(a + dt_bias)
 *
 * conv1d is the depthwise Conv1d of the pages' module listings (kernel_size 4, padding 3,
 * groups = channels, no bias), causal: channel c at token t is
 * sum_{i=0..3} conv_weight[c][i] * x_{t-3+i}[c].  C = 2*HK*Dk + HV*Dv channels in the
 * order q (head-major), k, v.
 *
 *   layout GDN_LAYOUT_QKV (Qwen3.5):
 *     proj    [T_total, C] dtype       in_proj_qkv output
 *     proj_b  [T_total, HV] dtype      in_proj_b output;  proj_a [T_total, HV] in_proj_a
 *   layout GDN_LAYOUT_QKVZ (Qwen3-Next), regrouped on the fly:
 *     proj    [T_total, HK*(2*Dk + 2*r*Dv)] dtype, r = HV/HK: per key head its query,
 *             its key, the values of its r value heads, then their output gates
 *     proj_b  [T_total, HK*2*r] dtype: per key head the r value heads' b, then their a;
 *     proj_a  unused (NULL)
 *     gate_z  [T_total, HV, Dv] dtype receives the output gates z (for the gated norm),
 *             or NULL
 *   conv_weight  [C, 4] float32 (a Conv1d weight [C, 1, 4]; tap 3 is the current token)
 *   A_log, dt_bias [HV] float32
 *   conv_state_in  [N, 3, C] dtype: the three inputs before each sequence, oldest first
 *                  (a prompt's continuation, or the decode cache), or NULL (zeros: the
 *                  start of a prompt)
 *   conv_state_out [N, 3, C] dtype: the three inputs before the token after each
 *                  sequence, or NULL; may be conv_state_in (updated in place)
 *   cu_seqlens     [N+1] int32 device token offsets, or NULL: N sequences of
 *                  T_total / N tokens (a decode step is N sequences of one token)
 *   queries, keys  [T_total, HK, Dk] dtype;  values [T_total, HV, Dv] dtype
 *   beta, decays   [T_total, HV] float32
 * Dk = Dv in {32, 64, 128}; HV % HK == 0.  T_total == 0 with conv_state_out copies the
 * states.  All pointers 16-byte aligned, tensors contiguous.
 * Errors: GDN_ERR_INVALID_ARG (null pointer, bad sizes, T_total % N != 0 without
 * cu_seqlens), GDN_ERR_UNSUPPORTED, GDN_ERR_MISALIGNED, GDN_ERR_CUDA.  cu_seqlens is not
 * validated on the device: it must be nondecreasing from 0 to T_total.
 */
int gdn_conv_gate_prologue(const void *proj, const void *proj_b, const void *proj_a,
                           gdn_proj_layout layout, const float *conv_weight,
                           const float *A_log, const float *dt_bias,
                           const void *conv_state_in, void *conv_state_out,
                           const int32_t *cu_seqlens, int N, int64_t T_total,
                           int HK, int HV, int Dk, int Dv, gdn_dtype dtype,
                           void *queries, void *keys, void *values, void *gate_z,
                           float *beta, float *decays, void *cuda_stream);

/*
 * Gated RMS norm of the mixer output, the step that follows the rule in the mixer
 * (qwen3_5_text page, Notes -> "The DeltaNet mixer": out = out_proj(norm(y,
 * gate=silu(z))), "gain: weight"; the DeltaNet's own output norm multiplies by its
 * weight, not by 1 + weight, Notes -> "The readout is the plain projection").  For each
 * row of Dv values (one token of one value head):
 *
 *     out_c = y_c / sqrt(mean_c(y^2) + norm_eps) * norm_weight_c * silu(gate_z_c)
 *
 * The pages give no epsilon (1e-6 is the usual choice) and do not spell out the order
 * inside norm(): the gate multiplies after the norm and the gain.
 *   y, gate_z, out  [rows, Dv]  dtype, contiguous; out may be y (in place)
 *   norm_weight     [Dv]        float32, shared by all heads
 * Dv in {32, 64, 128}.  rows == 0 is allowed.  norm_eps must be finite and >= 0.
 * Errors: GDN_ERR_INVALID_ARG (null pointer, rows < 0, bad eps), GDN_ERR_UNSUPPORTED
 * (Dv, dtype), GDN_ERR_MISALIGNED (a pointer not 16-byte aligned), GDN_ERR_CUDA.
 */
int gdn_gated_rmsnorm(const void *y, const void *gate_z, const float *norm_weight, void *out,
                      int64_t rows, int Dv, gdn_dtype dtype, float norm_eps, void *cuda_stream);

/*
 * gdn_decode_step with the gated RMS norm above fused into the same kernel: `out`
 * receives norm(y, gate=silu(gate_z)) * norm_weight, formed from the fp32 y of the whole
 * head (y itself is never rounded to dtype or written).
 *   gate_z       [B, HV, Dv]  dtype
 *   norm_weight  [Dv]         float32
 * Everything else (arguments, in-place state, errors) as gdn_decode_step; gate_z or
 * norm_weight NULL, or a negative or non-finite norm_eps, is GDN_ERR_INVALID_ARG.
 */
int gdn_decode_step_gated(const void *queries, const void *keys, const void *values,
                          const float *decays, const float *beta,
                          float *state, void *out,
                          const void *gate_z, const float *norm_weight, float norm_eps,
                          int B, int HK, int HV, int Dk, int Dv, gdn_dtype dtype,
                          float scale, int use_qk_l2norm, void *cuda_stream);

/*
 * gdn_prefill for callers that cannot allocate device memory (no counterpart on the
 * pages: it exists for deployments, not for the method).  Engines that carve up
 * device memory once in their own pool, plugins that only see the buffers their
 * host hands them, and paths where an allocation (and the device synchronisation it
 * may cause) is not allowed can call this instead: it takes no workspace and uses a
 * scratch array of 64 MiB that the library keeps in device memory.
 *
 *   Arguments, layouts, results and error codes are those of gdn_prefill, minus the
 *   workspace.  Shapes whose scratch would exceed 64 MiB are rejected with
 *   GDN_ERR_WORKSPACE (for 128 x 128 bf16 heads a record is 58 KiB per 64-token chunk
 *   and value head: B * ceil(T / 64) * HV records must fit, at most 1129 of them, e.g.
 *   T = 2240 tokens at 32 value heads uses 66.5 MB).
 *   - The array is a file-scope __device__ variable: every GPU that loads the
 *     library holds its 64 MiB until the process exits.
 *   - The first call on each device looks up the array's device address (with that
 *     device current) and caches it; make that first call before any stream capture.
 *     A lookup that fails is not cached: the next call tries again.
 *   - All calls share the one array and it keeps the last call's contents; the call
 *     clears the status word it reads, everything else is written before it is read.
 *     Calls whose GPU work overlaps (two streams, two host threads) race on it: order
 *     them on one stream or serialise them.
 *   - Errors found on the device (a bounded wait that timed out) go to the status word
 *     at the start of the array; read it with gdn_prefill_noalloc_status() before the
 *     next call clears it.  gdn_workspace_status() does not apply (there is no caller
 *     workspace).
 * No cudaMalloc, cudaFree or allocating library routine is called.
 */
int gdn_prefill_noalloc(const void *queries, const void *keys, const void *values,
                        const float *decays, const float *beta, const float *initial_state,
                        void *out, float *final_state, float *states,
                        int B, int T, int HK, int HV, int Dk, int Dv, gdn_dtype dtype,
                        float scale, int use_qk_l2norm, void *cuda_stream);

/*
 * The device status word of the last gdn_prefill_noalloc on the current device: GDN_OK
 * or the GDN_ERR_* code its kernels recorded (GDN_ERR_TIMEOUT for a bounded wait that
 * gave up).  Enqueues a 4-byte copy on `cuda_stream` (the stream the prefill ran on) and
 * waits for that stream.  Returns GDN_OK, GDN_ERR_INVALID_ARG for a null `status`, or
 * GDN_ERR_CUDA when the copy fails.  Allocates nothing.
 */
int gdn_prefill_noalloc_status(void *cuda_stream, int *status);

/*
 * Layout of the recurrent state buffer [batch, value_heads, key_dim,
 * value_dim] float32, row = key index, column = value index (the pages'
 * State layout).  The kernels use this layout internally too, so a cache
 * buffer of this layout is passed to them as is.  Host-only; never fails
 * for positive sizes.
 */
typedef struct {
    size_t bytes;          /* total bytes for `batch` states                    */
    size_t bytes_per_head; /* key_dim * value_dim * 4                           */
    int64_t stride[4];     /* element strides of [batch, head, key, value]      */
    int64_t shape[4];
    int alignment;         /* required pointer alignment in bytes (16)          */
} gdn_state_layout_t;

int gdn_state_layout(int batch, int HV, int Dk, int Dv, gdn_state_layout_t *layout);

/*
 * Bytes of device workspace gdn_prefill / gdn_prefill_varlen need for
 * `T_total` tokens in `n_seqs` sequences (B for gdn_prefill), whatever the dtype
 * (the larger of the two paths' needs).  Host-only.  Returns 0 for invalid sizes.
 */
size_t gdn_prefill_workspace_size(int64_t T_total, int n_seqs, int HV, int Dk, int Dv);

/*
 * The same for a given dtype: exactly what the path that shape and dtype take needs
 * (128 x 128 bf16 heads take the tensor-core path, 58 KiB per (chunk, value head);
 * the other shapes and fp32 the CUDA-core path, 4 * (64 (Dk + Dv + 64) + 320) bytes;
 * either path also a 4-byte flag per (chunk, value head) and a few KiB of header).
 * A workspace of this size is accepted by calls with that dtype.  Host-only.
 * Returns 0 for invalid sizes or dtype.
 */
size_t gdn_prefill_workspace_size_for(int64_t T_total, int n_seqs, int HV, int Dk, int Dv,
                                      gdn_dtype dtype);

/*
 * Read the device status word a prefill wrote into `workspace`: GDN_OK, or
 * the GDN_ERR_* code of an error found in device data.  Enqueues a 4-byte
 * copy on `cuda_stream` and waits for that stream.  Returns GDN_OK or
 * GDN_ERR_CUDA / GDN_ERR_INVALID_ARG for the read itself.
 */
int gdn_workspace_status(const void *workspace, void *cuda_stream, int *status);

/* Static description of a status code (never NULL). */
const char *gdn_status_string(int status);

/* ABI version: major * 10000 + minor * 100 + patch. */
int gdn_abi_version(void);

/*
 * Self-test of the bounded waits (no counterpart on the pages: failure handling of this
 * library).  Every wait of the tensor-core kernels on an mbarrier phase gives up after a
 * time limit and records GDN_ERR_TIMEOUT instead of hanging.  This call launches one
 * thread on `cuda_stream` that waits, with the same helper, on a phase that nothing
 * completes, for `limit_ns` nanoseconds (1 ns .. 2 s), then writes status[0] =
 * GDN_ERR_TIMEOUT (or GDN_OK, which would mean the wait returned without the phase
 * completing, i.e. a broken wait) and status[1] = the microseconds it waited.  `status`
 * is a device pointer to two int32 owned by the caller (4-byte aligned).  Returns
 * GDN_ERR_INVALID_ARG / GDN_ERR_MISALIGNED for bad arguments, GDN_ERR_CUDA if the
 * launch fails, otherwise GDN_OK (asynchronous: read status after synchronising).
 */
int gdn_selftest_wait_timeout(int32_t *status, uint64_t limit_ns, void *cuda_stream);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H */
