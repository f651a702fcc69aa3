// gdn_internal.cuh -- shared definitions of the CUDA path (not part of the ABI).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "gdn.h"

namespace gdn {

constexpr int kChunk = 64;            // tokens per chunk of the chunked prefill
constexpr float kL2Eps = 1e-6f;       // l2norm(x) = x / sqrt(sum x^2 + eps)

// Workspace header: status words, then one flag word per chain of the tensor-core path,
// then the chunk table of a packed batch.
constexpr size_t kWsHeader = 256;     // int32 status[64]: [0] status, [1] number of chunks,
                                      // [2] work units claimed by the chain kernel, [3] prep
                                      // items claimed below the limit, [4] prep CTAs that stay
                                      // beside the chain, [5] prep items claimed past the limit
enum { kStatusWord = 0, kChunkCountWord = 1, kClaimWord = 2, kPrepClaimWord = 3, kPrepStayWord = 4,
       kPrepClaimPastWord = 5 };
// value slices per (sequence, value head) chain of the tensor-core prefill
constexpr int kChainSlices = 4;
// bytes of the chain flag words (one per (sequence, value head, value slice)), 256-aligned;
// zero before the chain kernel runs, like the status words
inline size_t chain_flag_bytes(int n_seqs, int HV) {
    return ((size_t)n_seqs * HV * kChainSlices * sizeof(int32_t) + 255) / 256 * 256;
}

// bytes of the record-ready flags (one per (chunk, value head)), 256-aligned: with the
// prep running beside the chain, the chain takes a record once its flag is set
inline size_t ready_flag_bytes(int max_chunks, int HV) {
    return ((size_t)max_chunks * HV * sizeof(int32_t) + 255) / 256 * 256;
}

// Everything a prefill launch needs; passed by value to the kernels.
struct PrefillParams {
    const void *q, *k, *v;        // [T_total, HK, Dk], [T_total, HV, Dv]
    const float *g, *beta;        // [T_total, HV]
    const float *s0;              // [N, HV, Dk, Dv] or null
    void *out;                    // [T_total, HV, Dv]
    float *s_final;               // [N, HV, Dk, Dv]
    float *states;                // [T_total, HV, Dk, Dv] or null
    const int32_t *cu_seqlens;    // [N+1] or null (equal lengths T_seq)
    int N, T_seq;
    int64_t T_total;
    int HK, HV, Dk, Dv;
    float scale;
    int l2norm;
    int max_chunks;               // grid bound on chunks
    int32_t *status;              // workspace status words
    int32_t *chunk_seq;           // [max_chunks] sequence of chunk (packed batches)
    int32_t *chunk_first;         // [N + 1] first chunk of each sequence (packed batches)
    int32_t *seq_order;           // [N] sequences by decreasing chunk count (packed batches)
    int32_t *chain_flags;         // [N * HV * kChainSlices] (tensor-core chain hand-offs)
    int32_t *ready;               // [max_chunks * HV] record-ready flags (tensor-core path)
    float *rec;                   // per (chunk, value head) records of the prep pass
    size_t rec_floats;            // floats per record
};

// Record of one (chunk, value head) written by the prep pass (all float32):
//   W    [C][Dk]  = T diag(beta * gamma * rk) K       (rows t >= len are zero)
//   Ut   [C][Dv]  = T diag(beta) V
//   P    [C][C]   = e^{G_t - G_j} rq_t rk_j (q_t . k_j) for j <= t, else 0
//   qd   [C]      = rq_t * gamma_t            kd [C] = rk_t e^{G_last - G_t}
//   rk   [C]      = key normaliser            alpha [C] = e^{g_t}
//   misc [C]      = { gamma_last, ... }
inline size_t record_floats(int Dk, int Dv) {
    return (size_t)kChunk * (Dk + Dv + kChunk) + 5 * kChunk;
}

size_t prefill_workspace_bytes(int64_t T_total, int n_seqs, int HV, int Dk, int Dv);
size_t prefill_workspace_bytes_for(int64_t T_total, int n_seqs, int HV, int Dk, int Dv, gdn_dtype dtype);
int max_chunks_for(int64_t T_total, int n_seqs, bool packed, int T_seq);

// Launchers (return cudaError_t of the launches).
cudaError_t launch_prefill_generic(const PrefillParams &p, gdn_dtype dtype, cudaStream_t st);
cudaError_t launch_chunk_table(const PrefillParams &p, cudaStream_t st);
// Tensor-core path (key_dim = value_dim = 128, bf16): prep + chain kernels.
bool tc_supported(int Dk, int Dv, gdn_dtype dtype);
size_t tc_record_bytes();
cudaError_t launch_prefill_tc(const PrefillParams &p, cudaStream_t st);
// gate_z == nullptr: out = y; otherwise out = norm(y, gate=silu(gate_z)) * norm_weight
cudaError_t launch_decode(const void *q, const void *k, const void *v, const float *g,
                          const float *beta, float *state, void *out, int B, int HK, int HV,
                          int Dk, int Dv, gdn_dtype dtype, float scale, int l2norm,
                          const void *gate_z, const float *norm_weight, float norm_eps,
                          cudaStream_t st);
// The step before the rule: conv + SiLU of the cat(q, k, v) channels, gates; the conv
// state after each sequence when state_out is given (may be state_in)
cudaError_t launch_prologue(const void *proj, const void *proj_b, const void *proj_a, int layout,
                            const float *conv_w, const float *A_log, const float *dt_bias,
                            const void *state_in, void *state_out, const int32_t *cu, int N,
                            int T_seq, int64_t T, int HK, int HV, int Dk, int Dv, gdn_dtype dtype,
                            void *q, void *k, void *v, void *z, float *beta, float *g,
                            cudaStream_t st);
// Gated RMS norm of rows of Dv values: out = y / sqrt(mean(y^2) + eps) * w * silu(z)
cudaError_t launch_gated_norm(const void *y, const void *z, const float *w, void *out, int64_t rows,
                              int Dv, gdn_dtype dtype, float eps, cudaStream_t st);

// ---------------------------------------------------------------- device helpers
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

// silu(x) = x sigmoid(x) from the MUFU exponential and the approximate division (a few
// parts in 1e6 relative; x -> -inf gives -0, x -> +inf gives x)
__device__ __forceinline__ float silu_f(float x) { return __fdividef(x, 1.f + __expf(-x)); }

// packed fp32 pairs: one instruction for two lanes of arithmetic
__device__ __forceinline__ uint64_t f2pack(float a, float b) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ void f2unpack(uint64_t r, float &a, float &b) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t fmul2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
// silu of a pair: x / (1 + e^{-x}) with the MUFU exponential and reciprocal
__device__ __forceinline__ uint64_t silu2(uint64_t x) {
    const uint64_t t = fmul2(x, f2pack(-1.4426950408889634f, -1.4426950408889634f));
    float t0, t1;
    f2unpack(t, t0, t1);
    float e0, e1;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e0) : "f"(t0));
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e1) : "f"(t1));
    const uint64_t d = fadd2(f2pack(e0, e1), f2pack(1.f, 1.f));
    float d0, d1;
    f2unpack(d, d0, d1);
    float r0, r1;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r0) : "f"(d0));
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r1) : "f"(d1));
    return fmul2(x, f2pack(r0, r1));
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

}  // namespace gdn
