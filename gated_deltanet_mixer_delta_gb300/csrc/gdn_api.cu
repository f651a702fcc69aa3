// gdn_api.cu -- the C ABI (include/gdn.h): argument checks, workspace layout, dispatch.
//
// Every check that can be made on the host is made here, before anything is
// enqueued; nothing here allocates device memory or keeps state between calls.
#include <math.h>
#include <stdint.h>
#include <string.h>

#include "gdn_internal.cuh"

namespace gdn {

static inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int max_chunks_for(int64_t T_total, int n_seqs, bool packed, int T_seq) {
    if (!packed) return n_seqs * ((T_seq + kChunk - 1) / kChunk);
    return (int)((T_total + kChunk - 1) / kChunk + n_seqs);
}

// header | chain flags[N*HV*kChainSlices] | ready flags[max_chunks][HV] |
// chunk_seq[max_chunks] | chunk_first[N+1] | seq_order[N] | records[max_chunks][HV]
static size_t table_bytes(int max_chunks, int n_seqs) {
    return round_up(sizeof(int32_t) * ((size_t)max_chunks + 2 * (size_t)n_seqs + 1), 256);
}

// bytes of one record of the path a shape and dtype take: the tensor-core path's operand
// images, or the CUDA-core path's fp32 record
static size_t record_bytes_for(int Dk, int Dv, gdn_dtype dtype) {
    return tc_supported(Dk, Dv, dtype) ? tc_record_bytes() : record_floats(Dk, Dv) * sizeof(float);
}

size_t prefill_workspace_bytes_for(int64_t T_total, int n_seqs, int HV, int Dk, int Dv, gdn_dtype dtype) {
    // sized for the packed bound, which also covers equal-length batches
    const int mc = max_chunks_for(T_total, n_seqs, true, 0);
    return kWsHeader + chain_flag_bytes(n_seqs, HV) + ready_flag_bytes(mc, HV) + table_bytes(mc, n_seqs) +
           (size_t)mc * HV * record_bytes_for(Dk, Dv, dtype);
}

size_t prefill_workspace_bytes(int64_t T_total, int n_seqs, int HV, int Dk, int Dv) {
    // without a dtype: enough for either path
    const size_t a = prefill_workspace_bytes_for(T_total, n_seqs, HV, Dk, Dv, GDN_BF16);
    const size_t b = prefill_workspace_bytes_for(T_total, n_seqs, HV, Dk, Dv, GDN_F32);
    return a > b ? a : b;
}

}  // namespace gdn

using namespace gdn;

namespace {

bool dim_ok(int d) { return d == 32 || d == 64 || d == 128; }
bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

int check_common(int HK, int HV, int Dk, int Dv, gdn_dtype dtype, float scale) {
    if (HK <= 0 || HV <= 0 || HV % HK != 0) return GDN_ERR_INVALID_ARG;
    if (!dim_ok(Dk) || Dv != Dk) return GDN_ERR_UNSUPPORTED;
    if (dtype != GDN_BF16 && dtype != GDN_F32) return GDN_ERR_UNSUPPORTED;
    if (isnan(scale) || isinf(scale)) return GDN_ERR_INVALID_ARG;
    return GDN_OK;
}

float resolve_scale(float scale, int Dk) { return scale > 0.f ? scale : 1.0f / sqrtf((float)Dk); }

int prefill_common(const void *queries, const void *keys, const void *values,
                   const float *decays, const float *beta, const float *initial_state,
                   void *out, float *final_state, float *states, const int32_t *cu_seqlens,
                   int N, int T_seq, int64_t T_total, int HK, int HV, int Dk, int Dv,
                   gdn_dtype dtype, float scale, int use_qk_l2norm, void *workspace,
                   size_t workspace_bytes, void *cuda_stream, const void *gate_z = nullptr,
                   const float *norm_weight = nullptr, float norm_eps = 0.f) {
    int rc = check_common(HK, HV, Dk, Dv, dtype, scale);
    if (rc != GDN_OK) return rc;
    if (N < 0 || T_total < 0 || T_seq < 0) return GDN_ERR_INVALID_ARG;
    if (gate_z && T_total > 0 && !norm_weight) return GDN_ERR_INVALID_ARG;
    if (T_total > INT32_MAX || N > 65535 || HV > 65535) return GDN_ERR_UNSUPPORTED;
    if ((int64_t)N * HV * kChainSlices > INT32_MAX) return GDN_ERR_UNSUPPORTED;   // chain numbers
    if (N > 0 && !final_state) return GDN_ERR_INVALID_ARG;
    if (T_total > 0 && (!queries || !keys || !values || !decays || !beta || !out))
        return GDN_ERR_INVALID_ARG;
    if (cu_seqlens == nullptr && N > 0 && T_seq > 0 && (int64_t)N * T_seq != T_total)
        return GDN_ERR_INVALID_ARG;
    const void *ptrs[] = {queries, keys, values, decays, beta, initial_state, out,
                          final_state, states, cu_seqlens, gate_z, norm_weight};
    for (const void *p : ptrs)
        if (p && !aligned16(p)) return GDN_ERR_MISALIGNED;
    // final_state may be initial_state (in place); no other overlap is checked here
    if (!workspace) return GDN_ERR_WORKSPACE;
    if ((uintptr_t)workspace & 255u) return GDN_ERR_MISALIGNED;
    if (workspace_bytes < prefill_workspace_bytes_for(T_total, N, HV, Dk, Dv, dtype)) return GDN_ERR_WORKSPACE;

    cudaStream_t st = (cudaStream_t)cuda_stream;
    const bool packed = cu_seqlens != nullptr;
    const int mc = max_chunks_for(T_total, N, packed, T_seq);
    char *ws = (char *)workspace;
    PrefillParams p;
    memset(&p, 0, sizeof p);
    p.q = queries; p.k = keys; p.v = values; p.g = decays; p.beta = beta;
    p.s0 = initial_state; p.out = out; p.s_final = final_state; p.states = states;
    p.cu_seqlens = cu_seqlens;
    p.N = N; p.T_seq = T_seq; p.T_total = T_total;
    p.HK = HK; p.HV = HV; p.Dk = Dk; p.Dv = Dv;
    p.scale = resolve_scale(scale, Dk);
    p.l2norm = use_qk_l2norm ? 1 : 0;
    p.max_chunks = mc;
    const size_t flag_bytes = chain_flag_bytes(N, HV) + ready_flag_bytes(mc, HV);
    p.status = (int32_t *)ws;
    p.chain_flags = (int32_t *)(ws + kWsHeader);
    p.ready = (int32_t *)(ws + kWsHeader + chain_flag_bytes(N, HV));
    p.chunk_seq = (int32_t *)(ws + kWsHeader + flag_bytes);
    p.chunk_first = p.chunk_seq + mc;
    p.seq_order = p.chunk_first + N + 1;
    p.rec = (float *)(ws + kWsHeader + flag_bytes + table_bytes(mc, N));
    p.rec_floats = record_bytes_for(Dk, Dv, dtype) / sizeof(float);

    if (N == 0) {
        // nothing to run; leave a clean status word
        if (cudaMemsetAsync(workspace, 0, 2 * sizeof(int32_t), st) != cudaSuccess)
            return GDN_ERR_CUDA;
        return GDN_OK;
    }
    cudaError_t e = tc_supported(Dk, Dv, dtype) ? launch_prefill_tc(p, st)
                                                : launch_prefill_generic(p, dtype, st);
    // the gated norm runs over the outputs in place, on the same stream
    if (e == cudaSuccess && gate_z && T_total > 0)
        e = launch_gated_norm(out, gate_z, norm_weight, out, T_total * HV, Dv, dtype, norm_eps, st);
    return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

}  // namespace

extern "C" {

int gdn_prefill(const void *queries, const void *keys, const void *values, const float *decays,
                const float *beta, const float *initial_state, void *out, float *final_state,
                float *states, int B, int T, int HK, int HV, int Dk, int Dv, gdn_dtype dtype,
                float scale, int use_qk_l2norm, void *workspace, size_t workspace_bytes,
                void *cuda_stream) {
    if (B < 0 || T < 0) return GDN_ERR_INVALID_ARG;
    return prefill_common(queries, keys, values, decays, beta, initial_state, out, final_state,
                          states, nullptr, B, T, (int64_t)B * T, HK, HV, Dk, Dv, dtype, scale,
                          use_qk_l2norm, workspace, workspace_bytes, cuda_stream);
}

int gdn_prefill_varlen(const void *queries, const void *keys, const void *values,
                       const float *decays, const float *beta, const float *initial_state,
                       void *out, float *final_state, float *states, const int32_t *cu_seqlens,
                       int N, int T_total, int HK, int HV, int Dk, int Dv, gdn_dtype dtype,
                       float scale, int use_qk_l2norm, void *workspace, size_t workspace_bytes,
                       void *cuda_stream) {
    if (N < 0 || T_total < 0) return GDN_ERR_INVALID_ARG;
    if (!cu_seqlens) return GDN_ERR_INVALID_ARG;
    return prefill_common(queries, keys, values, decays, beta, initial_state, out, final_state,
                          states, cu_seqlens, N, 0, T_total, HK, HV, Dk, Dv, dtype, scale,
                          use_qk_l2norm, workspace, workspace_bytes, cuda_stream);
}

static int decode_common(const void *queries, const void *keys, const void *values,
                         const float *decays, const float *beta, float *state, void *out, int B,
                         int HK, int HV, int Dk, int Dv, gdn_dtype dtype, float scale,
                         int use_qk_l2norm, const void *gate_z, const float *norm_weight,
                         float norm_eps, void *cuda_stream) {
    int rc = check_common(HK, HV, Dk, Dv, dtype, scale);
    if (rc != GDN_OK) return rc;
    if (B < 0) return GDN_ERR_INVALID_ARG;
    if (B == 0) return GDN_OK;
    if (!queries || !keys || !values || !decays || !beta || !state || !out)
        return GDN_ERR_INVALID_ARG;
    const void *ptrs[] = {queries, keys, values, decays, beta, state, out, gate_z, norm_weight};
    for (const void *p : ptrs)
        if (p && !aligned16(p)) return GDN_ERR_MISALIGNED;
    if ((int64_t)B * HV > INT32_MAX) return GDN_ERR_UNSUPPORTED;
    cudaError_t e = launch_decode(queries, keys, values, decays, beta, state, out, B, HK, HV, Dk,
                                  Dv, dtype, resolve_scale(scale, Dk), use_qk_l2norm ? 1 : 0,
                                  gate_z, norm_weight, norm_eps, (cudaStream_t)cuda_stream);
    return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

int gdn_prefill_gated(const void *queries, const void *keys, const void *values,
                      const float *decays, const float *beta, const float *initial_state,
                      void *out, float *final_state, float *states, const void *gate_z,
                      const float *norm_weight, float norm_eps, int B, int T, int HK, int HV,
                      int Dk, int Dv, gdn_dtype dtype, float scale, int use_qk_l2norm,
                      void *workspace, size_t workspace_bytes, void *cuda_stream) {
    if (B < 0 || T < 0) return GDN_ERR_INVALID_ARG;
    if (!gate_z || !norm_weight || !(norm_eps >= 0.f) || isinf(norm_eps)) return GDN_ERR_INVALID_ARG;
    return prefill_common(queries, keys, values, decays, beta, initial_state, out, final_state,
                          states, nullptr, B, T, (int64_t)B * T, HK, HV, Dk, Dv, dtype, scale,
                          use_qk_l2norm, workspace, workspace_bytes, cuda_stream, gate_z,
                          norm_weight, norm_eps);
}

int gdn_prefill_varlen_gated(const void *queries, const void *keys, const void *values,
                             const float *decays, const float *beta, const float *initial_state,
                             void *out, float *final_state, float *states, const void *gate_z,
                             const float *norm_weight, float norm_eps,
                             const int32_t *cu_seqlens, int N, int T_total, int HK, int HV,
                             int Dk, int Dv, gdn_dtype dtype, float scale, int use_qk_l2norm,
                             void *workspace, size_t workspace_bytes, void *cuda_stream) {
    if (N < 0 || T_total < 0) return GDN_ERR_INVALID_ARG;
    if (!cu_seqlens) return GDN_ERR_INVALID_ARG;
    if (!gate_z || !norm_weight || !(norm_eps >= 0.f) || isinf(norm_eps)) return GDN_ERR_INVALID_ARG;
    return prefill_common(queries, keys, values, decays, beta, initial_state, out, final_state,
                          states, cu_seqlens, N, 0, T_total, HK, HV, Dk, Dv, dtype, scale,
                          use_qk_l2norm, workspace, workspace_bytes, cuda_stream, gate_z,
                          norm_weight, norm_eps);
}

int gdn_decode_step(const void *queries, const void *keys, const void *values,
                    const float *decays, const float *beta, float *state, void *out, int B,
                    int HK, int HV, int Dk, int Dv, gdn_dtype dtype, float scale,
                    int use_qk_l2norm, void *cuda_stream) {
    return decode_common(queries, keys, values, decays, beta, state, out, B, HK, HV, Dk, Dv,
                         dtype, scale, use_qk_l2norm, nullptr, nullptr, 0.f, cuda_stream);
}

int gdn_decode_step_gated(const void *queries, const void *keys, const void *values,
                          const float *decays, const float *beta, float *state, void *out,
                          const void *gate_z, const float *norm_weight, float norm_eps, int B,
                          int HK, int HV, int Dk, int Dv, gdn_dtype dtype, float scale,
                          int use_qk_l2norm, void *cuda_stream) {
    if (!gate_z || !norm_weight) return GDN_ERR_INVALID_ARG;
    if (!(norm_eps >= 0.f) || isinf(norm_eps)) return GDN_ERR_INVALID_ARG;
    return decode_common(queries, keys, values, decays, beta, state, out, B, HK, HV, Dk, Dv,
                         dtype, scale, use_qk_l2norm, gate_z, norm_weight, norm_eps, cuda_stream);
}

int gdn_conv_gate_prologue(const void *proj, const void *proj_b, const void *proj_a,
                           gdn_proj_layout layout, const float *conv_weight, const float *A_log,
                           const float *dt_bias, const void *conv_state_in, void *conv_state_out,
                           const int32_t *cu_seqlens, int N, int64_t T_total, int HK, int HV,
                           int Dk, int Dv, gdn_dtype dtype, void *queries, void *keys,
                           void *values, void *gate_z, float *beta, float *decays,
                           void *cuda_stream) {
    int rc = check_common(HK, HV, Dk, Dv, dtype, 1.f);
    if (rc != GDN_OK) return rc;
    if (layout != GDN_LAYOUT_QKV && layout != GDN_LAYOUT_QKVZ) return GDN_ERR_INVALID_ARG;
    if (N < 0 || T_total < 0) return GDN_ERR_INVALID_ARG;
    if (N > 65535) return GDN_ERR_UNSUPPORTED;
    if (!cu_seqlens && (N == 0 ? T_total != 0 : T_total % N != 0)) return GDN_ERR_INVALID_ARG;
    if (T_total > 0) {
        if (!proj || !proj_b || !conv_weight || !A_log || !dt_bias || !queries || !keys ||
            !values || !beta || !decays)
            return GDN_ERR_INVALID_ARG;
        if (layout == GDN_LAYOUT_QKV && !proj_a) return GDN_ERR_INVALID_ARG;
    }
    if (layout == GDN_LAYOUT_QKV && gate_z) return GDN_ERR_INVALID_ARG;
    const void *ptrs[] = {proj, proj_b, proj_a, conv_weight, A_log, dt_bias, conv_state_in,
                          conv_state_out, cu_seqlens, queries, keys, values, gate_z, beta, decays};
    for (const void *p : ptrs)
        if (p && !aligned16(p)) return GDN_ERR_MISALIGNED;
    const int T_seq = (!cu_seqlens && N > 0) ? (int)(T_total / N) : 0;
    if (!cu_seqlens && N > 0 && T_total / N > INT32_MAX) return GDN_ERR_UNSUPPORTED;
    cudaError_t e = launch_prologue(proj, proj_b, proj_a, (int)layout, conv_weight, A_log, dt_bias,
                                    conv_state_in, conv_state_out, cu_seqlens, N, T_seq, T_total,
                                    HK, HV, Dk, Dv, dtype, queries, keys, values, gate_z, beta,
                                    decays, (cudaStream_t)cuda_stream);
    return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

int gdn_gated_rmsnorm(const void *y, const void *gate_z, const float *norm_weight, void *out,
                      int64_t rows, int Dv, gdn_dtype dtype, float norm_eps, void *cuda_stream) {
    if (rows < 0 || !(norm_eps >= 0.f) || isinf(norm_eps)) return GDN_ERR_INVALID_ARG;
    if (!dim_ok(Dv)) return GDN_ERR_UNSUPPORTED;
    if (dtype != GDN_BF16 && dtype != GDN_F32) return GDN_ERR_UNSUPPORTED;
    if (rows == 0) return GDN_OK;
    if (!y || !gate_z || !norm_weight || !out) return GDN_ERR_INVALID_ARG;
    const void *ptrs[] = {y, gate_z, norm_weight, out};
    for (const void *p : ptrs)
        if (!aligned16(p)) return GDN_ERR_MISALIGNED;
    cudaError_t e = launch_gated_norm(y, gate_z, norm_weight, out, rows, Dv, dtype, norm_eps,
                                      (cudaStream_t)cuda_stream);
    return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

int gdn_state_layout(int batch, int HV, int Dk, int Dv, gdn_state_layout_t *layout) {
    if (!layout || batch < 0 || HV <= 0 || Dk <= 0 || Dv <= 0) return GDN_ERR_INVALID_ARG;
    layout->bytes_per_head = (size_t)Dk * Dv * sizeof(float);
    layout->bytes = (size_t)batch * HV * layout->bytes_per_head;
    layout->shape[0] = batch; layout->shape[1] = HV; layout->shape[2] = Dk; layout->shape[3] = Dv;
    layout->stride[3] = 1;
    layout->stride[2] = Dv;
    layout->stride[1] = (int64_t)Dk * Dv;
    layout->stride[0] = (int64_t)HV * Dk * Dv;
    layout->alignment = 16;
    return GDN_OK;
}

size_t gdn_prefill_workspace_size(int64_t T_total, int n_seqs, int HV, int Dk, int Dv) {
    if (T_total < 0 || n_seqs < 0 || HV <= 0 || !dim_ok(Dk) || !dim_ok(Dv)) return 0;
    return prefill_workspace_bytes(T_total, n_seqs, HV, Dk, Dv);
}

size_t gdn_prefill_workspace_size_for(int64_t T_total, int n_seqs, int HV, int Dk, int Dv, gdn_dtype dtype) {
    if (T_total < 0 || n_seqs < 0 || HV <= 0 || !dim_ok(Dk) || Dv != Dk) return 0;
    if (dtype != GDN_BF16 && dtype != GDN_F32) return 0;
    return prefill_workspace_bytes_for(T_total, n_seqs, HV, Dk, Dv, dtype);
}

int gdn_workspace_status(const void *workspace, void *cuda_stream, int *status) {
    if (!workspace || !status) return GDN_ERR_INVALID_ARG;
    int32_t v = 0;
    cudaStream_t st = (cudaStream_t)cuda_stream;
    if (cudaMemcpyAsync(&v, workspace, sizeof v, cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return GDN_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return GDN_ERR_CUDA;
    *status = v;
    return GDN_OK;
}

const char *gdn_status_string(int status) {
    switch (status) {
    case GDN_OK: return "ok";
    case GDN_ERR_INVALID_ARG: return "invalid argument";
    case GDN_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case GDN_ERR_MISALIGNED: return "pointer not aligned";
    case GDN_ERR_WORKSPACE: return "workspace missing or too small";
    case GDN_ERR_CUDA: return "CUDA launch or runtime error";
    case GDN_ERR_TIMEOUT: return "bounded device wait timed out";
    case GDN_ERR_BAD_SEQLENS: return "cu_seqlens is not 0 = c0 <= ... <= cN = T_total";
    default: return "unknown status";
    }
}

int gdn_abi_version(void) { return 100; }

}  // extern "C"
