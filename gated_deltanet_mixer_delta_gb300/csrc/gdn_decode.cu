// gdn_decode.cu -- one-token recurrent step of the gated delta rule, state in place.
//
// The decode kernel of the pages ("a decode step's recurrent one", qwen3_5_text
// page, linear_attn value table): per (sequence b, value head h) with key head
// j = h / (HV/HK), and S the cached state [Dk][Dv] (row = key index):
//
//     S' = a S  (a = e^g)      x = S'^T k^       y = S'^T q~
//     u  = beta (v - x)        S <- S' + k^ u^T  o = y + (k^ . q~) u
//
// The last line is the read-out after the write, (S' + k^ u^T)^T q~, expanded
// so that S is read once and written once.
//
// HBM-bound: 2 * Dk * Dv * 4 bytes of state move per (b, h) against a few
// hundred bytes of q, k, v, g, beta, o.  One CTA per (b, h) keeps its whole
// state tile in registers between the read and the write: every thread owns
// 4 consecutive value columns (one 16-byte vector) of Dk*Dv/1024 rows; a warp
// reads/writes whole 512-byte rows, so every access is a full, coalesced
// 128-bit transaction.  The two reductions over the key index (S^T k, S^T q)
// run first inside each thread over its rows, then across the row groups
// through shared memory.  All loads of the tile are issued before any is used.
//
// GATED: the output goes through the gated RMS norm that follows the rule in the
// mixer (out = norm(y, gate=silu(z)) * weight, qwen3_5_text page, "The DeltaNet
// mixer"), from the fp32 y of the CTA's whole head, so y never goes to memory.
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kDecodeThreads = 256;

template <int DK, int DV, typename Tin, bool GATED>
__global__ void __launch_bounds__(kDecodeThreads, 2)
decode_kernel(const Tin *__restrict__ q, const Tin *__restrict__ k, const Tin *__restrict__ v,
              const float *__restrict__ g, const float *__restrict__ beta,
              float *__restrict__ state, Tin *__restrict__ out, int HK, int HV, float scale,
              int l2norm, const Tin *__restrict__ gz, const float *__restrict__ gw, float eps) {
    constexpr int TPR = DV / 4;                    // threads per state row
    constexpr int NRG = kDecodeThreads / TPR;      // row groups
    constexpr int RPT = DK / NRG;                  // rows per thread
    static_assert(RPT >= 1 && DK % NRG == 0, "tile shape");

    __shared__ float s_q[DK], s_k[DK], s_u[DV];
    __shared__ float s_red[2][NRG][DV];
    __shared__ float s_scal[4];
    __shared__ float s_nrm[DV / 32];

    const int bh = blockIdx.x;                     // b * HV + h
    const int b = bh / HV, h = bh - b * HV;
    const int j = h / (HV / HK);
    const int tid = threadIdx.x;
    const int cg = tid % TPR, rg = tid / TPR;      // column group, row group
    float4 *S4 = reinterpret_cast<float4 *>(state + (size_t)bh * DK * DV);

    // 1. issue every load of the state tile
    float4 s[RPT];
#pragma unroll
    for (int a = 0; a < RPT; ++a) s[a] = __ldcs(&S4[(rg + a * NRG) * TPR + cg]);
    float gzv = 0.f, gwv = 0.f;                    // gate and gain of column tid
    if (GATED && tid < DV) {
        gzv = to_f32(gz[(size_t)bh * DV + tid]);
        gwv = gw[tid];
    }

    // 2. q, k of key head j; norms and q.k in warp 0
    const Tin *qr = q + ((size_t)b * HK + j) * DK;
    const Tin *kr = k + ((size_t)b * HK + j) * DK;
    for (int i = tid; i < DK; i += kDecodeThreads) {
        s_q[i] = to_f32(qr[i]);
        s_k[i] = to_f32(kr[i]);
    }
    __syncthreads();
    if (tid < 32) {
        float sq = 0.f, sk = 0.f, qk = 0.f;
        for (int i = tid; i < DK; i += 32) {
            float a = s_q[i], c = s_k[i];
            sq += a * a; sk += c * c; qk += a * c;
        }
        sq = warp_sum(sq); sk = warp_sum(sk); qk = warp_sum(qk);
        if (tid == 0) {
            float rq = l2norm ? scale * rsqrtf(sq + kL2Eps) : scale;
            float rk = l2norm ? rsqrtf(sk + kL2Eps) : 1.f;
            s_scal[0] = rq; s_scal[1] = rk; s_scal[2] = qk * rq * rk;
        }
    }

    // 3. per-thread partial S^T k and S^T q over its rows (raw q, k)
    float4 px = make_float4(0.f, 0.f, 0.f, 0.f), py = px;
#pragma unroll
    for (int a = 0; a < RPT; ++a) {
        const int i = rg + a * NRG;
        const float kk = s_k[i], qq = s_q[i];
        px.x += s[a].x * kk; px.y += s[a].y * kk; px.z += s[a].z * kk; px.w += s[a].w * kk;
        py.x += s[a].x * qq; py.y += s[a].y * qq; py.z += s[a].z * qq; py.w += s[a].w * qq;
    }
    *reinterpret_cast<float4 *>(&s_red[0][rg][cg * 4]) = px;
    *reinterpret_cast<float4 *>(&s_red[1][rg][cg * 4]) = py;
    __syncthreads();

    // 4. finish the reductions, form u and o
    const float alpha = expf(g[bh]);
    float yo = 0.f;                                // y of column tid
    if (tid < DV) {
        float x = 0.f, y = 0.f;
#pragma unroll 8
        for (int r = 0; r < NRG; ++r) { x += s_red[0][r][tid]; y += s_red[1][r][tid]; }
        const float rq = s_scal[0], rk = s_scal[1], kq = s_scal[2];
        const float vv = to_f32(v[(size_t)bh * DV + tid]);
        const float u = beta[bh] * (vv - alpha * rk * x);
        s_u[tid] = u;
        yo = alpha * rq * y + kq * u;
        if (GATED) {
            const float ss = warp_sum(yo * yo);      // DV is a multiple of 32: whole warps
            if ((tid & 31) == 0) s_nrm[tid >> 5] = ss;
        } else {
            out[(size_t)bh * DV + tid] = from_f32<Tin>(yo);
        }
    }
    __syncthreads();

    // 5. S <- a S + k^ u^T, written back in place
    const float rk = s_scal[1];
    const float4 u4 = *reinterpret_cast<const float4 *>(&s_u[cg * 4]);
#pragma unroll
    for (int a = 0; a < RPT; ++a) {
        const int i = rg + a * NRG;
        const float kk = rk * s_k[i];
        float4 o;
        o.x = alpha * s[a].x + kk * u4.x;
        o.y = alpha * s[a].y + kk * u4.y;
        o.z = alpha * s[a].z + kk * u4.z;
        o.w = alpha * s[a].w + kk * u4.w;
        __stcs(&S4[i * TPR + cg], o);
    }
    // the gated output once the state stores are on their way
    if (GATED && tid < DV) {
        float ss = 0.f;
#pragma unroll
        for (int w = 0; w < DV / 32; ++w) ss += s_nrm[w];
        const float inv = rsqrtf(ss * (1.f / DV) + eps);
        out[(size_t)bh * DV + tid] = from_f32<Tin>(yo * inv * gwv * silu_f(gzv));
    }
}

template <int DK, int DV, typename Tin>
cudaError_t launch_t(const void *q, const void *k, const void *v, const float *g,
                     const float *beta, float *state, void *out, int B, int HK, int HV,
                     float scale, int l2norm, const void *gz, const float *gw, float eps,
                     cudaStream_t st) {
    if (gz)
        decode_kernel<DK, DV, Tin, true><<<B * HV, kDecodeThreads, 0, st>>>(
            (const Tin *)q, (const Tin *)k, (const Tin *)v, g, beta, state, (Tin *)out, HK, HV,
            scale, l2norm, (const Tin *)gz, gw, eps);
    else
        decode_kernel<DK, DV, Tin, false><<<B * HV, kDecodeThreads, 0, st>>>(
            (const Tin *)q, (const Tin *)k, (const Tin *)v, g, beta, state, (Tin *)out, HK, HV,
            scale, l2norm, nullptr, nullptr, 0.f);
    return cudaGetLastError();
}

template <typename Tin>
cudaError_t dispatch_dims(int Dk, int Dv, const void *q, const void *k, const void *v,
                          const float *g, const float *beta, float *state, void *out, int B,
                          int HK, int HV, float scale, int l2norm, const void *gz,
                          const float *gw, float eps, cudaStream_t st) {
#define GDN_DEC_CASE(DK_, DV_)                                                             \
    if (Dk == DK_ && Dv == DV_)                                                            \
        return launch_t<DK_, DV_, Tin>(q, k, v, g, beta, state, out, B, HK, HV, scale,     \
                                       l2norm, gz, gw, eps, st);
    GDN_DEC_CASE(32, 32) GDN_DEC_CASE(64, 64) GDN_DEC_CASE(128, 128)
#undef GDN_DEC_CASE
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_decode(const void *q, const void *k, const void *v, const float *g,
                          const float *beta, float *state, void *out, int B, int HK, int HV,
                          int Dk, int Dv, gdn_dtype dtype, float scale, int l2norm,
                          const void *gate_z, const float *norm_weight, float norm_eps,
                          cudaStream_t st) {
    if (B == 0) return cudaSuccess;
    if (dtype == GDN_BF16)
        return dispatch_dims<__nv_bfloat16>(Dk, Dv, q, k, v, g, beta, state, out, B, HK, HV,
                                            scale, l2norm, gate_z, norm_weight, norm_eps, st);
    return dispatch_dims<float>(Dk, Dv, q, k, v, g, beta, state, out, B, HK, HV, scale,
                                l2norm, gate_z, norm_weight, norm_eps, st);
}

}  // namespace gdn
