// gdn_prologue.cu -- the step before the rule in the mixer (qwen3_5_text page, Notes ->
// "The DeltaNet mixer"; qwen3_next page, Notes -> "The DeltaNet mixer fuses its
// projections per key head"):
//
//     q, k, v = split(silu(conv1d(cat(q, k, v))))      causal depthwise conv, width 4
//     beta    = sigmoid(b)
//     g       = -exp(A_log) * softplus(a + dt_bias)
//
// from the projections' outputs, in either of the pages' layouts: the cat(q, k, v)
// channels as they come (in_proj_qkv, plus in_proj_b / in_proj_a), or Qwen3-Next's fused
// in_proj_qkvz / in_proj_ba grouped per key head (query, key, the values of the key head's
// value heads, then their output gates; b's then a's), regrouped on the fly.  The conv of
// channel c at token t is sum_i w[c][i] x_{t-3+i}[c] (tap 3 on the current token); inputs
// before a sequence's first token come from its carried conv state [N][3][C] (the three
// inputs before it, oldest first) or are zero.
//
// HBM-bound elementwise work: every conv thread owns 8 bytes of consecutive channels (4
// bf16 or 2 fp32, never straddling a head) over a tile of 16 tokens; it stages the tile's
// inputs and the three before it (mostly L2 hits) in shared memory with asynchronous
// copies, which hold no registers while in flight, so that several blocks fit on an SM;
// it runs a sliding three-token window in registers and writes the SiLU'd values into
// the queries / keys / values tensors of the rule.  One block per tile forms the gates;
// with the fused layout further blocks copy the output gates z out.  The conv state after
// each sequence is written by a second kernel, once every read of the incoming state is
// done (so the state can be updated in place).
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kProThreads = 256;
constexpr int kProTile = 16;                           // tokens per tile
constexpr int kProBatch = 8;                           // tokens whose loads go out together

struct ProParams {
    const void *proj, *proj_b, *proj_a;
    int layout;                                        // GDN_LAYOUT_QKV / GDN_LAYOUT_QKVZ
    const float *conv_w, *A_log, *dt_bias;
    const void *state_in;
    void *state_out;
    const int32_t *cu;                                 // [N+1] or nullptr (T_seq tokens each)
    int N, T_seq;
    int64_t T;
    int HK, HV, Dk, Dv;
    void *q, *k, *v, *z;
    float *beta, *g;
};

template <typename T> struct V16;
template <> struct V16<__nv_bfloat16> {
    static constexpr int E = 8;
    static __device__ __forceinline__ void get(const void *p, float (&x)[8]) {
        unpack(*reinterpret_cast<const uint4 *>(p), x);
    }
    static __device__ __forceinline__ void unpack(const uint4 &r, float (&x)[8]) {
        const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&r);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __bfloat1622float2(h[i]);
            x[2 * i] = f.x;
            x[2 * i + 1] = f.y;
        }
    }
    static __device__ __forceinline__ void put(void *p, const float (&x)[8]) {
        uint4 r;
        __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(&r);
#pragma unroll
        for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(x[2 * i], x[2 * i + 1]);
        *reinterpret_cast<uint4 *>(p) = r;
    }
};
template <> struct V16<float> {
    static constexpr int E = 4;
    static __device__ __forceinline__ void get(const void *p, float (&x)[4]) {
        unpack(*reinterpret_cast<const uint4 *>(p), x);
    }
    static __device__ __forceinline__ void unpack(const uint4 &r, float (&x)[4]) {
        x[0] = __uint_as_float(r.x); x[1] = __uint_as_float(r.y);
        x[2] = __uint_as_float(r.z); x[3] = __uint_as_float(r.w);
    }
    static __device__ __forceinline__ void put(void *p, const float (&x)[4]) {
        *reinterpret_cast<float4 *>(p) = make_float4(x[0], x[1], x[2], x[3]);
    }
};

// 8 bytes of T (4 bf16 or 2 fp32): the conv's per-thread channel group
template <typename T> struct V8;
template <> struct V8<__nv_bfloat16> {
    static constexpr int E = 4;
    static __device__ __forceinline__ void unpack(const uint2 &r, float (&x)[4]) {
        const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&r);
        const float2 a = __bfloat1622float2(h[0]), b = __bfloat1622float2(h[1]);
        x[0] = a.x; x[1] = a.y; x[2] = b.x; x[3] = b.y;
    }
    static __device__ __forceinline__ uint2 pack(const float (&x)[4]) {
        uint2 r;
        __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(&r);
        h[0] = __floats2bfloat162_rn(x[0], x[1]);
        h[1] = __floats2bfloat162_rn(x[2], x[3]);
        return r;
    }
};
template <> struct V8<float> {
    static constexpr int E = 2;
    static __device__ __forceinline__ void unpack(const uint2 &r, float (&x)[2]) {
        x[0] = __uint_as_float(r.x); x[1] = __uint_as_float(r.y);
    }
    static __device__ __forceinline__ uint2 pack(const float (&x)[2]) {
        return make_uint2(__float_as_uint(x[0]), __float_as_uint(x[1]));
    }
};

// 8-byte global -> shared copy that holds no register while in flight
__device__ __forceinline__ void cp_async8(void *sdst, const void *gsrc) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"((uint32_t)__cvta_generic_to_shared(sdst)),
                 "l"(gsrc)
                 : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ int64_t seq_start(const ProParams &p, int s) {
    return p.cu ? (int64_t)p.cu[s] : (int64_t)s * p.T_seq;
}
// the sequence holding token t (the last one starting at or before t; empty sequences
// before it are skipped by the caller's walk)
__device__ __forceinline__ int seq_of(const ProParams &p, int64_t t) {
    if (!p.cu) return p.T_seq > 0 ? (int)(t / p.T_seq) : 0;
    int lo = 0, hi = p.N - 1;                          // largest s with cu[s] <= t
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if ((int64_t)p.cu[mid] <= t) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// element offset of cat(q, k, v) channel c in a projection row, and the row width
__device__ __forceinline__ int64_t proj_col(const ProParams &p, int c) {
    if (p.layout == GDN_LAYOUT_QKV) return c;
    const int r = p.HV / p.HK, per = 2 * p.Dk + 2 * r * p.Dv;
    const int nq = p.HK * p.Dk;
    if (c < nq) return (int64_t)(c / p.Dk) * per + c % p.Dk;
    if (c < 2 * nq) return (int64_t)((c - nq) / p.Dk) * per + p.Dk + (c - nq) % p.Dk;
    const int cv = c - 2 * nq, h = cv / p.Dv, d = cv % p.Dv;
    return (int64_t)(h / r) * per + 2 * p.Dk + (h % r) * p.Dv + d;
}
__device__ __forceinline__ int64_t proj_width(const ProParams &p) {
    return p.layout == GDN_LAYOUT_QKV ? (int64_t)2 * p.HK * p.Dk + (int64_t)p.HV * p.Dv
                                      : (int64_t)p.HK * (2 * p.Dk + 2 * (p.HV / p.HK) * p.Dv);
}

// four blocks per SM (at most 64 registers a thread): the conv blocks' inputs in flight
// from four blocks rather than three hide HBM latency better (83 -> 88% of the copy
// bandwidth) than the few registers this spills cost
template <typename T>
__global__ void __launch_bounds__(kProThreads, 4)
prologue_kernel(ProParams p) {
    constexpr int E = V16<T>::E;                       // z copy: 16 bytes a thread
    constexpr int EC = V8<T>::E;                       // conv: 8 bytes a thread
    // the conv thread's inputs: the tile's tokens and the three before it
    __shared__ uint2 sx[kProTile + 3][kProThreads];
    const int C = 2 * p.HK * p.Dk + p.HV * p.Dv;
    const int nconv = (C / EC + kProThreads - 1) / kProThreads;
    const int nz = p.z ? ((p.HV * p.Dv) / E + kProThreads - 1) / kProThreads : 0;
    const int64_t tb = (int64_t)blockIdx.x * kProTile;   // token tile along x (no limit)
    const int64_t te = min(p.T, tb + kProTile);
    const int64_t W = proj_width(p);
    const T *proj = reinterpret_cast<const T *>(p.proj);
    const int bx = blockIdx.y;                            // conv / z / gate block

    if (bx < nconv) {
        // ---- conv + SiLU of EC consecutive channels
        const int c = (bx * kProThreads + threadIdx.x) * EC;
        if (c >= C) return;
        const int64_t col = proj_col(p, c);
        // every input row the tile may read, fetched asynchronously; a thread reads back
        // only its own slots, so no barrier is needed
#pragma unroll
        for (int i = 0; i < kProTile + 3; ++i) {
            const int64_t tau = tb - 3 + i;
            if (tau >= 0 && tau < te) cp_async8(&sx[i][threadIdx.x], proj + tau * W + col);
        }
        float w[4][EC];
#pragma unroll
        for (int e = 0; e < EC; ++e) {
            const float4 w4 = *reinterpret_cast<const float4 *>(p.conv_w + (size_t)(c + e) * 4);
            w[0][e] = w4.x; w[1][e] = w4.y; w[2][e] = w4.z; w[3][e] = w4.w;
        }
        const int nq = p.HK * p.Dk;
        T *dst;
        int64_t dstride;
        if (c < nq) { dst = reinterpret_cast<T *>(p.q) + c; dstride = nq; }
        else if (c < 2 * nq) { dst = reinterpret_cast<T *>(p.k) + (c - nq); dstride = nq; }
        else { dst = reinterpret_cast<T *>(p.v) + (c - 2 * nq); dstride = (int64_t)p.HV * p.Dv; }
        const T *sin = reinterpret_cast<const T *>(p.state_in);
        int s = seq_of(p, tb);
        int64_t t0 = seq_start(p, s), t1 = seq_start(p, s + 1);
        cp_async_wait_all();
        // x_tau of this thread's channels, tau in the sequence s or its three predecessors
        auto xin = [&](int64_t tau, float (&x)[EC]) {
            if (tau >= t0) {
                V8<T>::unpack(sx[tau - (tb - 3)][threadIdx.x], x);
            } else if (sin && tau >= t0 - 3) {
                V8<T>::unpack(*reinterpret_cast<const uint2 *>(sin + ((int64_t)s * 3 + 3 + (tau - t0)) * C + c), x);
            } else {
#pragma unroll
                for (int e = 0; e < EC; ++e) x[e] = 0.f;
            }
        };
        float x3[EC], x2[EC], x1[EC];                  // x_{t-3}, x_{t-2}, x_{t-1}
        xin(tb - 3, x3);
        xin(tb - 2, x2);
        xin(tb - 1, x1);
        // one token: the conv taps, SiLU, two channels per instruction
        auto conv_silu = [&](const float (&x0)[EC], float (&o)[EC]) {
#pragma unroll
            for (int e = 0; e < EC; e += 2) {
                uint64_t acc = fmul2(f2pack(w[0][e], w[0][e + 1]), f2pack(x3[e], x3[e + 1]));
                acc = ffma2(f2pack(w[1][e], w[1][e + 1]), f2pack(x2[e], x2[e + 1]), acc);
                acc = ffma2(f2pack(w[2][e], w[2][e + 1]), f2pack(x1[e], x1[e + 1]), acc);
                acc = ffma2(f2pack(w[3][e], w[3][e + 1]), f2pack(x0[e], x0[e + 1]), acc);
                f2unpack(silu2(acc), o[e], o[e + 1]);
            }
        };
        if (te - tb == kProTile && te <= t1) {
            // the common tile: whole, inside one sequence; straight-line code over its
            // tokens (the window shifts are renames), outputs one row stride apart
            T *o_t = dst + tb * dstride;
#pragma unroll
            for (int u = 0; u < kProTile; ++u) {
                float x0[EC], o[EC];
                V8<T>::unpack(sx[u + 3][threadIdx.x], x0);
                conv_silu(x0, o);
#pragma unroll
                for (int e = 0; e < EC; ++e) {
                    x3[e] = x2[e];
                    x2[e] = x1[e];
                    x1[e] = x0[e];
                }
                *reinterpret_cast<uint2 *>(o_t) = V8<T>::pack(o);
                o_t += dstride;
            }
            return;
        }
#pragma unroll 1
        for (int u = 0; u < kProTile; ++u) {
            const int64_t t = tb + u;
            if (t >= te) break;
            if (t >= t1) {
                // next non-empty sequence: its window comes from its carried state
                do {
                    ++s;
                    t0 = seq_start(p, s);
                    t1 = seq_start(p, s + 1);
                } while (t >= t1);
                xin(t - 3, x3);
                xin(t - 2, x2);
                xin(t - 1, x1);
            }
            float x0[EC], o[EC];
            V8<T>::unpack(sx[u + 3][threadIdx.x], x0);
            conv_silu(x0, o);
#pragma unroll
            for (int e = 0; e < EC; ++e) {
                x3[e] = x2[e];
                x2[e] = x1[e];
                x1[e] = x0[e];
            }
            *reinterpret_cast<uint2 *>(dst + t * dstride) = V8<T>::pack(o);
        }
    } else if (bx < nconv + nz) {
        // ---- output gates z of the fused layout, copied out per value head
        const int c = ((bx - nconv) * kProThreads + threadIdx.x) * E;   // h * Dv + d
        if (c >= p.HV * p.Dv) return;
        const int r = p.HV / p.HK, h = c / p.Dv, d = c % p.Dv;
        const int64_t col = (int64_t)(h / r) * (2 * p.Dk + 2 * r * p.Dv) + 2 * p.Dk + r * p.Dv +
                            (h % r) * p.Dv + d;
        T *zo = reinterpret_cast<T *>(p.z) + c;
        for (int64_t t8 = tb; t8 < te; t8 += kProBatch) {
            uint4 raw[kProBatch];
#pragma unroll
            for (int u = 0; u < kProBatch; ++u)
                if (t8 + u < te) raw[u] = *reinterpret_cast<const uint4 *>(proj + (t8 + u) * W + col);
#pragma unroll
            for (int u = 0; u < kProBatch; ++u)
                if (t8 + u < te) *reinterpret_cast<uint4 *>(zo + (t8 + u) * (int64_t)p.HV * p.Dv) = raw[u];
        }
    } else {
        // ---- gates of the tile's tokens
        const T *pb = reinterpret_cast<const T *>(p.proj_b);
        const T *pa = reinterpret_cast<const T *>(p.proj_a);
        const int r = p.HV / p.HK;
        const int n = (int)(te - tb) * p.HV;
        for (int i = threadIdx.x; i < n; i += kProThreads) {
            const int64_t t = tb + i / p.HV;
            const int h = i % p.HV;
            float bv, av;
            if (p.layout == GDN_LAYOUT_QKV) {
                bv = to_f32(pb[t * p.HV + h]);
                av = to_f32(pa[t * p.HV + h]);
            } else {
                const int64_t base = t * (int64_t)p.HK * 2 * r + (int64_t)(h / r) * 2 * r + h % r;
                bv = to_f32(pb[base]);
                av = to_f32(pb[base + r]);
            }
            const float u = av + p.dt_bias[h];
            const float sp = u > 0.f ? u + log1pf(expf(-u)) : log1pf(expf(u));
            p.beta[t * p.HV + h] = 1.f / (1.f + expf(-bv));
            p.g[t * p.HV + h] = -expf(p.A_log[h]) * sp;
        }
    }
}

// conv state after each sequence: its last three inputs (reaching back into the carried
// state for sequences shorter than three); every value is read before any is written,
// by the same thread, so state_out may be state_in
template <typename T>
__global__ void __launch_bounds__(kProThreads)
conv_state_kernel(ProParams p) {
    constexpr int E = V16<T>::E;
    const int C = 2 * p.HK * p.Dk + p.HV * p.Dv;
    const int c = (blockIdx.x * kProThreads + threadIdx.x) * E;
    const int s = blockIdx.y;
    if (c >= C) return;
    const int64_t t0 = seq_start(p, s), t1 = seq_start(p, s + 1);
    const int64_t W = proj_width(p), col = proj_col(p, c);
    const T *proj = reinterpret_cast<const T *>(p.proj);
    const T *sin = reinterpret_cast<const T *>(p.state_in);
    float x[3][E];
#pragma unroll
    for (int rr = 0; rr < 3; ++rr) {
        const int64_t tau = t1 - 3 + rr;
        if (tau >= t0) {
            V16<T>::get(proj + tau * W + col, x[rr]);
        } else if (sin) {
            V16<T>::get(sin + ((int64_t)s * 3 + 3 + (tau - t0)) * C + c, x[rr]);
        } else {
#pragma unroll
            for (int e = 0; e < E; ++e) x[rr][e] = 0.f;
        }
    }
    T *so = reinterpret_cast<T *>(p.state_out);
#pragma unroll
    for (int rr = 0; rr < 3; ++rr) V16<T>::put(so + ((int64_t)s * 3 + rr) * C + c, x[rr]);
}

template <typename T>
cudaError_t launch_t(const ProParams &p, cudaStream_t st) {
    constexpr int E = V16<T>::E, EC = V8<T>::E;
    const int C = 2 * p.HK * p.Dk + p.HV * p.Dv;
    const int nconv = (C / EC + kProThreads - 1) / kProThreads;
    const int nz = p.z ? ((p.HV * p.Dv) / E + kProThreads - 1) / kProThreads : 0;
    const int64_t tiles = (p.T + kProTile - 1) / kProTile;
    if (tiles > 0x7fffffffLL) return cudaErrorInvalidValue;
    if (tiles > 0) {
        prologue_kernel<T><<<dim3((unsigned)tiles, nconv + nz + 1), kProThreads, 0, st>>>(p);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    if (p.state_out && p.N > 0) {
        conv_state_kernel<T><<<dim3((unsigned)((C / E + kProThreads - 1) / kProThreads), (unsigned)p.N),
                               kProThreads, 0, st>>>(p);
        return cudaGetLastError();
    }
    return cudaSuccess;
}

}  // namespace

cudaError_t launch_prologue(const void *proj, const void *proj_b, const void *proj_a, int layout,
                            const float *conv_w, const float *A_log, const float *dt_bias,
                            const void *state_in, void *state_out, const int32_t *cu, int N,
                            int T_seq, int64_t T, int HK, int HV, int Dk, int Dv, gdn_dtype dtype,
                            void *q, void *k, void *v, void *z, float *beta, float *g,
                            cudaStream_t st) {
    ProParams p;
    p.proj = proj; p.proj_b = proj_b; p.proj_a = proj_a; p.layout = layout;
    p.conv_w = conv_w; p.A_log = A_log; p.dt_bias = dt_bias;
    p.state_in = state_in; p.state_out = state_out; p.cu = cu; p.N = N; p.T_seq = T_seq; p.T = T;
    p.HK = HK; p.HV = HV; p.Dk = Dk; p.Dv = Dv;
    p.q = q; p.k = k; p.v = v; p.z = z; p.beta = beta; p.g = g;
    return dtype == GDN_BF16 ? launch_t<__nv_bfloat16>(p, st) : launch_t<float>(p, st);
}

}  // namespace gdn
