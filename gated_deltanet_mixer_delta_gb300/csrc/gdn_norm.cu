// gdn_norm.cu -- gated RMS norm of the mixer output, the step that follows the rule
// (qwen3_5_text page, Notes -> "The DeltaNet mixer": out = out_proj(norm(y,
// gate=silu(z))), gain: weight; the DeltaNet's own output norm multiplies by its weight,
// Notes -> "The readout is the plain projection").  Per row of Dv values (one token of
// one value head):
//
//     out_c = y_c / sqrt(mean(y^2) + eps) * weight_c * silu(z_c),   silu(z) = z sigmoid(z)
//
// HBM-bound: a row moves 3 Dv elements (y and z in, out back) against ~8 Dv flops.  Every
// access is 16 bytes wide: a row is spread over Dv * sizeof(T) / 16 lanes (a 128-value bf16
// row over half a warp), the sum of squares closes with shuffles inside that lane group,
// and each thread handles one row; the grid covers every row (no grid-stride loop,
// so the hardware keeps every SM's warp slots filled to the end).
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kNormThreads = 256;
constexpr int kNormRowsPerThread = 1;

// 16 bytes of T as floats
template <typename T> struct Pack16;
template <> struct Pack16<__nv_bfloat16> {
    static constexpr int E = 8;
    static __device__ __forceinline__ void unpack(const uint4 &r, float (&v)[8]) {
        const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&r);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __bfloat1622float2(h[i]);
            v[2 * i] = f.x;
            v[2 * i + 1] = f.y;
        }
    }
    static __device__ __forceinline__ uint4 pack(const float (&v)[8]) {
        uint4 r;
        __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(&r);
#pragma unroll
        for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
        return r;
    }
};
template <> struct Pack16<float> {
    static constexpr int E = 4;
    static __device__ __forceinline__ void unpack(const uint4 &r, float (&v)[4]) {
        v[0] = __uint_as_float(r.x); v[1] = __uint_as_float(r.y);
        v[2] = __uint_as_float(r.z); v[3] = __uint_as_float(r.w);
    }
    static __device__ __forceinline__ uint4 pack(const float (&v)[4]) {
        return make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]), __float_as_uint(v[2]),
                          __float_as_uint(v[3]));
    }
};

template <int DV, typename T>
struct NormShape {
    static constexpr int E = Pack16<T>::E;          // elements per lane
    static constexpr int L = DV / E;                // lanes per row
    static constexpr int RW = 32 / L;               // rows per warp per step
    static constexpr int RB = (kNormThreads / 32) * RW * kNormRowsPerThread;   // rows per block
    static_assert(L >= 1 && L <= 32 && 32 % L == 0, "row layout");
};

template <int DV, typename T>
__global__ void __launch_bounds__(kNormThreads)
gated_norm_kernel(const T *__restrict__ y, const T *__restrict__ z, const float *__restrict__ w,
                  T *out, int64_t rows, float eps) {
    using S = NormShape<DV, T>;
    constexpr int E = S::E, L = S::L;
    const int lane = threadIdx.x & 31, l = lane % L;
    // rows of this thread: one per step, a block's worth of rows per step apart
    const int64_t step_rows = (int64_t)(kNormThreads / 32) * S::RW;
    const int64_t r0 = (int64_t)blockIdx.x * S::RB + (threadIdx.x >> 5) * S::RW + lane / L;
    float wt[E];
#pragma unroll
    for (int i = 0; i < E; i += 4) {
        const float4 w4 = *reinterpret_cast<const float4 *>(w + l * E + i);
        wt[i] = w4.x; wt[i + 1] = w4.y; wt[i + 2] = w4.z; wt[i + 3] = w4.w;
    }
    uint4 yr[kNormRowsPerThread], zr[kNormRowsPerThread];
#pragma unroll
    for (int k = 0; k < kNormRowsPerThread; ++k) {
        const int64_t r = r0 + k * step_rows;
        if (r < rows) {
            yr[k] = __ldcs(reinterpret_cast<const uint4 *>(y + r * DV) + l);
            zr[k] = __ldcs(reinterpret_cast<const uint4 *>(z + r * DV) + l);
        } else {
            yr[k] = zr[k] = make_uint4(0u, 0u, 0u, 0u);
        }
    }
#pragma unroll
    for (int k = 0; k < kNormRowsPerThread; ++k) {
        const int64_t r = r0 + k * step_rows;
        float yv[E], zv[E];
        Pack16<T>::unpack(yr[k], yv);
        Pack16<T>::unpack(zr[k], zv);
        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < E; ++i) ss += yv[i] * yv[i];
#pragma unroll
        for (int o = L / 2; o >= 1; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        const float inv = rsqrtf(ss * (1.f / DV) + eps);
        float o[E];
#pragma unroll
        for (int i = 0; i < E; ++i) o[i] = yv[i] * inv * wt[i] * silu_f(zv[i]);
        if (r < rows) __stcs(reinterpret_cast<uint4 *>(out + r * DV) + l, Pack16<T>::pack(o));
    }
}

template <int DV, typename T>
cudaError_t launch_t(const void *y, const void *z, const float *w, void *out, int64_t rows, float eps,
                     cudaStream_t st) {
    const int64_t blocks = (rows + NormShape<DV, T>::RB - 1) / NormShape<DV, T>::RB;
    if (blocks > 0x7fffffff) return cudaErrorInvalidValue;
    gated_norm_kernel<DV, T><<<(unsigned)blocks, kNormThreads, 0, st>>>(
        (const T *)y, (const T *)z, w, (T *)out, rows, eps);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gated_norm(const void *y, const void *z, const float *w, void *out, int64_t rows,
                              int Dv, gdn_dtype dtype, float eps, cudaStream_t st) {
    if (rows == 0) return cudaSuccess;
#define GDN_NORM_CASE(DV_)                                                                   \
    if (Dv == DV_)                                                                           \
        return dtype == GDN_BF16 ? launch_t<DV_, __nv_bfloat16>(y, z, w, out, rows, eps, st)  \
                                 : launch_t<DV_, float>(y, z, w, out, rows, eps, st);
    GDN_NORM_CASE(32) GDN_NORM_CASE(64) GDN_NORM_CASE(128)
#undef GDN_NORM_CASE
    return cudaErrorInvalidValue;
}

}  // namespace gdn
