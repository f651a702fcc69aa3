// gdn_prefill_tc.cu -- chunked prefill of the gated delta rule on the 5th-generation
// tensor cores (tcgen05 + TMEM + TMA), for key_dim = value_dim = 128 and bf16 inputs.
//
// Same chunk algebra as the CUDA-core path (chunks of C = 64 tokens; derived from the
// recurrence of the qwen3_5_text / qwen3_next pages, "The DeltaNet mixer"):
//   (I + A) U = diag(beta) V - diag(beta gamma) K^ S0,  A_tj = beta_t e^{G_t-G_j} k^_t.k^_j (j<t)
//   T = (I + A)^{-1},  W = T diag(beta gamma rk) K,  Ut = T diag(beta) V,  U = Ut - W S0
//   O = diag(rq gamma) Q S0 + P U,  P_tj = e^{G_t-G_j} rq_t rk_j q_t.k_j  (j <= t)
//   S_C = gamma_C S0 + K^T diag(rk e^{G_C-G}) U
// with raw bf16 q, k, v as MMA operands (exact) and every computed operand (T, W, P, U,
// S) split into a bf16 high part and a bf16 residual (hi + lo carries ~16 mantissa bits),
// products accumulated in fp32 in TMEM: x*y ~ hi(x)hi(y) + hi(x)lo(y) + lo(x)hi(y).
//
// Two kernels:
//  prep  -- one CTA per (chunk, value head), all independent: TMA the key tile, Gram
//           K K^T on the tensor core, norms, decay prefix, A, then T = (I + A)^{-1} by a
//           blocked forward substitution in fp32 (16 x 16 diagonal blocks, then block
//           rows).  Writes T and the per-token factors (18 KB per record).
//  chain -- one CTA per (sequence, value head, 32-wide value slice), the sequential
//           chunk loop, warp-specialised:
//             warp 0       TMA producer (key, query tiles, value slice; 2-stage ring)
//             warp 1       MMA issuer of the state-dependent products
//             warps 4-7    "pre" warpgroup, one chunk ahead: query norms, Q K^T -> P,
//                          T' = T diag(beta gamma rk), T'' = T diag(beta) as hi/lo
//                          operands, W^T = K^T T'^T and Ut = T'' V on the tensor core,
//                          W -> -W hi/lo operand
//             warps 8-11   epilogue warpgroup: holds the fp32 state slice in registers
//                          (thread i = key row i), forms U, Z = kd U, O, the new state,
//                          writes outputs (and the per-token states when asked).
// All waits are bounded; a timeout sets GDN_ERR_TIMEOUT in the status word and the CTA
// drains and exits.
#include <string.h>

#include "gdn_internal.cuh"
#include <cudaTypedefs.h>

#include "gdn_sm100.cuh"

namespace gdn {
namespace tc {

using namespace sm100;

constexpr int C = 64;          // chunk
constexpr int D = 128;         // key_dim = value_dim
constexpr int NV = 32;         // value columns per chain CTA
constexpr int kRecFloats = C * C + 8 * C;   // T, then 8 per-token factor rows
enum { SC_C1 = 0, SC_C2, SC_KD, SC_G, SC_RK, SC_ALPHA, SC_GAMMA, SC_MISC };

struct Params {
    const float *g, *beta, *s0;
    __nv_bfloat16 *out;
    float *s_final, *states;
    const int32_t *cu_seqlens;
    int N, T_seq, HK, HV;
    int64_t T_total;
    float scale;
    int l2norm;
    int max_chunks;
    int32_t *status, *chunk_seq, *chunk_first;
    float *rec;                  // [chunks][HV][kRecFloats]
};

// ------------------------------------------------------------------ shared helpers
struct SeqRange {
    int first, count;
    int64_t t0, t_end;
};

__device__ __forceinline__ bool seq_range(const Params &p, int s, SeqRange &r) {
    if (p.cu_seqlens) {
        if (p.status[kStatusWord] != GDN_OK) return false;
        r.first = p.chunk_first[s];
        r.count = p.chunk_first[s + 1] - r.first;
        r.t0 = p.cu_seqlens[s];
        r.t_end = p.cu_seqlens[s + 1];
    } else {
        const int cps = (p.T_seq + C - 1) / C;
        r.first = s * cps;
        r.count = cps;
        r.t0 = (int64_t)s * p.T_seq;
        r.t_end = r.t0 + p.T_seq;
    }
    return true;
}

__device__ __forceinline__ void set_error(const Params &p, int code) {
    atomicCAS(&p.status[kStatusWord], GDN_OK, code);
}

__device__ __forceinline__ void named_sync(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// bf16 hi/lo split of x: hi = bf16(x), lo = bf16(x - hi)
__device__ __forceinline__ void split_bf16(float x, __nv_bfloat16 &hi, __nv_bfloat16 &lo) {
    hi = __float2bfloat16_rn(x);
    lo = __float2bfloat16_rn(x - __bfloat162float(hi));
}

__device__ __forceinline__ uint32_t pack2(__nv_bfloat16 a, __nv_bfloat16 b) {
    return (uint32_t)__bfloat16_as_ushort(a) | ((uint32_t)__bfloat16_as_ushort(b) << 16);
}

// Write one 64-element fp32 row (scaled elementwise by f[]) as hi and lo bf16 rows of
// two K-major 128B-swizzled operand images ([rows][64 elements]).
__device__ __forceinline__ void store_row_hilo(uint8_t *img_hi, uint8_t *img_lo, int row,
                                               const float (&x)[64]) {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        uint32_t h[4], l[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            __nv_bfloat16 h0, l0, h1, l1;
            split_bf16(x[q * 8 + 2 * e], h0, l0);
            split_bf16(x[q * 8 + 2 * e + 1], h1, l1);
            h[e] = pack2(h0, h1);
            l[e] = pack2(l0, l1);
        }
        const uint32_t off = sw128_offset(row, q * 16);
        *reinterpret_cast<uint4 *>(img_hi + off) = make_uint4(h[0], h[1], h[2], h[3]);
        *reinterpret_cast<uint4 *>(img_lo + off) = make_uint4(l[0], l[1], l[2], l[3]);
    }
}

// ================================================================== prep kernel
// smem: key tile (2 x 8 KB, 128B swizzle) | A [64][65] | T [64][65] | X [16][65] | factors
constexpr int kPrepThreads = 128;
constexpr int LDA = C + 1;
constexpr size_t kPrepSmem = 1024 /*align*/ + 16384 + 3 * C * LDA * 4 + 8 * C * 4 + 64;

__global__ void __launch_bounds__(kPrepThreads)
prep_kernel(const __grid_constant__ CUtensorMap mapK, Params p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t su = smem_u32(smem_raw);
    uint8_t *sm = smem_raw + (((su + 1023u) & ~1023u) - su);
    uint8_t *sK = sm;                                   // [2][64][128 B]
    float *sA = reinterpret_cast<float *>(sm + 16384);  // [64][65]
    float *sT = sA + C * LDA;                           // [64][65]
    float *sX = sT + C * LDA;                           // [64][65] scratch (16 rows used)
    float *sG = sX + C * LDA;                           // decay prefix
    float *sB = sG + C;                                 // beta
    float *sRk = sB + C;                                // key normaliser
    float *sg = sRk + C;                                // g
    uint64_t *bar = reinterpret_cast<uint64_t *>(sg + 4 * C);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(bar + 2);

    const int c = blockIdx.x, h = blockIdx.y;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // chunk -> (sequence, first token, length)
    int64_t t0;
    int len;
    if (p.cu_seqlens) {
        if (p.status[kStatusWord] != GDN_OK || c >= p.status[kChunkCountWord]) return;
        const int s = p.chunk_seq[c];
        t0 = p.cu_seqlens[s] + (int64_t)(c - p.chunk_first[s]) * C;
        len = (int)min((int64_t)C, (int64_t)p.cu_seqlens[s + 1] - t0);
    } else {
        const int cps = (p.T_seq + C - 1) / C;
        if (cps == 0 || c >= p.N * cps) return;
        const int s = c / cps, local = c - s * cps;
        t0 = (int64_t)s * p.T_seq + (int64_t)local * C;
        len = min(C, p.T_seq - local * C);
    }
    const int j = h / (p.HV / p.HK);

    if (tid == 0) {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        fence_mbar_init();
        prefetch_tensormap(&mapK);
    }
    if (warp == 0) { tmem_alloc(tslot, 64); tmem_relinquish(); }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;

    if (tid == 0) {
        mbar_arrive_expect_tx(&bar[0], 16384);
        tma_load_3d(sK, &mapK, &bar[0], 0, j, (int)t0);
        tma_load_3d(sK + 8192, &mapK, &bar[0], 64, j, (int)t0);
    }
    // gates of the chunk and the decay prefix (two warps, shuffle scan)
    if (tid < C) {
        const bool in = tid < len;
        const size_t gi = (size_t)(t0 + tid) * p.HV + h;
        float gv = in ? p.g[gi] : 0.f;
        sg[tid] = gv;
        sB[tid] = in ? p.beta[gi] : 0.f;
        float x = gv;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            float y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        sG[tid] = x;   // inclusive within the warp
    }
    bool ok = mbar_wait(&bar[0], 0);
    __syncthreads();
    if (tid >= 32 && tid < C) sG[tid] += sG[31];
    tc_fence_after();
    if (tid == 0 && ok) {
        const uint32_t idesc = instr_desc(64, 64, kFmtBF16, 0, 0);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            const uint32_t a = smem_u32(sK + (ks >> 2) * 8192 + (ks & 3) * 32);
            mma_bf16(tmem, smem_desc(a, 16, 1024, kSwizzle128B), smem_desc(a, 16, 1024, kSwizzle128B),
                     idesc, ks > 0);
        }
        mma_commit(&bar[1]);
    }
    ok = ok && mbar_wait(&bar[1], 0);
    __syncthreads();
    tc_fence_after();
    if (!ok) {
        if (tid == 0) set_error(p, GDN_ERR_TIMEOUT);
        tc_fence_before();
        __syncthreads();
        if (warp == 0) tmem_dealloc(tmem, 64);
        return;
    }
    // Gram rows: M = 64 layout, row t in lane 16 * warp + (lane < 16)
    float kk[64];
    {
        float v[32];
        const uint32_t ta = tmem + ((uint32_t)(warp * 32) << 16);
        tmem_ld32(ta, v);
        tmem_ld_wait();
#pragma unroll
        for (int q = 0; q < 32; ++q) kk[q] = v[q];
        tmem_ld32(ta + 32, v);
        tmem_ld_wait();
#pragma unroll
        for (int q = 0; q < 32; ++q) kk[32 + q] = v[q];
    }
    const int t = warp * 16 + lane;          // valid for lane < 16
    if (lane < 16) {
        float diag = 0.f;
#pragma unroll
        for (int q = 0; q < 64; ++q) diag = (q == t) ? kk[q] : diag;
        sRk[t] = p.l2norm ? rsqrtf(diag + kL2Eps) : 1.f;
    }
    __syncthreads();
    if (lane < 16) {
        const float bt = sB[t], Gt = sG[t], rt = sRk[t];
        const bool live = t < len;
#pragma unroll
        for (int q = 0; q < 64; ++q) {
            float a = 0.f;
            if (live && q < t) a = bt * expf(Gt - sG[q]) * rt * sRk[q] * kk[q];
            sA[t * LDA + q] = a;
        }
    }
    // zero T (upper part stays zero)
    for (int e = tid; e < C * LDA; e += kPrepThreads) sT[e] = 0.f;
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 64);

    // ---- T = (I + A)^{-1}: 16 x 16 diagonal blocks by forward substitution
    if (tid < C) {
        const int b = tid >> 4, cc = tid & 15, base = b * 16;
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            float acc = (r == cc) ? 1.f : 0.f;
#pragma unroll
            for (int k = 0; k < r; ++k) acc -= sA[(base + r) * LDA + base + k] * x[k];
            x[r] = (r < cc) ? 0.f : acc;
        }
#pragma unroll
        for (int r = 0; r < 16; ++r) sT[(base + r) * LDA + base + cc] = x[r];
    }
    __syncthreads();
    // ---- block rows i = 1..3: X = A[i-block, 0:16i] T[0:16i, 0:16i]; T[i, 0:16i] = -T_ii X
    for (int i = 1; i < 4; ++i) {
        const int ncol = 16 * i, nent = 16 * ncol;
        for (int e = tid; e < nent; e += kPrepThreads) {
            const int r = e / ncol, col = e - r * ncol;
            const float *arow = sA + (16 * i + r) * LDA;
            float acc = 0.f;
            for (int m = col; m < ncol; ++m) acc += arow[m] * sT[m * LDA + col];
            sX[r * LDA + col] = acc;
        }
        __syncthreads();
        for (int e = tid; e < nent; e += kPrepThreads) {
            const int r = e / ncol, col = e - r * ncol;
            const float *trow = sT + (16 * i + r) * LDA + 16 * i;
            float acc = 0.f;
            for (int m = 0; m <= r; ++m) acc += trow[m] * sX[m * LDA + col];
            sT[(16 * i + r) * LDA + col] = -acc;
        }
        __syncthreads();
    }

    // ---- record: T row-major, then the per-token factors
    float *rec = p.rec + ((size_t)c * p.HV + h) * kRecFloats;
    for (int e = tid; e < C * C; e += kPrepThreads) rec[e] = sT[(e >> 6) * LDA + (e & 63)];
    float *sc = rec + C * C;
    if (tid < C) {
        const bool in = tid < len;
        const float G = sG[tid], Gl = sG[len - 1], rk = sRk[tid], b = sB[tid];
        const float gam = expf(G);
        sc[SC_C1 * C + tid] = in ? b * gam * rk : 0.f;
        sc[SC_C2 * C + tid] = in ? b : 0.f;
        sc[SC_KD * C + tid] = in ? rk * expf(Gl - G) : 0.f;
        sc[SC_G * C + tid] = G;
        sc[SC_RK * C + tid] = in ? rk : 0.f;
        sc[SC_ALPHA * C + tid] = in ? expf(sg[tid]) : 0.f;
        sc[SC_GAMMA * C + tid] = in ? gam : 0.f;
        sc[SC_MISC * C + tid] = tid == 0 ? expf(Gl) : (tid == 1 ? (float)len : 0.f);
    }
}

// ================================================================== chain kernel
constexpr int kChainThreads = 384;
// shared memory map (bytes from a 1024-aligned base)
constexpr int kStageBytes = 16384 + 16384 + 4096;          // K | Q | V slice
constexpr int OFF_STAGE = 0;                               // [2]
constexpr int OFF_W = OFF_STAGE + 2 * kStageBytes;         // -W hi | lo   [2][64][128B] each
constexpr int OFF_P = OFF_W + 2 * 16384;                   // P hi | lo    [64][128B] each
constexpr int OFF_T1 = OFF_P + 2 * 8192;                   // T' hi | lo
constexpr int OFF_T2 = OFF_T1 + 2 * 8192;                  // T'' hi | lo
constexpr int OFF_VT = OFF_T2 + 2 * 8192;                  // V^T [32][128B]
constexpr int OFF_S = OFF_VT + 4096;                       // S hi | lo   [2][32][128B] each
constexpr int OFF_Z = OFF_S + 2 * 8192;                    // Z hi | lo   [32][128B]
constexpr int OFF_U = OFF_Z + 2 * 4096;                    // U hi | lo
constexpr int OFF_UF = OFF_U + 2 * 4096;                   // U fp32 [64][32] (states)
constexpr int OFF_SC = OFF_UF + C * NV * 4;                // factors [2][16][64] fp32
constexpr int OFF_BAR = OFF_SC + 2 * 16 * C * 4;
constexpr int kChainSmem = OFF_BAR + 256 + 1024;
// factor rows in smem (beyond the 8 record rows)
enum { SCX_RQ = 8, SCX_QD = 9 };

// TMEM columns
constexpr uint32_t TM_QK = 0, TM_W = 64, TM_U0 = 128, TM_QS = 192, TM_S = 224, TM_O = 256;
constexpr uint32_t kTmemCols = 512;

// barriers
enum {
    B_FULL0 = 0, B_FULL1, B_EMPTY0, B_EMPTY1, B_PRE_MMA, B_PRE_U, B_PRE_DONE, B_S_READY,
    B_D1, B_E1, B_D2, B_DO, B_DRAIN, B_DRAIN2, B_COUNT
};

__device__ __forceinline__ uint32_t lane_base(int warp) { return (uint32_t)((warp & 3) * 32) << 16; }

template <bool STATES>
__global__ void __launch_bounds__(kChainThreads, 1)
chain_kernel(const __grid_constant__ CUtensorMap mapK, const __grid_constant__ CUtensorMap mapQ,
             const __grid_constant__ CUtensorMap mapV, Params p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t su = smem_u32(smem_raw);
    uint8_t *sm = smem_raw + (((su + 1023u) & ~1023u) - su);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + OFF_BAR);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + OFF_BAR + 8 * B_COUNT);
    volatile int *s_err = reinterpret_cast<volatile int *>(sm + OFF_BAR + 8 * B_COUNT + 4);

    const int vs = blockIdx.x, h = blockIdx.y, s = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    SeqRange sr;
    if (!seq_range(p, s, sr)) return;
    const int j = h / (p.HV / p.HK);
    const int nch = sr.count;

    if (tid == 0) {
        mbar_init(&bars[B_FULL0], 1);
        mbar_init(&bars[B_FULL1], 1);
        mbar_init(&bars[B_EMPTY0], 2);      // MMA2 commit + epilogue warpgroup
        mbar_init(&bars[B_EMPTY1], 2);
        mbar_init(&bars[B_PRE_MMA], 1);
        mbar_init(&bars[B_PRE_U], 1);
        mbar_init(&bars[B_PRE_DONE], 128);
        mbar_init(&bars[B_S_READY], 128);
        mbar_init(&bars[B_D1], 1);
        mbar_init(&bars[B_E1], 128);
        mbar_init(&bars[B_D2], 1);
        mbar_init(&bars[B_DO], 1);
        mbar_init(&bars[B_DRAIN], 1);
        mbar_init(&bars[B_DRAIN2], 1);
        *s_err = 0;
        fence_mbar_init();
        if (nch > 0) {
            prefetch_tensormap(&mapK);
            prefetch_tensormap(&mapQ);
            prefetch_tensormap(&mapV);
        }
    }
    if (warp == 2) { tmem_alloc(tslot, kTmemCols); tmem_relinquish(); }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;

    auto fail = [&](void) {
        *s_err = 1;
        set_error(p, GDN_ERR_TIMEOUT);
    };
    auto wait = [&](int b, uint32_t parity) -> bool {
        if (*s_err) return false;
        if (!mbar_wait(&bars[b], parity)) { fail(); return false; }
        return true;
    };
    // Warpgroup-uniform wait: one elected thread polls, the warpgroup meets at a
    // named barrier, and every thread takes the same decision from the error flag.
    auto wg_wait = [&](int b, uint32_t parity, int bar_id, bool elected) -> bool {
        if (elected && !*s_err && !mbar_wait(&bars[b], parity)) fail();
        named_sync(bar_id, 128);
        return *s_err == 0;
    };

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            for (int cc = 0; cc < nch; ++cc) {
                const int st = cc & 1, u = cc >> 1;
                if (u >= 1 && !wait(B_EMPTY0 + st, (u - 1) & 1)) break;
                uint8_t *stg = sm + OFF_STAGE + st * kStageBytes;
                const int tok = (int)(sr.t0 + (int64_t)cc * C);
                mbar_arrive_expect_tx(&bars[B_FULL0 + st], kStageBytes);
                tma_load_3d(stg, &mapK, &bars[B_FULL0 + st], 0, j, tok);
                tma_load_3d(stg + 8192, &mapK, &bars[B_FULL0 + st], 64, j, tok);
                tma_load_3d(stg + 16384, &mapQ, &bars[B_FULL0 + st], 0, j, tok);
                tma_load_3d(stg + 24576, &mapQ, &bars[B_FULL0 + st], 64, j, tok);
                tma_load_3d(stg + 32768, &mapV, &bars[B_FULL0 + st], vs * NV, h, tok);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t id_64x32 = instr_desc(64, NV, kFmtBF16, 0, 0);
            const uint32_t id_128x32_amn = instr_desc(128, NV, kFmtBF16, 1, 0);
            bool issued = false;
            for (int cc = 0; cc < nch; ++cc) {
                const int st = cc & 1;
                uint8_t *stg = sm + OFF_STAGE + st * kStageBytes;
                if (!wait(B_FULL0 + st, (cc >> 1) & 1) || !wait(B_PRE_DONE, cc & 1) ||
                    !wait(B_S_READY, cc & 1))
                    break;
                tc_fence_after();
                // MMA1: D_U += (-W) S  (3 hi/lo terms);  D_QS = Q S  (2 terms)
                const uint32_t dU = tmem + TM_U0 + (uint32_t)(st * NV);
#pragma unroll 1
                for (int ks = 0; ks < 8; ++ks) {
                    const int kb = ks >> 2, ko = (ks & 3) * 32;
                    const uint32_t wh = smem_u32(sm + OFF_W + kb * 8192 + ko);
                    const uint32_t wl = wh + 16384;
                    const uint32_t sh = smem_u32(sm + OFF_S + kb * 4096 + ko);
                    const uint32_t sl = sh + 8192;
                    const uint32_t qa = smem_u32(stg + 16384 + kb * 8192 + ko);
                    mma_bf16(dU, smem_desc(wh, 16, 1024, kSwizzle128B), smem_desc(sh, 16, 1024, kSwizzle128B), id_64x32, 1);
                    mma_bf16(dU, smem_desc(wh, 16, 1024, kSwizzle128B), smem_desc(sl, 16, 1024, kSwizzle128B), id_64x32, 1);
                    mma_bf16(dU, smem_desc(wl, 16, 1024, kSwizzle128B), smem_desc(sh, 16, 1024, kSwizzle128B), id_64x32, 1);
                    mma_bf16(tmem + TM_QS, smem_desc(qa, 16, 1024, kSwizzle128B), smem_desc(sh, 16, 1024, kSwizzle128B), id_64x32, ks > 0);
                    mma_bf16(tmem + TM_QS, smem_desc(qa, 16, 1024, kSwizzle128B), smem_desc(sl, 16, 1024, kSwizzle128B), id_64x32, 1);
                }
                mma_commit(&bars[B_D1]);
                issued = true;
                if (!wait(B_E1, cc & 1)) break;
                tc_fence_after();
                // MMA2: D_S = K^T (Z hi + Z lo)   (A = key tile, MN-major)
#pragma unroll 1
                for (int ks = 0; ks < 4; ++ks) {
                    const uint32_t ka = smem_u32(stg + ks * 2048);
                    const uint32_t zh = smem_u32(sm + OFF_Z + ks * 32);
                    mma_bf16(tmem + TM_S, smem_desc(ka, 8192, 1024, kSwizzle128B), smem_desc(zh, 16, 1024, kSwizzle128B), id_128x32_amn, ks > 0);
                    mma_bf16(tmem + TM_S, smem_desc(ka, 8192, 1024, kSwizzle128B), smem_desc(zh + 4096, 16, 1024, kSwizzle128B), id_128x32_amn, 1);
                }
                mma_commit(&bars[B_D2]);
                mma_commit(&bars[B_EMPTY0 + st]);
                // MMA_O: D_O = P U  (3 hi/lo terms)
#pragma unroll 1
                for (int ks = 0; ks < 4; ++ks) {
                    const uint32_t ph = smem_u32(sm + OFF_P + ks * 32), pl = ph + 8192;
                    const uint32_t uh = smem_u32(sm + OFF_U + ks * 32), ul = uh + 4096;
                    mma_bf16(tmem + TM_O, smem_desc(ph, 16, 1024, kSwizzle128B), smem_desc(uh, 16, 1024, kSwizzle128B), id_64x32, ks > 0);
                    mma_bf16(tmem + TM_O, smem_desc(ph, 16, 1024, kSwizzle128B), smem_desc(ul, 16, 1024, kSwizzle128B), id_64x32, 1);
                    mma_bf16(tmem + TM_O, smem_desc(pl, 16, 1024, kSwizzle128B), smem_desc(uh, 16, 1024, kSwizzle128B), id_64x32, 1);
                }
                mma_commit(&bars[B_DO]);
            }
            if (issued) {   // let every MMA of this thread finish before teardown
                mma_commit(&bars[B_DRAIN]);
                mbar_wait(&bars[B_DRAIN], 0);
            }
        }
    } else if (warp >= 4 && warp < 8) {
        // ------------------------------------------------------------ pre warpgroup
        const int ptid = tid - 128, pw = warp & 3;
        const bool lead = (ptid == 0);
        const uint32_t lb = lane_base(warp);
        const uint32_t id_qk = instr_desc(64, 64, kFmtBF16, 0, 0);
        const uint32_t id_w = instr_desc(128, 64, kFmtBF16, 1, 0);
        const uint32_t id_u = instr_desc(64, NV, kFmtBF16, 0, 0);
        float *scs = reinterpret_cast<float *>(sm + OFF_SC);   // pre-private factors
        bool leader_issued = false;
        uint32_t pre_mma_phase = 0, pre_u_phase = 0;
        for (int cc = 0; cc < nch; ++cc) {
            const int st = cc & 1, u = cc >> 1;
            uint8_t *stg = sm + OFF_STAGE + st * kStageBytes;
            const float *rec = p.rec + ((size_t)(sr.first + cc) * p.HV + h) * kRecFloats;
            if (!wg_wait(B_FULL0 + st, u & 1, 1, lead)) break;
            // factors: c1, c2, G, rk from the record; rq from the query tile (the swizzle
            // only permutes 16-byte chunks inside a row, so the sum needs no unswizzle)
            for (int e = ptid; e < 8 * C; e += 128) scs[e] = rec[C * C + e];
            if (ptid < C) {
                float ss = 0.f;
#pragma unroll
                for (int kb = 0; kb < 2; ++kb)
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const uint4 w4 = *reinterpret_cast<const uint4 *>(stg + 16384 + kb * 8192 + ptid * 128 + q * 16);
                        const __nv_bfloat162 *b2 = reinterpret_cast<const __nv_bfloat162 *>(&w4);
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 f = __bfloat1622float2(b2[e]);
                            ss += f.x * f.x + f.y * f.y;
                        }
                    }
                scs[SCX_RQ * C + ptid] = p.l2norm ? p.scale * rsqrtf(ss + kL2Eps) : p.scale;
            }
            if (lead) {
                tc_fence_after();
                // Q K^T (M = 64, N = 64, K = 128) into D_QK
#pragma unroll 1
                for (int ks = 0; ks < 8; ++ks) {
                    const int kb = ks >> 2, ko = (ks & 3) * 32;
                    const uint32_t qa = smem_u32(stg + 16384 + kb * 8192 + ko);
                    const uint32_t ka = smem_u32(stg + kb * 8192 + ko);
                    mma_bf16(tmem + TM_QK, smem_desc(qa, 16, 1024, kSwizzle128B),
                             smem_desc(ka, 16, 1024, kSwizzle128B), id_qk, ks > 0);
                }
                leader_issued = true;
            }
            named_sync(1, 128);            // factors visible
            // T' = T diag(c1), T'' = T diag(c2) as hi/lo operands; V^T operand
            if (ptid < C) {
                const int t = ptid;
                float x[64];
                const float4 *tr = reinterpret_cast<const float4 *>(rec + t * C);
#pragma unroll
                for (int q = 0; q < 16; ++q) {
                    const float4 v4 = tr[q];
                    x[4 * q] = v4.x * scs[SC_C1 * C + 4 * q];
                    x[4 * q + 1] = v4.y * scs[SC_C1 * C + 4 * q + 1];
                    x[4 * q + 2] = v4.z * scs[SC_C1 * C + 4 * q + 2];
                    x[4 * q + 3] = v4.w * scs[SC_C1 * C + 4 * q + 3];
                }
                store_row_hilo(sm + OFF_T1, sm + OFF_T1 + 8192, t, x);
#pragma unroll
                for (int q = 0; q < 16; ++q) {
                    const float4 v4 = tr[q];
                    x[4 * q] = v4.x * scs[SC_C2 * C + 4 * q];
                    x[4 * q + 1] = v4.y * scs[SC_C2 * C + 4 * q + 1];
                    x[4 * q + 2] = v4.z * scs[SC_C2 * C + 4 * q + 2];
                    x[4 * q + 3] = v4.w * scs[SC_C2 * C + 4 * q + 3];
                }
                store_row_hilo(sm + OFF_T2, sm + OFF_T2 + 8192, t, x);
            } else {
                // V^T: [32 value rows][64 tokens] from the staged [64 tokens][32 values]
                const __nv_bfloat16 *vsrc = reinterpret_cast<const __nv_bfloat16 *>(stg + 32768);
                for (int e = ptid - 64; e < NV * 8; e += 64) {
                    const int cv = e >> 3, q = e & 7;
                    uint32_t w[4];
#pragma unroll
                    for (int ee = 0; ee < 4; ++ee)
                        w[ee] = pack2(vsrc[(q * 8 + 2 * ee) * NV + cv], vsrc[(q * 8 + 2 * ee + 1) * NV + cv]);
                    *reinterpret_cast<uint4 *>(sm + OFF_VT + sw128_offset(cv, q * 16)) =
                        make_uint4(w[0], w[1], w[2], w[3]);
                }
            }
            fence_async_smem();
            named_sync(1, 128);
            if (lead) {
                tc_fence_after();
                // W^T = K^T T'^T (M = 128 keys, N = 64 tokens, K = 64 tokens), A MN-major
#pragma unroll 1
                for (int ks = 0; ks < 4; ++ks) {
                    const uint32_t ka = smem_u32(stg + ks * 2048);
                    const uint32_t th = smem_u32(sm + OFF_T1 + ks * 32);
                    mma_bf16(tmem + TM_W, smem_desc(ka, 8192, 1024, kSwizzle128B),
                             smem_desc(th, 16, 1024, kSwizzle128B), id_w, ks > 0);
                    mma_bf16(tmem + TM_W, smem_desc(ka, 8192, 1024, kSwizzle128B),
                             smem_desc(th + 8192, 16, 1024, kSwizzle128B), id_w, 1);
                }
                mma_commit(&bars[B_PRE_MMA]);
            }
            // the previous chunk's MMA1 must have consumed the -W operand and, through the
            // s_ready handshake, the epilogue must be done with D_U[cc % 2]
            if (cc >= 1 && !wg_wait(B_D1, (cc - 1) & 1, 1, lead)) break;
            if (lead) {
                tc_fence_after();
                // Ut = T'' V into D_U[cc % 2] (M = 64, N = 32, K = 64)
                const uint32_t dU = tmem + TM_U0 + (uint32_t)(st * NV);
#pragma unroll 1
                for (int ks = 0; ks < 4; ++ks) {
                    const uint32_t ta = smem_u32(sm + OFF_T2 + ks * 32);
                    const uint32_t vb = smem_u32(sm + OFF_VT + ks * 32);
                    mma_bf16(dU, smem_desc(ta, 16, 1024, kSwizzle128B),
                             smem_desc(vb, 16, 1024, kSwizzle128B), id_u, ks > 0);
                    mma_bf16(dU, smem_desc(ta + 8192, 16, 1024, kSwizzle128B),
                             smem_desc(vb, 16, 1024, kSwizzle128B), id_u, 1);
                }
                mma_commit(&bars[B_PRE_U]);
            }
            // W^T from TMEM (lane = key i) -> -W hi/lo into the MMA1 A operand
            if (!wg_wait(B_PRE_MMA, pre_mma_phase & 1, 1, lead)) break;
            ++pre_mma_phase;
            tc_fence_after();
            {
                const int i = ptid;
                float wv[32];
                uint8_t *wh = sm + OFF_W + (i >> 6) * 8192;
                const uint32_t byte = (uint32_t)(i & 63) * 2;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    tmem_ld32(tmem + lb + TM_W + half * 32, wv);
                    tmem_ld_wait();
#pragma unroll
                    for (int q = 0; q < 32; ++q) {
                        __nv_bfloat16 hi, lo;
                        split_bf16(-wv[q], hi, lo);
                        const uint32_t off = sw128_offset(half * 32 + q, byte);
                        *reinterpret_cast<__nv_bfloat16 *>(wh + off) = hi;
                        *reinterpret_cast<__nv_bfloat16 *>(wh + 16384 + off) = lo;
                    }
                }
            }
            // P from Q K^T (rows t = 16 pw + lane, lane < 16), once the previous chunk's
            // MMA_O has consumed the P operand
            if (cc >= 1 && !wg_wait(B_DO, (cc - 1) & 1, 1, lead)) break;
            tc_fence_after();
            {
                float qk[64], v[32];
                tmem_ld32(tmem + lb + TM_QK, v);
                tmem_ld_wait();
#pragma unroll
                for (int q = 0; q < 32; ++q) qk[q] = v[q];
                tmem_ld32(tmem + lb + TM_QK + 32, v);
                tmem_ld_wait();
#pragma unroll
                for (int q = 0; q < 32; ++q) qk[32 + q] = v[q];
                if (lane < 16) {
                    const int t = pw * 16 + lane;
                    const float Gt = scs[SC_G * C + t], rq = scs[SCX_RQ * C + t];
#pragma unroll
                    for (int q = 0; q < 64; ++q)
                        qk[q] = (q <= t) ? expf(Gt - scs[SC_G * C + q]) * rq * scs[SC_RK * C + q] * qk[q] : 0.f;
                    store_row_hilo(sm + OFF_P, sm + OFF_P + 8192, t, qk);
                }
            }
            fence_async_smem();
            tc_fence_before();
            if (!wg_wait(B_PRE_U, pre_u_phase & 1, 1, lead)) break;
            ++pre_u_phase;
            mbar_arrive(&bars[B_PRE_DONE]);
        }
        if (lead && leader_issued) {
            mma_commit(&bars[B_DRAIN2]);
            mbar_wait(&bars[B_DRAIN2], 0);
        }
    } else if (warp >= 8) {
        // ------------------------------------------------------------ epilogue warpgroup
        const int i = tid - 256;            // key row of the state slice
        const bool lead = (i == 0);
        const uint32_t lb = lane_base(warp);
        const int ew = warp & 3;
        float S[NV];
        const size_t sbase = (((size_t)s * p.HV + h) * D + i) * D + (size_t)vs * NV;
        if (p.s0) {
#pragma unroll
            for (int q = 0; q < NV / 4; ++q) {
                const float4 v4 = reinterpret_cast<const float4 *>(p.s0 + sbase)[q];
                S[4 * q] = v4.x; S[4 * q + 1] = v4.y; S[4 * q + 2] = v4.z; S[4 * q + 3] = v4.w;
            }
        } else {
#pragma unroll
            for (int q = 0; q < NV; ++q) S[q] = 0.f;
        }
        auto write_state_operand = [&]() {
            uint8_t *img = sm + OFF_S + (i >> 6) * 4096;
            const uint32_t byte = (uint32_t)(i & 63) * 2;
#pragma unroll
            for (int c = 0; c < NV; ++c) {
                __nv_bfloat16 hi, lo;
                split_bf16(S[c], hi, lo);
                const uint32_t off = sw128_offset(c, byte);
                *reinterpret_cast<__nv_bfloat16 *>(img + off) = hi;
                *reinterpret_cast<__nv_bfloat16 *>(img + 8192 + off) = lo;
            }
        };
        write_state_operand();
        fence_async_smem();
        mbar_arrive(&bars[B_S_READY]);
        float *uf = reinterpret_cast<float *>(sm + OFF_UF);
        for (int cc = 0; cc < nch; ++cc) {
            const int st = cc & 1, u = cc >> 1;
            const uint8_t *stg = sm + OFF_STAGE + st * kStageBytes;
            const float *fac = p.rec + ((size_t)(sr.first + cc) * p.HV + h) * kRecFloats + C * C;
            const int64_t tok0 = sr.t0 + (int64_t)cc * C;
            const int len = (int)min((int64_t)C, sr.t_end - tok0);
            // the stage's tiles (query norms here, key rows for the states) are loaded
            if (!wg_wait(B_FULL0 + st, u & 1, 2, lead)) break;
            if (!wg_wait(B_D1, cc & 1, 2, lead)) break;
            tc_fence_after();
            // E1: U rows and Q S rows (M = 64 layout: row t = 16 ew + lane for lane < 16)
            float op[NV];
            {
                float uu[NV], qs[NV];
                tmem_ld32(tmem + lb + TM_U0 + (uint32_t)(st * NV), uu);
                tmem_ld32(tmem + lb + TM_QS, qs);
                tmem_ld_wait();
                if (lane < 16) {
                    const int t = ew * 16 + lane;
                    float ss = 0.f;
#pragma unroll
                    for (int kb = 0; kb < 2; ++kb)
#pragma unroll
                        for (int q = 0; q < 8; ++q) {
                            const uint4 w4 = *reinterpret_cast<const uint4 *>(stg + 16384 + kb * 8192 + t * 128 + q * 16);
                            const __nv_bfloat162 *b2 = reinterpret_cast<const __nv_bfloat162 *>(&w4);
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float2 f = __bfloat1622float2(b2[e]);
                                ss += f.x * f.x + f.y * f.y;
                            }
                        }
                    const float rq = p.l2norm ? p.scale * rsqrtf(ss + kL2Eps) : p.scale;
                    const float qd = rq * fac[SC_GAMMA * C + t], kd = fac[SC_KD * C + t];
                    const uint32_t byte = (uint32_t)t * 2;
#pragma unroll
                    for (int c = 0; c < NV; ++c) {
                        op[c] = qd * qs[c];
                        __nv_bfloat16 hi, lo;
                        const uint32_t off = sw128_offset(c, byte);
                        split_bf16(kd * uu[c], hi, lo);
                        *reinterpret_cast<__nv_bfloat16 *>(sm + OFF_Z + off) = hi;
                        *reinterpret_cast<__nv_bfloat16 *>(sm + OFF_Z + 4096 + off) = lo;
                        split_bf16(uu[c], hi, lo);
                        *reinterpret_cast<__nv_bfloat16 *>(sm + OFF_U + off) = hi;
                        *reinterpret_cast<__nv_bfloat16 *>(sm + OFF_U + 4096 + off) = lo;
                    }
                    if (STATES) {
#pragma unroll
                        for (int c = 0; c < NV; c += 4)
                            *reinterpret_cast<float4 *>(uf + t * NV + c) =
                                make_float4(uu[c], uu[c + 1], uu[c + 2], uu[c + 3]);
                    }
                }
            }
            fence_async_smem();
            tc_fence_before();
            mbar_arrive(&bars[B_E1]);
            // E2: new state (thread i = key row i)
            if (!wg_wait(B_D2, cc & 1, 2, lead)) break;
            tc_fence_after();
            float ds[NV];
            tmem_ld32(tmem + lb + TM_S, ds);
            tmem_ld_wait();
            const float gl = fac[SC_MISC * C + 0];
            if (STATES) {
                const uint8_t *ktile = stg + (i >> 6) * 8192;
                const uint32_t kbyte = (uint32_t)(i & 63) * 2;
                float run[NV];
#pragma unroll
                for (int c = 0; c < NV; ++c) run[c] = S[c];
                for (int t = 0; t < len; ++t) {
                    const float kt = __bfloat162float(
                        *reinterpret_cast<const __nv_bfloat16 *>(ktile + sw128_offset(t, kbyte)));
                    const float al = fac[SC_ALPHA * C + t], f = fac[SC_RK * C + t] * kt;
                    float *dst = p.states + (((size_t)(tok0 + t) * p.HV + h) * D + i) * D + (size_t)vs * NV;
                    const bool last = (t == len - 1);
#pragma unroll
                    for (int c = 0; c < NV; c += 4) {
                        const float4 u4 = *reinterpret_cast<const float4 *>(uf + t * NV + c);
                        run[c] = al * run[c] + f * u4.x;
                        run[c + 1] = al * run[c + 1] + f * u4.y;
                        run[c + 2] = al * run[c + 2] + f * u4.z;
                        run[c + 3] = al * run[c + 3] + f * u4.w;
                        const float4 o4 = last
                            ? make_float4(gl * S[c] + ds[c], gl * S[c + 1] + ds[c + 1],
                                          gl * S[c + 2] + ds[c + 2], gl * S[c + 3] + ds[c + 3])
                            : make_float4(run[c], run[c + 1], run[c + 2], run[c + 3]);
                        __stcs(reinterpret_cast<float4 *>(dst + c), o4);
                    }
                }
            }
#pragma unroll
            for (int c = 0; c < NV; ++c) S[c] = gl * S[c] + ds[c];
            write_state_operand();
            fence_async_smem();
            // outputs
            if (!wg_wait(B_DO, cc & 1, 2, lead)) break;
            tc_fence_after();
            {
                float dov[NV];
                tmem_ld32(tmem + lb + TM_O, dov);
                tmem_ld_wait();
                if (lane < 16) {
                    const int t = ew * 16 + lane;
                    if (t < len) {
                        __nv_bfloat16 *dst = p.out + ((size_t)(tok0 + t) * p.HV + h) * D + (size_t)vs * NV;
#pragma unroll
                        for (int c = 0; c < NV; c += 8) {
                            uint32_t w[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                w[e] = pack2(__float2bfloat16_rn(op[c + 2 * e] + dov[c + 2 * e]),
                                             __float2bfloat16_rn(op[c + 2 * e + 1] + dov[c + 2 * e + 1]));
                            *reinterpret_cast<uint4 *>(dst + c) = make_uint4(w[0], w[1], w[2], w[3]);
                        }
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(&bars[B_S_READY]);
            named_sync(2, 128);              // every reader of the stage and of uf is done
            if (lead) mbar_arrive(&bars[B_EMPTY0 + st]);
        }
        // final state slice
        if (!*s_err) {
#pragma unroll
            for (int q = 0; q < NV / 4; ++q)
                reinterpret_cast<float4 *>(p.s_final + sbase)[q] =
                    make_float4(S[4 * q], S[4 * q + 1], S[4 * q + 2], S[4 * q + 3]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 2) tmem_dealloc(tmem, kTmemCols);
}

// ================================================================== host side
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        cudaDriverEntryPointQueryResult q;
        void *f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess && q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }
    return fn;
}

// [T_total][heads][128] bf16 viewed as 3-D (element, head, token), box {box_x, 1, 64}
static bool make_map(CUtensorMap *m, const void *base, int heads, int64_t T_total, int box_x,
                     bool swizzle) {
    auto enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)heads, (cuuint64_t)T_total};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)heads * D * 2};
    cuuint32_t box[3] = {(cuuint32_t)box_x, 1, (cuuint32_t)C};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides,
                     box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace tc

size_t tc_record_bytes() { return (size_t)tc::kRecFloats * sizeof(float); }

bool tc_supported(int Dk, int Dv, gdn_dtype dtype) {
    return Dk == tc::D && Dv == tc::D && dtype == GDN_BF16;
}

cudaError_t launch_prefill_tc(const PrefillParams &pp, cudaStream_t st) {
    using namespace tc;
    cudaError_t e;
    if (pp.cu_seqlens) {
        if ((e = launch_chunk_table(pp, st)) != cudaSuccess) return e;
    }
    Params p;
    memset(&p, 0, sizeof p);
    p.g = pp.g; p.beta = pp.beta; p.s0 = pp.s0;
    p.out = (__nv_bfloat16 *)pp.out; p.s_final = pp.s_final; p.states = pp.states;
    p.cu_seqlens = pp.cu_seqlens; p.N = pp.N; p.T_seq = pp.T_seq; p.T_total = pp.T_total;
    p.HK = pp.HK; p.HV = pp.HV; p.scale = pp.scale; p.l2norm = pp.l2norm;
    p.max_chunks = pp.max_chunks; p.status = pp.status; p.chunk_seq = pp.chunk_seq;
    p.chunk_first = pp.chunk_first; p.rec = pp.rec;
    CUtensorMap mk, mq, mv;
    if (pp.T_total > 0) {
        if (!make_map(&mk, pp.k, pp.HK, pp.T_total, 64, true) ||
            !make_map(&mq, pp.q, pp.HK, pp.T_total, 64, true) ||
            !make_map(&mv, pp.v, pp.HV, pp.T_total, NV, false))
            return cudaErrorInvalidValue;
    } else {
        memset(&mk, 0, sizeof mk); memset(&mq, 0, sizeof mq); memset(&mv, 0, sizeof mv);
    }
    if (pp.max_chunks > 0) {
        if ((e = cudaFuncSetAttribute(prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)kPrepSmem)) != cudaSuccess)
            return e;
        prep_kernel<<<dim3(pp.max_chunks, pp.HV), kPrepThreads, kPrepSmem, st>>>(mk, p);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if (pp.N > 0) {
        auto kern = pp.states ? chain_kernel<true> : chain_kernel<false>;
        if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      kChainSmem)) != cudaSuccess)
            return e;
        kern<<<dim3(D / NV, pp.HV, pp.N), kChainThreads, kChainSmem, st>>>(mk, mq, mv, p);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace gdn
