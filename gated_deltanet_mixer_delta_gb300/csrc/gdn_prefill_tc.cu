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
//  prep  -- one CTA per (chunk, one or two value heads of a key head), all independent:
//           TMA the key and query tiles, Gram K K^T and Q K^T on the tensor core, norms,
//           decay prefix, A, then T = (I + A)^{-1} in place of A by a blocked forward
//           substitution in fp32 (16 x 16 diagonal blocks, then doubling),
//           W^T = K^T T'^T on the tensor core, P; writes -W (hi/lo), T'' (hi/lo) and P
//           as operand images, and the per-token factors.
//  chain -- one CTA per (sequence, value head, 32-wide value slice), the sequential
//           chunk loop (or, when an equal-length batch has more of these chains than the
//           GPU has SMs, one persistent CTA per SM running a stream of chain segments
//           whose states pass between CTAs), warp-specialised (256 threads): a TMA
//           producer warp, a warp that
//           issues the products off the chain's critical path, two output warps, and an
//           epilogue warpgroup that holds the fp32 state slice in registers (thread i =
//           key row i), forms U, Z = kd U and the new state, and issues the products
//           on the critical path itself.  Hi/lo operand pairs are stacked along M or N so
//           that one instruction covers several terms.
//  states -- only when per-token states are asked for: the chain leaves each chunk's U
//           rows and its carried state in the states tensor, and one CTA per (chunk,
//           value head, value slice), all independent, replays the recurrence over the
//           chunk's tokens from there (then a small kernel copies the final states).
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
// Record of one (chunk, value head), written by the prep kernel and bulk-copied as is
// into the chain kernel's shared memory.  Operand images are bf16, 128B-swizzled, ready
// for the tensor core:
//   -W hi, -W lo  [128 keys][64 tokens]   MN-major; stacked along M they are the A
//                                          operand [-W_hi; -W_lo] of (-W) S   16 KiB each
//   T'' hi, lo    [64 tokens][64 tokens]  K-major; stacked, the A operand of T'' V
//                                                                            8 KiB each
//   P             [64 tokens][64 tokens]  K-major A operand of P U          8 KiB
//   factors       8 rows of 64 floats (qd, kd, rk, alpha, misc, 3 unused)  2 KiB
constexpr int REC_WHI = 0, REC_WLO = 16384, REC_T2HI = 32768, REC_T2LO = 40960, REC_P = 49152,
              REC_F = 57344;
constexpr int kRecBytes = REC_F + 8 * C * 4;                // 58 KiB
enum { SC_QD = 0, SC_KD, SC_RK, SC_ALPHA, SC_MISC };

struct Params {
    const __nv_bfloat16 *k;      // keys [T_total][HK][128] (read by the states kernel)
    const float *g, *beta, *s0;
    __nv_bfloat16 *out;
    float *s_final, *states;
    const int32_t *cu_seqlens;
    int N, T_seq, HK, HV;
    int64_t T_total;
    float scale;
    int l2norm;
    int max_chunks;
    int32_t *status, *chunk_seq, *chunk_first, *seq_order;
    float *rec;                  // [chunks][HV] records of kRecBytes
    // the chain kernel's work-unit stream: a unit is a run of at most seg_len consecutive
    // chunks of one of the n_chains (sequence, value head, value slice) chains
    int32_t *chain_flags;        // [n_chains] segments of the chain whose end state is out
    int seg_len, n_chains, n_units;
    int states_overlap;          // the states kernel takes each segment as the stream ends it
    int final_direct;            // with per-token states, the stream writes the final states
                                 // too (final_state does not alias initial_state)
    // prep beside the chain: prep_items > 0 makes the prep grid persistent over that many
    // items; CTAs on SMs below prep_stay_sms keep claiming after prep_limit items, and
    // every record's flag in ready is set once the record is complete
    int32_t *ready;              // [chunks][HV] or null (the chain waits for the prep grid)
    int prep_items, prep_limit, prep_stay_sms;
    int prep_slots;              // prep CTAs resident at once (one CTA per item: L2 prefetch distance)
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
// the same for two values at once, packed (a in the low half): one conversion per word
__device__ __forceinline__ void split2_bf16(float a, float b, uint32_t &hi, uint32_t &lo) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    const float2 hf = __bfloat1622float2(h);
    float ra, rb;                                   // (a - hi, b - hi) in one instruction
    f2unpack(ffma2(f2pack(-1.f, -1.f), f2pack(hf.x, hf.y), f2pack(a, b)), ra, rb);
    const __nv_bfloat162 l = __floats2bfloat162_rn(ra, rb);
    hi = *reinterpret_cast<const uint32_t *>(&h);
    lo = *reinterpret_cast<const uint32_t *>(&l);
}

__device__ __forceinline__ uint32_t pack2(__nv_bfloat16 a, __nv_bfloat16 b) {
    return (uint32_t)__bfloat16_as_ushort(a) | ((uint32_t)__bfloat16_as_ushort(b) << 16);
}

// 32 consecutive elements of a row (chunks c0 .. c0+3 of 16 bytes) of two K-major,
// 128B-swizzled bf16 operand images: hi and lo parts of x.
__device__ __forceinline__ void store_half_row_hilo(uint8_t *img_hi, uint8_t *img_lo, int row,
                                                    int c0, const float (&x)[32]) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint32_t h[4], l[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) split2_bf16(x[q * 8 + 2 * e], x[q * 8 + 2 * e + 1], h[e], l[e]);
        const uint32_t off = sw128_offset(row, (c0 + q) * 16);
        *reinterpret_cast<uint4 *>(img_hi + off) = make_uint4(h[0], h[1], h[2], h[3]);
        *reinterpret_cast<uint4 *>(img_lo + off) = make_uint4(l[0], l[1], l[2], l[3]);
    }
}

// 32 consecutive elements of a row of one K-major, 128B-swizzled bf16 operand image.
__device__ __forceinline__ void store_half_row_bf16(uint8_t *img, int row, int c0,
                                                    const float (&x)[32]) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint32_t h[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const __nv_bfloat162 v = __floats2bfloat162_rn(x[q * 8 + 2 * e], x[q * 8 + 2 * e + 1]);
            h[e] = *reinterpret_cast<const uint32_t *>(&v);
        }
        *reinterpret_cast<uint4 *>(img + sw128_offset(row, (c0 + q) * 16)) = make_uint4(h[0], h[1], h[2], h[3]);
    }
}

// ================================================================== prep kernel
// One CTA per (chunk, HPC value heads that share a key head): HPC = 2 when the number of
// value heads per key head is even, else 1.  The key and query tiles, K K^T, Q K^T and the
// norms are shared by the CTA's heads, and the heads go through every step side by side,
// so that they share the barriers and their independent work fills each other's latency.
// The record images are assembled in shared memory and written with bulk copies (whole
// lines, off the threads' critical path).
// smem (from a 1024-aligned base):
//   key tile   [2][64][128 B], 128B swizzle (TMA)
//   query tile [2][64][128 B], 128B swizzle (TMA); once Q K^T is done it stages the P
//              images, then holds the X scratch of the solve ([HPC][1152] fp32), then
//              the T' hi/lo operand images of one head at a time
//   A/T [HPC][64][68] fp32: A of each head, overwritten in place by T = (I + A)^{-1},
//              then by the T'' images of the head, then (two heads) by -W of head 0
//   rk, rq | per head: G, G log2(e), beta, beta gamma rk | barriers
// After the last product the key and query tiles stage -W of the last head.
constexpr int kPrepThreads = 128;
constexpr int kPrepPerSm = 3;                                // CTAs per SM (launch bounds)
constexpr int LDA = C + 4;
constexpr int LDX = 36;                                      // X scratch rows (32 columns used)
constexpr int kXHead = 2 * 16 * LDX;                         // == 32 * LDX floats per head
constexpr int kPrepVecHead = 4;
template <int HPC>
constexpr size_t prep_smem_bytes() {
    return 1024 /*align*/ + 32768 + (size_t)HPC * C * LDA * 4 +
           (size_t)(2 + HPC * kPrepVecHead) * C * 4 + 64;
}
static_assert(5 * 8 + 5 * 4 <= 64, "barriers, TMEM slot, item, pending item and ticket words");
static_assert(2 * kXHead * 4 <= 16384, "solve scratch of two heads fits the query tile");
static_assert(2 * C * LDA * 4 >= 32768 && C * LDA * 4 >= 16384, "A/T tiles stage the images");
static_assert(REC_T2LO == REC_T2HI + 8192 && REC_WLO == REC_WHI + 16384, "record layout");
constexpr uint32_t kPrepTmemCols = 128;                      // K K^T | Q K^T, then W^T of head 0 | 1

// 2^x on the MUFU unit (relative error ~2^-22); underflows to 0.
__device__ __forceinline__ float ex2_fast(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float4 lds4(const float *p) { return *reinterpret_cast<const float4 *>(p); }
__device__ __forceinline__ void sts4(float *p, float a, float b, float c, float d) {
    *reinterpret_cast<float4 *>(p) = make_float4(a, b, c, d);
}
__device__ __forceinline__ float f4get(const float4 &v, int e) {
    return e == 0 ? v.x : (e == 1 ? v.y : (e == 2 ? v.z : v.w));
}

// One row of an M = 64 accumulator pair (columns c0 .. c0+63) spread over a warp: the
// rows sit in lanes 0-15 (row 16 * (warp % 4) + lane); lane l < 16 keeps columns 0-31
// of its row, lane l + 16 receives columns 32-63 of the same row.
__device__ __forceinline__ void tmem_row_split(uint32_t taddr, float (&x)[32]) {
    float v1[32], v2[32];
    tmem_ld32(taddr, v1);
    tmem_ld32(taddr + 32, v2);
    tmem_ld_wait();
    const int lane = threadIdx.x & 31, src = lane & 15, cb = lane >> 4;
#pragma unroll
    for (int q = 0; q < 32; ++q) {
        const float r2 = __shfl_sync(0xffffffffu, v2[q], src);
        x[q] = cb ? r2 : v1[q];
    }
}

// Off-diagonal block of T = (I + A)^{-1} from two diagonal blocks already in T, with A
// and T in one array (T overwrites A block by block):
//   X = A[rows, cols] T[cols, cols];  T[rows, cols] = -T[rows, rows] X
// for an N x N block (N = 16 or 32) at row offset r0 and column offset c0.  Thread
// (tr, tc) owns rows tr, tr + 8, .. (RT of them) and columns 4 tc .. 4 tc + 3 of the block:
// per k-step it reads one float4 of each of its rows and one float4 of the right-hand
// factor, so that the eight lanes of a quarter-warp hit distinct banks.  Full-length
// loops: T is zero above its diagonal and the A block read is wholly below it.  The A
// block is read by solve_tile and replaced by apply_tile; a barrier separates the two.
// The k-step loop is unrolled twice, not fully: the prep kernel is large and its three
// CTAs on an SM run different phases, so code size costs instruction fetch (full
// unrolling measured 1.8% slower for the prep, 1.9% for the B = 2 x 65536 call).
template <int N, int RT>
__device__ __forceinline__ void solve_tile(const float *sAT, float *sX, int r0, int c0, int tr, int tc) {
    uint64_t acc[RT][2];                                // column pairs (0, 1), (2, 3)
#pragma unroll
    for (int a = 0; a < RT; ++a) acc[a][0] = acc[a][1] = 0;
#pragma unroll 2
    for (int m4 = 0; m4 < N; m4 += 4) {
        float4 a4[RT];
#pragma unroll
        for (int a = 0; a < RT; ++a) a4[a] = lds4(sAT + (r0 + tr + 8 * a) * LDA + c0 + m4);
#pragma unroll
        for (int mm = 0; mm < 4; ++mm) {
            const float4 t4 = lds4(sAT + (c0 + m4 + mm) * LDA + c0 + 4 * tc);
            const uint64_t t01 = f2pack(t4.x, t4.y), t23 = f2pack(t4.z, t4.w);
#pragma unroll
            for (int a = 0; a < RT; ++a) {
                const float av = f4get(a4[a], mm);
                const uint64_t aa = f2pack(av, av);
                acc[a][0] = ffma2(aa, t01, acc[a][0]);
                acc[a][1] = ffma2(aa, t23, acc[a][1]);
            }
        }
    }
#pragma unroll
    for (int a = 0; a < RT; ++a) {
        float x0, x1, x2, x3;
        f2unpack(acc[a][0], x0, x1);
        f2unpack(acc[a][1], x2, x3);
        sts4(sX + (tr + 8 * a) * LDX + 4 * tc, x0, x1, x2, x3);
    }
}
template <int N, int RT>
__device__ __forceinline__ void apply_tile(float *sAT, const float *sX, int r0, int c0, int tr, int tc) {
    uint64_t acc[RT][2];                                // column pairs (0, 1), (2, 3)
#pragma unroll
    for (int a = 0; a < RT; ++a) acc[a][0] = acc[a][1] = 0;
#pragma unroll 2
    for (int m4 = 0; m4 < N; m4 += 4) {
        float4 t4[RT];
#pragma unroll
        for (int a = 0; a < RT; ++a) t4[a] = lds4(sAT + (r0 + tr + 8 * a) * LDA + r0 + m4);
#pragma unroll
        for (int mm = 0; mm < 4; ++mm) {
            const float4 x4 = lds4(sX + (m4 + mm) * LDX + 4 * tc);
            const uint64_t x01 = f2pack(x4.x, x4.y), x23 = f2pack(x4.z, x4.w);
#pragma unroll
            for (int a = 0; a < RT; ++a) {
                const float tv = f4get(t4[a], mm);
                const uint64_t tt = f2pack(tv, tv);
                acc[a][0] = ffma2(tt, x01, acc[a][0]);
                acc[a][1] = ffma2(tt, x23, acc[a][1]);
            }
        }
    }
#pragma unroll
    for (int a = 0; a < RT; ++a) {
        float x0, x1, x2, x3;
        f2unpack(acc[a][0], x0, x1);
        f2unpack(acc[a][1], x2, x3);
        sts4(sAT + (r0 + tr + 8 * a) * LDA + c0 + 4 * tc, -x0, -x1, -x2, -x3);
    }
}

// x (32 columns of a row of T) times diag(col) as hi/lo images (row t, chunks 4 half ..)
__device__ __forceinline__ void store_scaled_row(const float (&tv)[32], const float *col, int t,
                                                 int half, uint8_t *img_hi, uint8_t *img_lo) {
    float x[32];
#pragma unroll
    for (int q = 0; q < 32; q += 4) {
        const float4 c4 = lds4(col + half * 32 + q);
        f2unpack(fmul2(f2pack(tv[q], tv[q + 1]), f2pack(c4.x, c4.y)), x[q], x[q + 1]);
        f2unpack(fmul2(f2pack(tv[q + 2], tv[q + 3]), f2pack(c4.z, c4.w)), x[q + 2], x[q + 3]);
    }
    store_half_row_hilo(img_hi, img_lo, t, half * 4, x);
}

// W^T = K^T T'^T (M = 128 keys, N = 64 tokens, K = 64 tokens) into TMEM columns
// col .. col + 63; A is the key tile read MN-major, B the T' hi and lo images
__device__ __forceinline__ void issue_w(uint32_t tmem_col, const uint8_t *sK, const uint8_t *sT1,
                                        uint64_t *bar) {
    const uint32_t id_w = instr_desc(128, 64, kFmtBF16, 1, 0);
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
        const uint64_t ka = smem_desc(smem_u32(sK + ks * 2048), 8192, 1024, kSwizzle128B);
        const uint32_t th = smem_u32(sT1 + ks * 32);
        mma_bf16(tmem_col, ka, smem_desc(th, 16, 1024, kSwizzle128B), id_w, ks > 0);
        mma_bf16(tmem_col, ka, smem_desc(th + 8192, 16, 1024, kSwizzle128B), id_w, 1);
    }
    mma_commit(bar);
}

// -W hi/lo images (hi at img, lo at img + 16 KiB): thread i holds row i (key i) of W^T,
// i.e. row i of the MN-major operand of the chain's first product
__device__ __forceinline__ void stage_minus_w(uint32_t taddr, uint8_t *img, int tid) {
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        float wv[32];
        tmem_ld32(taddr + half * 32, wv);
        tmem_ld_wait();
#pragma unroll
        for (int q = 0; q < 32; ++q) wv[q] = -wv[q];
        store_half_row_hilo(img, img + 16384, tid, half * 4, wv);
    }
}

// Persistent prep (beside the chain kernel): a work item is a (chunk, value-head group).
// Items below p.prep_limit are handed out by one counter in the workspace header, the rest
// by a second one.  Every CTA takes items from the first; once it runs dry, a CTA on an SM
// whose index is below p.prep_stay_sms goes on with the second until no item is left, while
// the others leave, which frees their SMs for the chain's CTAs.  A CTA leaves only once some
// staying CTA has registered, so every item is always taken.  Plain atomic increments (a
// compare-and-swap loop starved the CTAs that lost its races for the whole grid).
// Where a prep item's chunk lies: the item number of the persistent prep (items chunk-major:
// the first chunk of every sequence and head group, then the second, ...; equal-length
// batches), else the CTA's grid position -- (head group, chunk counted from the last), so
// that the hardware starts the CTAs chunk-major from the last chunk and the records the
// chain reads first are the ones written last (most likely still in L2).  False for a
// chunk past the batch's end (a packed batch's chunk table may hold fewer chunks than the
// grid) or after a bad chunk table.
constexpr unsigned kGridY = 65535;                          // grid y limit: chunks beyond it in z
struct PrepChunk {
    int c, h0, len;
    int64_t t0;
};
template <int HPC>
__device__ __forceinline__ bool prep_chunk_locate(const Params &p, PrepChunk &w) {
    if (p.cu_seqlens) {
        if (p.status[kStatusWord] != GDN_OK || w.c < 0 || w.c >= p.status[kChunkCountWord]) return false;
        const int s = p.chunk_seq[w.c];
        w.t0 = p.cu_seqlens[s] + (int64_t)(w.c - p.chunk_first[s]) * C;
        w.len = (int)min((int64_t)C, (int64_t)p.cu_seqlens[s + 1] - w.t0);
    } else {
        const int cps = (p.T_seq + C - 1) / C;
        if (cps == 0 || w.c < 0 || w.c >= p.N * cps) return false;
        const int s = w.c / cps, local = w.c - s * cps;
        w.t0 = (int64_t)s * p.T_seq + (int64_t)local * C;
        w.len = min(C, p.T_seq - local * C);
    }
    return true;
}
// grid position (x = head group, y = chunk counted from the last)
template <int HPC>
__device__ __forceinline__ bool prep_chunk_at(const Params &p, unsigned gx, unsigned gy, PrepChunk &w) {
    w.h0 = (int)gx * HPC;
    const int count = p.cu_seqlens ? p.status[kChunkCountWord] : p.N * ((p.T_seq + C - 1) / C);
    w.c = count - 1 - (int)gy;
    return prep_chunk_locate<HPC>(p, w);
}
template <int HPC>
__device__ __forceinline__ bool prep_chunk(const Params &p, bool persist, int item, PrepChunk &w) {
    if (persist) {
        const int ny = p.HV / HPC, per = p.N * ny;
        const int local = item / per, r = item - local * per, sq = r / ny;
        w.c = sq * ((p.T_seq + C - 1) / C) + local;
        w.h0 = (r - sq * ny) * HPC;
        return prep_chunk_locate<HPC>(p, w);
    }
    return prep_chunk_at<HPC>(p, blockIdx.x, blockIdx.y + kGridY * blockIdx.z, w);
}

// The key and query tiles of a chunk (key head j) into the prep's tiles, completing bar.
__device__ __forceinline__ void prep_load_tiles(const CUtensorMap *mapK, const CUtensorMap *mapQ, uint8_t *sK,
                                                uint8_t *sQ, uint64_t *bar, int j, int64_t t0) {
    mbar_arrive_expect_tx(bar, 32768);
    tma_load_3d(sK, mapK, bar, 0, j, (int)t0);
    tma_load_3d(sK + 8192, mapK, bar, 64, j, (int)t0);
    tma_load_3d(sQ, mapQ, bar, 0, j, (int)t0);
    tma_load_3d(sQ + 8192, mapQ, bar, 64, j, (int)t0);
}

// An item is claimed in two steps, so that the atomic's round trip overlaps the item
// before: a ticket from the first counter, then the item it stands for.
__device__ __forceinline__ int prep_ticket(const Params &p) {
    return atomicAdd(&p.status[kPrepClaimWord], 1);
}
__device__ __forceinline__ int prep_item(const Params &p, int ticket, bool stay) {
    if (ticket < p.prep_limit) return ticket;
    if (!stay && *reinterpret_cast<volatile int32_t *>(&p.status[kPrepStayWord]) > 0) return -1;
    if (*reinterpret_cast<volatile int32_t *>(&p.status[kPrepClaimPastWord]) >= p.prep_items - p.prep_limit)
        return -1;
    const int k = p.prep_limit + atomicAdd(&p.status[kPrepClaimPastWord], 1);
    return k < p.prep_items ? k : -1;
}

// Sets the ready flags of the HPC records of item (c, h0) once its bulk stores are complete
// in global memory (the factor rows the other threads stored came before a CTA barrier).
template <int HPC>
__device__ __forceinline__ void prep_publish(const Params &p, int c, int h0) {
    bulk_wait_all();
    fence_async_global();
    asm volatile("fence.acq_rel.gpu;" ::: "memory");
#pragma unroll
    for (int i = 0; i < HPC; ++i)
        asm volatile("st.relaxed.gpu.global.s32 [%0], 1;" ::"l"(p.ready + (size_t)c * p.HV + h0 + i) : "memory");
}

// PERSIST == false: one CTA per item, launched as a (chunk, head group) grid.  PERSIST ==
// true: the persistent prep beside the chain (items claimed in chunk order, records'
// ready flags set).  Each schedule compiles only its own loop code.
template <int HPC, bool PERSIST>
__global__ void __launch_bounds__(kPrepThreads, kPrepPerSm)
prep_kernel(const __grid_constant__ CUtensorMap mapK, const __grid_constant__ CUtensorMap mapQ,
            Params p) {
    static_assert(HPC == 1 || HPC == 2, "one or two value heads per CTA");
    extern __shared__ uint8_t smem_raw[];
    const uint32_t su = smem_u32(smem_raw);
    uint8_t *sm = smem_raw + (((su + 1023u) & ~1023u) - su);
    uint8_t *sK = sm;                                   // [2][64][128 B]
    uint8_t *sQ = sm + 16384;                           // [2][64][128 B]
    float *sX = reinterpret_cast<float *>(sQ);          // [HPC][kXHead], during the solve
    uint8_t *sT1 = sQ;                                  // T' hi | lo images, after the solve
    float *sAT = reinterpret_cast<float *>(sm + 32768); // [HPC][64][68]
    uint8_t *sAT8 = sm + 32768;
    float *sRk = sAT + HPC * C * LDA;                   // key normaliser
    float *sRq = sRk + C;                               // query normaliser (with the scale)
    float *sV = sRq + C;                                // [HPC][4][64] per-head vectors
    uint64_t *bar = reinterpret_cast<uint64_t *>(sV + HPC * kPrepVecHead * C);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(bar + 5);
    volatile int *s_item = reinterpret_cast<volatile int *>(tslot + 1);
    // thread 0's bookkeeping of the persistent prep (kept out of registers): the item whose
    // records are written but whose flags are not yet set (chunk, first value head; chunk -1
    // for none), and the ticket of the next item
    volatile int *s_pend = s_item + 1, *s_ticket = s_item + 3;
    // per-head vectors: decay prefix (natural log), the same times log2(e), beta,
    // beta gamma rk (0 past the chunk end)
    auto vG = [&](int i) { return sV + (i * kPrepVecHead + 0) * C; };
    auto vG2 = [&](int i) { return sV + (i * kPrepVecHead + 1) * C; };
    auto vB = [&](int i) { return sV + (i * kPrepVecHead + 2) * C; };
    auto vC1 = [&](int i) { return sV + (i * kPrepVecHead + 3) * C; };

    // the chain kernel may be scheduled as soon as every prep CTA has started; it takes a
    // record once its ready flag is set (persistent prep), or after this grid completes
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool stay = PERSIST && sm_id() < (uint32_t)p.prep_stay_sms;
    PrepChunk w;
    if constexpr (!PERSIST) {
        if (!prep_chunk<HPC>(p, false, 0, w)) return;
    }
    // thread 0 starts the tile loads of an item as early as it can: the first item's at once,
    // (persistent prep) each later one's as soon as the item before has left the tiles; the
    // persistent prep sets an item's flags while the next item's tiles load, and takes the
    // next item's ticket before the current one ends
    if (tid == 0) {
        for (int b = 0; b < 5; ++b) mbar_init(&bar[b], 1);
        fence_mbar_init();
        prefetch_tensormap(&mapK);
        prefetch_tensormap(&mapQ);
        if constexpr (PERSIST) {
            if (stay) atomicAdd(&p.status[kPrepStayWord], 1);
            s_pend[0] = -1;
            const int first = prep_item(p, prep_ticket(p), stay);
            PrepChunk w1;
            if (first >= 0 && prep_chunk<HPC>(p, true, first, w1)) {
                prep_load_tiles(&mapK, &mapQ, sK, sQ, &bar[0], w1.h0 / (p.HV / p.HK), w1.t0);
                *s_item = first;
            } else {
                *s_item = -1;
            }
        } else {
            prep_load_tiles(&mapK, &mapQ, sK, sQ, &bar[0], w.h0 / (p.HV / p.HK), w.t0);
            // the tiles of the item the next wave of CTAs starts with (the CTA p.prep_slots
            // further on) into L2, so that its load does not wait for HBM.  Only the first
            // two waves do this: later the L2 is full of the records written since, and a
            // tile fetched a wave early is evicted before its load (measured at B = 2,
            // T = 65536: prep 2.5% slower with every wave prefetching).  Equal-length batches
            // only: a packed batch's chunk takes a chain of dependent loads to find.
            const unsigned b0 = blockIdx.x + gridDim.x * (blockIdx.y + kGridY * blockIdx.z);
            if (p.prep_slots > 0 && !p.cu_seqlens && b0 < 2u * (unsigned)p.prep_slots) {
                const unsigned b = b0 + p.prep_slots;
                PrepChunk w2;
                if (b < gridDim.x * gridDim.y * gridDim.z &&
                    prep_chunk_at<HPC>(p, b % gridDim.x, b / gridDim.x, w2)) {
                    const int j2 = w2.h0 / (p.HV / p.HK);
                    tma_prefetch_3d(&mapK, 0, j2, (int)w2.t0);
                    tma_prefetch_3d(&mapK, 64, j2, (int)w2.t0);
                    tma_prefetch_3d(&mapQ, 0, j2, (int)w2.t0);
                    tma_prefetch_3d(&mapQ, 64, j2, (int)w2.t0);
                }
            }
        }
    }
    if (warp == 0) { tmem_alloc(tslot, kPrepTmemCols); tmem_relinquish(); }
    if constexpr (PERSIST) __syncthreads();             // the first item, claimed by thread 0
    bool ok = true;
    uint32_t par = 0;                                   // parity of every barrier's phase
    for (;;) {
        // the item (its tiles are on their way); every thread finds its chunk
        if constexpr (PERSIST) {
            if (*s_item < 0 || !prep_chunk<HPC>(p, true, *s_item, w)) break;
        }
        const int c = w.c, h0 = w.h0, len = w.len;
        const int64_t t0 = w.t0;
        auto record = [&](int i) {
            return reinterpret_cast<uint8_t *>(p.rec) + ((size_t)c * p.HV + h0 + i) * kRecBytes;
        };
        {
            // gate thread (head gh, token gt): its gate and beta are requested before anything
            // waits, and it scans the decay prefix of its head (two warps per head)
            const int gh = tid >> 6, gt = tid & 63;
            const bool gthr = gh < HPC;
            const bool gin = gthr && gt < len;
            float g_in = 0.f, b_in = 0.f;
            if (gin) {
                const size_t gi = (size_t)(t0 + gt) * p.HV + h0 + gh;
                g_in = p.g[gi];
                b_in = p.beta[gi];
            }
            float Gx = g_in;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, Gx, o);
                if (lane >= o) Gx += y;
            }
            if (gthr) vG(gh)[gt] = Gx;                          // inclusive within the warp
            __syncthreads();
            tc_fence_after();
            const uint32_t tmem = *tslot;
            const uint32_t lb = (uint32_t)(warp * 32) << 16;    // this warp's TMEM lanes
            const int trow = warp * 16 + (lane & 15), tcb = lane >> 4;   // row / column half of
                                                                          // the M = 64 results
            const int hrow = tid >> 1, hhalf = tid & 1;         // row / column half, 2 threads a row
            float gr[32], qk[32];                               // Gram and Q K^T: row trow, 32 columns

            if (gthr) {
                if (gt >= 32) {
                    Gx += vG(gh)[31];
                    vG(gh)[gt] = Gx;
                }
                vG2(gh)[gt] = Gx * kLog2e;
                vB(gh)[gt] = b_in;
            }
            // the previous item's flags, while the tiles load
            if constexpr (PERSIST) {
                if (tid == 0 && s_pend[0] >= 0) {
                    prep_publish<HPC>(p, s_pend[0], s_pend[1]);
                    s_pend[0] = -1;
                }
            }
            ok = mbar_wait(&bar[0], par);
            if (__syncthreads_or(!ok)) goto item_fail;
            tc_fence_after();
            if (lane == 0 && warp < 2) {
                // Gram K K^T into columns 0-63 (thread 0), Q K^T into columns 64-127 (thread 32);
                // M = N = 64, K = 128
                const uint32_t idesc = instr_desc(64, 64, kFmtBF16, 0, 0);
                const uint8_t *aop = warp ? sQ : sK;
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t o = (ks >> 2) * 8192 + (ks & 3) * 32;
                    mma_bf16(tmem + warp * 64, smem_desc(smem_u32(aop + o), 16, 1024, kSwizzle128B),
                             smem_desc(smem_u32(sK + o), 16, 1024, kSwizzle128B), idesc, ks > 0);
                }
                mma_commit(&bar[1 + 2 * warp]);
            }
            // query normalisers: two threads per row; the 16-byte chunks are visited in an order
            // that keeps the eight lanes of a quarter-warp on distinct banks
            {
                const uint8_t *src = sQ + hhalf * 8192 + hrow * 128;
                float ss = 0.f;
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const int pc = q ^ (hrow & 7) ^ (hhalf * 4);
                    const uint4 w4 = *reinterpret_cast<const uint4 *>(src + pc * 16);
                    const __nv_bfloat162 *b2 = reinterpret_cast<const __nv_bfloat162 *>(&w4);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 f = __bfloat1622float2(b2[e]);
                        ss += f.x * f.x + f.y * f.y;
                    }
                }
                ss += __shfl_xor_sync(0xffffffffu, ss, 1);
                if (hhalf == 0) sRq[hrow] = p.l2norm ? p.scale * rsqrtf(ss + kL2Eps) : p.scale;
            }
            ok = mbar_wait(&bar[1], par) && mbar_wait(&bar[3], par);
            if (__syncthreads_or(!ok)) goto item_fail;
            tc_fence_after();
            // Gram and Q K^T rows into registers; the key normaliser from the Gram diagonal
            tmem_row_split(tmem + lb, gr);
            tmem_row_split(tmem + lb + 64, qk);
            {
                float diag = 0.f;
#pragma unroll
                for (int q = 0; q < 32; ++q) diag = (tcb * 32 + q == trow) ? gr[q] : diag;
                if ((trow >> 5) == tcb) sRk[trow] = p.l2norm ? rsqrtf(diag + kL2Eps) : 1.f;
            }
            tc_fence_before();
            __syncthreads();
            if (gthr) vC1(gh)[gt] = gin ? b_in * expf(Gx) * sRk[gt] : 0.f;
            {
                // per head: A_tj = beta_t e^{G_t-G_j} rk_t rk_j k_t.k_j (j < t) into shared memory
                // and P_tj = e^{G_t-G_j} rq_t rk_j q_t.k_j (j <= t) as an image in the free query
                // tile, one exponential for both
                const bool live = trow < len;
                const float rkt = sRk[trow], pt = sRq[trow];
#pragma unroll
                for (int i = 0; i < HPC; ++i) {
                    const float *G2 = vG2(i);
                    const float G2t = G2[trow], at = vB(i)[trow] * rkt;
                    float av[32], pv[32];
                    const uint64_t G2t2 = f2pack(G2t, G2t), at2 = f2pack(at, at), pt2 = f2pack(pt, pt);
#pragma unroll
                    for (int q4 = 0; q4 < 32; q4 += 4) {
                        const float4 g4 = lds4(G2 + tcb * 32 + q4), r4 = lds4(sRk + tcb * 32 + q4);
                        const float gv[4] = {g4.x, g4.y, g4.z, g4.w}, rv[4] = {r4.x, r4.y, r4.z, r4.w};
#pragma unroll
                        for (int qq = 0; qq < 4; qq += 2) {             // column pairs
                            const int q = q4 + qq, jj = tcb * 32 + q;
                            float d0, d1;                               // G_t - G_j (log2 units)
                            f2unpack(ffma2(f2pack(-1.f, -1.f), f2pack(gv[qq], gv[qq + 1]), G2t2), d0, d1);
                            // the exponent is selected before any product (past t it may be inf)
                            const float e0 = (jj <= trow && jj < len) ? ex2_fast(d0) : 0.f;
                            const float e1 = (jj + 1 <= trow && jj + 1 < len) ? ex2_fast(d1) : 0.f;
                            const uint64_t e2 = fmul2(f2pack(e0, e1), f2pack(rv[qq], rv[qq + 1]));
                            float a0, a1;
                            f2unpack(fmul2(fmul2(at2, e2), f2pack(gr[q], gr[q + 1])), a0, a1);
                            av[q] = (live && jj < trow) ? a0 : 0.f;
                            av[q + 1] = (live && jj + 1 < trow) ? a1 : 0.f;
                            f2unpack(fmul2(fmul2(pt2, e2), f2pack(qk[q], qk[q + 1])), pv[q], pv[q + 1]);
                        }
                    }
                    float *sA = sAT + i * C * LDA;
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        sts4(sA + trow * LDA + tcb * 32 + 4 * q, av[4 * q], av[4 * q + 1], av[4 * q + 2], av[4 * q + 3]);
                    store_half_row_bf16(sQ + i * 8192, trow, tcb * 4, pv);
                }
            }
            fence_async_smem();
            __syncthreads();
            if (tid == 0) {
#pragma unroll
                for (int i = 0; i < HPC; ++i) bulk_store(record(i) + REC_P, sQ + i * 8192, 8192);
                bulk_commit();
            }

            // ---- T = (I + A)^{-1}, in place: the four 16 x 16 diagonal blocks of each head by
            // forward substitution (one thread per column), written once every thread has read A
            {
                const int dh = tid >> 6, b = (tid >> 4) & 3, cc = tid & 15, base = b * 16;
                float *sA = sAT + (dh < HPC ? dh : 0) * C * LDA;
                float x[16];
                if (dh < HPC) {
#pragma unroll
                    for (int r = 0; r < 16; ++r) {
                        float acc = (r == cc) ? 1.f : 0.f;
#pragma unroll
                        for (int k4 = 0; k4 < r; k4 += 4) {
                            const float4 a4 = lds4(sA + (base + r) * LDA + base + k4);
                            const float aw[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk)
                                if (k4 + kk < r) acc -= aw[kk] * x[k4 + kk];
                        }
                        x[r] = (r < cc) ? 0.f : acc;
                    }
                }
                // the P images have left the query tile before it becomes the solve's scratch
                if (tid == 0) bulk_wait_read_all();
                __syncthreads();
                if (dh < HPC) {
#pragma unroll
                    for (int r = 0; r < 16; ++r) sA[(base + r) * LDA + base + cc] = x[r];
                }
                __syncthreads();
            }
            // ---- then by doubling, 64 threads per head: blocks (1,0) and (3,2) of 16 x 16 (a warp
            // each, 2 x 4 tiles), then block (1,0) of 32 x 32 (4 x 4 tiles): T_ij = -T_ii A_ij T_jj
            if ((tid >> 6) < HPC) {
                const int i = tid >> 6, pb = (tid >> 5) & 1;
                float *sATi = sAT + i * C * LDA, *sXi = sX + i * kXHead;
                solve_tile<16, 2>(sATi, sXi + pb * 16 * LDX, 16 + 32 * pb, 32 * pb, lane >> 2, lane & 3);
            }
            __syncthreads();
            if ((tid >> 6) < HPC) {
                const int i = tid >> 6, pb = (tid >> 5) & 1;
                float *sATi = sAT + i * C * LDA, *sXi = sX + i * kXHead;
                apply_tile<16, 2>(sATi, sXi + pb * 16 * LDX, 16 + 32 * pb, 32 * pb, lane >> 2, lane & 3);
            }
            __syncthreads();
            if ((tid >> 6) < HPC) {
                const int i = tid >> 6, t = tid & 63;
                solve_tile<32, 4>(sAT + i * C * LDA, sX + i * kXHead, 32, 0, t >> 3, t & 7);
            }
            __syncthreads();
            if ((tid >> 6) < HPC) {
                const int i = tid >> 6, t = tid & 63;
                apply_tile<32, 4>(sAT + i * C * LDA, sX + i * kXHead, 32, 0, t >> 3, t & 7);
            }
            __syncthreads();

            {
                // the ticket of the next item (its round trip overlaps the rest of this one)
                if constexpr (PERSIST) {
                    if (tid == 0) *s_ticket = prep_ticket(p);
                }
                // rows of T (two threads a row, 32 columns each) into registers, then:
                // T' = T diag(beta gamma rk) of head 0 as operand images for W in the query tile,
                // T'' = T diag(beta) of every head as images in place of its T, bulk-copied out
                float tv[HPC][32];
#pragma unroll
                for (int i = 0; i < HPC; ++i)
#pragma unroll
                    for (int q = 0; q < 32; q += 4) {
                        const float4 t4 = lds4(sAT + i * C * LDA + hrow * LDA + hhalf * 32 + q);
                        tv[i][q] = t4.x; tv[i][q + 1] = t4.y; tv[i][q + 2] = t4.z; tv[i][q + 3] = t4.w;
                    }
                store_scaled_row(tv[0], vC1(0), hrow, hhalf, sT1, sT1 + 8192);
                fence_async_smem();
                tc_fence_before();
                __syncthreads();
                tc_fence_after();
                if (tid == 0) issue_w(tmem, sK, sT1, &bar[2]);
#pragma unroll
                for (int i = 0; i < HPC; ++i)
                    store_scaled_row(tv[i], vB(i), hrow, hhalf, sAT8 + i * C * LDA * 4, sAT8 + i * C * LDA * 4 + 8192);
                // ---- per-token factors of every head (one coalesced row each)
                if (gthr) {
                    float *sc = reinterpret_cast<float *>(record(gh) + REC_F);
                    const float Gl = vG(gh)[len - 1], rk = sRk[gt];
                    sc[SC_QD * C + gt] = gin ? sRq[gt] * expf(Gx) : 0.f;
                    sc[SC_KD * C + gt] = gin ? rk * expf(Gl - Gx) : 0.f;
                    sc[SC_RK * C + gt] = gin ? rk : 0.f;
                    sc[SC_ALPHA * C + gt] = gin ? expf(g_in) : 0.f;
                    sc[SC_MISC * C + gt] = gt == 0 ? expf(Gl) : (gt == 1 ? (float)len : 0.f);
                }
                fence_async_smem();
                __syncthreads();
                if (tid == 0) {
#pragma unroll
                    for (int i = 0; i < HPC; ++i)
                        bulk_store(record(i) + REC_T2HI, sAT8 + i * C * LDA * 4, 16384);
                    bulk_commit();
                }
                ok = mbar_wait(&bar[2], par);
                if (__syncthreads_or(!ok)) goto item_fail;
                tc_fence_after();
                if constexpr (HPC == 2) {
                    // W of head 1 into columns 64-127 while -W of head 0 is staged in place of the
                    // T'' images (once their copies have read them)
                    store_scaled_row(tv[1], vC1(1), hrow, hhalf, sT1, sT1 + 8192);
                    fence_async_smem();
                    tc_fence_before();
                    __syncthreads();
                    tc_fence_after();
                    if (tid == 0) {
                        issue_w(tmem + 64, sK, sT1, &bar[4]);
                        bulk_wait_read_all();
                    }
                    __syncthreads();
                    stage_minus_w(tmem + lb, sAT8, tid);
                    fence_async_smem();
                    __syncthreads();
                    if (tid == 0) {
                        bulk_store(record(0) + REC_WHI, sAT8, 32768);
                        bulk_commit();
                    }
                    ok = mbar_wait(&bar[4], par);
                    if (__syncthreads_or(!ok)) goto item_fail;
                    tc_fence_after();
                }
            }
            // the next item (persistent prep), announced before the barrier below
            if constexpr (PERSIST) {
                if (tid == 0) *s_item = prep_item(p, *s_ticket, stay);
            }
            // -W of the last head, staged in the key and query tiles (free once its product is done)
            stage_minus_w(tmem + lb + (HPC - 1) * 64, sm, tid);
            fence_async_smem();
            tc_fence_before();
            __syncthreads();
            if (tid == 0) {
                bulk_store(record(HPC - 1) + REC_WHI, sm, 32768);
                bulk_commit();
                if constexpr (PERSIST) {
                    // the next item's tiles overwrite what the copies read; the records'
                    // flags are set once the copies are complete
                    bulk_wait_read_all();
                    s_pend[0] = c;
                    s_pend[1] = h0;
                    PrepChunk nw;
                    if (*s_item >= 0 && prep_chunk<HPC>(p, true, *s_item, nw))
                        prep_load_tiles(&mapK, &mapQ, sK, sQ, &bar[0], nw.h0 / (p.HV / p.HK), nw.t0);
                }
            }
        }
        if constexpr (!PERSIST) break;
        par ^= 1u;
        continue;
    item_fail:
        ok = false;
        break;
    }
    if (!ok && tid == 0) set_error(p, GDN_ERR_TIMEOUT);
    if constexpr (PERSIST) {
        if (tid == 0 && s_pend[0] >= 0) prep_publish<HPC>(p, s_pend[0], s_pend[1]);
    }
    // shared memory stays until every bulk copy has read it
    if (tid == 0) bulk_wait_read_all();
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(*tslot, kPrepTmemCols);
}

// ================================================================== chain kernel
// Operand shapes: hi/lo pairs are stacked so that one instruction covers several terms.
//   -W S      A = [-W_hi; -W_lo] (M = 128: two 64-token halves), B = [S_hi | S_lo]
//             (N = 64): rows 0-63 hold -W_hi S_hi and -W_hi S_lo, rows 64-127 -W_lo S_hi
//             (and the negligible -W_lo S_lo); two issuers take k-steps 0-3 and 4-7
//   T'' V     A = [T''_hi; T''_lo] (M = 128), B = V slice (N = 32)
//   K^T Z     A = key tile (M = 128 keys), B = [Z_hi | Z_lo] (N = 64); two issuers take
//             k-steps 0-1 and 2-3
//   Q S       A = [any; Q] (M = 128, the operand read from 8 KiB before the query tile,
//             so that the 64 live rows land in TMEM lanes 64-127), B = [S_hi | S_lo]
//   P U_hi    A = [any; P] the same way, B = U_hi (N = 32); an output row is
//             qd (Q S[:, 0:32] + Q S[:, 32:64]) + P U_hi
// Warp roles (256 threads):
//   warps 0-3  epilogue warpgroup: thread i holds key row i of the fp32 state slice in
//              registers; forms U (the two token halves of the stacked products are
//              combined through shared memory, each thread finishing 16 columns of one
//              token), Z = kd U and the new state; lane 0 of warps 1-3 issues the
//              products on the chain's critical path right after the step that enables
//              them (no hand-off): after the state update warps 1, 2 the k-step halves
//              of -W S of the next chunk, after U warps 2, 3 the k-step halves of K^T Z.
//   warp 4     TMEM owner; issues P U_hi of chunk cc once U of chunk cc is formed
//   warp 5     TMA producer; also issues T'' V of chunk cc + 1 as soon as it sees ring A
//              of chunk cc - 1 released, i.e. once -W S of chunk cc is done
//   warps 6-7  output warps: once -W S of chunk cc is done, lane 0 of each issues one
//              k-step half of Q S of chunk cc (so that it runs while U is formed, when the
//              tensor pipe is idle); then they read rows 64-127 of Q S and P U (TMEM lanes
//              64-127, one token per thread) and write the outputs
// A chunk's inputs come through two 2-deep rings that are released at different points:
//   ring A  -W hi/lo, T'' hi/lo (the first 48 KiB of the record) and the value slice
//           (64B swizzle: the MN-major B operand of T'' V as loaded); free once -W S and
//           T'' V of the chunk are done, so the next loads start early in the chunk
//   ring B  key and query tiles, P and the factor rows; free after the state update,
//           P U and the output warps' read of the factors
constexpr int kChainThreads = 256;
constexpr int kAW = 0, kAV = REC_P, kStageA = kAV + C * NV * 2;              // 52 KiB
constexpr int kBK = 0, kBQ = 16384, kBP = 32768, kBF = kBP + (REC_F - REC_P),
              kStageB = kBF + 8 * C * 4;                                     // 42 KiB
static_assert(REC_WHI == 0 && REC_P == REC_T2LO + 8192 && REC_F == REC_P + 8192, "record layout");
static_assert(kBP >= 8192 && kBQ >= 8192, "the stacked output operands read 8 KiB before P and Q");
// shared memory map (bytes from a 1024-aligned base)
constexpr int OFF_A = 0;                                   // [2] ring A
constexpr int OFF_B = OFF_A + 2 * kStageA;                 // [2] ring B
constexpr int OFF_S = OFF_B + 2 * kStageB;                 // [S_hi | S_lo] [128 keys][128B] MN-major
constexpr int OFF_Z = OFF_S + 16384;                       // [Z_hi | Z_lo] [64 tokens][128B] MN-major
constexpr int OFF_U = OFF_Z + 8192;                        // U_hi [64 tokens][64B] MN-major
constexpr int OFF_X = OFF_U + 4096;                        // fp32 [2][64][16] half-row exchange
                                                           // (16-byte chunks XOR-swizzled)
constexpr int OFF_BAR = OFF_X + C * NV * 4;                // barriers, TMEM slot, error flag
constexpr int OFF_DESC = OFF_BAR + 128;                    // chunk descriptors [4][8] int32
constexpr int kChainSmem = OFF_BAR + 256 + 1024;
static_assert(kStageA % 1024 == 0 && kStageB % 1024 == 0 && kAV % 1024 == 0 && kBQ % 1024 == 0,
              "swizzled operands need 1 KiB alignment");
static_assert(kChainSmem <= 232448, "shared memory");

// TMEM columns; M = 128 accumulators have row m in lane m
constexpr uint32_t TM_W = 0,      // -W S [2], k-steps 0-3 / 4-7 (N = 64 each)
                   TM_UT = 128,   // T'' V [2]           (N = 32 each)
                   TM_S = 192,    // K^T Z, k-steps 0-1  (N = 64)
                   TM_S2 = 256,   // K^T Z, k-steps 2-3  (N = 64)
                   TM_QS = 320,   // Q S [2], k-steps 0-3 / 4-7 (N = 64 each; rows 64-127 live)
                   TM_PU = 448;   // P U_hi              (N = 32; rows 64-127 live)
constexpr uint32_t kTmemCols = 512;

// barriers (arrival counts in brackets)
enum {
    B_FULLA0 = 0, B_FULLA1,    // [1 + tx] ring A stage loaded
    B_EMPTYA0, B_EMPTYA1,      // [1] ring A stage released
    B_FULLB0, B_FULLB1,        // [1 + tx] ring B stage loaded
    B_EMPTYB0, B_EMPTYB1,      // [4] ring B stage released (state update, P U done, both
                               // output warps have read the factors)
    B_D1,                      // [3] both halves of -W S and T'' V of the chunk are done
    B_D2,                      // [2] both halves of K^T Z of the chunk are done
    B_QSD,                     // [2] both halves of Q S of the chunk are done
    B_DO,                      // [1] P U_hi of the chunk is done
    B_OUT,                     // [2] the output warps have read Q S and P U
    B_E1DONE,                  // [1] Z and U_hi of the chunk are written
    B_DRAIN,                   // [8] every MMA of every issuer is done (teardown)
    B_COUNT
};

__device__ __forceinline__ uint32_t lane_base(int warp) { return (uint32_t)((warp & 3) * 32) << 16; }

// AND of a predicate over the 128 threads of the epilogue warpgroup (named barrier 1)
__device__ __forceinline__ bool wg_and(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, 1, 128, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v)
        : "memory");
    return r != 0;
}

// 8 fp32 values to global memory in one 32-byte store (a whole sector); dst 32-byte aligned
__device__ __forceinline__ void st_v8(float *dst, const float *x) {
    asm volatile("st.global.v8.f32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
                 :: "l"(dst), "f"(x[0]), "f"(x[1]), "f"(x[2]), "f"(x[3]), "f"(x[4]), "f"(x[5]), "f"(x[6]),
                    "f"(x[7])
                 : "memory");
}
// 4 fp32 values to global memory in one 16-byte streaming store; dst 16-byte aligned
__device__ __forceinline__ void st_cs_v4(float *dst, float a0, float a1, float a2, float a3) {
    asm volatile("st.global.cs.v4.f32 [%0], {%1, %2, %3, %4};"
                 :: "l"(dst), "f"(a0), "f"(a1), "f"(a2), "f"(a3) : "memory");
}

// 32 fp32 values -> one 128-byte row [hi | lo] of a 128B-swizzled bf16 image
__device__ __forceinline__ void store_row_hilo128(uint8_t *img, int row, const float (&x)[32]) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint32_t h[4], l[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) split2_bf16(x[q * 8 + 2 * e], x[q * 8 + 2 * e + 1], h[e], l[e]);
        *reinterpret_cast<uint4 *>(img + sw128_offset(row, q * 16)) = make_uint4(h[0], h[1], h[2], h[3]);
        *reinterpret_cast<uint4 *>(img + sw128_offset(row, 64 + q * 16)) = make_uint4(l[0], l[1], l[2], l[3]);
    }
}

// float offset of 16-byte chunk c (0-3) of row t in a [64][16] fp32 block whose chunks
// are XOR-swizzled so that eight consecutive rows hit eight different bank groups
__device__ __forceinline__ int xchg_off(int t, int c) { return t * 16 + ((c ^ ((t >> 1) & 3)) << 2); }

// Work units (equal-length batches whose chains outnumber the SMs).  A chain is one
// (sequence, value head, 32-wide value slice); its chunks are cut into segments of at
// most seg_len chunks, and the units are numbered segment-major (segment 0 of every
// chain, then segment 1, ...), so that the CTAs, one per SM, share the work evenly
// instead of running whole waves of chains.  CTA b takes unit b first; later units are
// claimed in order from an atomic counter by running CTAs, so a unit's predecessor (the
// previous segment of its chain) was taken earlier by a CTA that has started.  A
// segment's end state goes through global memory (the final-state slice, or with
// per-token states the slot of its last token) and a flag word per chain.
struct Unit {
    SeqRange sr;
    int s, h, vs, seg, c0, c1;      // chunks c0 .. c1 - 1 of the sequence
};

__device__ __forceinline__ bool unit_of(const Params &p, int u, Unit &w) {
    constexpr int SL = D / NV;
    int c = u, seg = 0;
    if (!p.cu_seqlens) {
        seg = u / p.n_chains;
        c = u - seg * p.n_chains;
    }
    const int per_seq = p.HV * SL;
    const int z = c / per_seq, rem = c - z * per_seq;
    w.h = rem / SL;
    w.vs = rem - w.h * SL;
    w.s = p.cu_seqlens ? p.seq_order[z] : z;
    if (!seq_range(p, w.s, w.sr)) return false;
    w.seg = seg;
    w.c0 = min(w.sr.count, seg * p.seg_len);
    w.c1 = min(w.sr.count, w.c0 + p.seg_len);
    return true;
}

// Descriptor of one chunk of a chain CTA's stream, written by the producer before it
// arms the chunk's ring barriers (whose phase then publishes it to the other warps).
enum { DW_TOK = 0, DW_LEN, DW_CHAIN, DW_SEG, DW_HEAD, DW_SLICE, kDescWords = 8 };
enum { DF_FIRST = 1, DF_LAST = 2, DF_END = 4, DF_STOP = 8 };   // DW_LEN bits 8 and up
constexpr int kDescSlots = 4;
static_assert(8 * B_COUNT + 8 <= OFF_DESC - OFF_BAR && OFF_DESC - OFF_BAR + kDescSlots * kDescWords * 4 <= 256,
              "barrier area");
static_assert(D / NV == kChainSlices, "chain flag words per value head");

// Flag words between CTAs: the writer publishes after a barrier that follows every
// participating thread's stores (the fence makes them visible at GPU scope first); the
// reader acquires before a barrier that precedes the other threads' loads.
__device__ __forceinline__ void flag_release(int32_t *f, int32_t v) {
    asm volatile("fence.acq_rel.gpu;\n\tst.relaxed.gpu.global.s32 [%0], %1;" ::"l"(f), "r"(v) : "memory");
}
__device__ __forceinline__ int32_t flag_acquire(const int32_t *f) {
    int32_t v;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(f) : "memory");
    return v;
}
__device__ __forceinline__ int32_t flag_relaxed(const int32_t *f) {
    int32_t v;
    asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(f) : "memory");
    return v;
}
// record-ready flags read ahead by the chain's producer in one round trip (each wait costs
// its producer ~0.75 us, which reaches the chain: with every record ready, 8 a round trip
// made the chain 6% slower than one that waits for the whole prep grid)
constexpr int kReadyAhead = 32;
// wait until *f >= want; gives up (false) after limit_ns
__device__ __forceinline__ bool flag_wait(const int32_t *f, int32_t want, uint64_t limit_ns = 1000000000ull) {
    if (flag_acquire(f) >= want) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        __nanosleep(128);
        if (flag_acquire(f) >= want) return true;
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
}

// The chain's wait for the record of chunk c (flags every `stride` words from `ready`):
// acquires its flag, reads the flags of up to kReadyAhead - 1 chunks after it in the same
// round trip, and returns the first chunk not known complete (-1 after a timeout).  Kept
// out of line: the chain kernel's speed depends on the size of its loop code.
__device__ __noinline__ int ready_wait(const int32_t *ready, int stride, int c, int nch) {
    if (!flag_wait(ready + (size_t)c * stride, 1)) return -1;
    int32_t f[kReadyAhead - 1];
#pragma unroll
    for (int i = 0; i < kReadyAhead - 1; ++i)
        f[i] = c + 1 + i < nch ? flag_relaxed(ready + (size_t)(c + 1 + i) * stride) : 0;
    int to = c + 1;
#pragma unroll
    for (int i = 0; i < kReadyAhead - 1; ++i)
        if (to == c + 1 + i && f[i] >= 1) to = c + 2 + i;
    // the flags read relaxed order the records' reads after this fence
    if (to > c + 1) asm volatile("fence.acq_rel.gpu;" ::: "memory");
    return to;
}

// UNITS == false: one CTA per chain, launched as a (value slice, value head, sequence)
// grid, packed batches' chains longest first (the hardware starts the CTAs in order).
// UNITS == true: the persistent work-unit stream above (equal-length batches whose chains
// outnumber the SMs).  The per-chunk work is the same code; only the loops around it and
// the source of a chunk's coordinates differ, and each schedule compiles only its own
// loops (the kernel's speed depends on the size of its loop code: instruction fetch).
// READY: the records come from the persistent prep beside the chain, each taken once its
// ready flag is set (one CTA per chain), instead of after the whole prep grid.
template <bool STATES, bool UNITS, bool READY>
__global__ void __launch_bounds__(kChainThreads, 1)
chain_kernel(const __grid_constant__ CUtensorMap mapK, const __grid_constant__ CUtensorMap mapQ,
             const __grid_constant__ CUtensorMap mapV, Params p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t su = smem_u32(smem_raw);
    uint8_t *sm = smem_raw + (((su + 1023u) & ~1023u) - su);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + OFF_BAR);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + OFF_BAR + 8 * B_COUNT);
    volatile int *s_err = reinterpret_cast<volatile int *>(sm + OFF_BAR + 8 * B_COUNT + 4);
    int32_t *descs = reinterpret_cast<int32_t *>(sm + OFF_DESC);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (p.cu_seqlens && p.status[kStatusWord] != GDN_OK) return;
    // the CTA's own chain (UNITS == false)
    int vs = 0, h = 0, s = 0, j = 0, nch = 0;
    SeqRange sr{};
    if constexpr (!UNITS) {
        vs = blockIdx.x;
        h = blockIdx.y;
        s = p.cu_seqlens ? p.seq_order[blockIdx.z] : (int)blockIdx.z;
        if (!seq_range(p, s, sr)) return;
        j = h / (p.HV / p.HK);
        nch = sr.count;
    }

    if (tid == 0) {
        for (int b = 0; b < 2; ++b) {
            mbar_init(&bars[B_FULLA0 + b], 1);
            mbar_init(&bars[B_EMPTYA0 + b], 1);
            mbar_init(&bars[B_FULLB0 + b], 1);
            mbar_init(&bars[B_EMPTYB0 + b], 4);
        }
        mbar_init(&bars[B_D1], 3);
        mbar_init(&bars[B_DO], 1);
        mbar_init(&bars[B_OUT], 2);
        mbar_init(&bars[B_D2], 2);
        mbar_init(&bars[B_QSD], 2);
        mbar_init(&bars[B_E1DONE], 1);
        mbar_init(&bars[B_DRAIN], 8);
        *s_err = 0;
        fence_mbar_init();
        if (UNITS ? p.n_units > 0 : nch > 0) {
            prefetch_tensormap(&mapK);
            prefetch_tensormap(&mapQ);
            prefetch_tensormap(&mapV);
        }
    }
    if (warp == 4) { tmem_alloc(tslot, kTmemCols); tmem_relinquish(); }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    // the stream's dependent grid (the states kernel, which takes each segment as it is
    // published) may be scheduled once every CTA of this grid has started
    if constexpr (UNITS) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    auto fail = [&](void) {
        *s_err = 1;
        set_error(p, GDN_ERR_TIMEOUT);
    };
    // single-thread wait (issuing lanes, producer)
    auto wait = [&](int b, uint32_t parity) -> bool {
        if (*s_err) return false;
        if (!mbar_wait(&bars[b], parity)) { fail(); return false; }
        return true;
    };
    auto ring_a = [&](int cc) { return sm + OFF_A + (cc & 1) * kStageA; };
    auto ring_b = [&](int cc) { return sm + OFF_B + (cc & 1) * kStageB; };
    auto desc = [&](int cc) { return descs + (cc & (kDescSlots - 1)) * kDescWords; };
    const uint32_t s_img = smem_u32(sm + OFF_S), z_img = smem_u32(sm + OFF_Z);

    // -W S of chunk cc from the state of chunk cc - 1, k-steps 4(w-1) .. 4(w-1)+3, issued
    // by lane 0 of epilogue warp w = 1 or 2 into its own accumulator; commit D1.  The
    // epilogue warpgroup has already seen ring A of chunk cc loaded.
    auto issue_ws = [&](int w, int cc) {
        tc_fence_after();
        constexpr uint32_t id_ws = instr_desc(128, 64, kFmtBF16, 1, 1);
        const uint32_t k0 = (uint32_t)(w - 1) * 4 * 2048;
        const uint64_t a0 = smem_desc(smem_u32(ring_a(cc) + kAW + REC_WHI) + k0, REC_WLO - REC_WHI, 1024,
                                      kSwizzle128B);
        const uint64_t b0 = smem_desc(s_img + k0, 16, 1024, kSwizzle128B);
        const uint32_t d = tmem + TM_W + (uint32_t)((w - 1) * 64);
#pragma unroll
        for (int q = 0; q < 4; ++q)
            mma_bf16(d, desc_adv(a0, q * 2048), desc_adv(b0, q * 2048), id_ws, q > 0);
        mma_commit(&bars[B_D1]);
    };

    if (warp == 5) {
        // ------------------------------------------------------------ TMA producer, T'' V
        if (lane == 0) {
            constexpr uint32_t id_u = instr_desc(128, NV, kFmtBF16, 0, 1);
            // T'' V of chunk c into D_UT[c % 2] (last read by the epilogue in chunk c - 2,
            // whose U was formed before -W S of chunk c - 1 was issued)
            auto issue_tv = [&](int c) -> bool {
                if (!wait(B_FULLA0 + (c & 1), (c >> 1) & 1)) return false;
                tc_fence_after();
                uint8_t *sa = ring_a(c);
                const uint64_t a0 = smem_desc(smem_u32(sa + kAW + REC_T2HI), 16, 1024, kSwizzle128B);
                const uint64_t b0 = smem_desc(smem_u32(sa + kAV), 16, 512, kSwizzle64B);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_bf16(tmem + TM_UT + (uint32_t)((c & 1) * NV), desc_adv(a0, ks * 32),
                             desc_adv(b0, ks * 1024), id_u, ks > 0);
                mma_commit(&bars[B_D1]);
                return true;
            };
            // the loads of chunk cc: ring A (the record's first 48 KiB and the value slice of
            // value head hh, slice vv), ring B (key and query tiles of key head jj, P and the
            // factor rows)
            auto load_a = [&](int cc, const uint8_t *rec, int tok, int hh, int vv) {
                uint8_t *sa = ring_a(cc);
                uint64_t *fa = &bars[B_FULLA0 + (cc & 1)];
                mbar_arrive_expect_tx(fa, kStageA);
                bulk_load(sa + kAW, rec, REC_P, fa);
                tma_load_3d(sa + kAV, &mapV, fa, vv * NV, hh, tok);
            };
            auto load_b = [&](int cc, const uint8_t *rec, int tok, int jj) {
                uint8_t *sb = ring_b(cc);
                uint64_t *fb = &bars[B_FULLB0 + (cc & 1)];
                mbar_arrive_expect_tx(fb, kStageB);
                tma_load_3d(sb + kBK, &mapK, fb, 0, jj, tok);
                tma_load_3d(sb + kBK + 8192, &mapK, fb, 64, jj, tok);
                tma_load_3d(sb + kBQ, &mapQ, fb, 0, jj, tok);
                tma_load_3d(sb + kBQ + 8192, &mapQ, fb, 64, jj, tok);
                bulk_load(sb + kBP, rec + REC_P, kStageB - kBP, fb);
            };
            bool issued = false;
            // the records come from the prep grid, which may still be running: with the
            // persistent prep beside the chain each record is taken once its ready flag is
            // set, otherwise once the whole prep grid has completed
            if constexpr (!READY) asm volatile("griddepcontrol.wait;" ::: "memory");
            if constexpr (!UNITS) {
                // records known complete: chunks below ready_to
                int ready_to = 0;
                // iteration cc: (once -W S of chunk cc - 2 is done) T'' V of chunk cc - 1, then
                // the loads of chunk cc; the last iteration only issues T'' V of chunk nch - 1.
                // T'' V of chunk 0 waits for its inputs, so it follows the loads of chunk 1.
                for (int cc = 0; cc <= nch; ++cc) {
                    const int st = cc & 1, u = cc >> 1;
                    if (cc >= 2 && !wait(B_EMPTYA0 + st, (u - 1) & 1)) break;
                    if (cc >= 2 || (cc == 1 && nch == 1)) {
                        if (!issue_tv(cc - 1)) break;
                        issued = true;
                    }
                    if (cc == nch) break;
                    const int tok = (int)(sr.t0 + (int64_t)cc * C);
                    const uint8_t *rec = reinterpret_cast<const uint8_t *>(p.rec) +
                                         ((size_t)(sr.first + cc) * p.HV + h) * kRecBytes;
                    if constexpr (READY) {
                        if (cc >= ready_to) {
                            // acquire the record's flag, then read the record with bulk copies;
                            // the flags of the next chunks are read in the same round trip
                            ready_to = ready_wait(p.ready + (size_t)sr.first * p.HV + h, p.HV, cc, nch);
                            if (ready_to < 0) { fail(); break; }
                            fence_async_global();
                        }
                    }
                    load_a(cc, rec, tok, h, vs);
                    if (u >= 1 && !wait(B_EMPTYB0 + st, (u - 1) & 1)) break;
                    load_b(cc, rec, tok, j);
                    if (cc == 1) {
                        if (!issue_tv(0)) break;
                        issued = true;
                    }
                }
            } else {
                Unit w;
                int k = 0, nk = 0;          // chunk k of the nk chunks of the current unit
                // the first unit of CTA b is unit b (a chain's first segment: no
                // predecessor); later ones come from the counter, after the grid's first round
                int next_u = blockIdx.x;
                // per unit: key head, chain number; per chunk (advanced after its loads):
                // first token and record
                int jj = 0, chain = 0, tok = 0;
                const uint8_t *rec = nullptr;
                const size_t rec_step = (size_t)p.HV * kRecBytes;
                // iteration cc (once -W S of chunk cc - 2 is done): the next chunk of the
                // stream (of the current unit, else of the next unit claimed that has chunks)
                // or the end of the stream, published in the chunk's descriptor, and T'' V of
                // chunk cc - 1
                for (int cc = 0;; ++cc) {
                    const int st = cc & 1, u = cc >> 1;
                    if (cc >= 2 && !wait(B_EMPTYA0 + st, (u - 1) & 1)) break;
                    bool stop = false;
                    while (k >= nk) {
                        const int un = next_u >= 0 ? next_u
                                     : p.n_units <= (int)gridDim.x ? p.n_units   // all were first ones
                                     : (int)gridDim.x + atomicAdd(&p.status[kClaimWord], 1);
                        next_u = -1;
                        if (un >= p.n_units || !unit_of(p, un, w)) { stop = true; break; }
                        k = 0;
                        nk = w.c1 - w.c0;
                        jj = w.h / (p.HV / p.HK);
                        chain = (w.s * p.HV + w.h) * (D / NV) + w.vs;
                        tok = (int)(w.sr.t0 + (int64_t)w.c0 * C);
                        rec = reinterpret_cast<const uint8_t *>(p.rec) +
                              ((size_t)(w.sr.first + w.c0) * p.HV + w.h) * kRecBytes;
                    }
                    int32_t *d = desc(cc);
                    if (stop) {
                        // an armed phase with no data: the other warps read the end marker
                        d[DW_LEN] = DF_STOP << 8;
                        mbar_arrive(&bars[B_FULLA0 + st]);
                    } else {
                        const int len = (int)min((int64_t)C, w.sr.t_end - tok);
                        const int fl = (k == 0 ? DF_FIRST : 0) | (k == nk - 1 ? DF_LAST : 0) |
                                       (w.c0 + k == w.sr.count - 1 ? DF_END : 0);
                        d[DW_TOK] = tok;
                        d[DW_LEN] = len | (fl << 8);
                        d[DW_CHAIN] = chain;
                        d[DW_SEG] = w.seg;
                        d[DW_HEAD] = w.h;
                        d[DW_SLICE] = w.vs;
                        load_a(cc, rec, tok, w.h, w.vs);
                    }
                    // T'' V of chunk cc - 1 goes ahead of ring B's wait (which ends only with
                    // the state update of chunk cc - 2), so that it runs before -W S of chunk
                    // cc - 1
                    if (cc >= 2 || (cc == 1 && stop)) {
                        if (!issue_tv(cc - 1)) break;
                        issued = true;
                    }
                    if (u >= 1 && !wait(B_EMPTYB0 + st, (u - 1) & 1)) break;
                    if (stop) {
                        mbar_arrive(&bars[B_FULLB0 + st]);
                        break;
                    }
                    load_b(cc, rec, tok, jj);
                    ++k;
                    tok += C;
                    rec += rec_step;
                    // T'' V of chunk 0 waits for its inputs, so it follows the loads of chunk 1
                    if (cc == 1) {
                        if (!issue_tv(0)) break;
                        issued = true;
                    }
                }
            }
            if (issued) mma_commit(&bars[B_DRAIN]);
            else mbar_arrive(&bars[B_DRAIN]);
        }
    } else if (warp == 4) {
        // ------------------------------------------------------------ off-path products
        if (lane == 0) {
            constexpr uint32_t id_o = instr_desc(128, NV, kFmtBF16, 0, 1);
            bool issued = false;
            for (int cc = 0; UNITS || cc < nch; ++cc) {
                // P U_hi (outputs only: one bf16 term) once U is formed and the output
                // warps have read the previous chunk's
                // polled without parking: the tensor pipe runs in order, and P U issued late
                // would sit in front of the next chunk's -W S.  At the end of a stream the
                // epilogue completes one more phase, and the chunk's descriptor says so.
                if (*s_err || !mbar_wait_spin(&bars[B_E1DONE], cc & 1)) { fail(); break; }
                if constexpr (UNITS) {
                    if (desc(cc)[DW_LEN] & (DF_STOP << 8)) break;
                }
                if (cc >= 1 && !wait(B_OUT, (cc - 1) & 1)) break;
                issued = true;
                tc_fence_after();
                {
                    const uint64_t a0 = smem_desc(smem_u32(ring_b(cc) + kBP - 8192), 16, 1024, kSwizzle128B);
                    const uint64_t b0 = smem_desc(smem_u32(sm + OFF_U), 16, 512, kSwizzle64B);
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_bf16(tmem + TM_PU, desc_adv(a0, ks * 32), desc_adv(b0, ks * 1024), id_o, ks > 0);
                    mma_commit(&bars[B_DO]);
                    mma_commit(&bars[B_EMPTYB0 + (cc & 1)]);
                }
            }
            if (issued) mma_commit(&bars[B_DRAIN]);
            else mbar_arrive(&bars[B_DRAIN]);
        }
    } else if (warp >= 6) {
        // ------------------------------------------------------------ output warps
        // thread = token t (TMEM lane 64 + t of the stacked output accumulator)
        const int t = tid - 192;
        const uint32_t lb = lane_base(warp);
        bool issued = false;
        for (int cc = 0; UNITS || cc < nch; ++cc) {
            // this thread's token, whether it is in the sequence, the value head and slice
            int64_t tok;
            bool live;
            int hh, vv;
            if constexpr (UNITS) {
                // ring B's phase publishes the chunk's descriptor (or the end of the stream)
                bool ok = !*s_err && mbar_wait(&bars[B_FULLB0 + (cc & 1)], (cc >> 1) & 1);
                if (!ok) fail();
                if (!__all_sync(0xffffffffu, ok)) break;
                const int32_t *d = desc(cc);
                const int dlen = d[DW_LEN];
                if (dlen & (DF_STOP << 8)) break;
                tok = (int64_t)d[DW_TOK] + t;
                live = t < (dlen & 255);
                hh = d[DW_HEAD];
                vv = d[DW_SLICE];
            } else {
                tok = sr.t0 + (int64_t)cc * C + t;
                live = tok < sr.t_end;
                hh = h;
                vv = vs;
            }
            // Q S of chunk cc, k-steps 4 (warp - 6) .. + 3: A = [any; Q] read from 8 KiB
            // before the query tile so that the live rows land in TMEM lanes 64-127.  The
            // state operand it reads was written before -W S of chunk cc was issued and is
            // rewritten only after QSD; both output warps have read Q S of chunk cc - 1 (OUT).
            if (lane == 0) {
                bool ok2 = wait(B_D1, cc & 1) && (UNITS || wait(B_FULLB0 + (cc & 1), (cc >> 1) & 1)) &&
                           (cc == 0 || wait(B_OUT, (cc - 1) & 1));
                if (ok2) {
                    tc_fence_after();
                    constexpr uint32_t id_qs = instr_desc(128, 64, kFmtBF16, 0, 1);
                    // k-steps 4 (warp - 6) + q: the query half (warp - 6) at 32 q bytes, the
                    // state rows at (4 (warp - 6) + q) 2 KiB
                    const uint32_t half = (uint32_t)(warp - 6);
                    const uint64_t a0 = smem_desc(smem_u32(ring_b(cc) + kBQ - 8192) + half * 8192, 16, 1024,
                                                  kSwizzle128B);
                    const uint64_t b0 = smem_desc(s_img + half * 4 * 2048, 16, 1024, kSwizzle128B);
                    const uint32_t dq = tmem + TM_QS + half * 64;
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        mma_bf16(dq, desc_adv(a0, q * 32), desc_adv(b0, q * 2048), id_qs, q > 0);
                    mma_commit(&bars[B_QSD]);
                    issued = true;
                }
            }
            __syncwarp();
            if constexpr (!UNITS) {
                bool ok = !*s_err && mbar_wait(&bars[B_FULLB0 + (cc & 1)], (cc >> 1) & 1);
                if (!ok) fail();
                if (!__all_sync(0xffffffffu, ok)) break;
            }
            // the chunk's query factor, then release ring B's factor rows
            const float qd = reinterpret_cast<const float *>(ring_b(cc) + kBF)[SC_QD * C + t];
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[B_EMPTYB0 + (cc & 1)]);
            bool ok = !*s_err && mbar_wait(&bars[B_QSD], cc & 1) && mbar_wait(&bars[B_DO], cc & 1);
            if (!ok) fail();
            if (!__all_sync(0xffffffffu, ok)) break;
            tc_fence_after();
            float o1[NV], o2[NV], o3[NV];
            tmem_ld32(tmem + lb + TM_QS, o1);
            tmem_ld32(tmem + lb + TM_QS + 32, o2);
            tmem_ld32(tmem + lb + TM_QS + 64, o3);
            tmem_ld_wait();
#pragma unroll
            for (int q = 0; q < NV; q += 2) {               // pairs: one instruction for two
                const uint64_t r = fadd2(f2pack(o1[q], o1[q + 1]), fadd2(f2pack(o2[q], o2[q + 1]),
                                                                          f2pack(o3[q], o3[q + 1])));
                f2unpack(r, o1[q], o1[q + 1]);
            }
            tmem_ld32(tmem + lb + TM_QS + 96, o2);
            tmem_ld32(tmem + lb + TM_PU, o3);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[B_OUT]);
            const uint64_t qd2 = f2pack(qd, qd);
#pragma unroll
            for (int q = 0; q < NV; q += 2) {
                const uint64_t r = ffma2(qd2, fadd2(f2pack(o1[q], o1[q + 1]), f2pack(o2[q], o2[q + 1])),
                                         f2pack(o3[q], o3[q + 1]));
                f2unpack(r, o1[q], o1[q + 1]);
            }
            if (live) {
                __nv_bfloat16 *dst = p.out + ((size_t)tok * p.HV + hh) * D + (size_t)vv * NV;
#pragma unroll
                for (int q = 0; q < NV; q += 8) {
                    uint32_t w[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        w[e] = pack2(__float2bfloat16_rn(o1[q + 2 * e]), __float2bfloat16_rn(o1[q + 2 * e + 1]));
                    *reinterpret_cast<uint4 *>(dst + q) = make_uint4(w[0], w[1], w[2], w[3]);
                }
            }
        }
        if (lane == 0) {
            if (issued) mma_commit(&bars[B_DRAIN]);
            else mbar_arrive(&bars[B_DRAIN]);
        }
    } else {
        // ------------------------------------------------------------ epilogue warpgroup
        const int i = tid;                  // key row of the state slice / row of the
                                            // M = 128 results
        const bool lead = (i == 0);
        const uint32_t lb = lane_base(warp);
        const int tk = i & 63, hf = i >> 6;        // token, column half handled in E1
        float S[NV];
        float *xf = reinterpret_cast<float *>(sm + OFF_X);
        // whole 32-byte sectors for the values left in the states tensor when its base
        // allows (every offset written below is a multiple of 64 bytes)
        const bool states32 = STATES && ((uintptr_t)p.states & 31u) == 0;
        // Up to four (barrier, parity) pairs, a negative barrier index being skipped: warp w
        // polls pair w (all its threads), then one barrier reduction over the warpgroup
        // joins them and makes the outcome uniform (a timeout anywhere stops every thread);
        // the barrier also orders every thread after the phases the other warps observed.
        auto wg_wait4 = [&](int b1, uint32_t p1, int b2, uint32_t p2, int b3, uint32_t p3,
                            int b4, uint32_t p4) -> bool {
            const int b = warp == 0 ? b1 : warp == 1 ? b2 : warp == 2 ? b3 : b4;
            const uint32_t par = warp == 0 ? p1 : warp == 1 ? p2 : warp == 2 ? p3 : p4;
            bool ok = !*s_err;
            if (ok && b >= 0 && !mbar_wait(&bars[b], par)) { fail(); ok = false; }
            return wg_and(ok);
        };
        // row i of a chain's slice in a [N][HV][D][D] fp32 state tensor (chains are numbered
        // (sequence, value head, slice)-major)
        auto slice_row = [&](int chain) -> size_t {
            return ((size_t)(chain / (D / NV)) * D + i) * D + (size_t)(chain % (D / NV)) * NV;
        };
        // the lead's end-state flag not yet published (the next segment of its chain waits)
        int32_t *pend = nullptr;
        int32_t pend_v = 0;
        // The state slice at the start of the unit of descriptor d: the initial state (zero
        // without one) for a chain's first segment, else the end state of the previous
        // segment once its CTA has published it (this CTA's own pending flag goes out first
        // if that means waiting); then its bf16 hi/lo operand image.
        auto unit_state = [&](const int32_t *d) -> bool {
            const int seg = d[DW_SEG];
            bool ok = !*s_err;
            if (lead && ok && seg > 0) {
                const int32_t *f = p.chain_flags + d[DW_CHAIN];
                if (flag_acquire(f) < seg) {
                    if (pend) { flag_release(pend, pend_v); pend = nullptr; }
                    if (!flag_wait(f, seg)) { fail(); ok = false; }
                }
            }
            if (!wg_and(ok)) return false;
            const float *src = nullptr;
            if (seg == 0) src = p.s0 ? p.s0 + slice_row(d[DW_CHAIN]) : nullptr;
            else if (STATES)
                src = p.states + ((size_t)(d[DW_TOK] - 1) * p.HV + d[DW_HEAD]) * (D * D) + (size_t)i * D +
                      (size_t)d[DW_SLICE] * NV;
            else src = p.s_final + slice_row(d[DW_CHAIN]);
            if (src) {
#pragma unroll
                for (int q = 0; q < NV / 4; ++q) {
                    const float4 v4 = __ldcg(reinterpret_cast<const float4 *>(src) + q);
                    S[4 * q] = v4.x; S[4 * q + 1] = v4.y; S[4 * q + 2] = v4.z; S[4 * q + 3] = v4.w;
                }
            } else {
#pragma unroll
                for (int q = 0; q < NV; ++q) S[q] = 0.f;
            }
            store_row_hilo128(sm + OFF_S, i, S);
            fence_async_smem();
            tc_fence_before();
            named_sync(1, 128);
            return true;
        };
        bool issued = false;                // this lane has issued tensor-core work
        // the state after a chunk's last token, with per-token states: the carried
        // chunk-form state
        auto state_out = [&](float *dst) {
            if (states32) {
#pragma unroll
                for (int q = 0; q < NV / 8; ++q) st_v8(dst + 8 * q, S + 8 * q);
            } else {
#pragma unroll
                for (int q = 0; q < NV / 4; ++q)
                    reinterpret_cast<float4 *>(dst)[q] = make_float4(S[4 * q], S[4 * q + 1], S[4 * q + 2],
                                                                     S[4 * q + 3]);
            }
        };
        // One chunk of the chain: E1 (U, Z = kd U, K^T Z) and E2 (the new state); then,
        // unless the chunk ends its unit, the next state operand, -W S of the next chunk
        // (issue_next) and, with per-token states, the carried state.  (tok0, len, hh, vv):
        // the chunk's first token and length, value head and value slice; wait_next: ring A
        // of the next chunk is armed (data, or the end of a stream).  Returns 0 (next chunk),
        // 1 (the chunk ends its unit: the state is in S), -1 (a wait gave up).
        auto chunk = [&](int cc, int64_t tok0, int len, int hh, int vv, bool wait_next, bool unit_end,
                         bool issue_next) -> int {
            const int st = cc & 1;
            uint8_t *sb = ring_b(cc);
            const float *F = reinterpret_cast<const float *>(sb + kBF);
            // ---- E1: U = rows 0-63 + rows 64-127 of (-W S + T'' V), Z = kd U; the previous
            // chunk's P U_hi must have read the U_hi image
            if (!wg_wait4(B_D1, cc & 1, B_FULLB0 + st, (cc >> 1) & 1, cc >= 1 ? B_DO : -1, (cc - 1) & 1,
                          -1, 0))
                return -1;
            if (lead) mbar_arrive(&bars[B_EMPTYA0 + st]);   // ring A of chunk cc is consumed
            tc_fence_after();
            const float kd = F[SC_KD * C + tk], gl = F[SC_MISC * C + 0];
            float uu[NV];
            {
                float a[NV], b[NV], c2[NV];
                tmem_ld32(tmem + lb + TM_UT + (uint32_t)(st * NV), uu);
                tmem_ld32(tmem + lb + TM_W, a);
                tmem_ld32(tmem + lb + TM_W + 32, b);
                tmem_ld_wait();
#pragma unroll
                for (int c = 0; c < NV; c += 2) {       // pairs: one instruction for two
                    const uint64_t r = fadd2(f2pack(uu[c], uu[c + 1]),
                                             fadd2(f2pack(a[c], a[c + 1]), f2pack(b[c], b[c + 1])));
                    f2unpack(r, uu[c], uu[c + 1]);
                }
                tmem_ld32(tmem + lb + TM_W + 64, a);
                tmem_ld32(tmem + lb + TM_W + 96, c2);
                tmem_ld_wait();
#pragma unroll
                for (int c = 0; c < NV; c += 2) {
                    const uint64_t r = fadd2(f2pack(uu[c], uu[c + 1]),
                                             fadd2(f2pack(a[c], a[c + 1]), f2pack(c2[c], c2[c + 1])));
                    f2unpack(r, uu[c], uu[c + 1]);
                }
            }
            // keep this thread's 16 columns, send the other 16 to the partner row (tk, 1 - hf)
            float u16[16], o16[16];
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                u16[k] = hf ? uu[16 + k] : uu[k];
                o16[k] = hf ? uu[k] : uu[16 + k];
            }
            {
                float *dst = xf + (1 - hf) * (C * 16);
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    *reinterpret_cast<float4 *>(dst + xchg_off(tk, c)) =
                        make_float4(o16[4 * c], o16[4 * c + 1], o16[4 * c + 2], o16[4 * c + 3]);
            }
            named_sync(1, 128);
            {
                const float *src = xf + hf * (C * 16);
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const float4 x4 = *reinterpret_cast<const float4 *>(src + xchg_off(tk, c));
                    const uint64_t r0 = fadd2(f2pack(u16[4 * c], u16[4 * c + 1]), f2pack(x4.x, x4.y));
                    const uint64_t r1 = fadd2(f2pack(u16[4 * c + 2], u16[4 * c + 3]), f2pack(x4.z, x4.w));
                    f2unpack(r0, u16[4 * c], u16[4 * c + 1]);
                    f2unpack(r1, u16[4 * c + 2], u16[4 * c + 3]);
                }
            }
            // columns 16 hf .. 16 hf + 15 of token tk: Z_hi, Z_lo (chunks 2 hf, 2 hf + 1 of
            // each half of the 128-byte row) and U_hi (chunks 2 hf, 2 hf + 1 of the 64-byte row)
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                uint32_t zh[4], zl[4], uh[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int c = 8 * q + 2 * e;
                    float z0, z1;
                    f2unpack(fmul2(f2pack(kd, kd), f2pack(u16[c], u16[c + 1])), z0, z1);
                    split2_bf16(z0, z1, zh[e], zl[e]);
                    const __nv_bfloat162 u2v = __floats2bfloat162_rn(u16[c], u16[c + 1]);
                    uh[e] = *reinterpret_cast<const uint32_t *>(&u2v);
                }
                const int ch = 2 * hf + q;
                *reinterpret_cast<uint4 *>(sm + OFF_Z + sw128_offset(tk, ch * 16)) = make_uint4(zh[0], zh[1], zh[2], zh[3]);
                *reinterpret_cast<uint4 *>(sm + OFF_Z + sw128_offset(tk, 64 + ch * 16)) = make_uint4(zl[0], zl[1], zl[2], zl[3]);
                *reinterpret_cast<uint4 *>(sm + OFF_U + sw64_offset(tk, ch * 16)) = make_uint4(uh[0], uh[1], uh[2], uh[3]);
            }
            if (STATES && tk < len - 1) {
                // U rows 0 .. len-2 of the chunk (fp32, this slice's columns) for the states
                // kernel, parked in the slot of the chunk's first token: row t at float t * D
                // (the states kernel reads them before it writes that slot)
                float *dst = p.states + ((size_t)tok0 * p.HV + hh) * (D * D) + (size_t)tk * D +
                             (size_t)vv * NV + hf * 16;
                if (states32) {
                    st_v8(dst, u16);
                    st_v8(dst + 8, u16 + 8);
                } else {
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        *reinterpret_cast<float4 *>(dst + 4 * c) =
                            make_float4(u16[4 * c], u16[4 * c + 1], u16[4 * c + 2], u16[4 * c + 3]);
                }
            }
            fence_async_smem();
            tc_fence_before();
            named_sync(1, 128);                 // Z and U complete
            if (lead) mbar_arrive(&bars[B_E1DONE]);
            if (lane == 0 && (warp == 2 || warp == 3)) {
                // K^T [Z_hi | Z_lo]: A = key tile read MN-major; k-steps 0-1 / 2-3
                tc_fence_after();
                constexpr uint32_t id_kz = instr_desc(128, 64, kFmtBF16, 1, 1);
                const uint32_t k0 = (uint32_t)(warp - 2) * 2 * 2048;
                const uint64_t a0 = smem_desc(smem_u32(sb + kBK) + k0, 8192, 1024, kSwizzle128B);
                const uint64_t b0 = smem_desc(z_img + k0, 16, 1024, kSwizzle128B);
                const uint32_t d = tmem + (warp == 2 ? TM_S : TM_S2);
#pragma unroll
                for (int q = 0; q < 2; ++q)
                    mma_bf16(d, desc_adv(a0, q * 2048), desc_adv(b0, q * 2048), id_kz, q > 0);
                mma_commit(&bars[B_D2]);
                issued = true;
            }
            __syncwarp();
            // ---- E2: new state (thread i = key row i).  Ring A of the next chunk is checked
            // here, for the -W S issued after the update: its loads start only once E1 of this
            // chunk has released the other stage, and waiting for them in E1 would put their
            // latency on the chain.
            if (!wg_wait4(B_D2, cc & 1, B_QSD, cc & 1, wait_next ? B_FULLA0 + (st ^ 1) : -1, ((cc + 1) >> 1) & 1,
                          -1, 0))
                return -1;
            tc_fence_after();
            float ds[NV];
            {
                float d2[NV], d3[NV], d4[NV];
                tmem_ld32(tmem + lb + TM_S, ds);
                tmem_ld32(tmem + lb + TM_S + 32, d2);
                tmem_ld32(tmem + lb + TM_S2, d3);
                tmem_ld32(tmem + lb + TM_S2 + 32, d4);
                tmem_ld_wait();
#pragma unroll
                for (int c = 0; c < NV; c += 2) {
                    const uint64_t r = fadd2(fadd2(f2pack(ds[c], ds[c + 1]), f2pack(d2[c], d2[c + 1])),
                                             fadd2(f2pack(d3[c], d3[c + 1]), f2pack(d4[c], d4[c + 1])));
                    f2unpack(r, ds[c], ds[c + 1]);
                }
            }
#pragma unroll
            for (int c = 0; c < NV; c += 2) {
                const uint64_t r = ffma2(f2pack(gl, gl), f2pack(S[c], S[c + 1]), f2pack(ds[c], ds[c + 1]));
                f2unpack(r, S[c], S[c + 1]);
            }
            if (unit_end) return 1;
            store_row_hilo128(sm + OFF_S, i, S);     // Q S of this chunk is done (QSD above)
            fence_async_smem();
            tc_fence_before();
            named_sync(1, 128);                 // the new state operand is complete
            if (lead) mbar_arrive(&bars[B_EMPTYB0 + st]);   // (with the P U commit)
            if (issue_next && lane == 0 && (warp == 1 || warp == 2)) {
                issue_ws(warp, cc + 1);
                issued = true;
            }
            __syncwarp();
            if (STATES)
                state_out(p.states + ((size_t)(tok0 + len - 1) * p.HV + hh) * (D * D) + (size_t)i * D +
                          (size_t)vv * NV);
            return 0;
        };
        if constexpr (!UNITS) {
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
            store_row_hilo128(sm + OFF_S, i, S);
            fence_async_smem();
            named_sync(1, 128);
            int nch_run = nch;
            if (nch > 0) {
                if (!wg_wait4(B_FULLA0, 0, -1, 0, -1, 0, -1, 0)) nch_run = 0;
                else if (lane == 0 && (warp == 1 || warp == 2)) {
                    issue_ws(warp, 0);
                    issued = true;
                }
                __syncwarp();
            }
            for (int cc = 0; cc < nch_run; ++cc) {
                const int64_t tok0 = sr.t0 + (int64_t)cc * C;
                const int len = (int)min((int64_t)C, sr.t_end - tok0);
                if (chunk(cc, tok0, len, h, vs, cc + 1 < nch, false, cc + 1 < nch) < 0) break;
            }
            if (lane == 0) {
                if (issued) mma_commit(&bars[B_DRAIN]);
                else mbar_arrive(&bars[B_DRAIN]);
            }
            // final state slice (with per-token states, a later kernel copies it from the last
            // token's state once nothing reads the initial state any more: they may alias)
            if (!STATES && !*s_err) {
#pragma unroll
                for (int q = 0; q < NV / 4; ++q)
                    reinterpret_cast<float4 *>(p.s_final + sbase)[q] =
                        make_float4(S[4 * q], S[4 * q + 1], S[4 * q + 2], S[4 * q + 3]);
            }
        } else {
            // ring A of the first chunk: its descriptor says what the stream holds
            bool run = wg_wait4(B_FULLA0, 0, -1, 0, -1, 0, -1, 0);
            int cc = 0;
            while (run) {
                // ---- the start of a unit (chunk cc, whose ring A has been seen armed): its
                // state, then -W S of its first chunk; the previous unit's end state is
                // published once that is on its way (or before any wait for another CTA)
                const int32_t *d0 = desc(cc);
                if ((d0[DW_LEN] & (DF_STOP << 8)) || !unit_state(d0)) break;
                if (lane == 0 && (warp == 1 || warp == 2)) {
                    issue_ws(warp, cc);
                    issued = true;
                }
                __syncwarp();
                if (pend) { flag_release(pend, pend_v); pend = nullptr; }
                // ---- the chunks of the unit (its descriptors stay in place for the whole
                // chunk: slot cc % 4 is rewritten for chunk cc + 4, after E1 of chunk cc + 2);
                // the last one returns after its state update
                int r;
                for (;; ++cc) {
                    const int32_t *dc = desc(cc);
                    const int dl = dc[DW_LEN];
                    r = chunk(cc, dc[DW_TOK], dl & 255, dc[DW_HEAD], dc[DW_SLICE], true, (dl >> 8) & DF_LAST, true);
                    if (r != 0) break;
                }
                if (r < 0) break;                   // a wait gave up
                // ---- the end of the unit (chunk cc): its end state goes out (the slot of
                // its last token, or the final-state slice: the final state, or the start of
                // the chain's next segment); then every thread's row is out and its reads of
                // ring B are done.  Ring A of chunk cc + 1 was seen in E2 of chunk cc.
                const int32_t *de = desc(cc);
                if (STATES) {
                    state_out(p.states + ((size_t)(de[DW_TOK] + (de[DW_LEN] & 255) - 1) * p.HV + de[DW_HEAD]) *
                                             (D * D) + (size_t)i * D + (size_t)de[DW_SLICE] * NV);
                    // the chain's final state, when nothing later reads the initial state
                    // through the same buffer
                    if (p.final_direct && (de[DW_LEN] & (DF_END << 8))) {
#pragma unroll
                        for (int q = 0; q < NV / 4; ++q)
                            reinterpret_cast<float4 *>(p.s_final + slice_row(de[DW_CHAIN]))[q] =
                                make_float4(S[4 * q], S[4 * q + 1], S[4 * q + 2], S[4 * q + 3]);
                    }
                }
                else {
#pragma unroll
                    for (int q = 0; q < NV / 4; ++q)
                        reinterpret_cast<float4 *>(p.s_final + slice_row(de[DW_CHAIN]))[q] =
                            make_float4(S[4 * q], S[4 * q + 1], S[4 * q + 2], S[4 * q + 3]);
                }
                named_sync(1, 128);
                if (lead) mbar_arrive(&bars[B_EMPTYB0 + (cc & 1)]);
                // (with per-token states also a chain's last segment: the states kernel waits)
                if (lead && (STATES || !(de[DW_LEN] & (DF_END << 8)))) {
                    pend = p.chain_flags + de[DW_CHAIN];
                    pend_v = de[DW_SEG] + 1;
                }
                ++cc;
            }
            if (lead && pend) flag_release(pend, pend_v);
            if (lead && !*s_err) mbar_arrive(&bars[B_E1DONE]);   // the end of the stream, for warp 4
            if (lane == 0) {
                if (issued) mma_commit(&bars[B_DRAIN]);
                else mbar_arrive(&bars[B_DRAIN]);
            }
        }
        if (lead) mbar_wait(&bars[B_DRAIN], 0);   // every MMA of the CTA has finished
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 4) tmem_dealloc(tmem, kTmemCols);
}
// ------------------------------------------------------------------ per-token states
// One CTA per (chunk, value head, 32-wide value slice), all independent.  It replays the
// recurrence S_t = alpha_t S_{t-1} + (rk_t k_t) u_t^T over the chunk's tokens but the last
// one, from the state before the chunk, with the chunk-form U rows: the same u_t as the
// token-by-token rule.  The chain kernel left in the states tensor the carried state after
// every chunk's last token (the state before chunk c > 0 of a sequence is the last
// per-token state of chunk c - 1; before the first chunk it is the initial state, or
// zero) and the chunk's U rows in the slot of its first token, columns of this slice;
// this CTA is the only reader of those rows and reads them all before it overwrites the
// slot.  Thread (r, cg) owns value columns 4 cg .. 4 cg + 3 of key rows r + 32 m, so a
// warp stores four whole 128-byte row segments per instruction.
constexpr int kStThreads = 256;

__global__ void __launch_bounds__(kStThreads)
states_kernel(Params p) {
    __shared__ float sF[C][D];                    // rk_t k_t[i]
    __shared__ __align__(16) float sU[C][NV];     // u_t, this slice's columns
    __shared__ float sAl[C];                      // alpha_t
    __shared__ int s_ok;
    // beside the chain's work-unit stream, the last CTA (started last) waits for the whole
    // stream grid first: this grid then ends only after it, so later work in the stream
    // finds every output and state in place
    if (p.states_overlap && blockIdx.x == gridDim.x - 1) asm volatile("griddepcontrol.wait;" ::: "memory");
    if (p.status[kStatusWord] != GDN_OK) return;
    int m = blockIdx.x, h = blockIdx.y, vs = blockIdx.z;
    if (p.states_overlap) {
        // running beside the chain's work-unit stream: CTAs in the order the stream ends
        // its segments (segment-major, then chain, then chunk); each waits until the
        // segment holding its chunk is published (its U rows and the carried state before
        // it are then in the states tensor)
        const int cps = (p.T_seq + C - 1) / C, L = p.seg_len;
        const int q = blockIdx.x, per_seg = p.n_chains * L;
        const int seg = q / per_seg, rem = q - seg * per_seg;
        const int chain = rem / L, cc0 = seg * L + (rem - (rem / L) * L);
        if (cc0 >= cps) return;
        vs = chain % (D / NV);
        h = (chain / (D / NV)) % p.HV;
        m = (chain / (D / NV) / p.HV) * cps + cc0;
        if (threadIdx.x == 0) {
            s_ok = flag_wait(p.chain_flags + chain, seg + 1);
            if (!s_ok) set_error(p, GDN_ERR_TIMEOUT);
        }
        __syncthreads();
        if (!s_ok) return;
    }
    int cc;
    int64_t t0;
    int len;
    int s;
    if (p.cu_seqlens) {
        if (m >= p.status[kChunkCountWord]) return;
        s = p.chunk_seq[m];
        cc = m - p.chunk_first[s];
        t0 = p.cu_seqlens[s] + (int64_t)cc * C;
        len = (int)min((int64_t)C, (int64_t)p.cu_seqlens[s + 1] - t0);
    } else {
        const int cps = (p.T_seq + C - 1) / C;
        if (cps == 0 || m >= p.N * cps) return;
        s = m / cps;
        cc = m - s * cps;
        t0 = (int64_t)s * p.T_seq + (int64_t)cc * C;
        len = min(C, p.T_seq - cc * C);
    }
    const int n = len - 1;                        // tokens whose states are written here
    if (n <= 0) return;
    const int j = h / (p.HV / p.HK);
    const int tid = threadIdx.x;
    const size_t slot = (size_t)D * D;            // floats per (token, value head)
    // the chunk's factor rows (written by the prep grid: complete and visible once the
    // chain, which waited for it before its first record, published the segment) and its
    // U rows (this slice's columns)
    const float *F = reinterpret_cast<const float *>(reinterpret_cast<const uint8_t *>(p.rec) +
                                                     ((size_t)m * p.HV + h) * kRecBytes + REC_F);
    const float *park = p.states + ((size_t)t0 * p.HV + h) * slot + (size_t)vs * NV;
    for (int e = tid; e < n * (NV / 4); e += kStThreads) {
        const int t = e >> 3, c4 = e & 7;
        *reinterpret_cast<float4 *>(&sU[t][4 * c4]) =
            *reinterpret_cast<const float4 *>(park + (size_t)t * D + 4 * c4);
    }
    for (int e = tid; e < n * (D / 8); e += kStThreads) {
        const int t = e >> 4, c8 = e & 15;
        const uint4 raw = *reinterpret_cast<const uint4 *>(p.k + ((size_t)(t0 + t) * p.HK + j) * D + 8 * c8);
        const float rk = F[SC_RK * C + t];
        const __nv_bfloat16 *kb = reinterpret_cast<const __nv_bfloat16 *>(&raw);
#pragma unroll
        for (int q = 0; q < 8; ++q) sF[t][8 * c8 + q] = rk * __bfloat162float(kb[q]);
    }
    if (tid < n) sAl[tid] = F[SC_ALPHA * C + tid];
    const int cg = tid & 7, r = tid >> 3;
    const float *src = cc > 0 ? p.states + ((size_t)(t0 - 1) * p.HV + h) * slot
                     : p.s0 ? p.s0 + ((size_t)s * p.HV + h) * slot : nullptr;
    float S[4][4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        float4 v4 = make_float4(0.f, 0.f, 0.f, 0.f);
        if (src) v4 = *reinterpret_cast<const float4 *>(src + (size_t)(r + 32 * q) * D + vs * NV + 4 * cg);
        S[q][0] = v4.x; S[q][1] = v4.y; S[q][2] = v4.z; S[q][3] = v4.w;
    }
    __syncthreads();                              // every U row is read before the slot is rewritten
    float *dst = p.states + ((size_t)t0 * p.HV + h) * slot + (size_t)vs * NV + 4 * cg;
    for (int t = 0; t < n; ++t, dst += (size_t)p.HV * slot) {
        const float al = sAl[t];
        const float4 u = *reinterpret_cast<const float4 *>(&sU[t][4 * cg]);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float f = sF[t][r + 32 * q];
            S[q][0] = al * S[q][0] + f * u.x;
            S[q][1] = al * S[q][1] + f * u.y;
            S[q][2] = al * S[q][2] + f * u.z;
            S[q][3] = al * S[q][3] + f * u.w;
            st_cs_v4(dst + (size_t)(r + 32 * q) * D, S[q][0], S[q][1], S[q][2], S[q][3]);
        }
    }
}

// Final states when per-token states are written: the last token's state (the carried
// chunk-form state), or the initial state (zero without one) for an empty sequence.  It
// runs after the states kernel, the last reader of the initial states, so a final state
// buffer that aliases the initial one is safe.
__global__ void __launch_bounds__(256)
final_from_states_kernel(Params p) {
    if (p.status[kStatusWord] != GDN_OK) return;
    const int h = blockIdx.x, s = blockIdx.y;
    int64_t t0, t_end;
    if (p.cu_seqlens) {
        t0 = p.cu_seqlens[s];
        t_end = p.cu_seqlens[s + 1];
    } else {
        t0 = (int64_t)s * p.T_seq;
        t_end = t0 + p.T_seq;
    }
    const size_t slot = (size_t)D * D;
    const float4 *src = t_end > t0 ? reinterpret_cast<const float4 *>(p.states + ((size_t)(t_end - 1) * p.HV + h) * slot)
                      : p.s0 ? reinterpret_cast<const float4 *>(p.s0 + ((size_t)s * p.HV + h) * slot)
                             : nullptr;
    float4 *dst = reinterpret_cast<float4 *>(p.s_final + ((size_t)s * p.HV + h) * slot);
    for (int e = threadIdx.x; e < D * D / 4; e += 256) dst[e] = src ? src[e] : make_float4(0.f, 0.f, 0.f, 0.f);
}

// ================================================================== host side
// the driver's tensor-map encoder, looked up once per process (a function-local static
// is initialised exactly once even when several host threads launch at the same time)
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        cudaDriverEntryPointQueryResult q;
        void *f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess && q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
        return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
    }();
    return fn;
}

// [T_total][heads][128] bf16 viewed as 3-D (element, head, token), box {box_x, 1, 64}
static bool make_map(CUtensorMap *m, const void *base, int heads, int64_t T_total, int box_x,
                     CUtensorMapSwizzle swizzle) {
    auto enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)heads, (cuuint64_t)T_total};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)heads * D * 2};
    cuuint32_t box[3] = {(cuuint32_t)box_x, 1, (cuuint32_t)C};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides,
                     box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     swizzle,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace tc

namespace tc {

struct ChainPlan {
    int n_chains, seg_len, n_units, grid;
};

// The work-unit stream of an equal-length batch: while its chains fit on the SMs, one
// unit per chain (and the fixed-chain kernel runs instead); otherwise segments of seg_len
// chunks, chosen to minimise the estimated makespan ceil(units / SMs) * (seg_len +
// kUnitCost) in chunk periods, kUnitCost standing for the hand-off of a segment's state
// between CTAs; one CTA per SM at most (its shared memory and TMEM allow no more).
constexpr double kUnitCost = 0.5;

// Beside the states kernel (per-token states of an equal-length batch): segments of
// kOverlapSeg chunks, so that the first states CTAs find work early, and about a sixth of
// the SMs for the stream.  A stream CTA ends a chunk per ~2.5 us; a states CTA writes a
// chunk's states (1 MiB a 32-wide slice) in ~100 us, five to an SM, so ~17 stream CTAs keep
// 135 SMs of states CTAs busy; more take SMs from the writes the call is bound by (measured
// at B = 4, T = 1024: 16 CTAs starve the writes, 25 give 90.7% of HBM, 38 give 87.5%).
constexpr int kOverlapSeg = 4;

static ChainPlan plan_overlap(const PrefillParams &pp, int n_sm) {
    ChainPlan c;
    c.n_chains = pp.N * pp.HV * (D / NV);
    const int n = (pp.T_seq + C - 1) / C;
    c.seg_len = n < kOverlapSeg ? (n > 0 ? n : 1) : kOverlapSeg;
    c.n_units = n > 0 ? c.n_chains * ((n + c.seg_len - 1) / c.seg_len) : 0;
    const int g = (n_sm + 5) / 6;
    c.grid = c.n_units < g ? c.n_units : g;
    if (c.grid < 1) c.grid = 1;
    return c;
}

static ChainPlan plan_chain(const PrefillParams &pp, int n_sm) {
    ChainPlan c;
    c.n_chains = pp.N * pp.HV * (D / NV);
    if (n_sm < 1) n_sm = 1;
    const int n = (pp.T_seq + C - 1) / C;
    c.seg_len = n > 0 ? n : 1;
    if (n > 1 && c.n_chains > n_sm) {
        double best = -1.0;
        for (int r = 1; r <= n; ++r) {
            const int L = (n + r - 1) / r;
            if (r > 1 && L == (n + r - 2) / (r - 1)) continue;   // the same segment length
            const int rr = (n + L - 1) / L;
            const double waves = ((double)c.n_chains * rr + n_sm - 1) / n_sm;
            const double cost = (double)(int64_t)waves * (L + kUnitCost);
            if (best < 0.0 || cost < best) {
                best = cost;
                c.seg_len = L;
            }
        }
    }
    c.n_units = n > 0 ? c.n_chains * ((n + c.seg_len - 1) / c.seg_len) : 0;
    c.grid = c.n_units < n_sm ? c.n_units : n_sm;
    if (c.grid < 1) c.grid = 1;
    return c;
}

// The prep beside the chain.  When an equal-length batch runs one chain CTA per chain and
// leaves SMs free, the prep grid is made persistent (one CTA per prep slot, `per_sm` to an
// SM) and the chain kernel starts at once: the prep CTAs on the SMs the chain leaves free
// produce every record, in chunk order, while the others leave at the start (the limit of
// items they may take is zero).  This pays where those CTAs keep ahead of the chain: one
// item time for the first chunk's records, then a chunk's records in less than a chunk
// period.  Otherwise (fewer free SMs than that, e.g. 24 beside the 128 chains of 32 value
// heads) every prep CTA takes items until none is left and the chain starts after them.
// The estimate uses costs measured on GB300 at T = 4096 (microseconds): a prep item with
// three CTAs to an SM (one value head, two value heads), a chunk of the chain.
constexpr double kPrepItemUs[2] = {11.0, 17.0};
constexpr double kChainChunkUs = 1.5;
constexpr double kPrepMargin = 0.8;        // the staying CTAs' rate is taken at 80% of that

struct PrepPlan {
    int items, limit, stay_sms, grid;
};

// limit == items: no prep beside the chain
static PrepPlan plan_prep(int n_items, int items_per_chunk, int chunks_per_seq, int chain_ctas,
                          int n_sm, int per_sm, int hpc) {
    PrepPlan pl;
    pl.items = n_items;
    pl.limit = n_items;
    pl.stay_sms = 0;
    pl.grid = n_items < per_sm * n_sm ? n_items : per_sm * n_sm;
    const int stay = n_sm - chain_ctas;
    if (stay <= 0 || n_items <= 0 || per_sm <= 0) return pl;
    const double item_us = kPrepItemUs[hpc - 1];
    const double rate = kPrepMargin * per_sm * stay / item_us;       // items per microsecond
    const double chain_us = (chunks_per_seq - 1) * kChainChunkUs;
    if (rate * kChainChunkUs >= items_per_chunk && per_sm * stay >= items_per_chunk &&
        rate * (item_us + chain_us) >= n_items) {
        pl.limit = 0;
        pl.stay_sms = stay;
    }
    return pl;
}

}  // namespace tc

size_t tc_record_bytes() { return (size_t)tc::kRecBytes; }

bool tc_supported(int Dk, int Dv, gdn_dtype dtype) {
    return Dk == tc::D && Dv == tc::D && dtype == GDN_BF16;
}

cudaError_t launch_prefill_tc(const PrefillParams &pp, cudaStream_t st) {
    using namespace tc;
    cudaError_t e;
    // the caller sized the workspace for records of rec_floats floats
    if ((size_t)pp.rec_floats * sizeof(float) < (size_t)kRecBytes) return cudaErrorInvalidValue;
    // the chain's schedule (equal-length batches): the work-unit stream where the chains are
    // cut into segments, else one CTA per chain; with per-token states the stream runs
    // beside the states kernel (see below)
    const bool overlap = pp.states && !pp.cu_seqlens && pp.max_chunks > 0;
    const int hpc = (pp.HV / pp.HK) % 2 == 0 ? 2 : 1;
    ChainPlan plan = {0, 1, 0, 1};
    int dev = 0, n_sm = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if (!pp.cu_seqlens && pp.N > 0) plan = overlap ? plan_overlap(pp, n_sm) : plan_chain(pp, n_sm);
    const bool units = overlap || plan.n_units > plan.n_chains;
    // the prep kernel of a schedule: one CTA per item, or the persistent prep beside the chain
    auto prep_fn = [&](bool persist) {
        return hpc == 2 ? (persist ? prep_kernel<2, true> : prep_kernel<2, false>)
                        : (persist ? prep_kernel<1, true> : prep_kernel<1, false>);
    };
    const size_t prep_smem = hpc == 2 ? prep_smem_bytes<2>() : prep_smem_bytes<1>();
    // prep CTAs an SM holds, from the kernel's registers and shared memory (the occupancy
    // calculator answered one where three run)
    auto ctas_per_sm = [&](bool persist, int &per_sm) -> cudaError_t {
        cudaFuncAttributes fa;
        int smem_sm = 0, regs_sm = 0, reserved = 0;
        cudaError_t r = cudaFuncGetAttributes(&fa, prep_fn(persist));
        if (r == cudaSuccess) r = cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
        if (r == cudaSuccess) r = cudaDeviceGetAttribute(&regs_sm, cudaDevAttrMaxRegistersPerMultiprocessor, dev);
        if (r == cudaSuccess) r = cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev);
        if (r != cudaSuccess) return r;
        const size_t smem_cta = prep_smem + fa.sharedSizeBytes + (size_t)reserved;
        const int regs_cta = (fa.numRegs * 32 + 255) / 256 * 256 * (kPrepThreads / 32);
        per_sm = kPrepPerSm;
        if (smem_cta > 0 && (int)((size_t)smem_sm / smem_cta) < per_sm) per_sm = (int)((size_t)smem_sm / smem_cta);
        if (regs_cta > 0 && regs_sm / regs_cta < per_sm) per_sm = regs_sm / regs_cta;
        return cudaSuccess;
    };
    // the prep beside the chain: equal-length batches with one CTA per chain
    bool beside = !pp.cu_seqlens && !units && pp.max_chunks > 0 && pp.N > 0;
    PrepPlan prep = {0, 0, 0, 0};
    if (beside) {
        int per_sm = 0;
        if ((e = ctas_per_sm(true, per_sm)) != cudaSuccess) return e;
        const int ny = pp.HV / hpc;
        if (per_sm >= 1)
            prep = plan_prep(pp.max_chunks * ny, pp.N * ny, (pp.T_seq + C - 1) / C, plan.n_chains, n_sm,
                             per_sm, hpc);
        beside = per_sm >= 1 && prep.limit < prep.items;
    }
    if (pp.cu_seqlens) {
        if ((e = launch_chunk_table(pp, st)) != cudaSuccess) return e;
    } else {
        // the kernels only ever move the status word from GDN_OK to an error code, so it
        // starts clean here (a reused workspace may hold the last call's error), with the
        // claim counters, the work-unit stream's hand-off flags (right after the header) and,
        // with the prep beside the chain, the record-ready flags (right after those)
        const size_t clear = (size_t)((const char *)pp.chain_flags - (const char *)pp.status) +
                             chain_flag_bytes(pp.N, pp.HV) +
                             (beside ? ready_flag_bytes(pp.max_chunks, pp.HV) : 0);
        if ((e = cudaMemsetAsync(pp.status, 0, clear, st)) != cudaSuccess) return e;
    }
    Params p;
    memset(&p, 0, sizeof p);
    p.k = (const __nv_bfloat16 *)pp.k; p.g = pp.g; p.beta = pp.beta; p.s0 = pp.s0;
    p.out = (__nv_bfloat16 *)pp.out; p.s_final = pp.s_final; p.states = pp.states;
    p.cu_seqlens = pp.cu_seqlens; p.N = pp.N; p.T_seq = pp.T_seq; p.T_total = pp.T_total;
    p.HK = pp.HK; p.HV = pp.HV; p.scale = pp.scale; p.l2norm = pp.l2norm;
    p.max_chunks = pp.max_chunks; p.status = pp.status; p.chunk_seq = pp.chunk_seq;
    p.chunk_first = pp.chunk_first; p.seq_order = pp.seq_order; p.rec = pp.rec;
    p.chain_flags = pp.chain_flags;
    if (beside) {
        p.ready = pp.ready;
        p.prep_items = prep.items;
        p.prep_limit = prep.limit;
        p.prep_stay_sms = prep.stay_sms;
    } else if (pp.max_chunks > 0 && !pp.cu_seqlens) {
        int per_sm = 0;
        if ((e = ctas_per_sm(false, per_sm)) != cudaSuccess) return e;
        p.prep_slots = per_sm * n_sm;
    }
    CUtensorMap mk, mq, mv;
    if (pp.T_total > 0) {
        if (!make_map(&mk, pp.k, pp.HK, pp.T_total, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !make_map(&mq, pp.q, pp.HK, pp.T_total, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !make_map(&mv, pp.v, pp.HV, pp.T_total, NV, CU_TENSOR_MAP_SWIZZLE_64B))
            return cudaErrorInvalidValue;
    } else {
        memset(&mk, 0, sizeof mk); memset(&mq, 0, sizeof mq); memset(&mv, 0, sizeof mv);
    }
    if (pp.max_chunks > 0) {
        // value heads in pairs when each key head serves an even number of them; one CTA
        // per item, or the persistent grid of the prep beside the chain.  All of the SM's
        // unified memory as shared memory, so that three prep CTAs fit.
        const auto kern = prep_fn(beside);
        if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)prep_smem)) != cudaSuccess ||
            (e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                      (int)cudaSharedmemCarveoutMaxShared)) != cudaSuccess)
            return e;
        const unsigned mc = (unsigned)pp.max_chunks;
        const dim3 grid = beside ? dim3(prep.grid)
                                 : dim3(pp.HV / hpc, mc < kGridY ? mc : kGridY, (mc + kGridY - 1) / kGridY);
        kern<<<grid, kPrepThreads, prep_smem, st>>>(mk, mq, p);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if (pp.N > 0) {
        // the work-unit stream only where an equal-length batch's chains are cut into
        // segments; otherwise one CTA per chain (packed batches: longest first, in the
        // order the hardware starts the CTAs)
        // With per-token states (equal-length batches) the stream runs on half the SMs and
        // the states kernel beside it on the other half, taking each segment as the stream
        // publishes it: the states are bound by HBM writes, the stream by its latency.
        p.n_chains = plan.n_chains;
        p.seg_len = plan.seg_len;
        p.n_units = plan.n_units;
        p.states_overlap = overlap ? 1 : 0;
        p.final_direct = overlap && pp.s_final != pp.s0 ? 1 : 0;
        auto kern = units ? (pp.states ? chain_kernel<true, true, false> : chain_kernel<false, true, false>)
                          : pp.states ? chain_kernel<true, false, false>
                                      : (beside ? chain_kernel<false, false, true> : chain_kernel<false, false, false>);
        if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      kChainSmem)) != cudaSuccess)
            return e;
        // programmatic dependent launch: the chain's CTAs may start (barriers, TMEM, the
        // initial state) while the last prep CTAs finish; its producer waits for the prep
        // grid before the first record copy
        cudaLaunchConfig_t cfg;
        memset(&cfg, 0, sizeof cfg);
        cfg.gridDim = units ? dim3(plan.grid) : dim3(D / NV, pp.HV, pp.N);
        cfg.blockDim = dim3(kChainThreads);
        cfg.dynamicSmemBytes = kChainSmem;
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = pp.max_chunks > 0 ? 1 : 0;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if ((e = cudaLaunchKernelEx(&cfg, kern, mk, mq, mv, p)) != cudaSuccess) return e;
        if (pp.states) {
            if (overlap) {
                // a programmatic dependent of the stream: its CTAs start once every stream
                // CTA has, on the SMs the stream leaves free
                const int n = (pp.T_seq + C - 1) / C;
                const int64_t ctas = (int64_t)((n + plan.seg_len - 1) / plan.seg_len) * plan.n_chains * plan.seg_len;
                if (ctas > 0x7fffffffLL) return cudaErrorInvalidValue;
                cudaLaunchConfig_t sc;
                memset(&sc, 0, sizeof sc);
                sc.gridDim = dim3((unsigned)ctas);
                sc.blockDim = dim3(kStThreads);
                sc.stream = st;
                cudaLaunchAttribute sa[1];
                sa[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
                sa[0].val.programmaticStreamSerializationAllowed = 1;
                sc.attrs = sa;
                sc.numAttrs = 1;
                if ((e = cudaLaunchKernelEx(&sc, states_kernel, p)) != cudaSuccess) return e;
            } else if (pp.max_chunks > 0) {
                states_kernel<<<dim3(pp.max_chunks, pp.HV, D / NV), kStThreads, 0, st>>>(p);
                if ((e = cudaGetLastError()) != cudaSuccess) return e;
            }
            if (!p.final_direct) {
                final_from_states_kernel<<<dim3(pp.HV, pp.N), 256, 0, st>>>(p);
                if ((e = cudaGetLastError()) != cudaSuccess) return e;
            }
        }
    }
    return cudaSuccess;
}

}  // namespace gdn
