// gdn_prefill_generic.cu -- chunked prefill of the gated delta rule, CUDA-core version.
//
// The prompt kernel of the pages ("a prompt's chunked one", qwen3_5_text page,
// linear_attn value table) written as chunks of C = 64 tokens.  The chunk
// algebra is derived from the recurrence (the pages give none).  Inside a chunk
// with entering state S0, G_t = g_1 + ... + g_t, gamma_t = e^{G_t}, k^_t = rk_t k_t,
// q~_t = rq_t q_t:
//
//   u_t = beta_t (v_t - e^{g_t} S_{t-1}^T k^_t)  unrolls to  (I + A) U = diag(beta) V -
//   diag(beta gamma) K^ S0,   A_tj = beta_t e^{G_t - G_j} (k^_t . k^_j)  (j < t),
//
// so with T = (I + A)^{-1}:  U = Ut - W S0,  Ut = T diag(beta) V,  W = T diag(beta gamma) K^,
//   O   = diag(gamma) Q~ S0 + P U,   P_tj = e^{G_t - G_j} (q~_t . k^_j)  (j <= t),
//   S_C = gamma_C S0 + K^T diag(e^{G_C - G}) U.
// Only non-positive decay differences are ever exponentiated.
//
// Three kernels:
//   chunk_table  (packed batches only) chunk -> sequence map from cu_seqlens,
//                validated on the device (status word, never a trap);
//   prep         one CTA per (chunk, value head), all in parallel: norms, decay
//                prefix, A and P, the triangular solve for T, W and Ut;
//   scan         one CTA per (sequence, value head, 32-wide value block): the
//                sequential chunk loop carrying S0 in shared memory; writes O,
//                the final state and, optionally, the state after every token
//                (S_t = e^{g_t} S_{t-1} + k^_t u_t^T, with the chunk-end state
//                taken from the chunk form so the last one equals final_state).
//
// This version runs every product on the CUDA cores in fp32: it is the shape-
// generic path (key_dim = value_dim in {32, 64, 128}; bf16 or fp32 inputs).
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int C = kChunk;
constexpr int kThreads = 256;

struct ChunkInfo {
    int seq;        // sequence index
    int64_t t0;     // first token (row of the packed layout)
    int len;        // tokens in this chunk (1..C)
};

__device__ __forceinline__ bool chunk_info(const PrefillParams &p, int c, ChunkInfo &ci) {
    if (p.cu_seqlens) {
        if (p.status[kStatusWord] != GDN_OK) return false;
        if (c >= p.status[kChunkCountWord]) return false;
        const int s = p.chunk_seq[c];
        const int local = c - p.chunk_first[s];
        const int64_t a = p.cu_seqlens[s], e = p.cu_seqlens[s + 1];
        ci.seq = s;
        ci.t0 = a + (int64_t)local * C;
        ci.len = (int)min((int64_t)C, e - ci.t0);
        return true;
    }
    const int cps = (p.T_seq + C - 1) / C;
    if (cps == 0 || c >= p.N * cps) return false;
    ci.seq = c / cps;
    const int local = c - ci.seq * cps;
    ci.t0 = (int64_t)ci.seq * p.T_seq + (int64_t)local * C;
    ci.len = min(C, p.T_seq - local * C);
    return true;
}

// ------------------------------------------------------------------ chunk table
// One CTA: checks 0 = cu[0] <= cu[1] <= ... <= cu[N] = T_total, counts the chunks
// of every sequence, and writes chunk_first (exclusive prefix) and chunk_seq.
constexpr int kMaxRanked = 1024;

__global__ void __launch_bounds__(1024) chunk_table_kernel(PrefillParams p) {
    __shared__ int s_bad;
    __shared__ int s_carry;
    __shared__ int s_scan[1024];
    const int tid = threadIdx.x;
    if (tid == 0) { s_bad = 0; s_carry = 0; }
    __syncthreads();
    for (int i = tid; i < p.N; i += blockDim.x) {
        const int a = p.cu_seqlens[i], b = p.cu_seqlens[i + 1];
        if (b < a) atomicOr(&s_bad, 1);
    }
    if (tid == 0 && (p.cu_seqlens[0] != 0 || (int64_t)p.cu_seqlens[p.N] != p.T_total))
        atomicOr(&s_bad, 1);
    __syncthreads();
    if (s_bad) {
        if (tid == 0) { p.status[kStatusWord] = GDN_ERR_BAD_SEQLENS; p.status[kChunkCountWord] = 0; }
        return;
    }
    // exclusive prefix of per-sequence chunk counts, 1024 sequences at a time
    for (int base = 0; base < p.N; base += blockDim.x) {
        const int i = base + tid;
        int cnt = 0;
        if (i < p.N) cnt = (p.cu_seqlens[i + 1] - p.cu_seqlens[i] + C - 1) / C;
        s_scan[tid] = cnt;
        __syncthreads();
        for (int off = 1; off < (int)blockDim.x; off <<= 1) {
            int x = tid >= off ? s_scan[tid - off] : 0;
            __syncthreads();
            s_scan[tid] += x;
            __syncthreads();
        }
        const int incl = s_scan[tid] + s_carry;
        if (i < p.N) {
            const int first = incl - cnt;
            p.chunk_first[i] = first;
            for (int c = 0; c < cnt; ++c) p.chunk_seq[first + c] = i;
        }
        __syncthreads();
        if (tid == blockDim.x - 1) s_carry = incl;
        __syncthreads();
    }
    if (tid == 0) p.chunk_first[p.N] = s_carry;
    // longest sequences first: seq_order[rank] = sequence, rank = number of sequences with
    // more chunks (ties by index), so that the sequential kernels start the longest chains
    // first; above kMaxRanked sequences the order is the identity
    __syncthreads();
    if (p.N <= kMaxRanked) {
        if (tid < p.N) s_scan[tid] = (p.cu_seqlens[tid + 1] - p.cu_seqlens[tid] + C - 1) / C;
        __syncthreads();
        if (tid < p.N) {
            const int ci = s_scan[tid];
            int rank = 0;
            for (int j2 = 0; j2 < p.N; ++j2) {
                const int cj = s_scan[j2];
                rank += (cj > ci) || (cj == ci && j2 < tid);
            }
            p.seq_order[rank] = tid;
        }
    } else {
        for (int i = tid; i < p.N; i += blockDim.x) p.seq_order[i] = i;
    }
    if (tid == 0) {
        p.status[kChunkCountWord] = s_carry;
        p.status[kStatusWord] = GDN_OK;
    }
}

// ------------------------------------------------------------------ prep
template <int DK, int DV>
struct PrepSmem {
    static constexpr int LDK = DK + 1, LDV = DV + 1, LDC = C + 1;
    static constexpr size_t floats = (size_t)C * LDK * 2 + (size_t)C * LDV + (size_t)C * LDC * 2 + 8 * C;
    static constexpr size_t bytes = floats * sizeof(float);
};

template <int DK, int DV, typename Tin>
__global__ void __launch_bounds__(kThreads) prep_kernel(PrefillParams p) {
    using L = PrepSmem<DK, DV>;
    extern __shared__ float sm[];
    float *sK = sm;                        // [C][LDK]  raw keys, later beta gamma rk K
    float *sQ = sK + C * L::LDK;           // [C][LDK]  raw queries
    float *sV = sQ + C * L::LDK;           // [C][LDV]  values, later beta V
    float *sA = sV + C * L::LDV;           // [C][LDC]  A (strictly lower)
    float *sT = sA + C * L::LDC;           // [C][LDC]  T = (I + A)^{-1}
    float *sG = sT + C * L::LDC;           // [C] decay prefix G
    float *sB = sG + C;                    // [C] beta
    float *sRk = sB + C;                   // [C] key normaliser
    float *sRq = sRk + C;                  // [C] query normaliser (incl. scale)
    float *sg = sRq + C;                   // [C] g

    ChunkInfo ci;
    const int c = blockIdx.x, h = blockIdx.y;
    if (!chunk_info(p, c, ci)) return;
    const int j = h / (p.HV / p.HK);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const Tin *q = (const Tin *)p.q, *k = (const Tin *)p.k, *v = (const Tin *)p.v;

    // load the chunk (rows >= len are zero)
    for (int e = tid; e < C * DK; e += kThreads) {
        const int t = e / DK, i = e - t * DK;
        float qq = 0.f, kk = 0.f;
        if (t < ci.len) {
            const size_t row = ((size_t)(ci.t0 + t) * p.HK + j) * DK + i;
            qq = to_f32(q[row]);
            kk = to_f32(k[row]);
        }
        sQ[t * L::LDK + i] = qq;
        sK[t * L::LDK + i] = kk;
    }
    for (int e = tid; e < C * DV; e += kThreads) {
        const int t = e / DV, i = e - t * DV;
        sV[t * L::LDV + i] = t < ci.len ? to_f32(v[((size_t)(ci.t0 + t) * p.HV + h) * DV + i]) : 0.f;
    }
    if (tid < C) {
        const bool in = tid < ci.len;
        const size_t gi = (size_t)(ci.t0 + tid) * p.HV + h;
        sg[tid] = in ? p.g[gi] : 0.f;
        sB[tid] = in ? p.beta[gi] : 0.f;
    }
    __syncthreads();

    // norms (one warp per row) and the decay prefix
    for (int t = warp; t < C; t += kThreads / 32) {
        float sq = 0.f, sk = 0.f;
        for (int i = lane; i < DK; i += 32) {
            const float a = sQ[t * L::LDK + i], b = sK[t * L::LDK + i];
            sq += a * a; sk += b * b;
        }
        sq = warp_sum(sq); sk = warp_sum(sk);
        if (lane == 0) {
            sRq[t] = p.l2norm ? p.scale * rsqrtf(sq + kL2Eps) : p.scale;
            sRk[t] = p.l2norm ? rsqrtf(sk + kL2Eps) : 1.f;
        }
    }
    if (tid == 0) {
        float acc = 0.f;
        for (int t = 0; t < C; ++t) { acc += sg[t]; sG[t] = acc; }
    }
    __syncthreads();

    // Gram tiles: KK^T and QK^T (raw), 4x4 register tile per thread
    float *rec = p.rec + ((size_t)c * p.HV + h) * p.rec_floats;
    float *gW = rec;
    float *gUt = gW + C * DK;
    float *gP = gUt + C * DV;
    float *gqd = gP + C * C;
    float *gkd = gqd + C;
    float *grk = gkd + C;
    float *galpha = grk + C;
    float *gmisc = galpha + C;
    {
        const int ty = tid >> 4, tx = tid & 15;
        float kk[4][4] = {}, qk[4][4] = {};
        for (int i = 0; i < DK; ++i) {
            float kt[4], qt[4], kj[4];
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                kt[a] = sK[(ty + 16 * a) * L::LDK + i];
                qt[a] = sQ[(ty + 16 * a) * L::LDK + i];
                kj[a] = sK[(tx + 16 * a) * L::LDK + i];
            }
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    kk[a][b] += kt[a] * kj[b];
                    qk[a][b] += qt[a] * kj[b];
                }
        }
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            const int t = ty + 16 * a;
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                const int jj = tx + 16 * b;
                const bool live = t < ci.len;
                const float dec = (jj <= t) ? expf(sG[t] - sG[jj]) : 0.f;
                sA[t * L::LDC + jj] = (live && jj < t) ? sB[t] * dec * sRk[t] * sRk[jj] * kk[a][b] : 0.f;
                gP[t * C + jj] = (live && jj <= t) ? dec * sRq[t] * sRk[jj] * qk[a][b] : 0.f;
            }
        }
    }
    __syncthreads();

    // T = (I + A)^{-1}: column c solved by thread c with forward substitution
    if (tid < C) {
        const int col = tid;
        for (int t = 0; t < C; ++t) {
            float acc = (t == col) ? 1.f : 0.f;
            for (int jj = 0; jj < t; ++jj) acc -= sA[t * L::LDC + jj] * sT[jj * L::LDC + col];
            sT[t * L::LDC + col] = (t < col) ? 0.f : acc;
        }
    }
    // fold the row factors of W and Ut into K and V
    const float Glast = sG[ci.len - 1];
    for (int e = tid; e < C * DK; e += kThreads) {
        const int t = e / DK, i = e - t * DK;
        sK[t * L::LDK + i] *= sB[t] * expf(sG[t]) * sRk[t];
    }
    for (int e = tid; e < C * DV; e += kThreads) {
        const int t = e / DV, i = e - t * DV;
        sV[t * L::LDV + i] *= sB[t];
    }
    if (tid < C) {
        const bool in = tid < ci.len;
        gqd[tid] = in ? sRq[tid] * expf(sG[tid]) : 0.f;
        gkd[tid] = in ? sRk[tid] * expf(Glast - sG[tid]) : 0.f;
        grk[tid] = in ? sRk[tid] : 0.f;
        galpha[tid] = in ? expf(sg[tid]) : 0.f;
        gmisc[tid] = tid == 0 ? expf(Glast) : 0.f;
    }
    __syncthreads();

    // W = T (beta gamma rk K), Ut = T (beta V): rows ty + 16 a, columns tx + 16 b
    {
        const int ty = tid >> 4, tx = tid & 15;
        constexpr int NB = DK / 16;
        float acc[4][NB] = {};
        for (int jj = 0; jj < C; ++jj) {
            float tt[4], kv[NB];
#pragma unroll
            for (int a = 0; a < 4; ++a) tt[a] = sT[(ty + 16 * a) * L::LDC + jj];
#pragma unroll
            for (int b = 0; b < NB; ++b) kv[b] = sK[jj * L::LDK + tx + 16 * b];
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int b = 0; b < NB; ++b) acc[a][b] += tt[a] * kv[b];
        }
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int b = 0; b < NB; ++b) gW[(ty + 16 * a) * DK + tx + 16 * b] = acc[a][b];
    }
    {
        const int ty = tid >> 4, tx = tid & 15;
        constexpr int NB = DV / 16;
        float acc[4][NB] = {};
        for (int jj = 0; jj < C; ++jj) {
            float tt[4], vv[NB];
#pragma unroll
            for (int a = 0; a < 4; ++a) tt[a] = sT[(ty + 16 * a) * L::LDC + jj];
#pragma unroll
            for (int b = 0; b < NB; ++b) vv[b] = sV[jj * L::LDV + tx + 16 * b];
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int b = 0; b < NB; ++b) acc[a][b] += tt[a] * vv[b];
        }
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int b = 0; b < NB; ++b) gUt[(ty + 16 * a) * DV + tx + 16 * b] = acc[a][b];
    }
}

// ------------------------------------------------------------------ scan
constexpr int VB = 32;   // value columns per scan CTA

template <int DK>
struct ScanSmem {
    static constexpr int LDK = DK + 1, LDC = C + 1, LDS = VB + 1;
    static constexpr size_t floats =
        (size_t)DK * LDS + (size_t)C * LDK * 3 + (size_t)C * LDC + (size_t)C * LDS + 5 * C;
    static constexpr size_t bytes = floats * sizeof(float);
};

template <int DK, int DV, typename Tin, bool STATES>
__global__ void __launch_bounds__(kThreads) scan_kernel(PrefillParams p) {
    using L = ScanSmem<DK>;
    extern __shared__ float sm[];
    float *sS = sm;                        // [DK][LDS] state block S0
    float *sW = sS + DK * L::LDS;          // [C][LDK]
    float *sQ = sW + C * L::LDK;           // [C][LDK] raw queries
    float *sK = sQ + C * L::LDK;           // [C][LDK] raw keys
    float *sP = sK + C * L::LDK;           // [C][LDC]
    float *sU = sP + C * L::LDC;           // [C][LDS] Ut, then U
    float *sqd = sU + C * L::LDS;
    float *skd = sqd + C;
    float *srk = skd + C;
    float *sal = srk + C;
    float *smisc = sal + C;

    const int vb = blockIdx.x, h = blockIdx.y, s = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int j = h / (p.HV / p.HK);
    const int c0v = vb * VB;

    int first, count;
    int64_t seq_t0;
    if (p.cu_seqlens) {
        if (p.status[kStatusWord] != GDN_OK) return;
        first = p.chunk_first[s];
        count = p.chunk_first[s + 1] - first;
        seq_t0 = p.cu_seqlens[s];
    } else {
        const int cps = (p.T_seq + C - 1) / C;
        first = s * cps;
        count = cps;
        seq_t0 = (int64_t)s * p.T_seq;
    }

    if (!p.cu_seqlens && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 && tid == 0)
        p.status[kStatusWord] = GDN_OK;

    // entering state block
    const size_t sbase = ((size_t)s * p.HV + h) * DK * DV;
    for (int e = tid; e < DK * VB; e += kThreads) {
        const int i = e / VB, cc = e - i * VB;
        sS[i * L::LDS + cc] = p.s0 ? p.s0[sbase + (size_t)i * DV + c0v + cc] : 0.f;
    }

    const Tin *q = (const Tin *)p.q, *k = (const Tin *)p.k;
    Tin *out = (Tin *)p.out;
    constexpr int RK = DK / 8;      // state rows per thread in the update (rows warp + 8 a)
    for (int cc = 0; cc < count; ++cc) {
        const int c = first + cc;
        const int64_t t0 = seq_t0 + (int64_t)cc * C;
        const float *rec = p.rec + ((size_t)c * p.HV + h) * p.rec_floats;
        const float *gW = rec, *gUt = gW + C * DK, *gP = gUt + C * DV, *gqd = gP + C * C;
        int len;
        if (p.cu_seqlens) len = (int)min((int64_t)C, (int64_t)p.cu_seqlens[s + 1] - t0);
        else len = min(C, p.T_seq - cc * C);

        __syncthreads();   // previous chunk done with the buffers
        for (int e = tid; e < C * DK; e += kThreads) {
            const int t = e / DK, i = e - t * DK;
            sW[t * L::LDK + i] = gW[e];
            float qq = 0.f, kk = 0.f;
            if (t < len) {
                const size_t row = ((size_t)(t0 + t) * p.HK + j) * DK + i;
                qq = to_f32(q[row]);
                kk = to_f32(k[row]);
            }
            sQ[t * L::LDK + i] = qq;
            sK[t * L::LDK + i] = kk;
        }
        for (int e = tid; e < C * C; e += kThreads) {
            const int t = e / C, jj = e - t * C;
            sP[t * L::LDC + jj] = gP[e];
        }
        for (int e = tid; e < C * VB; e += kThreads) {
            const int t = e / VB, cc2 = e - t * VB;
            sU[t * L::LDS + cc2] = gUt[t * DV + c0v + cc2];
        }
        for (int e = tid; e < 5 * C; e += kThreads) sqd[e] = gqd[e];   // qd, kd, rk, alpha, misc
        __syncthreads();

        // U = Ut - W S0: rows warp + 8 a, column lane
        float u[C / 8];
#pragma unroll
        for (int a = 0; a < C / 8; ++a) {
            const int t = warp + 8 * a;
            float acc = 0.f;
            for (int i = 0; i < DK; ++i) acc += sW[t * L::LDK + i] * sS[i * L::LDS + lane];
            u[a] = sU[t * L::LDS + lane] - acc;
        }
        __syncthreads();
#pragma unroll
        for (int a = 0; a < C / 8; ++a) sU[(warp + 8 * a) * L::LDS + lane] = u[a];
        __syncthreads();

        // O = diag(qd) Q S0 + P U
#pragma unroll
        for (int a = 0; a < C / 8; ++a) {
            const int t = warp + 8 * a;
            float acc = 0.f, acc2 = 0.f;
            for (int i = 0; i < DK; ++i) acc += sQ[t * L::LDK + i] * sS[i * L::LDS + lane];
            for (int jj = 0; jj <= t; ++jj) acc2 += sP[t * L::LDC + jj] * sU[jj * L::LDS + lane];
            if (t < len)
                out[((size_t)(t0 + t) * p.HV + h) * DV + c0v + lane] = from_f32<Tin>(sqd[t] * acc + acc2);
        }

        // S_C = gamma_C S0 + K^T diag(kd) U: rows warp + 8 a, column lane
        const float gC = smisc[0];
        float sn[RK];
#pragma unroll
        for (int a = 0; a < RK; ++a) {
            const int i = warp + 8 * a;
            float acc = 0.f;
            for (int t = 0; t < C; ++t) acc += sK[t * L::LDK + i] * skd[t] * sU[t * L::LDS + lane];
            sn[a] = gC * sS[i * L::LDS + lane] + acc;
        }
        if (STATES) {
            // state after every token: recurrence from S0, chunk form at the chunk end
            float run[RK];
#pragma unroll
            for (int a = 0; a < RK; ++a) run[a] = sS[(warp + 8 * a) * L::LDS + lane];
            for (int t = 0; t < len; ++t) {
                float *dst = p.states + ((size_t)(t0 + t) * p.HV + h) * DK * DV + c0v + lane;
                const float al = sal[t], uk = srk[t] * sU[t * L::LDS + lane];
                const bool last = (t == len - 1);
#pragma unroll
                for (int a = 0; a < RK; ++a) {
                    const int i = warp + 8 * a;
                    run[a] = al * run[a] + sK[t * L::LDK + i] * uk;
                    __stcs(dst + (size_t)i * DV, last ? sn[a] : run[a]);
                }
            }
        }
        __syncthreads();
#pragma unroll
        for (int a = 0; a < RK; ++a) sS[(warp + 8 * a) * L::LDS + lane] = sn[a];
    }
    __syncthreads();
    for (int e = tid; e < DK * VB; e += kThreads) {
        const int i = e / VB, cc = e - i * VB;
        p.s_final[sbase + (size_t)i * DV + c0v + cc] = sS[i * L::LDS + cc];
    }
}

template <typename K>
cudaError_t set_smem(K kernel, size_t bytes) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

template <int DK, int DV, typename Tin>
cudaError_t run(const PrefillParams &p, cudaStream_t st) {
    cudaError_t e;
    if (p.cu_seqlens) {
        chunk_table_kernel<<<1, 1024, 0, st>>>(p);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if (p.max_chunks > 0) {
        auto kp = prep_kernel<DK, DV, Tin>;
        if ((e = set_smem(kp, PrepSmem<DK, DV>::bytes)) != cudaSuccess) return e;
        kp<<<dim3(p.max_chunks, p.HV), kThreads, PrepSmem<DK, DV>::bytes, st>>>(p);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if (p.N > 0) {
        auto ks = p.states ? scan_kernel<DK, DV, Tin, true> : scan_kernel<DK, DV, Tin, false>;
        if ((e = set_smem(ks, ScanSmem<DK>::bytes)) != cudaSuccess) return e;
        ks<<<dim3(DV / VB, p.HV, p.N), kThreads, ScanSmem<DK>::bytes, st>>>(p);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    return cudaSuccess;
}

template <typename Tin>
cudaError_t dispatch(const PrefillParams &p, cudaStream_t st) {
#define GDN_PF_CASE(DK_, DV_) \
    if (p.Dk == DK_ && p.Dv == DV_) return run<DK_, DV_, Tin>(p, st);
    GDN_PF_CASE(32, 32) GDN_PF_CASE(64, 64) GDN_PF_CASE(128, 128)
#undef GDN_PF_CASE
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_chunk_table(const PrefillParams &p, cudaStream_t st) {
    chunk_table_kernel<<<1, 1024, 0, st>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_prefill_generic(const PrefillParams &p, gdn_dtype dtype, cudaStream_t st) {
    return dtype == GDN_BF16 ? dispatch<__nv_bfloat16>(p, st) : dispatch<float>(p, st);
}

}  // namespace gdn
