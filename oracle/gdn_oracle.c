/*
 * gdn_oracle.c -- fp64 CPU oracle for the gated delta rule.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's
 * CPU-baseline leg load this library.  It shares no code, header, table or
 * helper with the CUDA path, and it is deliberately plain and slow: one
 * token at a time, one (sequence, value head) chain at a time, in double
 * precision, in the order the rule is stated.
 *
 * What it computes (qwen3_5_text page, Notes -> "The DeltaNet mixer";
 * qwen3_next page, Notes -> "The DeltaNet mixer fuses its projections per
 * key head"): for each value head the mixer keeps a state S of shape
 * [key_dim][value_dim] (row = key index, column = value index, as in the
 * State layout [batch heads key_dim value_dim] of the linear_attn value
 * table).  For every token t:
 *
 *     q <- l2norm(q_t) * scale,  k <- l2norm(k_t)        (scale = key_dim^-1/2)
 *     S <- exp(g_t) * S                                  (decays.exp() is the
 *                                                          fraction kept)
 *     u <- beta_t * (v_t - S^T k)                         (delta correction,
 *                                                          against decayed S)
 *     S <- S + k u^T
 *     o_t <- S^T q                                        (read out after the
 *                                                          write)
 *
 * The value head h reads key head h / (HV/HK): the queries and keys are
 * repeat_interleave'd up to the value heads, heads 2j and 2j+1 being copies
 * of key head j (qwen3_5_text page, "The DeltaNet mixer").
 *
 * A state passed in is the recurrent state entering the prompt; NULL means
 * the start of a prompt, i.e. S = 0 (linear_attn value table, state_input).
 *
 * Readings where the pages are silent:
 *   - l2norm(x) = x / sqrt(sum(x^2) + 1e-6);  an all-zero row stays zero.
 *   - decays are natural-log, finite and <= 0 (not validated here).
 */
#include <math.h>
#include <pthread.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define GDN_ORACLE_L2NORM_EPS 1e-6

/* l2norm(x) = x / sqrt(sum x^2 + eps), in place. */
static void oracle_l2norm(double *x, int n)
{
    double ss = 0.0;
    for (int i = 0; i < n; ++i) ss += x[i] * x[i];
    double inv = 1.0 / sqrt(ss + GDN_ORACLE_L2NORM_EPS);
    for (int i = 0; i < n; ++i) x[i] *= inv;
}

/*
 * One (sequence, value head) chain over T tokens.
 *
 * Row t of each input is found at base + t * stride (in doubles); within a row
 * the Dk (queries, keys) or Dv (values, outputs) elements are contiguous.
 * g and beta are scalars per token at g[t * gb_stride], beta[t * gb_stride].
 * s0 / s_final / states[t] are [Dk][Dv] row-major.  s0 may be NULL (zeros);
 * s_final may be NULL; states may be NULL.  s0 and s_final may alias.
 * Returns 0, or -1 when a scratch allocation fails.
 */
int gdn_oracle_chain(int T, int Dk, int Dv,
                     const double *q, ptrdiff_t q_stride,
                     const double *k, ptrdiff_t k_stride,
                     const double *v, ptrdiff_t v_stride,
                     const double *g, const double *beta, ptrdiff_t gb_stride,
                     const double *s0,
                     double *o, ptrdiff_t o_stride,
                     double *s_final,
                     double *states, ptrdiff_t states_stride,
                     double scale, int use_qk_l2norm)
{
    double *S = (double *)calloc((size_t)Dk * Dv, sizeof(double));
    double *qt = (double *)malloc(sizeof(double) * (size_t)Dk);
    double *kt = (double *)malloc(sizeof(double) * (size_t)Dk);
    double *u = (double *)malloc(sizeof(double) * (size_t)Dv);
    if (!S || !qt || !kt || !u) {
        free(S); free(qt); free(kt); free(u);
        return -1;
    }
    if (s0) memcpy(S, s0, sizeof(double) * (size_t)Dk * Dv);

    for (int t = 0; t < T; ++t) {
        const double *qrow = q + (ptrdiff_t)t * q_stride;
        const double *krow = k + (ptrdiff_t)t * k_stride;
        const double *vrow = v + (ptrdiff_t)t * v_stride;
        for (int i = 0; i < Dk; ++i) { qt[i] = qrow[i]; kt[i] = krow[i]; }
        if (use_qk_l2norm) { oracle_l2norm(qt, Dk); oracle_l2norm(kt, Dk); }
        for (int i = 0; i < Dk; ++i) qt[i] *= scale;

        /* decay first */
        double alpha = exp(g[(ptrdiff_t)t * gb_stride]);
        for (int e = 0; e < Dk * Dv; ++e) S[e] *= alpha;

        /* u = beta * (v - S^T k) against the decayed state */
        double b = beta[(ptrdiff_t)t * gb_stride];
        for (int c = 0; c < Dv; ++c) {
            double sk = 0.0;
            for (int i = 0; i < Dk; ++i) sk += S[(size_t)i * Dv + c] * kt[i];
            u[c] = b * (vrow[c] - sk);
        }
        /* S = S + k u^T */
        for (int i = 0; i < Dk; ++i)
            for (int c = 0; c < Dv; ++c) S[(size_t)i * Dv + c] += kt[i] * u[c];

        /* o = S^T q, read after the write */
        double *orow = o + (ptrdiff_t)t * o_stride;
        for (int c = 0; c < Dv; ++c) {
            double acc = 0.0;
            for (int i = 0; i < Dk; ++i) acc += S[(size_t)i * Dv + c] * qt[i];
            orow[c] = acc;
        }
        if (states)
            memcpy(states + (ptrdiff_t)t * states_stride, S, sizeof(double) * (size_t)Dk * Dv);
    }
    if (s_final) memcpy(s_final, S, sizeof(double) * (size_t)Dk * Dv);
    free(S); free(qt); free(kt); free(u);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* All chains of a packed batch, threaded over (sequence, value head).       */

typedef struct {
    const double *queries, *keys, *values, *decays, *beta, *initial_state;
    double *out, *final_state, *states;
    const int64_t *cu_seqlens;
    int N, HK, HV, Dk, Dv, use_qk_l2norm;
    double scale;
    const int32_t *chains;   /* chain ids (seq * HV + h) or NULL = all */
    int n_chains;
    int next;                /* next chain to take (under lock) */
    int err;
    pthread_mutex_t lock;
} oracle_job;

static void *oracle_worker(void *arg)
{
    oracle_job *J = (oracle_job *)arg;
    for (;;) {
        pthread_mutex_lock(&J->lock);
        int idx = J->next++;
        pthread_mutex_unlock(&J->lock);
        if (idx >= J->n_chains) break;
        int chain = J->chains ? J->chains[idx] : idx;
        int s = chain / J->HV, h = chain % J->HV;
        int r = J->HV / J->HK;
        int j = h / r;                               /* key head of value head h */
        int64_t t0 = J->cu_seqlens[s], T = J->cu_seqlens[s + 1] - t0;
        size_t dd = (size_t)J->Dk * J->Dv;
        const double *s0 = J->initial_state ? J->initial_state + ((size_t)s * J->HV + h) * dd : NULL;
        double *sf = J->final_state ? J->final_state + ((size_t)s * J->HV + h) * dd : NULL;
        double *st = J->states ? J->states + ((size_t)t0 * J->HV + h) * dd : NULL;
        int rc = gdn_oracle_chain(
            (int)T, J->Dk, J->Dv,
            J->queries + ((size_t)t0 * J->HK + j) * J->Dk, (ptrdiff_t)J->HK * J->Dk,
            J->keys + ((size_t)t0 * J->HK + j) * J->Dk, (ptrdiff_t)J->HK * J->Dk,
            J->values + ((size_t)t0 * J->HV + h) * J->Dv, (ptrdiff_t)J->HV * J->Dv,
            J->decays + (size_t)t0 * J->HV + h, J->beta + (size_t)t0 * J->HV + h, J->HV,
            s0,
            J->out + ((size_t)t0 * J->HV + h) * J->Dv, (ptrdiff_t)J->HV * J->Dv,
            sf,
            st, (ptrdiff_t)J->HV * (ptrdiff_t)dd,
            J->scale, J->use_qk_l2norm);
        if (rc) {
            pthread_mutex_lock(&J->lock);
            J->err = rc;
            pthread_mutex_unlock(&J->lock);
        }
    }
    return NULL;
}

/*
 * Packed layout: token rows of all sequences are concatenated, sequence s
 * owning rows [cu_seqlens[s], cu_seqlens[s+1]).  A [B, T, ...] batch is the
 * same thing with cu_seqlens = {0, T, 2T, ..., BT}.
 *   queries, keys  [T_total, HK, Dk]      values, out  [T_total, HV, Dv]
 *   decays, beta   [T_total, HV]
 *   initial_state, final_state  [N, HV, Dk, Dv]  (initial may be NULL)
 *   states         [T_total, HV, Dk, Dv] or NULL
 * chains: optional list of chain ids s*HV+h to compute (others untouched).
 * Returns 0 on success, -1 on a bad argument or allocation failure.
 */
int gdn_oracle_forward(const double *queries, const double *keys, const double *values,
                       const double *decays, const double *beta,
                       const double *initial_state,
                       double *out, double *final_state, double *states,
                       const int64_t *cu_seqlens, int N, int HK, int HV, int Dk, int Dv,
                       double scale, int use_qk_l2norm,
                       const int32_t *chains, int n_chains, int n_threads)
{
    if (N < 0 || HK <= 0 || HV <= 0 || Dk <= 0 || Dv <= 0 || HV % HK != 0) return -1;
    if (!cu_seqlens || !queries || !keys || !values || !decays || !beta || !out) return -1;
    for (int s = 0; s < N; ++s)
        if (cu_seqlens[s + 1] < cu_seqlens[s]) return -1;
    oracle_job J;
    memset(&J, 0, sizeof J);
    J.queries = queries; J.keys = keys; J.values = values; J.decays = decays; J.beta = beta;
    J.initial_state = initial_state; J.out = out; J.final_state = final_state; J.states = states;
    J.cu_seqlens = cu_seqlens; J.N = N; J.HK = HK; J.HV = HV; J.Dk = Dk; J.Dv = Dv;
    J.scale = scale; J.use_qk_l2norm = use_qk_l2norm;
    J.chains = chains;
    J.n_chains = chains ? n_chains : N * HV;
    pthread_mutex_init(&J.lock, NULL);
    if (n_threads < 1) n_threads = 1;
    if (n_threads > J.n_chains) n_threads = J.n_chains > 0 ? J.n_chains : 1;
    pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)n_threads);
    if (!tid) return -1;
    int started = 0;
    for (int i = 0; i < n_threads; ++i)
        if (pthread_create(&tid[i], NULL, oracle_worker, &J) == 0) ++started;
    if (started == 0) oracle_worker(&J);
    for (int i = 0; i < started; ++i) pthread_join(tid[i], NULL);
    free(tid);
    pthread_mutex_destroy(&J.lock);
    return J.err;
}

/*
 * Gated RMS norm of the mixer's output (qwen3_5_text page, Notes -> "The DeltaNet
 * mixer": out = out_proj(norm(y, gate=silu(z))), "gain: weight"; the DeltaNet's own
 * output norm multiplies by its weight, not by 1 + weight, Notes -> "The readout is the
 * plain projection").  For each row of Dv values (one token of one value head):
 *
 *     r     = 1 / sqrt(mean_c(y_c^2) + eps)
 *     out_c = y_c * r * weight_c * silu(z_c),    silu(z) = z / (1 + exp(-z))
 *
 * Readings where the pages are silent: the mean runs over the head's Dv values, the
 * weight has Dv entries shared by all heads, and the gate multiplies after the norm
 * and the gain.  rows = number of rows; y, z, out are [rows][Dv], weight is [Dv].
 * Returns 0, or -1 on a bad argument.
 */
int gdn_oracle_gated_rmsnorm(const double *y, const double *z, const double *weight, double *out,
                             int64_t rows, int Dv, double eps)
{
    if (!y || !z || !weight || !out || rows < 0 || Dv <= 0 || eps < 0.0) return -1;
    for (int64_t r = 0; r < rows; ++r) {
        const double *yr = y + r * Dv, *zr = z + r * Dv;
        double *orow = out + r * Dv;
        double ms = 0.0;
        for (int c = 0; c < Dv; ++c) ms += yr[c] * yr[c];
        ms /= (double)Dv;
        const double inv = 1.0 / sqrt(ms + eps);
        for (int c = 0; c < Dv; ++c) {
            const double gate = zr[c] / (1.0 + exp(-zr[c]));
            orow[c] = yr[c] * inv * weight[c] * gate;
        }
    }
    return 0;
}

/*
 * The step before the rule in the mixer (qwen3_5_text page, Notes -> "The DeltaNet
 * mixer"; qwen3_next page, Notes -> "The DeltaNet mixer fuses its projections per key
 * head"):
 *
 *     q, k, v = split(silu(conv1d(cat(q, k, v))))     causal, width 4
 *     beta    = sigmoid(b)
 *     g       = -exp(A_log) * softplus(a + dt_bias)
 *
 * conv1d is the depthwise Conv1d of the module listings (kernel_size 4, padding 3,
 * groups = channels, no bias), cut to the causal outputs: for channel c of token t,
 *
 *     conv_t[c] = sum_{i=0..3} w[c][i] * x_{t-3+i}[c]
 *
 * where x_tau for tau before the sequence's first token is 0 at the start of a prompt, or
 * comes from the carried conv state: state[s][3 + tau - start][c] holds x_tau for
 * tau = start-3 .. start-1 (rows 0, 1, 2 = the third-last, second-last and last input
 * before the sequence).  The state after the sequence (the last three inputs, reaching
 * back into the carried state for sequences shorter than three) goes to state_out.
 *
 *   x      [T][C]   conv inputs (cat(q, k, v) channels)     y [T][C] = silu(conv)
 *   b, a   [T][HV]                                          beta, g [T][HV]
 *   w      [C][4];  A_log, dt_bias [HV]
 *   state_in / state_out  [N][3][C] or NULL;  cu [N+1] token offsets of the sequences
 * Returns 0, or -1 on a bad argument.
 */
int gdn_oracle_conv_gate(const double *x, const double *b, const double *a, const double *w,
                         const double *A_log, const double *dt_bias, const double *state_in,
                         double *state_out, const int64_t *cu, int N, int C, int HV,
                         double *y, double *beta, double *g)
{
    if (!x || !w || !cu || !y || N < 0 || C <= 0 || HV < 0) return -1;
    if (HV > 0 && (!b || !a || !A_log || !dt_bias || !beta || !g)) return -1;
    for (int s = 0; s < N; ++s) {
        const int64_t t0 = cu[s], t1 = cu[s + 1];
        if (t1 < t0) return -1;
        /* input of channel c at token tau (tau < t0 reaches into the carried state) */
#define ORACLE_X(tau, c)                                                                   \
    ((tau) >= t0 ? x[(tau) * C + (c)]                                                      \
                 : ((tau) >= t0 - 3 && state_in ? state_in[((int64_t)s * 3 + 3 + ((tau) - t0)) * C + (c)] \
                                                : 0.0))
        for (int64_t t = t0; t < t1; ++t) {
            for (int c = 0; c < C; ++c) {
                double acc = 0.0;
                for (int i = 0; i < 4; ++i) acc += w[c * 4 + i] * ORACLE_X(t - 3 + i, c);
                y[t * C + c] = acc / (1.0 + exp(-acc));
            }
            for (int h = 0; h < HV; ++h) {
                const double bb = b[t * HV + h], aa = a[t * HV + h] + dt_bias[h];
                beta[t * HV + h] = 1.0 / (1.0 + exp(-bb));
                /* softplus(u) = log(1 + e^u), written so that it neither overflows nor
                 * loses the small values */
                const double sp = aa > 0.0 ? aa + log1p(exp(-aa)) : log1p(exp(aa));
                g[t * HV + h] = -exp(A_log[h]) * sp;
            }
        }
        if (state_out)
            for (int r = 0; r < 3; ++r)
                for (int c = 0; c < C; ++c)
                    state_out[((int64_t)s * 3 + r) * C + c] = ORACLE_X(t1 - 3 + r, c);
#undef ORACLE_X
    }
    return 0;
}
