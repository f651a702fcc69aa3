"""Pins of the fp64 oracle to facts that do not come from the oracle itself.

Each test names what fixes the expected value: a closed form the rule reduces
to, an invariant of the mathematics, a worked example computed by hand, the
pages' own statements (qwen3_5_text page, Notes -> "The DeltaNet mixer";
qwen3_next page, Notes -> "The DeltaNet mixer fuses its projections per key
head"), or an independent solve of the same result.  Together they are meant
to fail on a plausible slip anywhere in the oracle: a dropped term, a wrong
sign, a transposed state, the wrong key head, readout before the write, the
decay applied after the write, a missing l2 norm or scale.
"""
import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng_seed = 20261202


def _rng(k=0):
    return np.random.default_rng(rng_seed + k)


def _l2n(x):
    return x / np.sqrt((x * x).sum(-1, keepdims=True) + 1e-6)


def _rand_case(rng, B, T, HK, HV, Dk, Dv, s0=False, g_scale=1.0):
    q = rng.standard_normal((B, T, HK, Dk))
    k = rng.standard_normal((B, T, HK, Dk))
    v = rng.standard_normal((B, T, HV, Dv))
    g = -np.log1p(np.exp(rng.standard_normal((B, T, HV)))) * g_scale
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((B, T, HV))))
    st = rng.standard_normal((B, HV, Dk, Dv)) * 0.3 if s0 else None
    return q, k, v, g, beta, st


# ---------------------------------------------------------------- hand example
def _parse_golden(path):
    out = {}
    for line in open(path):
        line = line.split("#", 1)[0].strip()
        if not line:
            continue
        name, rest = line.split(None, 1)
        if ";" in rest:
            out[name] = np.array([[float(x) for x in r.split()] for r in rest.split(";")])
        else:
            out[name] = np.array([[float(x) for x in r.split()] for r in rest.split("|")])
    return out


@pytest.mark.parametrize("case,l2", [("raw", False), ("normed", True)])
def test_hand_worked_example(oracle_mod, case, l2):
    """tests/golden/hand_T2_Dk2_Dv2.txt: two tokens computed by hand (decay, delta
    write against the decayed state, read after the write, S[key][value])."""
    G = _parse_golden(os.path.join(GOLDEN, "hand_T2_Dk2_Dv2.txt"))
    p = lambda f: G[f"{case}.{f}"]
    q = p("q").reshape(1, 2, 1, 2)
    k = p("k").reshape(1, 2, 1, 2)
    v = p("v").reshape(1, 2, 1, 2)
    g = p("g").reshape(1, 2, 1)
    b = p("beta").reshape(1, 2, 1)
    o, sf, _ = oracle_mod.forward(q, k, v, g, b, scale=None if l2 else 1.0, use_qk_l2norm=l2)
    tol = 1e-6 if l2 else 1e-14
    np.testing.assert_allclose(o.reshape(2, 2), p("o"), atol=tol, rtol=0)
    np.testing.assert_allclose(sf.reshape(2, 2), p("S_final"), atol=tol, rtol=0)


# ---------------------------------------------------------------- closed forms
@pytest.mark.parametrize("Dk,Dv", [(5, 7), (32, 32), (128, 128)])
def test_single_token_closed_form(oracle_mod, Dk, Dv):
    """T = 1 from a zero state: o = beta (q~ . k^) v and S = beta k^ v^T, with
    q~ = l2norm(q) Dk^-1/2 and k^ = l2norm(k) (the rule's closed form at T=1)."""
    rng = _rng(1)
    q, k, v, g, beta, _ = _rand_case(rng, 3, 1, 2, 4, Dk, Dv)
    o, sf, _ = oracle_mod.forward(q, k, v, g, beta)
    for b in range(3):
        for h in range(4):
            j = h // 2
            qt = _l2n(q[b, 0, j]) * Dk ** -0.5
            kt = _l2n(k[b, 0, j])
            bb = beta[b, 0, h]
            np.testing.assert_allclose(o[b, 0, h], bb * (qt @ kt) * v[b, 0, h], rtol=1e-12, atol=1e-14)
            np.testing.assert_allclose(sf[b, h], bb * np.outer(kt, v[b, 0, h]), rtol=1e-12, atol=1e-14)


def test_beta_zero_no_decay(oracle_mod):
    """beta = 0, g = 0: nothing is written.  From zero, o = 0 and S = 0; from S0,
    S stays S0 and o_t = S0^T q~_t."""
    rng = _rng(2)
    q, k, v, g, beta, s0 = _rand_case(rng, 2, 9, 1, 2, 6, 4, s0=True)
    z = np.zeros_like(g)
    o, sf, _ = oracle_mod.forward(q, k, v, z, z)
    assert np.all(o == 0) and np.all(sf == 0)
    o, sf, _ = oracle_mod.forward(q, k, v, z, z, initial_state=s0)
    np.testing.assert_allclose(sf, s0, rtol=0, atol=0)
    for b in range(2):
        for h in range(2):
            qt = _l2n(q[b, :, 0]) * 6 ** -0.5
            np.testing.assert_allclose(o[b, :, h], qt @ s0[b, h], rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("with_s0", [False, True])
def test_orthonormal_keys_projection(oracle_mod, with_s0):
    """beta = 1, g = 0, keys orthonormal (T <= Dk): every write makes S^T k_t = v_t and
    later writes along orthogonal keys leave it so (Widrow-Hoff projection), while S^T x
    for x orthogonal to all keys stays S0^T x."""
    rng = _rng(3)
    Dk, Dv, T = 16, 8, 11
    Qm, _ = np.linalg.qr(rng.standard_normal((Dk, Dk)))
    keys = Qm[:, :T].T                                  # T orthonormal rows
    k = keys.reshape(1, T, 1, Dk)
    q = rng.standard_normal((1, T, 1, Dk))
    v = rng.standard_normal((1, T, 1, Dv))
    s0 = rng.standard_normal((1, 1, Dk, Dv)) if with_s0 else None
    # keys already unit length: the l2 norm is switched off so that "exactly" holds to
    # rounding (its 1e-6 epsilon would shorten k^ by ~5e-7).
    o, sf, _ = oracle_mod.forward(q, k, v, np.zeros((1, T, 1)), np.ones((1, T, 1)),
                                  initial_state=s0, use_qk_l2norm=False)
    S = sf[0, 0]
    for i in range(T):
        np.testing.assert_allclose(S.T @ keys[i], v[0, i, 0], rtol=0, atol=1e-12)
    comp = Qm[:, T:]
    base = s0[0, 0] if with_s0 else np.zeros((Dk, Dv))
    np.testing.assert_allclose(comp.T @ S, comp.T @ base, rtol=0, atol=1e-12)


def test_fully_forgetting_decay(oracle_mod):
    """g -> -inf (g = -1e4, exp underflows to 0): a token sees only its own key and
    value: o_t = beta_t (q~_t . k^_t) v_t, and S_T = beta_T k^_T v_T^T."""
    rng = _rng(4)
    q, k, v, g, beta, s0 = _rand_case(rng, 2, 7, 2, 2, 8, 5, s0=True)
    g = np.full_like(g, -1e4)
    o, sf, _ = oracle_mod.forward(q, k, v, g, beta, initial_state=s0)
    for b in range(2):
        for h in range(2):
            qt = _l2n(q[b, :, h]) * 8 ** -0.5
            kt = _l2n(k[b, :, h])
            exp_o = (beta[b, :, h] * (qt * kt).sum(-1))[:, None] * v[b, :, h]
            np.testing.assert_allclose(o[b, :, h], exp_o, rtol=1e-12, atol=1e-14)
            np.testing.assert_allclose(sf[b, h], beta[b, -1, h] * np.outer(kt[-1], v[b, -1, h]),
                                       rtol=1e-12, atol=1e-14)


# ---------------------------------------------------------------- invariants
def test_prefill_then_decode_equals_prefill(oracle_mod):
    """The prompt kernel and the decode kernel continue one state (state_input is a copy
    of the cache's buffer): prefill(t) then T-t decode steps = prefill(T)."""
    rng = _rng(5)
    q, k, v, g, beta, s0 = _rand_case(rng, 3, 20, 2, 4, 8, 6, s0=True)
    o_full, s_full, _ = oracle_mod.forward(q, k, v, g, beta, initial_state=s0)
    t = 13
    o_a, s, _ = oracle_mod.forward(q[:, :t], k[:, :t], v[:, :t], g[:, :t], beta[:, :t],
                                   initial_state=s0)
    np.testing.assert_allclose(o_a, o_full[:, :t], rtol=0, atol=1e-12)
    for i in range(t, 20):
        o_i, s = oracle_mod.decode_step(q[:, i], k[:, i], v[:, i], g[:, i], beta[:, i], s)
        np.testing.assert_allclose(o_i, o_full[:, i], rtol=0, atol=1e-12)
    np.testing.assert_allclose(s, s_full, rtol=0, atol=1e-12)


def test_linear_in_values_and_state(oracle_mod):
    """For fixed q, k, g, beta the map (V, S0) -> (O, S_T) is linear."""
    rng = _rng(6)
    q, k, v1, g, beta, s1 = _rand_case(rng, 1, 12, 1, 2, 6, 5, s0=True)
    v2 = rng.standard_normal(v1.shape)
    s2 = rng.standard_normal(s1.shape)
    a, c = 0.7, -1.3
    o1, f1, _ = oracle_mod.forward(q, k, v1, g, beta, initial_state=s1)
    o2, f2, _ = oracle_mod.forward(q, k, v2, g, beta, initial_state=s2)
    o3, f3, _ = oracle_mod.forward(q, k, a * v1 + c * v2, g, beta, initial_state=a * s1 + c * s2)
    np.testing.assert_allclose(o3, a * o1 + c * o2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(f3, a * f1 + c * f2, rtol=0, atol=1e-12)


def test_gqa_interleave(oracle_mod):
    """Queries and keys are repeat_interleave'd to the value heads: heads 2j and 2j+1
    read key head j (not head h mod HK)."""
    rng = _rng(7)
    q, k, v, g, beta, s0 = _rand_case(rng, 2, 10, 2, 4, 8, 8, s0=True)
    o, sf, _ = oracle_mod.forward(q, k, v, g, beta, initial_state=s0)
    o_r, sf_r, _ = oracle_mod.forward(np.repeat(q, 2, axis=2), np.repeat(k, 2, axis=2), v, g,
                                      beta, initial_state=s0)
    np.testing.assert_array_equal(o, o_r)
    np.testing.assert_array_equal(sf, sf_r)
    o_t, _, _ = oracle_mod.forward(np.tile(q, (1, 1, 2, 1)), np.tile(k, (1, 1, 2, 1)), v, g,
                                   beta, initial_state=s0)
    assert np.abs(o_t - o).max() > 1e-3        # the modulo mapping is a different result


def test_l2norm_makes_scale_irrelevant_and_matters(oracle_mod):
    """With the in-kernel l2 norm, positive row scalings of q and k do not change the
    result (up to the 1e-6 epsilon); turning the norm off changes it by a lot (the pages
    report a 42% error in a final state without it)."""
    rng = _rng(8)
    q, k, v, g, beta, _ = _rand_case(rng, 1, 16, 2, 2, 16, 16)
    o, sf, _ = oracle_mod.forward(q, k, v, g, beta)
    sq = rng.uniform(0.2, 5.0, q.shape[:-1] + (1,))
    sk = rng.uniform(0.2, 5.0, k.shape[:-1] + (1,))
    o2, sf2, _ = oracle_mod.forward(q * sq, k * sk, v, g, beta)
    np.testing.assert_allclose(o2, o, rtol=0, atol=1e-6)
    np.testing.assert_allclose(sf2, sf, rtol=0, atol=1e-6)
    o3, sf3, _ = oracle_mod.forward(q, k, v, g, beta, use_qk_l2norm=False)
    rel = np.linalg.norm(sf3 - sf) / np.linalg.norm(sf)
    assert rel > 0.1


def test_zero_rows_stay_finite(oracle_mod):
    """An all-zero query or key row gives zeros, not NaN (l2 norm with epsilon)."""
    rng = _rng(9)
    q, k, v, g, beta, _ = _rand_case(rng, 1, 6, 1, 1, 8, 8)
    q[0, 2] = 0
    k[0, 3] = 0
    o, sf, _ = oracle_mod.forward(q, k, v, g, beta)
    assert np.isfinite(o).all() and np.isfinite(sf).all()
    assert np.all(o[0, 2] == 0)


def test_packed_equals_separate(oracle_mod):
    """A packed batch with cu_seqlens (zero-length sequences allowed) equals the
    sequences run one by one; a zero-length sequence returns its initial state."""
    rng = _rng(10)
    lens = [5, 0, 17, 1, 9]
    cu = np.concatenate([[0], np.cumsum(lens)])
    Tt = cu[-1]
    q, k, v, g, beta, _ = _rand_case(rng, 1, Tt, 2, 4, 8, 6)
    s0 = rng.standard_normal((len(lens), 4, 8, 6))
    o, sf, st = oracle_mod.forward(q, k, v, g, beta, initial_state=s0, cu_seqlens=cu,
                                   want_states=True)
    for i, L in enumerate(lens):
        a, b = cu[i], cu[i + 1]
        if L == 0:
            np.testing.assert_array_equal(sf[i], s0[i])
            continue
        oi, fi, sti = oracle_mod.forward(q[:, a:b], k[:, a:b], v[:, a:b], g[:, a:b],
                                         beta[:, a:b], initial_state=s0[i:i + 1],
                                         want_states=True)
        np.testing.assert_array_equal(o[:, a:b], oi)
        np.testing.assert_array_equal(sf[i], fi[0])
        np.testing.assert_array_equal(st[:, a:b], sti)
        np.testing.assert_array_equal(sti[0, -1], fi[0])


def test_chain_entry_matches_forward(oracle_mod):
    """The single-chain entry used for sampled checks is the same computation."""
    rng = _rng(11)
    q, k, v, g, beta, s0 = _rand_case(rng, 2, 13, 2, 4, 8, 6, s0=True)
    o, sf, st = oracle_mod.forward(q, k, v, g, beta, initial_state=s0, want_states=True)
    for b, h in [(0, 0), (1, 3), (0, 2)]:
        oc, fc, sc = oracle_mod.chain(q[b, :, h // 2], k[b, :, h // 2], v[b, :, h],
                                      g[b, :, h], beta[b, :, h], initial_state=s0[b, h],
                                      want_states=True)
        np.testing.assert_array_equal(oc, o[b, :, h])
        np.testing.assert_array_equal(fc, sf[b, h])
        np.testing.assert_array_equal(sc, st[b, :, h])


def test_chain_subset_only_touches_listed(oracle_mod):
    rng = _rng(12)
    q, k, v, g, beta, _ = _rand_case(rng, 2, 5, 1, 2, 4, 4)
    o, sf, _ = oracle_mod.forward(q, k, v, g, beta, chains=[1, 2])
    assert np.isnan(o[0, :, 0]).all() and np.isfinite(o[0, :, 1]).all()
    assert np.isfinite(o[1, :, 0]).all() and np.isnan(o[1, :, 1]).all()


# ---------------------------------------------------------------- independent solve
def _wy_one_chunk(q, k, v, g, beta, s0, scale):
    """The whole sequence as one chunk, solved in closed form with numpy:
    with G_t = sum_{s<=t} g_s, A_tj = beta_t e^{G_t-G_j} (k^_t . k^_j) for j < t,
    (I + A) U = diag(beta) (V - diag(e^G) K^ S0), O = diag(e^G) Q~ S0 + (M o Q~K^^T) U
    with M_tj = e^{G_t-G_j} for j <= t, S_T = e^{G_T} S0 + sum_j e^{G_T-G_j} k^_j u_j^T.
    Derived by unrolling the recurrence over one chunk; np.linalg.solve does the
    triangular solve."""
    T = q.shape[0]
    qn = _l2n(q) * scale
    kn = _l2n(k)
    G = np.cumsum(g)
    D = np.exp(G[:, None] - G[None, :])
    low = np.tril(np.ones((T, T)), -1)
    A = beta[:, None] * D * (kn @ kn.T) * low
    rhs = beta[:, None] * (v - np.exp(G)[:, None] * (kn @ s0))
    U = np.linalg.solve(np.eye(T) + A, rhs)
    P = D * (qn @ kn.T) * np.tril(np.ones((T, T)))
    O = np.exp(G)[:, None] * (qn @ s0) + P @ U
    ST = np.exp(G[-1]) * s0 + (np.exp(G[-1] - G)[:, None] * kn).T @ U
    return O, ST


@pytest.mark.parametrize("T,Dk,Dv,g_scale", [(1, 8, 8, 1.0), (37, 16, 12, 1.0),
                                             (64, 32, 32, 0.05), (128, 32, 16, 0.01)])
def test_matches_independent_one_chunk_solve(oracle_mod, T, Dk, Dv, g_scale):
    rng = _rng(13 + T)
    q, k, v, g, beta, s0 = _rand_case(rng, 1, T, 1, 1, Dk, Dv, s0=True, g_scale=g_scale)
    o, sf, _ = oracle_mod.forward(q, k, v, g, beta, initial_state=s0)
    O, ST = _wy_one_chunk(q[0, :, 0], k[0, :, 0], v[0, :, 0], g[0, :, 0], beta[0, :, 0],
                          s0[0, 0], Dk ** -0.5)
    np.testing.assert_allclose(o[0, :, 0], O, rtol=0, atol=1e-10)
    np.testing.assert_allclose(sf[0, 0], ST, rtol=0, atol=1e-10)


def _chunked(q, k, v, g, beta, s0, scale, C=64, single_stage=False):
    """The chunk form over chunks of C tokens, carrying the state between chunks (the
    algebra of the tensor-core prefill).  Per chunk, with G the decay prefix restarted at
    the chunk, gamma = e^G, T = (I + A)^{-1}, Ut = T diag(beta) V, W = T diag(beta gamma) K^:
        U = Ut - W S,  O = diag(gamma) Q~ S + P U,  S' = gamma_C S + (diag(e^{G_C-G}) K^)^T U.
    single_stage: the same through S' = M S + N and O = R S + P Ut with
    M = gamma_C I - Kd^T W, N = Kd^T Ut, R = diag(gamma) Q~ - P W.
    Also returns every token's state, replayed from the state before its chunk with the
    chunk's U rows: S_t = e^{g_t} S_{t-1} + k^_t u_t^T."""
    Tn, Dk = q.shape
    qn, kn = _l2n(q) * scale, _l2n(k)
    S = s0.copy()
    O = np.zeros_like(v)
    states = np.zeros((Tn, Dk, v.shape[1]))
    for c0 in range(0, Tn, C):
        sl = slice(c0, min(Tn, c0 + C))
        n = sl.stop - sl.start
        G = np.cumsum(g[sl])
        gam = np.exp(G)
        D = np.exp(G[:, None] - G[None, :])
        A = beta[sl][:, None] * D * (kn[sl] @ kn[sl].T) * np.tril(np.ones((n, n)), -1)
        Tinv = np.linalg.inv(np.eye(n) + A)
        Ut = Tinv @ (beta[sl][:, None] * v[sl])
        W = Tinv @ ((beta[sl] * gam)[:, None] * kn[sl])
        P = D * (qn[sl] @ kn[sl].T) * np.tril(np.ones((n, n)))
        Kd = np.exp(G[-1] - G)[:, None] * kn[sl]
        U = Ut - W @ S
        Sp = S.copy()
        for t in range(n):
            Sp = np.exp(g[sl][t]) * Sp + np.outer(kn[sl][t], U[t])
            states[sl.start + t] = Sp
        if single_stage:
            M = gam[-1] * np.eye(Dk) - Kd.T @ W
            R = gam[:, None] * qn[sl] - P @ W
            O[sl] = R @ S + P @ Ut
            S = M @ S + Kd.T @ Ut
        else:
            O[sl] = gam[:, None] * (qn[sl] @ S) + P @ U
            S = gam[-1] * S + Kd.T @ U
    return O, S, states


@pytest.mark.parametrize("single_stage", [False, True])
@pytest.mark.parametrize("T,g_scale", [(150, 0.05), (129, 1.0), (64, 0.5)])
def test_matches_chunked_form_over_several_chunks(oracle_mod, T, g_scale, single_stage):
    """Chunks of 64 carrying the state (tails of 22 and 1 tokens), the per-token states
    replayed from each chunk's U rows, and the single-stage rewrite of the state update
    and outputs: all equal the token-by-token rule."""
    rng = _rng(40 + T)
    q, k, v, g, beta, s0 = _rand_case(rng, 1, T, 1, 1, 16, 12, s0=True, g_scale=g_scale)
    o, sf, st = oracle_mod.forward(q, k, v, g, beta, initial_state=s0, want_states=True)
    O, ST, states = _chunked(q[0, :, 0], k[0, :, 0], v[0, :, 0], g[0, :, 0], beta[0, :, 0],
                             s0[0, 0], 16 ** -0.5, single_stage=single_stage)
    np.testing.assert_allclose(O, o[0, :, 0], rtol=0, atol=1e-10)
    np.testing.assert_allclose(ST, sf[0, 0], rtol=0, atol=1e-10)
    np.testing.assert_allclose(states, st[0, :, 0], rtol=0, atol=1e-10)


def test_per_token_states_are_the_running_state(oracle_mod):
    """states[t] is the state after token t: o_t = states[t]^T q~_t and the last one is
    the final state."""
    rng = _rng(14)
    q, k, v, g, beta, s0 = _rand_case(rng, 1, 10, 1, 1, 6, 5, s0=True)
    o, sf, st = oracle_mod.forward(q, k, v, g, beta, initial_state=s0, want_states=True)
    qn = _l2n(q[0, :, 0]) * 6 ** -0.5
    for t in range(10):
        np.testing.assert_allclose(o[0, t, 0], st[0, t, 0].T @ qn[t], rtol=0, atol=1e-13)
    np.testing.assert_array_equal(st[0, -1, 0], sf[0, 0])


# ---------------------------------------------------------------- gated RMS norm
def test_gated_norm_hand_worked_example(oracle_mod):
    """tests/golden/gated_norm_hand_Dv4.txt: two rows computed by hand (mean over the
    head's values, gain = weight, silu gate after the norm)."""
    G = _parse_golden(os.path.join(GOLDEN, "gated_norm_hand_Dv4.txt"))
    for r in range(2):
        out = oracle_mod.gated_rmsnorm(G["y"][r:r + 1], G["z"][r:r + 1], G["weight"][r], eps=0.0)
        np.testing.assert_allclose(out[0], G["out"][r], atol=1e-15, rtol=0)


def _norm_case(rng, rows, Dv):
    y = rng.standard_normal((rows, Dv)) * np.exp(rng.standard_normal((rows, 1)))
    z = rng.standard_normal((rows, Dv)) * 2.0
    w = 1.0 + 0.3 * rng.standard_normal(Dv)
    return y, z, w


@pytest.mark.parametrize("Dv", [4, 32, 128])
def test_gated_norm_gate_is_silu_after_the_norm(oracle_mod, Dv):
    """silu(z) - silu(-z) = z, so out(y, z) - out(y, -z) = y r w z when the gate
    multiplies after the norm (r does not depend on z); and rms(y r) = 1 at eps = 0
    (the mean, not the sum, of the squares)."""
    y, z, w = _norm_case(_rng(50 + Dv), 9, Dv)
    d = oracle_mod.gated_rmsnorm(y, z, w, eps=0.0) - oracle_mod.gated_rmsnorm(y, -z, w, eps=0.0)
    yr = d / (w[None, :] * z)
    np.testing.assert_allclose(np.sqrt((yr * yr).mean(-1)), 1.0, rtol=1e-12)
    np.testing.assert_allclose(yr / y, (yr / y)[:, :1].repeat(Dv, 1), rtol=1e-11)


def test_gated_norm_invariances(oracle_mod):
    """At eps = 0 the norm ignores a positive scale of its row and is odd in y; the gain
    is the weight itself (weight 0 gives 0, not the gate); rows do not interact."""
    y, z, w = _norm_case(_rng(60), 6, 16)
    o = oracle_mod.gated_rmsnorm(y, z, w, eps=0.0)
    np.testing.assert_allclose(oracle_mod.gated_rmsnorm(37.5 * y, z, w, eps=0.0), o, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(oracle_mod.gated_rmsnorm(-y, z, w, eps=0.0), -o, rtol=0, atol=0)
    assert np.all(oracle_mod.gated_rmsnorm(y, z, np.zeros_like(w)) == 0.0)
    y2 = y.copy()
    y2[3] *= 1e3
    o2 = oracle_mod.gated_rmsnorm(y2, z, w, eps=0.0)
    np.testing.assert_array_equal(np.delete(o2, 3, 0), np.delete(o, 3, 0))


def test_gated_norm_epsilon_and_zero_rows(oracle_mod):
    """eps sits inside the root next to the mean square: a constant row c with c^2 = eps
    comes out at 1/sqrt(2) of its eps-free value; an all-zero row stays zero (finite)."""
    c = 1e-3
    y = np.full((1, 8), c)
    z = np.linspace(-3, 3, 8)[None, :]
    w = np.linspace(0.5, 1.5, 8)
    ratio = oracle_mod.gated_rmsnorm(y, z, w, eps=c * c) / oracle_mod.gated_rmsnorm(y, z, w, eps=0.0)
    np.testing.assert_allclose(ratio, 2 ** -0.5, rtol=1e-12)
    zero = oracle_mod.gated_rmsnorm(np.zeros((2, 8)), np.ones((2, 8)), w)
    assert np.all(zero == 0.0)


# ---------------------------------------------------------------- conv + gates prologue
def _conv_case(rng, T, C, HV=2):
    x = rng.standard_normal((1, T, C))
    b = rng.standard_normal((1, T, HV)) * 3
    a = rng.standard_normal((1, T, HV)) * 3
    w = rng.standard_normal((C, 4))
    al = rng.standard_normal(HV)
    db = rng.standard_normal(HV)
    return x, b, a, w, al, db


def _conv_only(oracle_mod, x, w, **kw):
    """The convolution itself: silu(u) - silu(-u) = u and the convolution is odd in x."""
    HV = 1
    z = np.zeros(x.shape[:-1] + (HV,))
    yp = oracle_mod.conv_gate(x, z, z, w, np.zeros(HV), np.zeros(HV), **kw)[0]
    kw2 = dict(kw)
    if kw2.get("conv_state") is not None:
        kw2["conv_state"] = -kw2["conv_state"]
    ym = oracle_mod.conv_gate(-x, z, z, w, np.zeros(HV), np.zeros(HV), **kw2)[0]
    return yp - ym


def test_conv_impulse_response_is_causal_depthwise_width_4(oracle_mod):
    """A unit input on one channel at token 2 comes out on that channel only, at tokens
    2, 3, 4, 5, weighted by taps 3, 2, 1, 0 (tap 3 on the current token), and nowhere
    else: causal, depthwise, width 4 (Conv1d(kernel_size=4, padding=3, groups=C))."""
    T, C = 9, 3
    w = _rng(70).standard_normal((C, 4))
    x = np.zeros((1, T, C))
    x[0, 2, 1] = 1.0
    conv = _conv_only(oracle_mod, x, w)[0]
    expect = np.zeros((T, C))
    expect[2:6, 1] = w[1, ::-1]
    np.testing.assert_allclose(conv, expect, atol=1e-15, rtol=1e-14)


def test_conv_state_continues_the_sequence(oracle_mod):
    """Prefill of t tokens, then the rest from the carried state, then token by token
    (decode), all equal one pass over the whole sequence; a sequence shorter than three
    tokens carries part of the incoming state on."""
    x, b, a, w, al, db = _conv_case(_rng(71), 11, 5)
    full = oracle_mod.conv_gate(x, b, a, w, al, db, want_state=True)
    p1 = oracle_mod.conv_gate(x[:, :4], b[:, :4], a[:, :4], w, al, db, want_state=True)
    p2 = oracle_mod.conv_gate(x[:, 4:], b[:, 4:], a[:, 4:], w, al, db, conv_state=p1[3],
                              want_state=True)
    for i in range(3):
        np.testing.assert_array_equal(np.concatenate([p1[i], p2[i]], 1), full[i])
    np.testing.assert_array_equal(p2[3], full[3])
    st = None
    for t in range(11):
        y, _, _, st = oracle_mod.conv_gate(x[:, t:t + 1], b[:, t:t + 1], a[:, t:t + 1], w, al, db,
                                           conv_state=st, want_state=True)
        np.testing.assert_array_equal(y[0, 0], full[0][0, t])
    # a 1-token sequence: the window slides by one
    s_in = _rng(72).standard_normal((1, 3, 5))
    _, _, _, s_out = oracle_mod.conv_gate(x[:, :1], b[:, :1], a[:, :1], w, al, db, conv_state=s_in,
                                          want_state=True)
    np.testing.assert_array_equal(s_out[0], np.stack([s_in[0, 1], s_in[0, 2], x[0, 0]]))


def test_conv_packed_equals_separate(oracle_mod):
    """Packed sequences restart their windows at each sequence start (from their own
    carried state), exactly as separate runs."""
    lens = [5, 1, 0, 7]
    cu = np.concatenate([[0], np.cumsum(lens)])
    x, b, a, w, al, db = _conv_case(_rng(73), int(cu[-1]), 4)
    st = _rng(74).standard_normal((len(lens), 3, 4))
    y, be, g, so = oracle_mod.conv_gate(x, b, a, w, al, db, conv_state=st, cu_seqlens=cu,
                                        want_state=True)
    for s, (p, e) in enumerate(zip(cu[:-1], cu[1:])):
        ys, bs, gs, ss = oracle_mod.conv_gate(x[:, p:e], b[:, p:e], a[:, p:e], w, al, db,
                                              conv_state=st[s:s + 1], want_state=True)
        np.testing.assert_array_equal(y[:, p:e], ys)
        np.testing.assert_array_equal(g[:, p:e], gs)
        np.testing.assert_array_equal(so[s], ss[0])
    np.testing.assert_array_equal(so[2], st[2])          # empty sequence: state unchanged


def test_gates_closed_forms(oracle_mod):
    """beta = sigmoid(b): 1/2 at 0, sigmoid(b) + sigmoid(-b) = 1.  g = -exp(A_log)
    softplus(a + dt_bias): -ln 2 at 0; softplus(u) - softplus(-u) = u gives
    g(a) - g(-a) = -exp(A_log) a; dt_bias adds to a; no overflow at |a| = 50, and g <= 0."""
    T, HV = 6, 3
    x = np.zeros((1, T, 1))
    w = np.zeros((1, 4))
    bvals = np.array([0.0, 1.0, -2.5, 7.0, -40.0, 40.0])[None, :, None].repeat(HV, 2)
    a = np.array([0.0, 0.3, -1.2, 3.0, 50.0, -50.0])[None, :, None].repeat(HV, 2)
    al = np.array([0.0, np.log(2.0), -1.0])
    zero = np.zeros(HV)
    _, beta, g, _ = oracle_mod.conv_gate(x, bvals, a, w, al, zero)
    _, beta_m, g_m, _ = oracle_mod.conv_gate(x, -bvals, -a, w, al, zero)
    assert beta[0, 0, 0] == 0.5
    np.testing.assert_allclose(beta + beta_m, 1.0, rtol=1e-15)
    np.testing.assert_allclose(g[0, 0], -np.exp(al) * np.log(2.0), rtol=1e-15)
    np.testing.assert_allclose(g - g_m, -np.exp(al)[None, None, :] * a, rtol=1e-12, atol=1e-14)
    assert np.all(g <= 0.0) and np.all(np.isfinite(g))
    db = np.array([0.5, -0.25, 2.0])
    _, _, g_db, _ = oracle_mod.conv_gate(x, bvals, a, w, al, db)
    _, _, g_sh, _ = oracle_mod.conv_gate(x, bvals, a + db[None, None, :], w, al, zero)
    np.testing.assert_allclose(g_db, g_sh, rtol=1e-15)


def test_regroup_matches_the_hand_listed_layout(oracle_mod):
    """tests/golden/regroup_qkvz_hk2_hv4_d2.txt: the columns each field takes, listed by
    hand from the page's description of the per-key-head layout."""
    G = _parse_golden(os.path.join(GOLDEN, "regroup_qkvz_hk2_hv4_d2.txt"))
    qkvz = np.arange(24, dtype=float)[None, :]
    ba = np.arange(8, dtype=float)[None, :]
    q, k, v, z, b, a = oracle_mod.regroup_qkvz(qkvz, ba, HK=2, HV=4, Dk=2, Dv=2)
    for name, got in zip("qkvzba", (q, k, v, z, b, a)):
        np.testing.assert_array_equal(got[0].reshape(G[name].shape), G[name])


def test_split_matches_the_hand_listed_layout(oracle_mod):
    """tests/golden/split_qkv_hk2_hv4_dk2_dv3.txt: the channels each of q, k, v takes out of
    the conv output, listed by hand from the page's cat(q, k, v) (q heads, then k heads,
    then v heads, each head contiguous).  Value heads wider than key heads, so a reshape
    with the head and width axes swapped, a v taken before k, or a width taken from the
    wrong field all move some channel."""
    G = _parse_golden(os.path.join(GOLDEN, "split_qkv_hk2_hv4_dk2_dv3.txt"))
    y = np.arange(20, dtype=float)[None, :]
    q, k, v = oracle_mod.split_qkv(y, HK=2, HV=4, Dk=2, Dv=3)
    assert q.shape == (1, 2, 2) and k.shape == (1, 2, 2) and v.shape == (1, 4, 3)
    for name, got in zip("qkv", (q, k, v)):
        np.testing.assert_array_equal(got[0], G[name])
