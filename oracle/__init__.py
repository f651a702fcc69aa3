"""fp64 CPU oracle for the gated delta rule -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It shares nothing with the CUDA path:
the arithmetic lives in ``gdn_oracle.c`` (plain C, double precision, one
token at a time), and this module only converts arrays to float64 and calls
it through ctypes.

Rule (qwen3_5_text page, Notes -> "The DeltaNet mixer"; qwen3_next page,
Notes -> "The DeltaNet mixer fuses its projections per key head"), per value
head h with key head h // (HV // HK):

    S <- exp(g_t) S ;  u = beta_t (v_t - S^T k_t) ;  S <- S + k_t u^T ;  o_t = S^T q_t

with k_t = l2norm(k_t), q_t = l2norm(q_t) * Dk**-0.5.  State layout
[.., key_dim, value_dim] (linear_attn value table, State).

Pins: every function here is checked in ``tests/test_oracle_pins.py``
against closed forms (T=1 output, beta=0, g -> -inf), the Widrow-Hoff
projection property with orthonormal keys, an independent one-chunk WY/UT
solve, continuation, linearity and the GQA interleave of the pages; the
gated RMS norm of the output against a hand-worked example, the identity
silu(z) - silu(-z) = z, its scale invariance and the unit RMS of the
normalised row; the convolution of the step before the rule by its impulse
response (causal, depthwise, width 4), continuation through the carried conv
state and packed-vs-separate runs; the gates by closed forms and the
softplus odd-part identity; the regroup of the fused projections against a
hand-listed column layout; the split of the conv output into queries, keys
and values against a hand-listed channel layout.
"""
import ctypes
import os

import numpy as np

from .build import build_oracle

_lib = None


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build_oracle())
        dp = ctypes.POINTER(ctypes.c_double)
        lib.gdn_oracle_forward.restype = ctypes.c_int
        lib.gdn_oracle_forward.argtypes = [
            dp, dp, dp, dp, dp, dp, dp, dp, dp,
            ctypes.POINTER(ctypes.c_int64), ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_int,
            ctypes.POINTER(ctypes.c_int32), ctypes.c_int, ctypes.c_int]
        lib.gdn_oracle_chain.restype = ctypes.c_int
        lib.gdn_oracle_chain.argtypes = [
            ctypes.c_int, ctypes.c_int, ctypes.c_int,
            dp, ctypes.c_ssize_t, dp, ctypes.c_ssize_t, dp, ctypes.c_ssize_t,
            dp, dp, ctypes.c_ssize_t, dp, dp, ctypes.c_ssize_t, dp, dp, ctypes.c_ssize_t,
            ctypes.c_double, ctypes.c_int]
        lib.gdn_oracle_conv_gate.restype = ctypes.c_int
        lib.gdn_oracle_conv_gate.argtypes = [dp, dp, dp, dp, dp, dp, dp, dp,
                                             ctypes.POINTER(ctypes.c_int64), ctypes.c_int,
                                             ctypes.c_int, ctypes.c_int, dp, dp, dp]
        lib.gdn_oracle_gated_rmsnorm.restype = ctypes.c_int
        lib.gdn_oracle_gated_rmsnorm.argtypes = [dp, dp, dp, dp, ctypes.c_int64, ctypes.c_int,
                                                 ctypes.c_double]
        _lib = lib
    return _lib


def _f64(x):
    """Exact upcast to a C-contiguous float64 numpy array (bf16/fp32 -> fp64 is exact)."""
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor
        x = x.detach().cpu().double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def forward(queries, keys, values, decays, beta, initial_state=None, cu_seqlens=None,
            scale=None, use_qk_l2norm=True, want_states=False, chains=None, n_threads=None):
    """Run the recurrence in fp64.

    Batched form: queries/keys [B, T, HK, Dk], values [B, T, HV, Dv],
    decays/beta [B, T, HV], initial_state [B, HV, Dk, Dv] or None.
    Packed (varlen) form: the same tensors with B == 1 and ``cu_seqlens``
    ([N+1] offsets); initial/final states are then [N, HV, Dk, Dv].

    Returns (out [.., HV, Dv], final_state [N or B, HV, Dk, Dv], states or None),
    all float64 numpy arrays.  ``chains`` (ids seq*HV + h) limits the work to
    those chains; other entries of the outputs are left as NaN.
    """
    q, k, v = _f64(queries), _f64(keys), _f64(values)
    g, b = _f64(decays), _f64(beta)
    s0 = _f64(initial_state)
    B, T, HK, Dk = q.shape
    HV, Dv = v.shape[2], v.shape[3]
    if cu_seqlens is None:
        cu = np.arange(B + 1, dtype=np.int64) * T
    else:
        if B != 1:
            raise ValueError("packed form needs batch 1")
        cu = np.ascontiguousarray(np.asarray(
            cu_seqlens.cpu() if hasattr(cu_seqlens, "cpu") else cu_seqlens, dtype=np.int64))
    N = len(cu) - 1
    if scale is None:
        scale = Dk ** -0.5
    out = np.full((B, T, HV, Dv), np.nan)
    final = np.full((N, HV, Dk, Dv), np.nan)
    states = np.full((B, T, HV, Dk, Dv), np.nan) if want_states else None
    ch = None
    n_ch = 0
    if chains is not None:
        ch = np.ascontiguousarray(np.asarray(chains, dtype=np.int32))
        n_ch = len(ch)
    rc = _load().gdn_oracle_forward(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(b), _ptr(s0),
        _ptr(out), _ptr(final), _ptr(states),
        cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), N, HK, HV, Dk, Dv,
        float(scale), int(bool(use_qk_l2norm)),
        None if ch is None else ch.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), n_ch,
        int(n_threads or default_threads()))
    if rc != 0:
        raise RuntimeError(f"gdn_oracle_forward failed ({rc})")
    return out, final, states


def decode_step(queries, keys, values, decays, beta, state, scale=None, use_qk_l2norm=True,
                n_threads=None):
    """One token per sequence: queries/keys [B, HK, Dk], values [B, HV, Dv],
    decays/beta [B, HV], state [B, HV, Dk, Dv] (not modified).

    Returns (out [B, HV, Dv], new_state [B, HV, Dk, Dv]) in float64.  This is
    the same recurrence over sequences of length one, started from ``state``.
    """
    q, k, v = _f64(queries), _f64(keys), _f64(values)
    g, b = _f64(decays), _f64(beta)
    B = q.shape[0]
    out, final, _ = forward(q.reshape(1, B, *q.shape[1:]), k.reshape(1, B, *k.shape[1:]),
                            v.reshape(1, B, *v.shape[1:]), g.reshape(1, B, -1),
                            b.reshape(1, B, -1), initial_state=state,
                            cu_seqlens=np.arange(B + 1), scale=scale,
                            use_qk_l2norm=use_qk_l2norm, n_threads=n_threads)
    return out.reshape(B, *out.shape[2:]), final


def chain(queries, keys, values, decays, beta, initial_state=None, scale=None,
          use_qk_l2norm=True, want_states=False):
    """One (sequence, value head) chain: queries/keys [T, Dk], values [T, Dv],
    decays/beta [T], initial_state [Dk, Dv] or None.

    Returns (out [T, Dv], final [Dk, Dv], states [T, Dk, Dv] or None) in float64.
    Used for sampled checks on workloads whose full fp64 copy would not fit.
    """
    q, k, v = _f64(queries), _f64(keys), _f64(values)
    g, b = _f64(decays), _f64(beta)
    s0 = _f64(initial_state)
    T, Dk = q.shape
    Dv = v.shape[1]
    if scale is None:
        scale = Dk ** -0.5
    out = np.zeros((T, Dv))
    final = np.zeros((Dk, Dv))
    states = np.zeros((T, Dk, Dv)) if want_states else None
    rc = _load().gdn_oracle_chain(
        T, Dk, Dv, _ptr(q), Dk, _ptr(k), Dk, _ptr(v), Dv, _ptr(g), _ptr(b), 1, _ptr(s0),
        _ptr(out), Dv, _ptr(final), _ptr(states), Dk * Dv, float(scale),
        int(bool(use_qk_l2norm)))
    if rc != 0:
        raise RuntimeError("gdn_oracle_chain failed")
    return out, final, states


GATED_NORM_EPS = 1e-6


def gated_rmsnorm(y, z, weight, eps=GATED_NORM_EPS):
    """Gated RMS norm of the mixer output, norm(y, gate=silu(z)) with gain = weight
    (qwen3_5_text page, Notes -> "The DeltaNet mixer"): per row of the last axis (Dv),
    y / sqrt(mean(y^2) + eps) * weight * silu(z).  y, z [..., Dv], weight [Dv].
    Returns float64 of y's shape."""
    yy, zz, ww = _f64(y), _f64(z), _f64(weight)
    Dv = yy.shape[-1]
    if zz.shape != yy.shape or ww.shape != (Dv,):
        raise ValueError("gated_rmsnorm: y, z must match and weight must be [Dv]")
    out = np.zeros_like(yy)
    rows = yy.size // Dv if Dv else 0
    rc = _load().gdn_oracle_gated_rmsnorm(_ptr(yy), _ptr(zz), _ptr(ww), _ptr(out), rows, Dv,
                                          float(eps))
    if rc != 0:
        raise RuntimeError("gdn_oracle_gated_rmsnorm failed")
    return out


def conv_gate(x, b, a, conv_weight, A_log, dt_bias, conv_state=None, cu_seqlens=None,
              want_state=False):
    """The step before the rule (qwen3_5_text page, Notes -> "The DeltaNet mixer"):
    y = silu(causal depthwise conv1d of width 4) over the cat(q, k, v) channels,
    beta = sigmoid(b), g = -exp(A_log) softplus(a + dt_bias).

    x [B, T, C]; b, a [B, T, HV]; conv_weight [C, 4] (tap 3 multiplies the current
    token); A_log, dt_bias [HV]; conv_state [N, 3, C] (the three inputs before each
    sequence, oldest first) or None for the start of a prompt.  Packed form: B == 1 and
    ``cu_seqlens`` [N+1].  Returns (y [B, T, C], beta [B, T, HV], g [B, T, HV],
    state_out [N, 3, C] or None), float64."""
    xx, bb, aa = _f64(x), _f64(b), _f64(a)
    w, al, db = _f64(conv_weight), _f64(A_log), _f64(dt_bias)
    B, T, C = xx.shape
    HV = bb.shape[-1]
    if cu_seqlens is None:
        cu = np.arange(B + 1, dtype=np.int64) * T
    else:
        if B != 1:
            raise ValueError("packed form needs batch 1")
        cu = np.ascontiguousarray(np.asarray(
            cu_seqlens.cpu() if hasattr(cu_seqlens, "cpu") else cu_seqlens, dtype=np.int64))
    N = len(cu) - 1
    st = _f64(conv_state)
    if st is not None and st.shape != (N, 3, C):
        raise ValueError("conv_state must be [N, 3, C]")
    y = np.zeros((B, T, C))
    beta = np.zeros((B, T, HV))
    g = np.zeros((B, T, HV))
    st_out = np.zeros((N, 3, C)) if want_state else None
    rc = _load().gdn_oracle_conv_gate(
        _ptr(xx), _ptr(bb), _ptr(aa), _ptr(w), _ptr(al), _ptr(db), _ptr(st), _ptr(st_out),
        cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), N, C, HV, _ptr(y), _ptr(beta), _ptr(g))
    if rc != 0:
        raise RuntimeError("gdn_oracle_conv_gate failed")
    return y, beta, g, st_out


def split_qkv(y, HK, HV, Dk, Dv):
    """split(...) of the mixer: the cat(q, k, v) channels of y [.., C] into queries
    [.., HK, Dk], keys [.., HK, Dk] and values [.., HV, Dv] (head-major channels)."""
    lead = y.shape[:-1]
    q = y[..., :HK * Dk].reshape(*lead, HK, Dk)
    k = y[..., HK * Dk:2 * HK * Dk].reshape(*lead, HK, Dk)
    v = y[..., 2 * HK * Dk:].reshape(*lead, HV, Dv)
    return q, k, v


def regroup_qkvz(qkvz, ba, HK, HV, Dk, Dv):
    """The regroup of the fused projections (qwen3_next page, Notes -> "The DeltaNet mixer
    fuses its projections per key head"): in_proj_qkvz holds, for each key head j, its
    query (Dk), its key (Dk), then the values of the r = HV/HK value heads it serves
    (r x Dv), then their output gates (r x Dv); in_proj_ba holds per key head the r
    value heads' b, then their a.  Returns (q [.., HK, Dk], k [.., HK, Dk],
    v [.., HV, Dv], z [.., HV, Dv], b [.., HV], a [.., HV]) as float64 views of the
    inputs' columns."""
    X, Y = _f64(qkvz), _f64(ba)
    r = HV // HK
    lead = X.shape[:-1]
    per = 2 * Dk + 2 * r * Dv
    if X.shape[-1] != HK * per or Y.shape[-1] != HK * 2 * r:
        raise ValueError("regroup_qkvz: widths do not match the head layout")
    Xh = X.reshape(*lead, HK, per)
    Yh = Y.reshape(*lead, HK, 2 * r)
    q = Xh[..., :Dk]
    k = Xh[..., Dk:2 * Dk]
    v = Xh[..., 2 * Dk:2 * Dk + r * Dv].reshape(*lead, HV, Dv)
    z = Xh[..., 2 * Dk + r * Dv:].reshape(*lead, HV, Dv)
    b = Yh[..., :r].reshape(*lead, HV)
    a = Yh[..., r:].reshape(*lead, HV)
    return q, k, v, z, b, a
