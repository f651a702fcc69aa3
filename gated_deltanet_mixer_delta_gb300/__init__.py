"""Gated delta rule kernels for GB300 (sm_103a): Python binding of ``libgdn.so``.

The gated delta rule is the recurrence of the Gated DeltaNet mixer in the
Qwen3.5 / Qwen3-Next hybrid models (qwen3_5_text page, Notes -> "The DeltaNet
mixer"; qwen3_next page, Notes -> "The DeltaNet mixer fuses its projections per
key head").  This module only marshals arguments: it checks tensors, allocates
outputs with PyTorch when the caller passes none, and calls the C ABI of
``include/gdn.h`` on the current CUDA stream (or on the ``stream`` given, which
then also owns every tensor the binding allocates).  Every step of the computation
runs in the library's CUDA kernels; there is no other implementation to fall
back to, and a missing library is an error.

Layouts (the pages' linear_attn value table):
    queries, keys  [B, T, HK, Dk]        values, out  [B, T, HV, Dv]
    decays, beta   [B, T, HV] float32    state        [B, HV, Dk, Dv] float32
    states         [B, T, HV, Dk, Dv] float32 (state after every token)
"""
import ctypes
import functools
import os

import torch

from . import build as _build

__all__ = ["prefill", "prefill_varlen", "decode_step", "gated_rmsnorm", "conv_gate_prologue",
           "state_layout", "workspace_size",
           "workspace_status", "selftest_wait_timeout", "GdnError", "library_path",
           "load_library", "abi"]

GDN_OK = 0
_STATUS = {0: "ok", -1: "invalid argument", -2: "unsupported shape or dtype",
           -3: "pointer not aligned", -4: "workspace missing or too small",
           -5: "CUDA launch or runtime error", -6: "bounded device wait timed out",
           -7: "cu_seqlens malformed"}
_DTYPES = {torch.bfloat16: 0, torch.float32: 1}


class GdnError(RuntimeError):
    def __init__(self, status, where=""):
        self.status = status
        super().__init__(f"{where}: {_STATUS.get(status, 'unknown status')} ({status})")


class _StateLayout(ctypes.Structure):
    _fields_ = [("bytes", ctypes.c_size_t), ("bytes_per_head", ctypes.c_size_t),
                ("stride", ctypes.c_int64 * 4), ("shape", ctypes.c_int64 * 4),
                ("alignment", ctypes.c_int)]


_lib = None


def library_path() -> str:
    return _build.LIB


def load_library(build_if_missing: bool = False):
    """Load libgdn.so (the C ABI).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB
    if not os.path.exists(path):
        if build_if_missing:
            _build.build()
        else:
            raise RuntimeError(f"libgdn.so not built ({path}); run "
                               "gated_deltanet_mixer_delta_gb300.build.build() first")
    lib = ctypes.CDLL(path)
    vp, fp, i, sz = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    f = ctypes.c_float
    lib.gdn_prefill.restype = i
    lib.gdn_prefill.argtypes = [vp, vp, vp, fp, fp, fp, vp, fp, fp, i, i, i, i, i, i, i, f, i,
                                vp, sz, vp]
    lib.gdn_prefill_varlen.restype = i
    lib.gdn_prefill_varlen.argtypes = [vp, vp, vp, fp, fp, fp, vp, fp, fp, vp, i, i, i, i, i, i,
                                       i, f, i, vp, sz, vp]
    lib.gdn_prefill_gated.restype = i
    lib.gdn_prefill_gated.argtypes = [vp, vp, vp, fp, fp, fp, vp, fp, fp, vp, fp, f, i, i, i, i,
                                      i, i, i, f, i, vp, sz, vp]
    lib.gdn_prefill_varlen_gated.restype = i
    lib.gdn_prefill_varlen_gated.argtypes = [vp, vp, vp, fp, fp, fp, vp, fp, fp, vp, fp, f, vp, i,
                                             i, i, i, i, i, i, f, i, vp, sz, vp]
    lib.gdn_decode_step.restype = i
    lib.gdn_decode_step.argtypes = [vp, vp, vp, fp, fp, fp, vp, i, i, i, i, i, i, f, i, vp]
    lib.gdn_decode_step_gated.restype = i
    lib.gdn_decode_step_gated.argtypes = [vp, vp, vp, fp, fp, fp, vp, vp, fp, f, i, i, i, i, i, i,
                                          f, i, vp]
    lib.gdn_conv_gate_prologue.restype = i
    lib.gdn_conv_gate_prologue.argtypes = [vp, vp, vp, i, fp, fp, fp, vp, vp, vp, i, ctypes.c_int64,
                                           i, i, i, i, i, vp, vp, vp, vp, fp, fp, vp]
    lib.gdn_gated_rmsnorm.restype = i
    lib.gdn_gated_rmsnorm.argtypes = [vp, vp, fp, vp, ctypes.c_int64, i, i, f, vp]
    lib.gdn_state_layout.restype = i
    lib.gdn_state_layout.argtypes = [i, i, i, i, ctypes.POINTER(_StateLayout)]
    lib.gdn_prefill_workspace_size.restype = sz
    lib.gdn_prefill_workspace_size.argtypes = [ctypes.c_int64, i, i, i, i]
    lib.gdn_prefill_workspace_size_for.restype = sz
    lib.gdn_prefill_workspace_size_for.argtypes = [ctypes.c_int64, i, i, i, i, i]
    lib.gdn_workspace_status.restype = i
    lib.gdn_workspace_status.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_int)]
    lib.gdn_status_string.restype = ctypes.c_char_p
    lib.gdn_status_string.argtypes = [i]
    lib.gdn_abi_version.restype = i
    lib.gdn_abi_version.argtypes = []
    lib.gdn_selftest_wait_timeout.restype = i
    lib.gdn_selftest_wait_timeout.argtypes = [vp, ctypes.c_uint64, vp]
    _lib = lib
    return lib


def abi():
    """The loaded ctypes library (raw C ABI)."""
    return load_library()


def _check(rc, where):
    if rc != GDN_OK:
        raise GdnError(rc, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _need(t, name, dtype=None, device=None, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def state_layout(batch, HV, Dk, Dv):
    """Shape, strides and bytes of the recurrent state buffer [batch, HV, Dk, Dv] float32."""
    lay = _StateLayout()
    _check(load_library().gdn_state_layout(batch, HV, Dk, Dv, ctypes.byref(lay)), "gdn_state_layout")
    return dict(bytes=lay.bytes, bytes_per_head=lay.bytes_per_head, stride=tuple(lay.stride),
                shape=tuple(lay.shape), alignment=lay.alignment)


def workspace_size(T_total, n_seqs, HV, Dk, Dv, dtype=None) -> int:
    """Workspace bytes of a prefill: for `dtype` (torch.bfloat16 / torch.float32) exactly
    what that path needs, without it enough for either."""
    lib = load_library()
    if dtype is None:
        return int(lib.gdn_prefill_workspace_size(T_total, n_seqs, HV, Dk, Dv))
    return int(lib.gdn_prefill_workspace_size_for(T_total, n_seqs, HV, Dk, Dv, _DTYPES[dtype]))


def workspace_status(workspace, stream=None) -> int:
    """Device status word of the last prefill that used ``workspace`` (0 = ok)."""
    st = ctypes.c_int(0)
    _check(load_library().gdn_workspace_status(_ptr(workspace), _stream(stream), ctypes.byref(st)),
           "gdn_workspace_status")
    return st.value


def selftest_wait_timeout(limit_ns, device=None, stream=None):
    """Run the library's bounded-wait self-test on the GPU: a wait on an mbarrier phase
    that nothing completes must give up after ``limit_ns`` and report GDN_ERR_TIMEOUT.
    Returns (status, microseconds waited)."""
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    status = torch.full((2,), 12345, dtype=torch.int32, device=dev)
    _check(load_library().gdn_selftest_wait_timeout(_ptr(status), int(limit_ns), _stream(stream)),
           "gdn_selftest_wait_timeout")
    torch.cuda.synchronize(dev)
    s = status.cpu().tolist()
    return int(s[0]), int(s[1])


def _on_stream(fn):
    """Run ``fn`` with its ``stream`` argument, when one is given, as torch's current
    stream.  Every tensor the binding allocates (outputs the caller did not pass, a
    default workspace) then belongs to the stream that the library's kernels use, so the
    caching allocator cannot hand a freed temporary to other work while those kernels
    still read or write it."""
    @functools.wraps(fn)
    def run(*args, stream=None, **kwargs):
        if stream is None:
            return fn(*args, stream=None, **kwargs)
        with torch.cuda.stream(stream):
            return fn(*args, stream=stream, **kwargs)
    return run


def _gated(gate, norm_weight, dtype, device, shape):
    """Checks the gated-norm arguments; True when they are given."""
    if (gate is None) != (norm_weight is None):
        raise ValueError("gate and norm_weight go together")
    if gate is None:
        return False
    _need(gate, "gate", dtype, device, shape)
    _need(norm_weight, "norm_weight", torch.float32, device, (shape[-1],))
    return True


def _workspace(workspace, nbytes, device):
    if workspace is None:
        return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
    _need(workspace, "workspace", torch.uint8, device)
    if workspace.numel() < nbytes:
        raise GdnError(-4, "workspace")
    return workspace


@_on_stream
def prefill(queries, keys, values, decays, beta, initial_state=None, *, scale=None,
            use_qk_l2norm=True, output_states=False, out=None, final_state=None, states=None,
            workspace=None, gate=None, norm_weight=None, norm_eps=1e-6, stream=None):
    """Chunked prefill over a batch of equal-length sequences (gdn_prefill).

    Returns ``(out, final_state, states)``; ``states`` is None unless
    ``output_states`` is set or a ``states`` tensor is passed.  With ``gate``
    ([B, T, HV, Dv], dtype of the values) and ``norm_weight`` ([Dv] float32) the gated
    RMS norm is formed in the same pass (gdn_prefill_gated): out is then
    norm(y, gate=silu(gate)) * norm_weight.
    """
    _need(queries, "queries")
    dev, dt = queries.device, queries.dtype
    if dt not in _DTYPES:
        raise ValueError("queries/keys/values must be bfloat16 or float32")
    B, T, HK, Dk = queries.shape
    HV, Dv = values.shape[2], values.shape[3]
    _need(keys, "keys", dt, dev, (B, T, HK, Dk))
    _need(values, "values", dt, dev, (B, T, HV, Dv))
    _need(decays, "decays", torch.float32, dev, (B, T, HV))
    _need(beta, "beta", torch.float32, dev, (B, T, HV))
    if initial_state is not None:
        _need(initial_state, "initial_state", torch.float32, dev, (B, HV, Dk, Dv))
    if out is None:
        out = torch.empty(B, T, HV, Dv, dtype=dt, device=dev)
    _need(out, "out", dt, dev, (B, T, HV, Dv))
    if final_state is None:
        final_state = torch.empty(B, HV, Dk, Dv, dtype=torch.float32, device=dev)
    _need(final_state, "final_state", torch.float32, dev, (B, HV, Dk, Dv))
    if states is None and output_states:
        states = torch.empty(B, T, HV, Dk, Dv, dtype=torch.float32, device=dev)
    if states is not None:
        _need(states, "states", torch.float32, dev, (B, T, HV, Dk, Dv))
    lib = load_library()
    nbytes = lib.gdn_prefill_workspace_size_for(B * T, B, HV, Dk, Dv, _DTYPES[dt])
    ws = _workspace(workspace, nbytes, dev)
    if _gated(gate, norm_weight, dt, dev, (B, T, HV, Dv)):
        rc = lib.gdn_prefill_gated(_ptr(queries), _ptr(keys), _ptr(values), _ptr(decays),
                                   _ptr(beta), _ptr(initial_state), _ptr(out), _ptr(final_state),
                                   _ptr(states), _ptr(gate), _ptr(norm_weight), float(norm_eps),
                                   B, T, HK, HV, Dk, Dv, _DTYPES[dt], float(scale or 0.0),
                                   int(bool(use_qk_l2norm)), _ptr(ws), ws.numel(), _stream(stream))
        _check(rc, "gdn_prefill_gated")
        return out, final_state, states
    rc = lib.gdn_prefill(_ptr(queries), _ptr(keys), _ptr(values), _ptr(decays), _ptr(beta),
                         _ptr(initial_state), _ptr(out), _ptr(final_state), _ptr(states),
                         B, T, HK, HV, Dk, Dv, _DTYPES[dt], float(scale or 0.0),
                         int(bool(use_qk_l2norm)), _ptr(ws), ws.numel(), _stream(stream))
    _check(rc, "gdn_prefill")
    return out, final_state, states


@_on_stream
def prefill_varlen(queries, keys, values, decays, beta, cu_seqlens, initial_state=None, *,
                   scale=None, use_qk_l2norm=True, output_states=False, out=None,
                   final_state=None, states=None, workspace=None, gate=None, norm_weight=None,
                   norm_eps=1e-6, stream=None):
    """Chunked prefill over sequences packed back to back (gdn_prefill_varlen).

    queries/keys [1, T_total, HK, Dk] (or [T_total, HK, Dk]), values [.., T_total, HV, Dv],
    decays/beta [.., T_total, HV], ``cu_seqlens`` int32 [N+1] on the device,
    initial_state [N, HV, Dk, Dv] or None.  Returns ``(out, final_state [N, HV, Dk, Dv],
    states)``; out and states keep the leading shape of ``values``.  ``gate`` and
    ``norm_weight`` as in :func:`prefill` (gdn_prefill_varlen_gated).
    """
    _need(queries, "queries")
    dev, dt = queries.device, queries.dtype
    if dt not in _DTYPES:
        raise ValueError("queries/keys/values must be bfloat16 or float32")
    lead = tuple(values.shape[:-2])
    T_total = queries.shape[-3]
    HK, Dk = queries.shape[-2], queries.shape[-1]
    HV, Dv = values.shape[-2], values.shape[-1]
    _need(cu_seqlens, "cu_seqlens", torch.int32, dev)
    N = cu_seqlens.numel() - 1
    if N < 0:
        raise ValueError("cu_seqlens needs at least one entry")
    _need(keys, "keys", dt, dev, queries.shape)
    _need(values, "values", dt, dev)
    _need(decays, "decays", torch.float32, dev, (*lead, HV))
    _need(beta, "beta", torch.float32, dev, (*lead, HV))
    if initial_state is not None:
        _need(initial_state, "initial_state", torch.float32, dev, (N, HV, Dk, Dv))
    if out is None:
        out = torch.empty(*lead, HV, Dv, dtype=dt, device=dev)
    _need(out, "out", dt, dev, values.shape)
    if final_state is None:
        final_state = torch.empty(N, HV, Dk, Dv, dtype=torch.float32, device=dev)
    _need(final_state, "final_state", torch.float32, dev, (N, HV, Dk, Dv))
    if states is None and output_states:
        states = torch.empty(*lead, HV, Dk, Dv, dtype=torch.float32, device=dev)
    if states is not None:
        _need(states, "states", torch.float32, dev, (*lead, HV, Dk, Dv))
    lib = load_library()
    nbytes = lib.gdn_prefill_workspace_size_for(T_total, N, HV, Dk, Dv, _DTYPES[dt])
    ws = _workspace(workspace, nbytes, dev)
    if _gated(gate, norm_weight, dt, dev, tuple(values.shape)):
        rc = lib.gdn_prefill_varlen_gated(
            _ptr(queries), _ptr(keys), _ptr(values), _ptr(decays), _ptr(beta),
            _ptr(initial_state), _ptr(out), _ptr(final_state), _ptr(states), _ptr(gate),
            _ptr(norm_weight), float(norm_eps), _ptr(cu_seqlens), N, T_total, HK, HV, Dk, Dv,
            _DTYPES[dt], float(scale or 0.0), int(bool(use_qk_l2norm)), _ptr(ws), ws.numel(),
            _stream(stream))
        _check(rc, "gdn_prefill_varlen_gated")
        return out, final_state, states
    rc = lib.gdn_prefill_varlen(_ptr(queries), _ptr(keys), _ptr(values), _ptr(decays),
                                _ptr(beta), _ptr(initial_state), _ptr(out), _ptr(final_state),
                                _ptr(states), _ptr(cu_seqlens), N, T_total, HK, HV, Dk, Dv,
                                _DTYPES[dt], float(scale or 0.0), int(bool(use_qk_l2norm)),
                                _ptr(ws), ws.numel(), _stream(stream))
    _check(rc, "gdn_prefill_varlen")
    return out, final_state, states


@_on_stream
def decode_step(queries, keys, values, decays, beta, state, *, scale=None, use_qk_l2norm=True,
                out=None, gate=None, norm_weight=None, norm_eps=1e-6, stream=None):
    """One decode step (gdn_decode_step): queries/keys [B, HK, Dk], values [B, HV, Dv],
    decays/beta [B, HV], state [B, HV, Dk, Dv] float32 updated in place.  Returns out
    [B, HV, Dv].  With ``gate`` ([B, HV, Dv], dtype of the values) and ``norm_weight``
    ([Dv] float32) the gated RMS norm is fused in (gdn_decode_step_gated): out is then
    norm(y, gate=silu(gate)) * norm_weight."""
    _need(queries, "queries")
    dev, dt = queries.device, queries.dtype
    if dt not in _DTYPES:
        raise ValueError("queries/keys/values must be bfloat16 or float32")
    B, HK, Dk = queries.shape
    HV, Dv = values.shape[1], values.shape[2]
    _need(keys, "keys", dt, dev, (B, HK, Dk))
    _need(values, "values", dt, dev, (B, HV, Dv))
    _need(decays, "decays", torch.float32, dev, (B, HV))
    _need(beta, "beta", torch.float32, dev, (B, HV))
    _need(state, "state", torch.float32, dev, (B, HV, Dk, Dv))
    if out is None:
        out = torch.empty(B, HV, Dv, dtype=dt, device=dev)
    _need(out, "out", dt, dev, (B, HV, Dv))
    if (gate is None) != (norm_weight is None):
        raise ValueError("gate and norm_weight go together")
    if gate is not None:
        _need(gate, "gate", dt, dev, (B, HV, Dv))
        _need(norm_weight, "norm_weight", torch.float32, dev, (Dv,))
        rc = load_library().gdn_decode_step_gated(
            _ptr(queries), _ptr(keys), _ptr(values), _ptr(decays), _ptr(beta), _ptr(state),
            _ptr(out), _ptr(gate), _ptr(norm_weight), float(norm_eps), B, HK, HV, Dk, Dv,
            _DTYPES[dt], float(scale or 0.0), int(bool(use_qk_l2norm)), _stream(stream))
        _check(rc, "gdn_decode_step_gated")
        return out
    rc = load_library().gdn_decode_step(_ptr(queries), _ptr(keys), _ptr(values), _ptr(decays),
                                        _ptr(beta), _ptr(state), _ptr(out), B, HK, HV, Dk, Dv,
                                        _DTYPES[dt], float(scale or 0.0),
                                        int(bool(use_qk_l2norm)), _stream(stream))
    _check(rc, "gdn_decode_step")
    return out


@_on_stream
def gated_rmsnorm(y, gate, norm_weight, *, eps=1e-6, out=None, stream=None):
    """Gated RMS norm of the mixer output (gdn_gated_rmsnorm): y, gate [..., Dv] (bf16 or
    float32, same dtype), norm_weight [Dv] float32.  Returns
    y / sqrt(mean(y^2) + eps) * norm_weight * silu(gate) per row of Dv; ``out`` may be y."""
    _need(y, "y")
    dev, dt = y.device, y.dtype
    if dt not in _DTYPES:
        raise ValueError("y must be bfloat16 or float32")
    Dv = y.shape[-1]
    _need(gate, "gate", dt, dev, tuple(y.shape))
    _need(norm_weight, "norm_weight", torch.float32, dev, (Dv,))
    if out is None:
        out = torch.empty_like(y)
    _need(out, "out", dt, dev, tuple(y.shape))
    rows = y.numel() // Dv if Dv else 0
    rc = load_library().gdn_gated_rmsnorm(_ptr(y), _ptr(gate), _ptr(norm_weight), _ptr(out), rows,
                                          Dv, _DTYPES[dt], float(eps), _stream(stream))
    _check(rc, "gdn_gated_rmsnorm")
    return out


LAYOUTS = {"qkv": 0, "qkvz": 1}


@_on_stream
def conv_gate_prologue(proj, proj_b, proj_a, conv_weight, A_log, dt_bias, *, HK, HV, Dk, Dv,
                       layout="qkv", conv_state=None, conv_state_out=None, cu_seqlens=None,
                       stream=None):
    """The step before the rule (gdn_conv_gate_prologue): from the projections' outputs
    proj [B, T, W] (layout "qkv": the cat(q, k, v) channels, with proj_b, proj_a
    [B, T, HV]; layout "qkvz": Qwen3-Next's per-key-head fused layout, with proj_b the
    fused b/a [B, T, 2 HV] and proj_a None), conv_weight [C, 4], A_log and dt_bias [HV]
    (float32), the carried conv_state [N, 3, C] or None.  ``conv_state_out`` receives the
    state after each sequence (it may be conv_state).  Packed form: B == 1 and
    ``cu_seqlens`` [N+1] int32.  Returns a dict with queries, keys [B, T, HK, Dk],
    values [B, T, HV, Dv], beta, decays [B, T, HV] float32 and, for "qkvz", z
    [B, T, HV, Dv]."""
    _need(proj, "proj")
    dev, dt = proj.device, proj.dtype
    if dt not in _DTYPES:
        raise ValueError("proj must be bfloat16 or float32")
    B, T = proj.shape[0], proj.shape[1]
    lay = LAYOUTS[layout]
    C = 2 * HK * Dk + HV * Dv
    if cu_seqlens is not None:
        if B != 1:
            raise ValueError("packed form needs batch 1")
        _need(cu_seqlens, "cu_seqlens", torch.int32, dev)
        N = cu_seqlens.numel() - 1
    else:
        N = B
    _need(proj_b, "proj_b", dt, dev)
    if lay == 0:
        _need(proj_a, "proj_a", dt, dev, tuple(proj_b.shape))
    _need(conv_weight, "conv_weight", torch.float32, dev, (C, 4))
    _need(A_log, "A_log", torch.float32, dev, (HV,))
    _need(dt_bias, "dt_bias", torch.float32, dev, (HV,))
    if conv_state is not None:
        _need(conv_state, "conv_state", dt, dev, (N, 3, C))
    if conv_state_out is not None:
        _need(conv_state_out, "conv_state_out", dt, dev, (N, 3, C))
    o = dict(queries=torch.empty(B, T, HK, Dk, dtype=dt, device=dev),
             keys=torch.empty(B, T, HK, Dk, dtype=dt, device=dev),
             values=torch.empty(B, T, HV, Dv, dtype=dt, device=dev),
             beta=torch.empty(B, T, HV, dtype=torch.float32, device=dev),
             decays=torch.empty(B, T, HV, dtype=torch.float32, device=dev))
    if lay == 1:
        o["z"] = torch.empty(B, T, HV, Dv, dtype=dt, device=dev)
    rc = load_library().gdn_conv_gate_prologue(
        _ptr(proj), _ptr(proj_b), _ptr(proj_a), lay, _ptr(conv_weight), _ptr(A_log),
        _ptr(dt_bias), _ptr(conv_state), _ptr(conv_state_out), _ptr(cu_seqlens), N, B * T,
        HK, HV, Dk, Dv, _DTYPES[dt], _ptr(o["queries"]), _ptr(o["keys"]), _ptr(o["values"]),
        _ptr(o.get("z")), _ptr(o["beta"]), _ptr(o["decays"]), _stream(stream))
    _check(rc, "gdn_conv_gate_prologue")
    return o
