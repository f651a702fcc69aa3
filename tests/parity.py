"""Parity helpers: compare the CUDA path with the fp64 oracle.

Tolerances (stated by the target of the build, for bf16 inputs with fp32
accumulation): outputs within max-abs 2e-2; states within relative Frobenius
error 1e-3, taken per (sequence, value head) and gated on the worst one.  For
float32 inputs the outputs carry no bf16 rounding, so the bound is tightened to
1e-4 (fp32 arithmetic over chunk algebra of depth ~C = 64 gives errors of a few
1e-6 on outputs of magnitude ~1).
"""
import concurrent.futures as cf
import os

import numpy as np
import torch

import oracle

O_ATOL_BF16 = 2e-2
O_ATOL_F32 = 1e-4
STATE_RFRO = 1e-3
STATE_ABS_FLOOR = 1e-9      # used when the reference state has norm below 1e-6


def o_atol(dtype):
    return O_ATOL_BF16 if dtype == torch.bfloat16 else O_ATOL_F32


def max_abs(a, b):
    a = a.detach().double().cpu().numpy() if isinstance(a, torch.Tensor) else np.asarray(a)
    b = b.detach().double().cpu().numpy() if isinstance(b, torch.Tensor) else np.asarray(b)
    assert a.shape == b.shape, (a.shape, b.shape)
    if a.size == 0:
        return 0.0
    return float(np.abs(a - b).max())


def rel_fro(gpu, ref):
    """||gpu - ref||_F / ||ref||_F over the last two axes; returns an array over the rest
    (an absolute error where ||ref|| < 1e-6, compared against the floor by the caller)."""
    g = gpu.detach().double().cpu().numpy() if isinstance(gpu, torch.Tensor) else np.asarray(gpu)
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    num = np.sqrt(((g - r) ** 2).sum(axis=(-1, -2)))
    den = np.sqrt((r ** 2).sum(axis=(-1, -2)))
    small = den < 1e-6
    out = np.where(small, num, num / np.where(small, 1.0, den))
    return out, small


def assert_states_close(gpu, ref, what="state"):
    err, small = rel_fro(gpu, ref)
    bad_rel = (~small) & (err > STATE_RFRO)
    bad_abs = small & (err > STATE_ABS_FLOOR)
    worst = float(err[~small].max()) if (~small).any() else 0.0
    assert not bad_rel.any() and not bad_abs.any(), \
        f"{what}: worst relative Frobenius error {worst:.3e} (bound {STATE_RFRO})"
    return worst


def assert_out_close(gpu, ref, dtype, what="out"):
    e = max_abs(gpu, ref)
    assert e <= o_atol(dtype), f"{what}: max-abs error {e:.3e} (bound {o_atol(dtype)})"
    return e


def oracle_chains(inp, chains, cu=None, want_states=False, threads=None):
    """Run the oracle on selected (sequence, value head) chains of a batch.

    ``inp`` holds queries/keys [B,T,HK,Dk], values [B,T,HV,Dv], decays/beta [B,T,HV] and
    initial_state (or None), on any device; with ``cu`` (offsets) the batch is packed
    (B = 1) and sequence i owns tokens cu[i]:cu[i+1].  Returns {(seq, h): (o, final, states)}
    in float64; chains run concurrently (ctypes drops the GIL)."""
    HK = inp["queries"].shape[2]
    HV = inp["values"].shape[2]
    r = HV // HK
    cu_l = None if cu is None else [int(x) for x in (cu.tolist() if hasattr(cu, "tolist") else cu)]

    def one(sh):
        s, h = sh
        if cu_l is None:
            b, a, e = s, 0, inp["queries"].shape[1]
        else:
            b, a, e = 0, cu_l[s], cu_l[s + 1]
        j = h // r
        s0 = inp.get("initial_state")
        return sh, oracle.chain(
            inp["queries"][b, a:e, j].cpu(), inp["keys"][b, a:e, j].cpu(),
            inp["values"][b, a:e, h].cpu(), inp["decays"][b, a:e, h].cpu(),
            inp["beta"][b, a:e, h].cpu(),
            initial_state=None if s0 is None else s0[s, h].cpu(), want_states=want_states)

    n = threads or len(os.sched_getaffinity(0))
    with cf.ThreadPoolExecutor(max_workers=max(1, min(n, len(chains)))) as ex:
        return dict(ex.map(one, chains))
