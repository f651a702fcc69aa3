"""Seeded synthetic inputs for the gated delta rule.

This module holds no arithmetic of the rule itself: it draws the tensors that
both the CUDA path and the fp64 oracle are fed (the same bits go to both), and
names the workloads the tests and the bench use.  Shapes follow the models on
the pages: Qwen3-Next-80B-A3B (16 key heads over 32 value heads, 128 x 128
heads; qwen3_next page, Config and Notes), Qwen3.5 (16 key heads over 16, 32 or
48 value heads; qwen3_5_text page, "The DeltaNet mixer").

Recipe (all draws from one ``torch.Generator`` seeded per workload, in a fixed
order: queries, keys, values, decays, beta, initial state, lengths first for
packed batches):
  * queries, keys, values ~ N(0, 1) in float32, then cast to the workload's
    dtype (bf16 by round-to-nearest-even, or kept float32);
  * decays  g = -softplus(N(0, 1)) - shift  (float32, <= 0);
  * beta    = sigmoid(N(0, 1))                 (float32, in (0, 1));
  * initial state ~ N(0, std^2) float32 when the workload has one.
Value ranges match what the pages report for a trained model: query norms
0.09-4.1 before the kernel's l2 norm, per-head kept fractions exp(g) from 0.05
to above 0.999 (qwen3_5_text page, "The DeltaNet mixer").
"""
from dataclasses import dataclass
from typing import Optional

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    T: int
    HK: int
    HV: int
    Dk: int
    Dv: int
    dtype: torch.dtype
    seed: int
    qk_prenorm: bool = False          # q, k L2-normalised when drawn
    g_shift: float = 0.0              # g = -softplus(N(0,1)) - g_shift
    init_state_std: Optional[float] = None
    n_seqs: int = 0                   # > 0: packed batch of that many sequences
    len_range: tuple = (0, 0)         # inclusive range of packed lengths
    emit_states: bool = False
    decode_steps: int = 0             # > 0: a decode workload of that many steps
    notes: str = ""


WORKLOADS = {
    w.name: w for w in [
        Workload("tiny_T64_H2_d32_f32", B=1, T=64, HK=2, HV=2, Dk=32, Dv=32,
                 dtype=torch.float32, seed=1001, qk_prenorm=True,
                 notes="tiny prefill, fp32, zero initial state"),
        Workload("next_prefill_T4096_hk16_hv32_d128", B=1, T=4096, HK=16, HV=32, Dk=128, Dv=128,
                 dtype=torch.bfloat16, seed=1002,
                 notes="Qwen3-Next-shaped prefill, zero initial state"),
        Workload("varlen8_512to8192_hk16_hv32_d128", B=1, T=0, HK=16, HV=32, Dk=128, Dv=128,
                 dtype=torch.bfloat16, seed=1003, init_state_std=0.02, n_seqs=8,
                 len_range=(512, 8192),
                 notes="8 packed sequences with per-sequence initial states"),
        Workload("decode_B256_hk16_hv32_d128", B=256, T=1, HK=16, HV=32, Dk=128, Dv=128,
                 dtype=torch.bfloat16, seed=1004, init_state_std=0.02, decode_steps=128,
                 notes="decode step, state [256,32,128,128] fp32 updated in place"),
        Workload("long_prefill_B2_T65536_hk16_hv32_d128", B=2, T=65536, HK=16, HV=32, Dk=128,
                 Dv=128, dtype=torch.bfloat16, seed=1005, g_shift=0.01,
                 notes="long-context prefill, zero initial state"),
        Workload("states_B4_T1024_hk16_hv32_d128", B=4, T=1024, HK=16, HV=32, Dk=128, Dv=128,
                 dtype=torch.bfloat16, seed=1006, g_shift=0.01, emit_states=True,
                 notes="prefill emitting per-token states [4,1024,32,128,128] fp32"),
        # head layouts of other sizes of the family (qwen3_5_text page, "The DeltaNet
        # mixer": 0.8B and 2B 16 key heads over 16 value heads, 27B over 48)
        Workload("qwen35_27b_prefill_T4096_hk16_hv48_d128", B=1, T=4096, HK=16, HV=48, Dk=128,
                 Dv=128, dtype=torch.bfloat16, seed=1007,
                 notes="27B-shaped prefill (three value heads per key head)"),
        Workload("qwen35_0p8b_prefill_T4096_hk16_hv16_d128", B=1, T=4096, HK=16, HV=16, Dk=128,
                 Dv=128, dtype=torch.bfloat16, seed=1008,
                 notes="0.8B-shaped prefill (one value head per key head)"),
    ]
}


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def draw_lengths(n: int, lo: int, hi: int, seed: int) -> list:
    """n integer lengths uniform on [lo, hi] (inclusive), drawn on the CPU."""
    g = _gen(seed, "cpu")
    return torch.randint(lo, hi + 1, (n,), generator=g).tolist()


def draw_inputs(B, T, HK, HV, Dk, Dv, dtype=torch.bfloat16, seed=0, *, qk_prenorm=False,
                g_shift=0.0, init_state_std=None, n_states=None, device="cpu"):
    """Draw one batch.  Returns a dict with queries/keys [B,T,HK,Dk], values [B,T,HV,Dv]
    (``dtype``), decays/beta [B,T,HV] float32 and initial_state [n_states or B,HV,Dk,Dv]
    float32 or None.  All tensors live on ``device``; the same seed gives the same bits on
    the same device type."""
    g = _gen(seed, device)
    f32 = dict(dtype=torch.float32, device=device, generator=g)
    q = torch.randn(B, T, HK, Dk, **f32)
    k = torch.randn(B, T, HK, Dk, **f32)
    if qk_prenorm:
        q = q / q.norm(dim=-1, keepdim=True)
        k = k / k.norm(dim=-1, keepdim=True)
    v = torch.randn(B, T, HV, Dv, **f32)
    decays = -torch.nn.functional.softplus(torch.randn(B, T, HV, **f32)) - g_shift
    beta = torch.sigmoid(torch.randn(B, T, HV, **f32))
    s0 = None
    if init_state_std is not None:
        s0 = torch.randn(n_states if n_states is not None else B, HV, Dk, Dv, **f32) * init_state_std
    return dict(queries=q.to(dtype), keys=k.to(dtype), values=v.to(dtype),
                decays=decays.contiguous(), beta=beta.contiguous(), initial_state=s0)


def workload_inputs(w: Workload, device="cpu", T_override: Optional[int] = None):
    """Inputs of a named prefill workload (packed ones get ``cu_seqlens`` int32 on
    ``device`` and ``lengths``)."""
    if w.n_seqs:
        lengths = draw_lengths(w.n_seqs, *w.len_range, seed=w.seed)
        total = sum(lengths)
        d = draw_inputs(1, total, w.HK, w.HV, w.Dk, w.Dv, w.dtype, w.seed + 100_000,
                        qk_prenorm=w.qk_prenorm, g_shift=w.g_shift,
                        init_state_std=w.init_state_std, n_states=w.n_seqs, device=device)
        cu = torch.tensor([0] + list(torch.tensor(lengths).cumsum(0).tolist()),
                          dtype=torch.int32, device=device)
        d["cu_seqlens"] = cu
        d["lengths"] = lengths
        return d
    T = T_override or w.T
    return draw_inputs(w.B, T, w.HK, w.HV, w.Dk, w.Dv, w.dtype, w.seed,
                       qk_prenorm=w.qk_prenorm, g_shift=w.g_shift,
                       init_state_std=w.init_state_std, device=device)


def decode_inputs(w: Workload, steps: Optional[int] = None, device="cpu"):
    """Decode workload: initial_state [B,HV,Dk,Dv] and per-step inputs stacked on a
    leading step axis: queries/keys [S,B,HK,Dk], values [S,B,HV,Dv], decays/beta [S,B,HV]."""
    S = steps or w.decode_steps
    d = draw_inputs(S, w.B, w.HK, w.HV, w.Dk, w.Dv, w.dtype, w.seed, g_shift=w.g_shift,
                    device=device)
    g = _gen(w.seed + 7, device)
    d["initial_state"] = torch.randn(w.B, w.HV, w.Dk, w.Dv, dtype=torch.float32, device=device,
                                     generator=g) * w.init_state_std
    return d
