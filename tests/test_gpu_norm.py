"""GPU parity of the gated RMS norm of the mixer output (gdn_gated_rmsnorm, and fused
into the decode step: gdn_decode_step_gated) against the fp64 oracle.

Tolerances, from the arithmetic: the kernels compute in fp32, where the mean of squares
over at most 128 values, rsqrt, exp and the products keep ~2e-5 relative error; a bf16
result then adds its rounding (8 significant bits: at most 2^-8 relative).  So
|gpu - ref| <= rtol |ref| with rtol = 2e-5 (fp32) or 2^-8 + 2e-5 -> 4e-3 (bf16), plus 1e-7
absolute for values that underflow to zero.  The fused decode normalises its own fp32 y: an error dy of y moves
the output by about |weight silu(z)| dy / rms(y), and the fp32 step keeps dy below 1e-3
rms(y), which adds 1e-3 |weight silu(z)|."""
import numpy as np
import pytest
import torch

import workloads
from parity import assert_states_close, oracle_chains

pytestmark = pytest.mark.gpu
import oracle  # noqa: E402

RTOL = {torch.float32: 2e-5, torch.bfloat16: 4e-3}


@pytest.fixture(scope="module")
def gdn():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gated_deltanet_mixer_delta_gb300 as m
    m.build.build()
    m.load_library()
    return m


def _norm_inputs(rows, Dv, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    y = torch.randn(rows, Dv, generator=g) * torch.exp(torch.randn(rows, 1, generator=g))
    z = torch.randn(rows, Dv, generator=g) * 2.0
    w = 1.0 + 0.3 * torch.randn(Dv, generator=g)
    if rows > 2:
        y[1] = 0.0                                   # an all-zero row stays zero
    return y.to(dtype), z.to(dtype), w.float()


def _assert_close(got, ref, rtol, extra=None, what="out"):
    got = got.double().cpu().numpy()
    bound = rtol * np.abs(ref) + 1e-7 + (0.0 if extra is None else extra)
    err = np.abs(got - ref)
    worst = np.unravel_index(np.argmax(err - bound), err.shape) if err.size else None
    assert np.all(err <= bound), f"{what}: err {err[worst]:.3g} > bound {bound[worst]:.3g} at {worst}"


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("Dv", [32, 64, 128])
@pytest.mark.parametrize("rows", [1, 7, 1029])
def test_gated_norm_matches_oracle(gdn, rows, Dv, dtype):
    y, z, w = _norm_inputs(rows, Dv, dtype, seed=rows * 7 + Dv)
    out = gdn.gated_rmsnorm(y.cuda(), z.cuda(), w.cuda())
    torch.cuda.synchronize()
    ref = oracle.gated_rmsnorm(y, z, w)
    _assert_close(out, ref, RTOL[dtype])


def test_gated_norm_in_place_and_eps(gdn):
    y, z, w = _norm_inputs(300, 128, torch.bfloat16, seed=3)
    yc, zc, wc = y.cuda(), z.cuda(), w.cuda()
    a = gdn.gated_rmsnorm(yc, zc, wc, eps=1e-2)
    b = yc.clone()
    gdn.gated_rmsnorm(b, zc, wc, eps=1e-2, out=b)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    _assert_close(a, oracle.gated_rmsnorm(y, z, w, eps=1e-2), RTOL[torch.bfloat16])
    empty = torch.empty(0, 128, dtype=torch.bfloat16, device="cuda")
    assert gdn.gated_rmsnorm(empty, empty, wc).numel() == 0


def test_gated_norm_on_a_prefill_output(gdn):
    """The norm applied to the headline-shaped prefill output (one layer, all 32 value
    heads of a 4096-token prompt), sampled rows against the oracle."""
    w = workloads.WORKLOADS["next_prefill_T4096_hk16_hv32_d128"]
    d = workloads.workload_inputs(w, device="cuda")
    y, _, _ = gdn.prefill(d["queries"], d["keys"], d["values"], d["decays"], d["beta"])
    g = torch.Generator(device="cuda").manual_seed(11)
    z = torch.randn(y.shape, generator=g, device="cuda").to(y.dtype)
    wt = 1.0 + 0.3 * torch.randn(128, generator=g, device="cuda")
    out = gdn.gated_rmsnorm(y, z, wt)
    torch.cuda.synchronize()
    idx = torch.randint(0, y.shape[1], (64,), generator=torch.Generator().manual_seed(2))
    ys, zs, os_ = (t[0, idx].reshape(-1, 128).cpu() for t in (y, z, out))
    _assert_close(os_, oracle.gated_rmsnorm(ys, zs, wt.cpu()), RTOL[y.dtype])


@pytest.mark.parametrize("D,dtype", [(128, torch.bfloat16), (64, torch.float32), (32, torch.bfloat16)])
def test_fused_decode_norm_matches_oracle(gdn, D, dtype):
    B, HK, HV = 5, 2, 4
    d = workloads.draw_inputs(1, B, HK, HV, D, D, dtype, seed=77 + D)
    args = [d[k][0].contiguous() for k in ("queries", "keys", "values", "decays", "beta")]
    gen = torch.Generator().manual_seed(9)
    s0 = torch.randn(B, HV, D, D, generator=gen) * 0.3
    z = (torch.randn(B, HV, D, generator=gen) * 2.0).to(dtype)
    wt = 1.0 + 0.3 * torch.randn(D, generator=gen)
    st_gated, st_plain = s0.cuda(), s0.cuda()
    cu = [a.cuda() for a in args]
    out = gdn.decode_step(*cu, st_gated, gate=z.cuda(), norm_weight=wt.cuda())
    gdn.decode_step(*cu, st_plain)
    torch.cuda.synchronize()
    y_ref, s_ref = oracle.decode_step(*args, s0.double().numpy())
    ref = oracle.gated_rmsnorm(y_ref, z, wt)
    gate = np.abs(wt.double().numpy() * (z.double() * torch.sigmoid(z.double())).numpy())
    _assert_close(out, ref, RTOL[dtype], extra=1e-3 * gate)
    assert torch.equal(st_gated, st_plain)              # the norm leaves the state step alone
    assert_states_close(st_gated, s_ref, "state")


def _norm_bound(y_ref, z, wt, rtol, ytol):
    """Per element: rtol |ref| plus the rule's output bound ytol on y carried through the
    norm (|weight silu(z)| ytol / rms(y))."""
    zz = z.double().cpu().numpy() if hasattr(z, "cpu") else z
    gate = np.abs(wt.double().cpu().numpy() * zz / (1 + np.exp(-zz)))
    rms = np.sqrt((y_ref ** 2).mean(-1, keepdims=True))
    return ytol * gate / np.maximum(rms, 1e-3)


@pytest.mark.parametrize("D,dtype", [(128, torch.bfloat16), (32, torch.float32)])
def test_fused_prefill_norm_matches_oracle(gdn, D, dtype):
    """gdn_prefill_gated (the prefill, then the norm over its output in place) on the
    tensor-core and the CUDA-core shapes, against the oracle's norm of the oracle's y; the
    final state is the ungated prefill's, bit for bit."""
    B, T, HK, HV = 2, 130, 2, 4
    d = workloads.draw_inputs(B, T, HK, HV, D, D, dtype, seed=61 + D, init_state_std=0.02)
    g = torch.Generator().manual_seed(62)
    z = (torch.randn(B, T, HV, D, generator=g) * 2.0).to(dtype)
    wt = 1.0 + 0.3 * torch.randn(D, generator=g)
    c = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    args = [c[k] for k in ("queries", "keys", "values", "decays", "beta")]
    out, fin, _ = gdn.prefill(*args, c["initial_state"], gate=z.cuda(), norm_weight=wt.cuda())
    y, fin0, _ = gdn.prefill(*args, c["initial_state"])
    torch.cuda.synchronize()
    assert torch.equal(fin, fin0)
    y_ref, _, _ = oracle.forward(d["queries"], d["keys"], d["values"], d["decays"], d["beta"],
                                 d["initial_state"])
    ref = oracle.gated_rmsnorm(y_ref, z, wt)
    ytol = 2e-2 if dtype == torch.bfloat16 else 1e-4
    _assert_close(out, ref, RTOL[dtype], extra=_norm_bound(y_ref, z, wt, RTOL[dtype], ytol))


def test_fused_prefill_norm_packed_sequences(gdn):
    """gdn_prefill_varlen_gated over packed sequences (one shorter than a chunk, one
    ragged over three chunks, one empty) with initial states, against the oracle."""
    lens = [10, 0, 150, 64]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T = int(cu[-1])
    d = workloads.draw_inputs(1, T, 2, 4, 128, 128, torch.bfloat16, 63, init_state_std=0.02,
                              n_states=len(lens))
    g = torch.Generator().manual_seed(64)
    z = torch.randn(1, T, 4, 128, generator=g).to(torch.bfloat16)
    wt = 1.0 + 0.3 * torch.randn(128, generator=g)
    c = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    cu_d = torch.from_numpy(cu).cuda()
    out, fin, _ = gdn.prefill_varlen(c["queries"], c["keys"], c["values"], c["decays"], c["beta"],
                                     cu_d, c["initial_state"], gate=z.cuda(), norm_weight=wt.cuda())
    _, fin0, _ = gdn.prefill_varlen(c["queries"], c["keys"], c["values"], c["decays"], c["beta"],
                                    cu_d, c["initial_state"])
    torch.cuda.synchronize()
    assert torch.equal(fin, fin0)
    y_ref, _, _ = oracle.forward(d["queries"], d["keys"], d["values"], d["decays"], d["beta"],
                                 d["initial_state"], cu_seqlens=cu)
    ref = oracle.gated_rmsnorm(y_ref, z, wt)
    _assert_close(out, ref, RTOL[torch.bfloat16],
                  extra=_norm_bound(y_ref, z, wt, RTOL[torch.bfloat16], 2e-2))


def test_fused_prefill_norm_at_qwen3_next_shape(gdn):
    """The headline-shaped prompt (4096 tokens, 16/32 heads) through gdn_prefill_gated:
    sampled value heads against the oracle, and every head bit for bit against the two
    calls it stands for (prefill, then the norm kernel)."""
    w = workloads.WORKLOADS["next_prefill_T4096_hk16_hv32_d128"]
    d = workloads.workload_inputs(w, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(65)
    z = torch.randn(1, w.T, w.HV, 128, generator=g, device="cuda").to(torch.bfloat16)
    wt = 1.0 + 0.3 * torch.randn(128, generator=g, device="cuda")
    args = [d[k] for k in ("queries", "keys", "values", "decays", "beta")]
    out, fin, _ = gdn.prefill(*args, gate=z, norm_weight=wt)
    y, fin0, _ = gdn.prefill(*args)
    unfused = gdn.gated_rmsnorm(y, z, wt)
    torch.cuda.synchronize()
    assert torch.equal(fin, fin0)
    assert torch.equal(out, unfused)
    chains = oracle_chains({k: v.cpu() if isinstance(v, torch.Tensor) else v for k, v in d.items()},
                           [(0, h) for h in (0, 17, 31)])
    zc = z[0].cpu()
    for (s, h), (o_r, _, _) in chains.items():
        ref = oracle.gated_rmsnorm(o_r, zc[:, h], wt.cpu())
        _assert_close(out[0, :, h], ref, RTOL[torch.bfloat16],
                      extra=_norm_bound(o_r, zc[:, h], wt, RTOL[torch.bfloat16], 2e-2),
                      what=f"head {h}")
