"""GPU parity of the step before the rule (gdn_conv_gate_prologue: causal depthwise conv
of width 4 + SiLU over the cat(q, k, v) channels, beta = sigmoid(b),
g = -exp(A_log) softplus(a + dt_bias)) in both projection layouts against the fp64 oracle.

Tolerances, from the arithmetic: the kernel sums four fp32 products and applies expf /
log1pf, ~1e-6 relative to the sum of the terms' magnitudes (inputs O(1): 1e-5 absolute
covers it); a bf16 output adds its rounding, at most 2^-8 relative."""
import numpy as np
import pytest
import torch

import workloads
from parity import assert_out_close, assert_states_close, oracle_chains

pytestmark = pytest.mark.gpu
import oracle  # noqa: E402

RTOL = {torch.float32: 1e-5, torch.bfloat16: 4e-3}


@pytest.fixture(scope="module")
def gdn():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gated_deltanet_mixer_delta_gb300 as m
    m.build.build()
    m.load_library()
    return m


def _close(got, ref, rtol, atol=1e-5, what=""):
    got = got.double().cpu().numpy()
    err = np.abs(got - ref)
    bound = rtol * np.abs(ref) + atol
    i = np.unravel_index(np.argmax(err - bound), err.shape)
    assert np.all(err <= bound), f"{what}: err {err[i]:.3g} > {bound[i]:.3g} at {i}"


def _params(HK, HV, D, seed, dtype, layout, B, T, with_state):
    g = torch.Generator().manual_seed(seed)
    C = 2 * HK * D + HV * D
    r = HV // HK
    W = C if layout == "qkv" else HK * (2 * D + 2 * r * D)
    proj = torch.randn(B, T, W, generator=g).to(dtype)
    if layout == "qkv":
        pb = torch.randn(B, T, HV, generator=g).mul(2).to(dtype)
        pa = torch.randn(B, T, HV, generator=g).mul(2).to(dtype)
    else:
        pb = torch.randn(B, T, 2 * HV, generator=g).mul(2).to(dtype)
        pa = None
    w = torch.randn(C, 4, generator=g) * 0.5
    al = torch.randn(HV, generator=g) * 0.5
    db = torch.randn(HV, generator=g) * 0.5
    st = torch.randn(B, 3, C, generator=g).to(dtype) if with_state else None
    return proj, pb, pa, w, al, db, st


def _oracle(proj, pb, pa, w, al, db, st, HK, HV, D, layout, cu=None):
    if layout == "qkv":
        x, b, a = proj, pb, pa
        z = None
    else:
        q, k, v, z, b, a = oracle.regroup_qkvz(proj, pb, HK, HV, D, D)
        lead = q.shape[:-2]
        x = np.concatenate([q.reshape(*lead, -1), k.reshape(*lead, -1), v.reshape(*lead, -1)], -1)
    y, beta, g, so = oracle.conv_gate(x, b, a, w, al, db, conv_state=st, cu_seqlens=cu,
                                      want_state=True)
    q, k, v = oracle.split_qkv(y, HK, HV, D, D)
    return dict(queries=q, keys=k, values=v, beta=beta, decays=g, z=z, state=so)


def _cuda(*ts):
    return [None if t is None else t.cuda() for t in ts]


@pytest.mark.parametrize("layout", ["qkv", "qkvz"])
@pytest.mark.parametrize("HK,HV,D,dtype", [(2, 4, 128, torch.bfloat16), (2, 6, 64, torch.bfloat16),
                                            (1, 2, 32, torch.float32), (3, 3, 128, torch.bfloat16)])
@pytest.mark.parametrize("with_state", [False, True])
def test_prologue_matches_oracle(gdn, layout, HK, HV, D, dtype, with_state):
    B, T = 2, 70                                   # 70 tokens: full 8-token tiles and a tail
    proj, pb, pa, w, al, db, st = _params(HK, HV, D, 5 + HV + D, dtype, layout, B, T, with_state)
    C = 2 * HK * D + HV * D
    so = torch.full((B, 3, C), 7.0, dtype=dtype, device="cuda")
    cp, cb, ca, cw, cal, cdb, cst = _cuda(proj, pb, pa, w, al, db, st)
    out = gdn.conv_gate_prologue(cp, cb, ca, cw, cal, cdb, HK=HK, HV=HV, Dk=D, Dv=D, layout=layout,
                                 conv_state=cst, conv_state_out=so)
    torch.cuda.synchronize()
    ref = _oracle(proj, pb, pa, w, al, db, st, HK, HV, D, layout)
    for key in ("queries", "keys", "values"):
        _close(out[key], ref[key], RTOL[dtype], what=key)
    for key in ("beta", "decays"):
        _close(out[key], ref[key], 1e-5, 1e-6, what=key)
    assert np.array_equal(so.double().cpu().numpy(), ref["state"])     # a copy of inputs
    if layout == "qkvz":
        assert np.array_equal(out["z"].double().cpu().numpy(), ref["z"])


@pytest.mark.parametrize("layout", ["qkv", "qkvz"])
def test_prologue_packed_sequences_and_in_place_state(gdn, layout):
    """Packed sequences (some shorter than the window, one empty, one spanning several
    tiles) with their own carried conv states, the states updated in place; against the
    oracle and bitwise against separate calls."""
    HK, HV, D, dtype = 2, 4, 128, torch.bfloat16
    lens = [40, 1, 2, 0, 33, 5]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T = int(cu[-1])
    proj, pb, pa, w, al, db, _ = _params(HK, HV, D, 17, dtype, layout, 1, T, False)
    C = 2 * HK * D + HV * D
    st = torch.randn(len(lens), 3, C, generator=torch.Generator().manual_seed(18)).to(dtype)
    cp, cb, ca, cw, cal, cdb, cst = _cuda(proj, pb, pa, w, al, db, st)
    st_before = cst.clone()
    out = gdn.conv_gate_prologue(cp, cb, ca, cw, cal, cdb, HK=HK, HV=HV, Dk=D, Dv=D, layout=layout,
                                 conv_state=cst, conv_state_out=cst,
                                 cu_seqlens=torch.from_numpy(cu).cuda())
    torch.cuda.synchronize()
    ref = _oracle(proj, pb, pa, w, al, db, st, HK, HV, D, layout, cu=cu)
    for key in ("queries", "keys", "values"):
        _close(out[key], ref[key], RTOL[dtype], what=key)
    assert np.array_equal(cst.double().cpu().numpy(), ref["state"])
    for s in range(len(lens)):
        a, b = int(cu[s]), int(cu[s + 1])
        if a == b:
            continue
        # fresh (16-byte aligned) copies of the sequence's rows
        one = gdn.conv_gate_prologue(cp[:, a:b].clone(), cb[:, a:b].clone(),
                                     None if ca is None else ca[:, a:b].clone(),
                                     cw, cal, cdb, HK=HK, HV=HV, Dk=D, Dv=D, layout=layout,
                                     conv_state=st_before[s:s + 1].clone())
        for key in ("queries", "values", "decays") + (("z",) if layout == "qkvz" else ()):
            assert torch.equal(one[key][0], out[key][0, a:b])


def test_prologue_decode_steps_equal_one_pass(gdn):
    """T decode steps (N sequences of one token, the conv state carried in place) give
    bit for bit the outputs and the final state of one pass over the T tokens."""
    HK, HV, D, dtype, B, T = 2, 4, 128, torch.bfloat16, 3, 9
    proj, pb, pa, w, al, db, st = _params(HK, HV, D, 21, dtype, "qkvz", B, T, True)
    cp, cb, _, cw, cal, cdb, cst = _cuda(proj, pb, pa, w, al, db, st)
    C = 2 * HK * D + HV * D
    full_state = torch.empty(B, 3, C, dtype=dtype, device="cuda")
    full = gdn.conv_gate_prologue(cp, cb, None, cw, cal, cdb, HK=HK, HV=HV, Dk=D, Dv=D,
                                  layout="qkvz", conv_state=cst, conv_state_out=full_state)
    state = cst.clone()
    for t in range(T):
        o = gdn.conv_gate_prologue(cp[:, t:t + 1].clone(), cb[:, t:t + 1].clone(), None,
                                   cw, cal, cdb, HK=HK, HV=HV, Dk=D, Dv=D, layout="qkvz",
                                   conv_state=state, conv_state_out=state)
        for key in ("queries", "keys", "values", "z", "beta", "decays"):
            assert torch.equal(o[key][:, 0], full[key][:, t]), (key, t)
    assert torch.equal(state, full_state)


def test_mixer_core_at_qwen3_next_shape(gdn):
    """The fused projections of a 4096-token prompt at the Qwen3-Next shape through the
    prologue (regroup, conv, gates), the chunked rule and the gated norm.  Each step is
    held to the oracle of that step on the inputs the GPU gave it (the rule's inputs are
    bf16 tensors: an fp64 prologue would hand the rule other values): the prologue on
    every token and channel, the rule and the norm on sampled value heads."""
    w = workloads.WORKLOADS["next_prefill_T4096_hk16_hv32_d128"]
    HK, HV, D, T = w.HK, w.HV, w.Dk, w.T
    proj, pb, _, cw, al, db, _ = _params(HK, HV, D, 23, torch.bfloat16, "qkvz", 1, T, False)
    cp, cb, cw_, cal, cdb = _cuda(proj, pb, cw, al, db)
    pro = gdn.conv_gate_prologue(cp, cb, None, cw_, cal, cdb, HK=HK, HV=HV, Dk=D, Dv=D,
                                 layout="qkvz")
    y, fin, _ = gdn.prefill(pro["queries"], pro["keys"], pro["values"], pro["decays"], pro["beta"])
    nw = (1.0 + 0.3 * torch.randn(D, generator=torch.Generator().manual_seed(3))).cuda()
    out = gdn.gated_rmsnorm(y, pro["z"], nw)
    torch.cuda.synchronize()
    ref = _oracle(proj, pb, None, cw, al, db, None, HK, HV, D, "qkvz")
    for key in ("queries", "keys", "values"):
        _close(pro[key], ref[key], RTOL[torch.bfloat16], what=key)
    for key in ("beta", "decays"):
        _close(pro[key], ref[key], 1e-5, 1e-6, what=key)
    d = {k: pro[k].cpu() for k in ("queries", "keys", "values", "decays", "beta")}
    d["initial_state"] = None
    heads = (0, 1, 31)
    chains = oracle_chains(d, [(0, h) for h in heads])
    zc = pro["z"][0].double().cpu().numpy()
    silu = lambda x: x / (1 + np.exp(-x))
    for (s, h), (o_r, f_r, _) in chains.items():
        assert_out_close(y[0, :, h], o_r, torch.bfloat16, f"head {h}")
        assert_states_close(fin[0, h], f_r, f"head {h}")
        nr = oracle.gated_rmsnorm(o_r, zc[:, h], nw.cpu())
        gate = np.abs(nw.double().cpu().numpy() * silu(zc[:, h]))
        yr = np.sqrt((o_r ** 2).mean(-1, keepdims=True))
        # the rule's 2e-2 output bound on y, carried through the norm, plus bf16 rounding
        extra = 2e-2 * gate / np.maximum(yr, 1e-3)
        _close(out[0, :, h], nr, 4e-3, 1e-5 + extra, what=f"norm head {h}")
