"""GPU parity of the one-token decode step (gdn_decode_step) against the fp64 oracle."""
import pytest
import torch

import workloads
from parity import assert_out_close, assert_states_close, oracle_chains

pytestmark = pytest.mark.gpu
import oracle  # noqa: E402


@pytest.fixture(scope="module")
def gdn():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gated_deltanet_mixer_delta_gb300 as m
    m.build.build()
    m.load_library()
    return m


@pytest.mark.parametrize("D,dtype", [(128, torch.bfloat16), (64, torch.bfloat16),
                                     (32, torch.float32), (128, torch.float32)])
def test_decode_steps_match_oracle(gdn, D, dtype):
    steps, B, HK, HV = 6, 3, 2, 4
    d = workloads.draw_inputs(steps, B, HK, HV, D, D, dtype, seed=31 + D)
    s0 = torch.randn(B, HV, D, D, generator=torch.Generator().manual_seed(5)) * 0.3
    state = s0.cuda()
    s_ref = s0.double().numpy()
    for i in range(steps):
        args = [d[k][i].contiguous() for k in ("queries", "keys", "values", "decays", "beta")]
        out = gdn.decode_step(*[a.cuda() for a in args], state)
        o_ref, s_ref = oracle.decode_step(*args, s_ref)
        torch.cuda.synchronize()
        assert_out_close(out, o_ref, dtype, f"step {i}")
        assert_states_close(state, s_ref, f"state after step {i}")


def test_decode_special_cases(gdn):
    """beta = 0 and g = 0 leave the state unchanged; g = -1e4 with a zero state gives
    o = beta (q~.k^) v (the closed forms the oracle is pinned to)."""
    B, HK, HV, D = 2, 1, 2, 128
    d = workloads.draw_inputs(1, B, HK, HV, D, D, torch.bfloat16, seed=41)
    q, k, v = (d[n][0].cuda() for n in ("queries", "keys", "values"))
    s0 = torch.randn(B, HV, D, D, device="cuda") * 0.1
    st = s0.clone()
    z = torch.zeros(B, HV, device="cuda")
    gdn.decode_step(q, k, v, z, z, st)
    assert torch.equal(st, s0)
    st = s0.clone()
    beta = d["beta"][0].cuda()
    out = gdn.decode_step(q, k, v, torch.full_like(z, -1e4), beta, st)
    o_ref, s_ref = oracle.decode_step(q.cpu(), k.cpu(), v.cpu(), torch.full((B, HV), -1e4),
                                      beta.cpu(), torch.zeros(B, HV, D, D))
    torch.cuda.synchronize()
    assert_out_close(out, o_ref, torch.bfloat16)
    assert_states_close(st, s_ref)


def test_decode_workload_128_steps(gdn):
    """B=256, 16 key / 32 value heads at 128x128, state [256,32,128,128] fp32 ~N(0,0.02),
    128 steps in place.  Checked on sampled chains against the oracle over all 128 tokens
    and, for every chain, against a prefill of the same 128 tokens from the same state."""
    w = workloads.WORKLOADS["decode_B256_hk16_hv32_d128"]
    d = workloads.decode_inputs(w, device="cuda")
    S = d["queries"].shape[0]
    state = d["initial_state"].clone()
    outs = []
    for i in range(S):
        outs.append(gdn.decode_step(d["queries"][i], d["keys"][i], d["values"][i],
                                    d["decays"][i], d["beta"][i], state))
    out = torch.stack(outs, 1)                         # [B, S, HV, D]
    torch.cuda.synchronize()
    # as a batch of prompts: [B, S, ...]
    seq = {n: d[n].transpose(0, 1).contiguous() for n in ("queries", "keys", "values", "decays", "beta")}
    seq["initial_state"] = d["initial_state"]
    o_pf, f_pf, _ = gdn.prefill(seq["queries"], seq["keys"], seq["values"], seq["decays"],
                                seq["beta"], seq["initial_state"])
    assert_out_close(out, o_pf.float(), torch.bfloat16, "decode vs prefill")
    assert_states_close(state, f_pf.cpu().double().numpy(), "decode vs prefill state")
    chains = [(0, 0), (17, 5), (100, 31), (255, 16), (128, 1), (63, 30)]
    ref = oracle_chains(seq, chains)
    for (b, h), (o_r, f_r, _) in ref.items():
        assert_out_close(out[b, :, h], o_r, torch.bfloat16, f"chain {(b, h)}")
        assert_states_close(state[b, h], f_r, f"chain {(b, h)}")
