"""GPU parity at the full sizes of the named workloads, in the launch configuration the
bench times: every (sequence, value head) chain against the fp64 oracle over all of its
tokens (the oracle runs chains in parallel on the host cores; large workloads go in
batches of chains so the fp64 references stay small)."""
import pytest
import torch

import workloads
from parity import assert_out_close, assert_states_close, oracle_chains

pytestmark = pytest.mark.gpu
import oracle  # noqa: E402

W = workloads.WORKLOADS


@pytest.fixture(scope="module")
def gdn():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gated_deltanet_mixer_delta_gb300 as m
    m.build.build()
    m.load_library()
    return m


def _ws(gdn, T_total, N, w):
    return torch.empty(gdn.workspace_size(T_total, N, w.HV, w.Dk, w.Dv), dtype=torch.uint8,
                       device="cuda")


def _check_chains(out, fin, d, chains, cu=None, batch=64, states=None, what=""):
    """Every listed chain: outputs and final state (and per-token states) against the
    oracle, `batch` chains at a time."""
    d = {k: (v.cpu() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    for i in range(0, len(chains), batch):
        part = chains[i:i + batch]
        ref = oracle_chains(d, part, cu=cu, want_states=states is not None)
        for (s, h), (o_r, f_r, s_r) in ref.items():
            if cu is None:
                o_g = out[s, :, h]
            else:
                o_g = out[0, int(cu[s]):int(cu[s + 1]), h]
            assert_out_close(o_g, o_r, torch.bfloat16, f"{what} chain {(s, h)}")
            assert_states_close(fin[s, h], f_r, f"{what} chain {(s, h)}")
            if states is not None:
                assert_states_close(states[s, :, h], s_r, f"{what} states of chain {(s, h)}")
        del ref


def test_next_prefill_T4096_all_chains(gdn):
    """Qwen3-Next-shaped prefill: B=1, T=4096, 16/32 heads, 128x128, zero initial state.
    Every (head) chain against the oracle."""
    w = W["next_prefill_T4096_hk16_hv32_d128"]
    d = workloads.workload_inputs(w, device="cuda")
    out, fin, _ = gdn.prefill(d["queries"], d["keys"], d["values"], d["decays"], d["beta"],
                              workspace=_ws(gdn, w.T, 1, w))
    torch.cuda.synchronize()
    o_ref, f_ref, _ = oracle.forward(d["queries"].cpu(), d["keys"].cpu(), d["values"].cpu(),
                                     d["decays"].cpu(), d["beta"].cpu())
    assert_out_close(out, o_ref, torch.bfloat16)
    assert_states_close(fin, f_ref)


def test_varlen_8_sequences(gdn):
    """8 packed sequences (lengths U{512..8192}), per-sequence initial states ~N(0,0.02):
    all 256 (sequence, value head) chains."""
    w = W["varlen8_512to8192_hk16_hv32_d128"]
    d = workloads.workload_inputs(w, device="cuda")
    T = d["queries"].shape[1]
    out, fin, _ = gdn.prefill_varlen(d["queries"], d["keys"], d["values"], d["decays"], d["beta"],
                                     d["cu_seqlens"], d["initial_state"],
                                     workspace=_ws(gdn, T, w.n_seqs, w))
    torch.cuda.synchronize()
    cu = d["cu_seqlens"].cpu()
    _check_chains(out, fin, d, [(s, h) for s in range(w.n_seqs) for h in range(w.HV)], cu=cu,
                  what="varlen")


def test_long_prefill_T65536(gdn):
    """B=2, T=65536, g = -softplus(N(0,1)) - 0.01: all 64 chains over all 65536 tokens."""
    w = W["long_prefill_B2_T65536_hk16_hv32_d128"]
    d = workloads.workload_inputs(w, device="cuda")
    out, fin, _ = gdn.prefill(d["queries"], d["keys"], d["values"], d["decays"], d["beta"],
                              workspace=_ws(gdn, w.B * w.T, w.B, w))
    torch.cuda.synchronize()
    _check_chains(out, fin, d, [(b, h) for b in range(w.B) for h in range(w.HV)], batch=16,
                  what="long")


def test_per_token_states_B4_T1024(gdn):
    """B=4, T=1024, states [4,1024,32,128,128] fp32 (8 GiB): every chain's per-token
    states against the oracle (8 chains at a time); the last state of every chain
    equals final_state."""
    w = W["states_B4_T1024_hk16_hv32_d128"]
    d = workloads.workload_inputs(w, device="cuda")
    out, fin, st = gdn.prefill(d["queries"], d["keys"], d["values"], d["decays"], d["beta"],
                               output_states=True, workspace=_ws(gdn, w.B * w.T, w.B, w))
    torch.cuda.synchronize()
    assert st.shape == (4, 1024, 32, 128, 128)
    assert torch.equal(st[:, -1], fin)
    _check_chains(out, fin, d, [(b, h) for b in range(w.B) for h in range(w.HV)], batch=8,
                  states=st, what="states")


@pytest.mark.parametrize("name", ["qwen35_27b_prefill_T4096_hk16_hv48_d128",
                                  "qwen35_0p8b_prefill_T4096_hk16_hv16_d128"])
def test_other_head_layouts_T4096(gdn, name):
    """Head layouts of other sizes of the family (three value heads per key head on 27B,
    one on 0.8B), T=4096: every value head against the oracle over every token."""
    w = W[name]
    d = workloads.workload_inputs(w, device="cuda")
    out, fin, _ = gdn.prefill(d["queries"], d["keys"], d["values"], d["decays"], d["beta"],
                              workspace=_ws(gdn, w.T, 1, w))
    torch.cuda.synchronize()
    _check_chains(out, fin, d, [(0, h) for h in range(w.HV)], what=name)
