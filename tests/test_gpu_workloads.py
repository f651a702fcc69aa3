"""GPU parity at the full sizes of the named workloads, in the launch configuration the
bench times.  Where the oracle can run every chain in seconds it does; otherwise it
checks sampled (sequence, value head) chains over all of their tokens."""
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
    all final states' chains for 3 heads of every sequence, outputs on the same chains."""
    w = W["varlen8_512to8192_hk16_hv32_d128"]
    d = workloads.workload_inputs(w, device="cuda")
    T = d["queries"].shape[1]
    out, fin, _ = gdn.prefill_varlen(d["queries"], d["keys"], d["values"], d["decays"], d["beta"],
                                     d["cu_seqlens"], d["initial_state"],
                                     workspace=_ws(gdn, T, w.n_seqs, w))
    torch.cuda.synchronize()
    cu = d["cu_seqlens"].cpu()
    chains = [(s, h) for s in range(w.n_seqs) for h in (0, 13, 31)]
    ref = oracle_chains(d, chains, cu=cu)
    for (s, h), (o_r, f_r, _) in ref.items():
        a, b = int(cu[s]), int(cu[s + 1])
        assert_out_close(out[0, a:b, h], o_r, torch.bfloat16, f"seq {s} head {h}")
        assert_states_close(fin[s, h], f_r, f"seq {s} head {h}")


def test_long_prefill_T65536(gdn):
    """B=2, T=65536, g = -softplus(N(0,1)) - 0.01: sampled chains over all 65536 tokens."""
    w = W["long_prefill_B2_T65536_hk16_hv32_d128"]
    d = workloads.workload_inputs(w, device="cuda")
    out, fin, _ = gdn.prefill(d["queries"], d["keys"], d["values"], d["decays"], d["beta"],
                              workspace=_ws(gdn, w.B * w.T, w.B, w))
    torch.cuda.synchronize()
    chains = [(0, 0), (0, 31), (1, 6), (1, 17)]
    ref = oracle_chains(d, chains)
    for (b, h), (o_r, f_r, _) in ref.items():
        assert_out_close(out[b, :, h], o_r, torch.bfloat16, f"chain {(b, h)}")
        assert_states_close(fin[b, h], f_r, f"chain {(b, h)}")


def test_per_token_states_B4_T1024(gdn):
    """B=4, T=1024, states [4,1024,32,128,128] fp32 (8 GiB): sampled chains' per-token
    states against the oracle; the last state of every chain equals final_state."""
    w = W["states_B4_T1024_hk16_hv32_d128"]
    d = workloads.workload_inputs(w, device="cuda")
    out, fin, st = gdn.prefill(d["queries"], d["keys"], d["values"], d["decays"], d["beta"],
                               output_states=True, workspace=_ws(gdn, w.B * w.T, w.B, w))
    torch.cuda.synchronize()
    assert st.shape == (4, 1024, 32, 128, 128)
    assert torch.equal(st[:, -1], fin)
    chains = [(0, 0), (1, 9), (2, 30), (3, 15)]
    ref = oracle_chains(d, chains, want_states=True)
    for (b, h), (o_r, f_r, s_r) in ref.items():
        assert_out_close(out[b, :, h], o_r, torch.bfloat16, f"chain {(b, h)}")
        assert_states_close(st[b, :, h], s_r, f"states of chain {(b, h)}")
        assert_states_close(fin[b, h], f_r, f"chain {(b, h)}")


@pytest.mark.parametrize("name,heads", [
    ("qwen35_27b_prefill_T4096_hk16_hv48_d128", (0, 1, 2, 25, 46, 47)),
    ("qwen35_0p8b_prefill_T4096_hk16_hv16_d128", (0, 7, 15)),
])
def test_other_head_layouts_T4096(gdn, name, heads):
    """Head layouts of other sizes of the family (three value heads per key head on 27B,
    one on 0.8B), T=4096: sampled value heads (all three of key head 0 on 27B) against
    the oracle over every token."""
    w = W[name]
    d = workloads.workload_inputs(w, device="cuda")
    out, fin, _ = gdn.prefill(d["queries"], d["keys"], d["values"], d["decays"], d["beta"],
                              workspace=_ws(gdn, w.T, 1, w))
    torch.cuda.synchronize()
    ref = oracle_chains(d, [(0, h) for h in heads])
    for (s, h), (o_r, f_r, _) in ref.items():
        assert_out_close(out[0, :, h], o_r, torch.bfloat16, f"head {h}")
        assert_states_close(fin[0, h], f_r, f"head {h}")
