"""The tensor-core prefill with its prep running beside the chain.  When an equal-length
batch's chains (one CTA per (sequence, value head, 32-wide value slice)) leave enough SMs
free, the prep grid is persistent: its CTAs on the SMs the chain does not need produce the
per-chunk records in chunk order and set a ready flag per record, and the chain kernel
starts at once, taking each record when its flag is set.  A packed batch always runs the
prep first, one CTA per item, and the chain after it.  The arithmetic of every step is the
same, so the two schedules must agree bit for bit; both are checked against the fp64
oracle too.  The workspace header tells which schedule ran: word 4 counts the prep CTAs
that stayed beside the chain (zero when the prep ran first)."""
import pytest
import torch

import workloads
from parity import assert_out_close, assert_states_close

pytestmark = pytest.mark.gpu
import oracle  # noqa: E402  (test infrastructure)

STAY_WORD = 4


@pytest.fixture(scope="module")
def gdn():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gated_deltanet_mixer_delta_gb300 as m
    m.build.build()
    m.load_library()
    return m


def _run_both(gdn, B, T, HK, HV, seed):
    d = workloads.draw_inputs(B, T, HK, HV, 128, 128, torch.bfloat16, seed, init_state_std=0.02)
    g = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    ws = torch.empty(gdn.workspace_size(B * T, B, HV, 128, 128, dtype=torch.bfloat16),
                     dtype=torch.uint8, device="cuda")
    out, fin, _ = gdn.prefill(g["queries"], g["keys"], g["values"], g["decays"], g["beta"],
                              g["initial_state"], workspace=ws)
    torch.cuda.synchronize()
    stayed = int(ws[:64].view(torch.int32)[STAY_WORD])
    # the same sequences as one packed batch: the prep runs first
    flat = lambda x: x.reshape(1, B * T, *x.shape[2:]).contiguous()
    cu = torch.arange(0, B * T + 1, T, dtype=torch.int32, device="cuda")
    pout, pfin, _ = gdn.prefill_varlen(flat(g["queries"]), flat(g["keys"]), flat(g["values"]),
                                       flat(g["decays"]), flat(g["beta"]), cu,
                                       g["initial_state"], workspace=ws)
    torch.cuda.synchronize()
    return d, out, fin, pout.reshape(out.shape), pfin, stayed


@pytest.mark.parametrize("B,T,HK,HV", [(1, 1000, 16, 16), (2, 700, 2, 4), (1, 64 * 9 + 17, 4, 12)])
def test_prep_beside_chain_matches_packed_run_and_oracle(gdn, B, T, HK, HV):
    d, out, fin, pout, pfin, stayed = _run_both(gdn, B, T, HK, HV, 900 + B + HV)
    assert stayed > 0, "the prep did not run beside the chain"
    assert torch.equal(out, pout) and torch.equal(fin, pfin)
    o_ref, f_ref, _ = oracle.forward(d["queries"], d["keys"], d["values"], d["decays"], d["beta"],
                                     d["initial_state"])
    assert_out_close(out, o_ref, torch.bfloat16)
    assert_states_close(fin, f_ref)


def test_prep_first_where_the_chain_fills_the_gpu(gdn):
    """32 value heads: 128 chain CTAs leave too few SMs for the prep to keep ahead, so it
    runs first (no CTA stays); the result is the same either way."""
    if torch.cuda.get_device_properties(0).multi_processor_count > 200:
        pytest.skip("more SMs than the schedule this checks assumes")
    _, out, fin, pout, pfin, stayed = _run_both(gdn, 1, 640, 16, 32, 907)
    assert stayed == 0
    assert torch.equal(out, pout) and torch.equal(fin, pfin)


def test_repeated_calls_reuse_the_flags(gdn):
    """The ready flags and claim counters start from zero on every call (a reused workspace
    holds the last call's flags): a second call on new inputs must not take stale records."""
    d1 = workloads.draw_inputs(1, 900, 8, 8, 128, 128, torch.bfloat16, 931)
    d2 = workloads.draw_inputs(1, 900, 8, 8, 128, 128, torch.bfloat16, 932)
    ws = torch.empty(gdn.workspace_size(900, 1, 8, 128, 128, dtype=torch.bfloat16),
                     dtype=torch.uint8, device="cuda")
    outs = []
    for d in (d1, d2):
        g = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
        o, f, _ = gdn.prefill(g["queries"], g["keys"], g["values"], g["decays"], g["beta"], None,
                              workspace=ws)
        outs.append((o, f))
    torch.cuda.synchronize()
    for d, (o, f) in zip((d1, d2), outs):
        o_ref, f_ref, _ = oracle.forward(d["queries"], d["keys"], d["values"], d["decays"],
                                         d["beta"], None)
        assert_out_close(o, o_ref, torch.bfloat16)
        assert_states_close(f, f_ref)
