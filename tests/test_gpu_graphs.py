"""The prefill, the packed prefill and the decode step captured in one CUDA graph.

Every one of these calls is ordered on the caller's stream, allocates nothing and waits
for nothing on the host, so a serving loop can capture a whole step (prefill of a prompt,
then decode steps that continue its state) and replay it.  Replays must give the same
bits as direct calls, replay after replay.
"""
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gdn():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gated_deltanet_mixer_delta_gb300 as m
    m.build.build()
    m.load_library()
    return m


def _cuda(d):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}


def test_prefill_and_decode_replayed_from_a_cuda_graph(gdn):
    names = ("queries", "keys", "values", "decays", "beta")
    # equal-length batch: 2 x 150 tokens (chunks of 64, 64, 22), 2 key / 4 value heads
    d = _cuda(workloads.draw_inputs(2, 150, 2, 4, 128, 128, torch.bfloat16, 91,
                                    init_state_std=0.02))
    # packed batch: lengths 70, 0, 5 (a zero-length sequence keeps its initial state)
    lens = [70, 0, 5]
    p = _cuda(workloads.draw_inputs(1, sum(lens), 2, 4, 128, 128, torch.bfloat16, 93,
                                    init_state_std=0.02, n_states=len(lens)))
    cu = torch.tensor([0, 70, 70, 75], dtype=torch.int32, device="cuda")
    # one decode token per sequence of the batch
    n = workloads.draw_inputs(1, 2, 2, 4, 128, 128, torch.bfloat16, 92)
    step = [n[k][0].cuda() for k in names]

    # direct calls
    out_ref, fin_ref, _ = gdn.prefill(*(d[k] for k in names), d["initial_state"])
    o_ref = gdn.decode_step(*step, fin_ref)              # fin_ref continues in place
    pout_ref, pfin_ref, _ = gdn.prefill_varlen(*(p[k] for k in names), cu, p["initial_state"])
    torch.cuda.synchronize()

    # the same work captured once, outputs preallocated
    out, fin, o = torch.empty_like(out_ref), torch.empty_like(fin_ref), torch.empty_like(o_ref)
    pout, pfin = torch.empty_like(pout_ref), torch.empty_like(pfin_ref)
    ws = torch.empty(gdn.workspace_size(2 * 150, 2, 4, 128, 128), dtype=torch.uint8, device="cuda")
    pws = torch.empty(gdn.workspace_size(sum(lens), len(lens), 4, 128, 128), dtype=torch.uint8,
                      device="cuda")
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        gdn.prefill(*(d[k] for k in names), d["initial_state"], out=out, final_state=fin,
                    workspace=ws)
        gdn.decode_step(*step, fin, out=o)
        gdn.prefill_varlen(*(p[k] for k in names), cu, p["initial_state"], out=pout,
                           final_state=pfin, workspace=pws)
    for _ in range(3):
        for t in (out, fin, o, pout, pfin):
            t.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, out_ref) and torch.equal(fin, fin_ref) and torch.equal(o, o_ref)
        assert torch.equal(pout, pout_ref) and torch.equal(pfin, pfin_ref)
        assert gdn.workspace_status(pws) == 0
