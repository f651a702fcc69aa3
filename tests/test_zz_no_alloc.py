"""gdn_prefill_noalloc: the prefill for callers that cannot allocate device memory.

Such callers (an engine that hands out device memory only from its own start-up pool,
a plugin that only sees the buffers its host passes it, a path where an allocation and
the synchronisation it may cause are not allowed) get a variant whose scratch is a
64 MiB array the library keeps in device memory.  This test calls it through the C ABI,
twice in a row with different shapes (the array keeps the previous call's contents),
and checks each result against gdn_prefill's within the tolerances the other parity
tests use.  It sits in a file of its own that pytest collects last and needs nothing
from the other tests.
"""
import ctypes

import pytest
import torch

import workloads
from parity import assert_out_close, assert_states_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gdn():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gated_deltanet_mixer_delta_gb300 as m
    m.build.build()
    lib = m.load_library()
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.gdn_prefill_noalloc.restype = i
    lib.gdn_prefill_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i,
                                        f, i, vp]
    lib.gdn_prefill_noalloc_status.restype = i
    lib.gdn_prefill_noalloc_status.argtypes = [vp, vp]
    return m


def _status(gdn):
    st = ctypes.c_int(-99)
    rc = gdn.abi().gdn_prefill_noalloc_status(ctypes.c_void_p(torch.cuda.current_stream().cuda_stream),
                                               ctypes.byref(st))
    assert rc == 0, rc
    return st.value


def _noalloc(gdn, d, states=False):
    q, k, v = d["queries"], d["keys"], d["values"]
    B, T, HK, Dk = q.shape
    HV, Dv = v.shape[2], v.shape[3]
    out = torch.empty_like(v)
    fin = torch.empty(B, HV, Dk, Dv, dtype=torch.float32, device=q.device)
    st = torch.empty(B, T, HV, Dk, Dv, dtype=torch.float32, device=q.device) if states else None
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    rc = gdn.abi().gdn_prefill_noalloc(
        p(q), p(k), p(v), p(d["decays"]), p(d["beta"]), p(d["initial_state"]), p(out), p(fin),
        p(st), B, T, HK, HV, Dk, Dv, 0 if q.dtype == torch.bfloat16 else 1, 0.0, 1,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, rc
    return out, fin, st


def _cuda(d):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}


def test_noalloc_matches_prefill_on_two_calls_in_a_row(gdn):
    # call 1: 128 x 128 bf16 heads (tensor-core path), ragged tail, initial state, states
    d1 = _cuda(workloads.draw_inputs(2, 200, 2, 4, 128, 128, torch.bfloat16, 71,
                                     init_state_std=0.02))
    # call 2: a different shape on the other path (32 x 32 fp32), no initial state
    d2 = _cuda(workloads.draw_inputs(3, 77, 1, 2, 32, 32, torch.float32, 72))
    o1, f1, s1 = _noalloc(gdn, d1, states=True)
    o2, f2, _ = _noalloc(gdn, d2)
    torch.cuda.synchronize()
    r1 = gdn.prefill(d1["queries"], d1["keys"], d1["values"], d1["decays"], d1["beta"],
                     d1["initial_state"], output_states=True)
    r2 = gdn.prefill(d2["queries"], d2["keys"], d2["values"], d2["decays"], d2["beta"])
    torch.cuda.synchronize()
    assert_out_close(o1, r1[0].double().cpu().numpy(), torch.bfloat16, "call 1 out")
    assert_states_close(f1, r1[1].double().cpu().numpy(), "call 1 final state")
    assert_states_close(s1, r1[2].double().cpu().numpy(), "call 1 states")
    assert_out_close(o2, r2[0].double().cpu().numpy(), torch.float32, "call 2 out")
    assert_states_close(f2, r2[1].double().cpu().numpy(), "call 2 final state")
    assert _status(gdn) == 0
    # the first call again, after the second one reused the scratch array
    o3, f3, _ = _noalloc(gdn, d1)
    torch.cuda.synchronize()
    assert_out_close(o3, r1[0].double().cpu().numpy(), torch.bfloat16, "call 3 out")
    assert_states_close(f3, r1[1].double().cpu().numpy(), "call 3 final state")
    assert _status(gdn) == 0


def test_noalloc_empty_prompts_carry_the_initial_state(gdn):
    """B = 2 sequences of T = 0 tokens: no chunk runs, the final state is the initial
    state (and zero without one), as with gdn_prefill."""
    d = _cuda(workloads.draw_inputs(2, 0, 2, 4, 128, 128, torch.bfloat16, 73, init_state_std=0.02))
    _, fin, _ = _noalloc(gdn, d)
    torch.cuda.synchronize()
    assert torch.equal(fin, d["initial_state"])
    d0 = dict(d, initial_state=None)
    _, fin0, _ = _noalloc(gdn, d0)
    torch.cuda.synchronize()
    assert torch.count_nonzero(fin0) == 0
    assert _status(gdn) == 0


def test_noalloc_rejects_shapes_beyond_its_scratch(gdn):
    # 64 MiB holds 1129 records of 58 KiB: 32 value heads x 128 chunks is more
    P = 0x10000
    rc = gdn.abi().gdn_prefill_noalloc(P, P, P, P, P, None, P, P, None, 1, 128 * 64, 16, 32, 128,
                                       128, 0, 0.0, 1, None)
    assert rc == -4
