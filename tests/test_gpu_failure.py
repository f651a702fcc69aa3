"""Failure handling on the GPU without a fault: the bounded waits of the tensor-core
kernels give up after their limit and report GDN_ERR_TIMEOUT instead of hanging, and the
context stays usable afterwards.  The wait that runs out is on an mbarrier phase that
nothing completes (gdn_selftest_wait_timeout), with a 2 ms limit."""
import pytest
import torch

import workloads
from parity import assert_out_close, assert_states_close

pytestmark = pytest.mark.gpu
import oracle  # noqa: E402  (test infrastructure)

GDN_ERR_TIMEOUT = -6


@pytest.fixture(scope="module")
def gdn():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gated_deltanet_mixer_delta_gb300 as m
    m.build.build()
    m.load_library()
    return m


def test_wait_without_arrival_times_out(gdn):
    status, waited_us = gdn.selftest_wait_timeout(2_000_000)
    assert status == GDN_ERR_TIMEOUT
    assert 2000 <= waited_us < 1_000_000


def test_context_usable_after_a_timeout(gdn):
    gdn.selftest_wait_timeout(1_000_000)
    d = workloads.draw_inputs(1, 130, 2, 4, 128, 128, torch.bfloat16, 91, init_state_std=0.02)
    g = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    out, fin, _ = gdn.prefill(g["queries"], g["keys"], g["values"], g["decays"], g["beta"],
                              g["initial_state"])
    torch.cuda.synchronize()
    o_ref, f_ref, _ = oracle.forward(d["queries"], d["keys"], d["values"], d["decays"], d["beta"],
                                     d["initial_state"])
    assert_out_close(out, o_ref, torch.bfloat16)
    assert_states_close(fin, f_ref, "final_state")
