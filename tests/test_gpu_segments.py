"""The tensor-core chain kernel's work units on the GPU.  When the (sequence, value head,
value slice) chains outnumber the SMs, each chain is cut into segments of consecutive
chunks.  CTAs claim the segments in segment-major order, and each segment's end state
passes to the CTA that takes the next one.  With 152 SMs, 2 x 32 value heads of 1019
tokens (16 chunks, the last of 59 tokens) make 256 chains of four 4-chunk segments.
Checks: every chain against the fp64 oracle, and bitwise equality with the same
sequences run one per call (128 chains: one unit each, never cut).  The same holds with
the cache updated in place, and with per-token states (512 chains of two 8-chunk
segments at 4 x 32 heads)."""
import pytest
import torch

import workloads
from parity import assert_out_close, assert_states_close, oracle_chains

pytestmark = pytest.mark.gpu
import oracle  # noqa: E402,F401  (test infrastructure)

T = 16 * 64 - 5


@pytest.fixture(scope="module")
def gdn():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gated_deltanet_mixer_delta_gb300 as m
    m.build.build()
    m.load_library()
    return m


def _draw(B, seed):
    d = workloads.draw_inputs(B, T, 16, 32, 128, 128, torch.bfloat16, seed, init_state_std=0.02)
    return d, {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}


def _one_sequence(gdn, g, b, states=False):
    sl = lambda x: x[b:b + 1].contiguous()
    return gdn.prefill(sl(g["queries"]), sl(g["keys"]), sl(g["values"]), sl(g["decays"]),
                       sl(g["beta"]), sl(g["initial_state"]), output_states=states)


def test_segmented_chains_match_oracle(gdn):
    d, g = _draw(2, 610)
    out, fin, _ = gdn.prefill(g["queries"], g["keys"], g["values"], g["decays"], g["beta"],
                              g["initial_state"])
    torch.cuda.synchronize()
    ref = oracle_chains(d, [(s, h) for s in range(2) for h in range(32)])
    for (s, h), (o_r, f_r, _) in ref.items():
        assert_out_close(out[s, :, h], o_r, torch.bfloat16, f"chain {(s, h)}")
        assert_states_close(fin[s, h], f_r, f"chain {(s, h)}")


def test_segments_are_bitwise_the_uncut_chain(gdn):
    """The hand-off is an exact fp32 copy of the state and every chunk does the same
    arithmetic, so cutting a chain changes no bit of its outputs or final state."""
    _, g = _draw(2, 611)
    out, fin, _ = gdn.prefill(g["queries"], g["keys"], g["values"], g["decays"], g["beta"],
                              g["initial_state"])
    for b in range(2):
        ob, fb, _ = _one_sequence(gdn, g, b)
        assert torch.equal(ob[0], out[b]) and torch.equal(fb[0], fin[b])
    # and the same call twice: the CTAs that take each segment differ, the bits do not
    out2, fin2, _ = gdn.prefill(g["queries"], g["keys"], g["values"], g["decays"], g["beta"],
                                g["initial_state"])
    assert torch.equal(out, out2) and torch.equal(fin, fin2)


def test_segmented_chains_with_the_cache_in_place(gdn):
    """final_state = initial_state: a chain's first segment reads the initial slice before
    any segment of that chain writes it, and the hand-offs go through the same buffer."""
    _, g = _draw(2, 612)
    ref_out, ref_fin, _ = gdn.prefill(g["queries"], g["keys"], g["values"], g["decays"], g["beta"],
                                      g["initial_state"].clone())
    cache = g["initial_state"].clone()
    out, fin, _ = gdn.prefill(g["queries"], g["keys"], g["values"], g["decays"], g["beta"],
                              cache, final_state=cache)
    assert fin.data_ptr() == cache.data_ptr()
    assert torch.equal(out, ref_out) and torch.equal(cache, ref_fin)


def test_segmented_chains_with_per_token_states(gdn):
    """Per-token states: a segment starts from the carried state its predecessor left in
    the slot of its last token.  Outputs, every per-token state and the final states are
    bitwise those of one call per sequence."""
    d = workloads.draw_inputs(4, T, 16, 32, 128, 128, torch.bfloat16, 613, init_state_std=0.02)
    g = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    out, fin, st = gdn.prefill(g["queries"], g["keys"], g["values"], g["decays"], g["beta"],
                               g["initial_state"], output_states=True)
    assert torch.equal(st[:, -1], fin)
    for b in (0, 3):
        ob, fb, sb = _one_sequence(gdn, g, b, states=True)
        assert torch.equal(ob[0], out[b]) and torch.equal(fb[0], fin[b])
        assert torch.equal(sb[0], st[b])
        del sb
    del st
    torch.cuda.empty_cache()
    ref = oracle_chains(d, [(1, h) for h in range(0, 32, 5)])
    for (s, h), (o_r, f_r, _) in ref.items():
        assert_out_close(out[s, :, h], o_r, torch.bfloat16, f"chain {(s, h)}")
        assert_states_close(fin[s, h], f_r, f"chain {(s, h)}")
