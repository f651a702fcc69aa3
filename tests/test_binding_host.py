"""Host-side behaviour of the Python binding (no GPU needed)."""
import contextlib
import inspect

import torch

import gated_deltanet_mixer_delta_gb300 as gdn


def test_calls_with_a_stream_run_and_allocate_on_it(monkeypatch):
    """With ``stream`` given, the call body (its allocations and its launches) runs with
    that stream current; without one, nothing is switched."""
    entered = []

    @contextlib.contextmanager
    def fake_stream(s):
        entered.append(s)
        yield

    monkeypatch.setattr(torch.cuda, "stream", fake_stream)
    seen = []

    @gdn._on_stream
    def call(x, *, stream=None):
        seen.append((x, stream, list(entered)))
        return x + 1

    assert call(1) == 2 and seen[-1] == (1, None, [])
    token = object()
    assert call(2, stream=token) == 3 and seen[-1] == (2, token, [token])


def test_public_calls_take_a_keyword_only_stream():
    for fn in (gdn.prefill, gdn.prefill_varlen, gdn.decode_step, gdn.gated_rmsnorm,
               gdn.conv_gate_prologue):
        params = inspect.signature(fn).parameters
        assert params["stream"].kind is inspect.Parameter.KEYWORD_ONLY, fn.__name__
        assert params["stream"].default is None, fn.__name__
