"""Host logic of LatentMoELayer.steps_from_host (no GPU): the double-buffered
device slots, the order of copies and steps, and the layer's own buffers after
the call. CUDA streams and events are stand-ins that run in program order, and
the layer's step is replaced by dx = x + dout on the slot's buffers, so every
step's gradient is known."""
import types
from unittest import mock

import pytest
import torch

from sparse_moe_layer_topk_gb300.layer import LatentMoELayer


class _Stream:
    def __init__(self, *a, **k):
        pass

    def wait_event(self, e):
        assert e is not None and e.recorded, "waits on an event that was never recorded"


class _Event:
    def __init__(self, *a, **k):
        self.recorded = False

    def record(self, stream=None):
        self.recorded = True


class _Ctx:
    def __init__(self, s):
        pass

    def __enter__(self):
        return self

    def __exit__(self, *a):
        return False


class _Layer(LatentMoELayer):
    """The pipeline of LatentMoELayer around a stand-in step: dx = x + dout."""

    def __init__(self, T, d):  # no device buffers beyond dx
        self.dx = torch.zeros(T, d)
        self.captures = 0

    def forward(self, x, stream=None):
        self.x = x

    def backward(self, dout, stream=None):
        self.dx.copy_(self.x + dout)
        return self.dx

    def capture_halves(self, x, dout):
        # the graphs replay the step on the buffers they were captured with:
        # the forward keeps a copy of x, the backward writes dx = x + dout
        self.captures += 1
        dx = self.dx
        seen = torch.zeros_like(x)
        fwd = types.SimpleNamespace(replay=lambda: seen.copy_(x))
        bwd = types.SimpleNamespace(replay=lambda: dx.copy_(seen + dout))
        return fwd, bwd


@pytest.mark.parametrize("graphs", [False, True])
@pytest.mark.parametrize("n", [1, 2, 5])
def test_each_step_gets_its_own_inputs_and_gradient(graphs, n):
    T, d = 4, 8
    layer = _Layer(T, d)
    own = layer.dx
    xs = [torch.full((T, d), float(10 * i + 1)) for i in range(n)]
    gs = [torch.full((T, d), float(i + 0.5)) for i in range(n)]
    outs = [torch.zeros(T, d) for _ in range(n)]
    with mock.patch.object(torch.cuda, "current_stream", lambda *a: _Stream()), \
            mock.patch.object(torch.cuda, "Stream", _Stream), \
            mock.patch.object(torch.cuda, "Event", _Event), \
            mock.patch.object(torch.cuda, "stream", _Ctx):
        layer.steps_from_host(xs, gs, outs, graphs=graphs)
        for i in range(n):
            assert torch.equal(outs[i], xs[i] + gs[i]), i
        assert layer.dx is own  # the layer's own gradient buffer again
        # a second call reuses the slots (and, with graphs, the captured steps)
        outs2 = [torch.zeros(T, d) for _ in range(n)]
        layer.steps_from_host(xs[::-1], gs[::-1], outs2, graphs=graphs)
    for i in range(n):
        assert torch.equal(outs2[i], xs[n - 1 - i] + gs[n - 1 - i]), i
    assert layer.dx is own
    assert layer.captures == (2 if graphs else 0)
