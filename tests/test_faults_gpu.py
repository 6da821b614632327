"""Failure detection without a GPU fault: a host-chosen skipped completion
signal in the forward ring makes the consumer's bounded wait run out; the call
records MOK_ERR_TIMEOUT, every CTA unwinds, and the context stays usable."""

import pytest
import torch

from _helpers import require_gpu

pytestmark = pytest.mark.gpu


def test_skipped_ring_signal_times_out_and_context_survives():
    require_gpu()
    from mixture_experts_layer_side_gb300 import _lib
    from mixture_experts_layer_side_gb300.inputs import Shape, make_inputs
    from mixture_experts_layer_side_gb300.layer import MoKLayer
    shape = Shape(512, 256, 256, 8, 2)
    inp = {k: v.cuda() for k, v in make_inputs(shape, "uniform", seed=9, device="cpu").items()}
    bad = MoKLayer(shape, minibatch_rows=128, ring_slots=2, debug_flags=_lib.MOK_DEBUG_SKIP_RING_SIGNAL)
    bad.build_schedule(inp["idx"])
    bad.forward(inp["x"], inp["s"], inp["W1"], inp["W3"], inp["W2"])
    assert _lib.mok_check(bad.ws) == 6  # MOK_ERR_TIMEOUT
    # the same process and context keep working
    good = MoKLayer(shape)
    good.build_schedule(inp["idx"])
    out1 = good.forward(inp["x"], inp["s"], inp["W1"], inp["W3"], inp["W2"])
    good.check()
    out2 = good.forward(inp["x"], inp["s"], inp["W1"], inp["W3"], inp["W2"])
    good.check()
    assert torch.equal(out1, out2)


def test_skipped_ring_signal_in_the_single_launch_forward():
    """The same skipped signal inside mok_forward_fused: the schedule items,
    the ring and the combine phase all unwind through their bounded waits."""
    require_gpu()
    from mixture_experts_layer_side_gb300 import _lib
    from mixture_experts_layer_side_gb300.inputs import Shape, make_inputs
    from mixture_experts_layer_side_gb300.layer import MoKLayer
    shape = Shape(512, 256, 256, 8, 2)
    inp = {k: v.cuda() for k, v in make_inputs(shape, "uniform", seed=9, device="cpu").items()}
    bad = MoKLayer(shape, minibatch_rows=128, ring_slots=2, debug_flags=_lib.MOK_DEBUG_SKIP_RING_SIGNAL)
    bad.forward_fused(inp["idx"], inp["x"], inp["s"], inp["W1"], inp["W3"], inp["W2"])
    assert _lib.mok_check(bad.ws) == 6  # MOK_ERR_TIMEOUT
    good = MoKLayer(shape)
    out1 = good.forward_fused(inp["idx"], inp["x"], inp["s"], inp["W1"], inp["W3"], inp["W2"])
    good.check()
    good.build_schedule(inp["idx"])
    out2 = good.forward(inp["x"], inp["s"], inp["W1"], inp["W3"], inp["W2"])
    good.check()
    assert torch.equal(out1, out2)
