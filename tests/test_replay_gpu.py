"""Bounded-memory backward (replay = 1): the forward context keeps [h|u] of
the last ring_slots minibatches only and the backward recomputes GEMM1 for
the others.  Outputs and gradients must be bitwise those of the saved
context (which the oracle tests pin), at every ring size, and the context
must be ring_slots minibatches large."""

import pytest
import torch

from _helpers import assert_bf16_close, np64, poisoned_outputs, require_gpu
from oracle import moe

pytestmark = pytest.mark.gpu


def run(shape, routing, seed, inp=None, **kw):
    from mixture_experts_layer_side_gb300.inputs import make_inputs
    from mixture_experts_layer_side_gb300.layer import MoKLayer
    if inp is None:
        inp = {k: v.cuda() for k, v in make_inputs(shape, routing, seed=seed, device="cpu").items()}
    layer = MoKLayer(shape, **kw)
    layer.build_schedule(inp["idx"])
    out, grads = poisoned_outputs(layer)
    layer.forward(inp["x"], inp["s"], inp["W1"], inp["W3"], inp["W2"], out=out)
    layer.backward(inp["x"], inp["s"], inp["W1"], inp["W3"], inp["W2"], inp["dout"], grads=grads)
    layer.check()
    return inp, out, grads, layer.ctx.numel()


CASES = [((4096, 256, 128, 16, 4), "zipf", 128, 2), ((4096, 256, 128, 16, 4), "zipf", 256, 3),
         ((256, 256, 128, 8, 2), "uniform", 0, 0), ((512, 384, 128, 24, 4), "hot", 256, 3),
         ((3000, 256, 128, 20, 2), "hot", 128, 2)]


@pytest.mark.parametrize("shape,routing,mb,slots", CASES)
def test_replay_is_bitwise_equal_to_the_saved_context(shape, routing, mb, slots):
    require_gpu()
    from mixture_experts_layer_side_gb300.inputs import Shape
    S = Shape(*shape)
    inp, out_a, g_a, ctx_a = run(S, routing, 31, minibatch_rows=mb, ring_slots=slots)
    _, out_b, g_b, ctx_b = run(S, routing, 31, inp=inp, minibatch_rows=mb, ring_slots=slots, replay=True)
    assert ctx_b <= ctx_a
    assert torch.equal(out_a, out_b)
    for k in g_a:
        assert torch.equal(g_a[k], g_b[k]), k


def test_replay_matches_oracle_with_a_small_ring():
    require_gpu()
    from mixture_experts_layer_side_gb300.inputs import Shape
    S = Shape(1024, 256, 128, 12, 4)
    inp, out, grads, ctx = run(S, "zipf", 32, minibatch_rows=128, ring_slots=2, replay=True)
    assert ctx == 2 * 128 * 2 * 128 * 2
    a = {k: np64(v) if v.dtype != torch.int32 else v.cpu().numpy() for k, v in inp.items()}
    ref_out, _ = moe.forward(a["x"], a["idx"], a["s"], a["W1"], a["W3"], a["W2"])
    dX, dW1, dW3, dW2, ds = moe.backward(a["x"], a["idx"], a["s"], a["W1"], a["W3"], a["W2"], a["dout"])
    assert_bf16_close(np64(out), ref_out, "out")
    for name, ref in (("dX", dX), ("dW1", dW1), ("dW3", dW3), ("dW2", dW2), ("ds", ds)):
        assert_bf16_close(np64(grads[name]), ref, name)


def test_replay_full_size_dsv3():
    """DeepSeek-V3 shape, default minibatch and ring: the context shrinks
    from every padded row to four minibatches, results bitwise unchanged."""
    require_gpu()
    from mixture_experts_layer_side_gb300.inputs import WORKLOADS, make_inputs
    shape, routing, _ = WORKLOADS["dsv3"]
    inp = make_inputs(shape, routing, seed=1000, device="cuda")
    _, out_a, g_a, ctx_a = run(shape, routing, 0, inp=inp)
    _, out_b, g_b, ctx_b = run(shape, routing, 0, inp=inp, replay=True)
    assert ctx_b * 8 < ctx_a
    assert torch.equal(out_a, out_b)
    for k in g_a:
        assert torch.equal(g_a[k], g_b[k]), k


def run_mx(shape, routing, seed, inp=None, **kw):
    from mixture_experts_layer_side_gb300.inputs import make_inputs
    from mixture_experts_layer_side_gb300.layer import MoKLayer
    if inp is None:
        inp = {k: v.cuda() for k, v in make_inputs(shape, routing, seed=seed, device="cpu").items()}
    layer = MoKLayer(shape, precision="mxfp8", **kw)
    wq = layer.quantize_weights(inp["W1"], inp["W3"], inp["W2"])
    layer.build_schedule(inp["idx"])
    out, grads = poisoned_outputs(layer)
    layer.forward(inp["x"], inp["s"], *wq["fwd"], out=out)
    wb = wq["bwd_replay"] if kw.get("replay") else wq["bwd"]
    layer.backward(inp["x"], inp["s"], *wb, inp["dout"], grads=grads)
    layer.check()
    return inp, out, grads, layer.ctx.numel()


@pytest.mark.parametrize("shape,routing,mb,slots,flags", [
    ((4096, 256, 128, 16, 4), "zipf", 128, 2, 0), ((4096, 256, 256, 16, 4), "zipf", 256, 3, 0),
    ((512, 384, 128, 24, 4), "hot", 256, 3, 0), ((3000, 256, 128, 20, 2), "hot", 128, 2, 64 | 4)])
def test_mxfp8_replay_is_bitwise_equal_to_the_saved_context(shape, routing, mb, slots, flags):
    """MXFP8 bounded-memory backward: GEMM1 recomputed from x quantised along
    H and the forward orientation of W1 / W3 gives the forward's [h|u] bit
    for bit, so every output and gradient equals the saved context's."""
    require_gpu()
    from mixture_experts_layer_side_gb300.inputs import Shape
    S = Shape(*shape)
    kw = dict(minibatch_rows=mb, ring_slots=slots, debug_flags=flags)
    inp, out_a, g_a, ctx_a = run_mx(S, routing, 33, **kw)
    _, out_b, g_b, ctx_b = run_mx(S, routing, 33, inp=inp, replay=True, **kw)
    assert ctx_b < ctx_a
    assert torch.equal(out_a, out_b)
    for k in g_a:
        assert torch.equal(g_a[k], g_b[k]), k
