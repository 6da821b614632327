"""A whole layer step (schedule, forward, backward) captured into one CUDA
graph: the library only enqueues on the caller's stream, so the captured
step replays bitwise like the eager one, for new inputs copied into the
captured buffers, BF16 and MXFP8."""

import pytest
import torch

from _helpers import require_gpu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("precision", ["bf16", "mxfp8"])
def test_captured_step_replays_bitwise(precision):
    require_gpu()
    from mixture_experts_layer_side_gb300.inputs import Shape, make_inputs
    from mixture_experts_layer_side_gb300.layer import MoKLayer
    S = Shape(1024, 256, 256, 16, 4)
    a = {k: v.cuda() for k, v in make_inputs(S, "zipf", seed=41, device="cpu").items()}
    b = {k: v.cuda() for k, v in make_inputs(S, "zipf", seed=42, device="cpu").items()}
    layer = MoKLayer(S, precision=precision, minibatch_rows=256, ring_slots=2)
    if precision == "mxfp8":
        wq = layer.quantize_weights(a["W1"], a["W3"], a["W2"])
        wf, wb = wq["fwd"], wq["bwd"]
    else:
        wf = wb = (a["W1"], a["W3"], a["W2"])
    # the captured step reads its inputs from these buffers
    buf = {k: a[k].clone() for k in ("x", "idx", "s", "dout")}
    out = torch.empty((S.T, S.H), dtype=torch.bfloat16, device="cuda")
    grads = layer.alloc_grads()

    def step():
        layer.build_schedule(buf["idx"])
        layer.forward(buf["x"], buf["s"], *wf, out=out)
        layer.backward(buf["x"], buf["s"], *wb, buf["dout"], grads=grads)

    def eager(inp):
        for k in buf:
            buf[k].copy_(inp[k])
        step()
        torch.cuda.synchronize()
        layer.check()
        return out.clone(), {k: v.clone() for k, v in grads.items()}

    ref_a, ref_b = eager(a), eager(b)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()  # warm-up on the capture stream (kernel attributes set outside the capture)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for inp, ref in ((a, ref_a), (b, ref_b), (a, ref_a)):
        for k in buf:
            buf[k].copy_(inp[k])
        graph.replay()
        torch.cuda.synchronize()
        layer.check()
        assert torch.equal(out, ref[0])
        for k in ref[1]:
            assert torch.equal(grads[k], ref[1][k]), k
