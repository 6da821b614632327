"""The single-launch forward (mok_forward_fused: the schedule's histogram,
scan and placement items, the ring's GEMM tiles and the combine in one
persistent launch) against mok_build_schedule + mok_forward on the same
inputs: the schedule arrays, out and the saved context bitwise equal, the
backward that follows bitwise equal, the oracle on one case, and an
out-of-range expert id reported as the schedule reports it."""

import numpy as np
import pytest
import torch

from _helpers import assert_bf16_close, np64, require_gpu
from oracle import moe

pytestmark = pytest.mark.gpu

CASES = [
    ((256, 256, 128, 8, 2), "uniform", {}),
    ((300, 256, 256, 6, 3), "zipf", {}),
    # 16 empty experts, half the tokens on one expert
    ((512, 384, 128, 24, 4), "hot", {}),
    ((1, 128, 128, 1, 1), "uniform", {}),
    ((512, 128, 128, 1024, 4), "uniform", {}),
    ((64, 256, 128, 40, 32), "uniform", {}),
    # several schedule chunks, small ring
    ((4096, 256, 256, 16, 4), "zipf", dict(minibatch_rows=256, ring_slots=2)),
    ((3000, 512, 256, 20, 2), "hot", dict(replay=True, minibatch_rows=384, ring_slots=3)),
]


def run(shape, routing, seed, fused, inp=None, **kw):
    from mixture_experts_layer_side_gb300.inputs import Shape, make_inputs
    from mixture_experts_layer_side_gb300.layer import MoKLayer
    S = Shape(*shape)
    if inp is None:
        inp = {k: v.cuda() for k, v in make_inputs(S, routing, seed=seed, device="cpu").items()}
    layer = MoKLayer(S, **kw)
    # an element the launch fails to write keeps this pattern
    layer.ws.fill_(0x55)
    layer.ctx.fill_(0x55)
    out = torch.full((S.T, S.H), float("nan"), dtype=torch.bfloat16, device="cuda")
    if fused:
        layer.forward_fused(inp["idx"], inp["x"], inp["s"], inp["W1"], inp["W3"], inp["W2"], out=out)
    else:
        layer.build_schedule(inp["idx"])
        layer.forward(inp["x"], inp["s"], inp["W1"], inp["W3"], inp["W2"], out=out)
    layer.check()
    sched = {n: a.clone() for n, a in layer.schedule_arrays().items()}
    ctx = layer.ctx.clone()
    grads = layer.backward(inp["x"], inp["s"], inp["W1"], inp["W3"], inp["W2"], inp["dout"])
    layer.check()
    return inp, out, sched, ctx, grads


@pytest.mark.parametrize("shape,routing,kw", CASES)
def test_fused_forward_is_bitwise_the_separate_launches(shape, routing, kw):
    require_gpu()
    inp, out_f, sch_f, ctx_f, g_f = run(shape, routing, 61, True, **kw)
    _, out_s, sch_s, ctx_s, g_s = run(shape, routing, 61, False, inp=inp, **kw)
    for name in ("counts", "offsets", "padded_offsets", "perm", "inv_perm", "pad_inv"):
        assert torch.equal(sch_f[name], sch_s[name]), name
    used = int(sch_s["padded_offsets"][-1])
    assert int(sch_f["header"][1]) == used and int(sch_f["header"][2]) == used // 128
    assert torch.equal(sch_f["pad_perm"][:used], sch_s["pad_perm"][:used])
    assert torch.equal(sch_f["tile_expert"][:used // 128], sch_s["tile_expert"][:used // 128])
    assert torch.equal(out_f, out_s)
    if not kw.get("replay"):
        row_bytes = 2 * shape[2] * 2
        assert torch.equal(ctx_f[:used * row_bytes], ctx_s[:used * row_bytes])
    for k in g_s:
        assert torch.equal(g_f[k], g_s[k]), k


def test_fused_forward_matches_oracle():
    require_gpu()
    inp, out, _, _, grads = run((700, 256, 256, 12, 4), "zipf", 62, True)
    a = {k: np64(v) if v.dtype != torch.int32 else v.cpu().numpy() for k, v in inp.items()}
    ref_out, _ = moe.forward(a["x"], a["idx"], a["s"], a["W1"], a["W3"], a["W2"])
    assert_bf16_close(np64(out), ref_out, "out")
    dX, dW1, dW3, dW2, ds = moe.backward(a["x"], a["idx"], a["s"], a["W1"], a["W3"], a["W2"], a["dout"])
    for name, ref in (("dX", dX), ("dW1", dW1), ("dW3", dW3), ("dW2", dW2), ("ds", ds)):
        assert_bf16_close(np64(grads[name]), ref, name)


def test_fused_forward_reports_a_bad_expert_index():
    require_gpu()
    from mixture_experts_layer_side_gb300 import _lib
    from mixture_experts_layer_side_gb300.inputs import Shape, make_inputs
    from mixture_experts_layer_side_gb300.layer import MoKLayer
    S = Shape(64, 128, 128, 8, 2)
    inp = {k: v.cuda() for k, v in make_inputs(S, "uniform", seed=63, device="cpu").items()}
    inp["idx"][5, 1] = 8
    layer = MoKLayer(S)
    layer.forward_fused(inp["idx"], inp["x"], inp["s"], inp["W1"], inp["W3"], inp["W2"])
    assert _lib.mok_check(layer.ws) == 5  # MOK_ERR_BAD_INDEX
    # the context stays usable: a clean call succeeds
    inp["idx"][5, 1] = 3
    out = layer.forward_fused(inp["idx"], inp["x"], inp["s"], inp["W1"], inp["W3"], inp["W2"])
    layer.check()
    assert torch.isfinite(out.float()).all()


def test_fused_forward_full_size_dsv3():
    """DeepSeek-V3 shape: bitwise equal to the separate launches."""
    require_gpu()
    from mixture_experts_layer_side_gb300.inputs import WORKLOADS, make_inputs
    shape, routing, _ = WORKLOADS["dsv3"]
    inp = make_inputs(shape, routing, seed=1000, device="cuda")
    from mixture_experts_layer_side_gb300.layer import MoKLayer
    outs = []
    for fused in (True, False):
        layer = MoKLayer(shape)
        if fused:
            out = layer.forward_fused(inp["idx"], inp["x"], inp["s"], inp["W1"], inp["W3"], inp["W2"])
        else:
            layer.build_schedule(inp["idx"])
            out = layer.forward(inp["x"], inp["s"], inp["W1"], inp["W3"], inp["W2"])
        layer.check()
        outs.append(out)
        del layer
    assert torch.equal(outs[0], outs[1])
    assert not torch.isnan(outs[0].float()).any()


def run_mx(shape, routing, seed, fused, inp=None, **kw):
    from mixture_experts_layer_side_gb300.inputs import Shape, make_inputs
    from mixture_experts_layer_side_gb300.layer import MoKLayer
    S = Shape(*shape)
    if inp is None:
        inp = {k: v.cuda() for k, v in make_inputs(S, routing, seed=seed, device="cpu").items()}
    layer = MoKLayer(S, precision="mxfp8", **kw)
    wq = layer.quantize_weights(inp["W1"], inp["W3"], inp["W2"])
    layer.ws.fill_(0x55)
    layer.ctx.fill_(0x55)
    out = torch.full((S.T, S.H), float("nan"), dtype=torch.bfloat16, device="cuda")
    if fused:
        layer.forward_fused(inp["idx"], inp["x"], inp["s"], *wq["fwd"], out=out)
    else:
        layer.build_schedule(inp["idx"])
        layer.forward(inp["x"], inp["s"], *wq["fwd"], out=out)
    layer.check()
    sched = {n: a.clone() for n, a in layer.schedule_arrays().items()}
    ctx = layer.ctx.clone()
    # (the bounded-memory backward also takes W1 / W3 in the forward orientation)
    grads = layer.backward(inp["x"], inp["s"], *wq["bwd_replay" if kw.get("replay") else "bwd"], inp["dout"])
    layer.check()
    return inp, out, sched, ctx, grads


@pytest.mark.parametrize("shape,routing,kw", CASES)
def test_mxfp8_fused_forward_is_bitwise_the_separate_launches(shape, routing, kw):
    """MXFP8: the placement items tile the placed rows' x scales for GEMM1
    and the ring gathers x's E4M3 rows by token; the separate launches read
    a token-sorted code copy and a scale tiling kernel's output.  Same
    schedule arrays, out, context and backward, bit for bit."""
    require_gpu()
    inp, out_f, sch_f, ctx_f, g_f = run_mx(shape, routing, 71, True, **kw)
    _, out_s, sch_s, ctx_s, g_s = run_mx(shape, routing, 71, False, inp=inp, **kw)
    for name in ("counts", "offsets", "padded_offsets", "perm", "inv_perm", "pad_inv"):
        assert torch.equal(sch_f[name], sch_s[name]), name
    used = int(sch_s["padded_offsets"][-1])
    assert torch.equal(sch_f["pad_perm"][:used], sch_s["pad_perm"][:used])
    assert torch.equal(out_f, out_s)
    assert not torch.isnan(out_f.float()).any()
    if not kw.get("replay"):
        row_bytes = 2 * shape[2] * 2
        assert torch.equal(ctx_f[:used * row_bytes], ctx_s[:used * row_bytes])
    for k in g_s:
        assert torch.equal(g_f[k], g_s[k]), k


def test_mxfp8_fused_forward_full_size_kimi():
    """Kimi-K2 shape in MXFP8: the single launch bitwise equal to the
    separate launches (out and context)."""
    require_gpu()
    from mixture_experts_layer_side_gb300.inputs import WORKLOADS, make_inputs
    from mixture_experts_layer_side_gb300.layer import MoKLayer
    shape, routing, _ = WORKLOADS["kimi_mxfp8"]
    inp = make_inputs(shape, routing, seed=1001, device="cuda")
    res = []
    for fused in (True, False):
        layer = MoKLayer(shape, precision="mxfp8")
        wq = layer.quantize_weights(inp["W1"], inp["W3"], inp["W2"])
        if fused:
            out = layer.forward_fused(inp["idx"], inp["x"], inp["s"], *wq["fwd"])
        else:
            layer.build_schedule(inp["idx"])
            out = layer.forward(inp["x"], inp["s"], *wq["fwd"])
        layer.check()
        used = int(layer.schedule_arrays()["padded_offsets"][-1])
        res.append((out, layer.ctx[:used * 2 * shape.I * 2].clone()))
        del layer, wq
    assert torch.equal(res[0][0], res[1][0])
    assert torch.equal(res[0][1], res[1][1])
    assert not torch.isnan(res[0][0].float()).any()
