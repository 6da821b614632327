"""Parity at the benchmark workloads' full sizes, in the launch configuration
bench.py times, on sampled outputs the float64 oracle computes exactly:

* one token: its out, dX and ds rows depend only on that token and its k
  experts, so the oracle runs on that one-token sub-problem;
* the smallest and the largest non-empty expert: an expert's dW1, dW3, dW2
  depend only on the tokens routed to it, so the oracle runs on those tokens
  with k = 1 (same row order, so the same MXFP8 row blocks).  The largest
  expert (8,077 routed rows on the DeepSeek-V3-shaped workload) runs on the
  long-K CTA-pair weight-gradient path at its full K.

The Kimi-K2-shaped minibatch sweep also checks that every ring size gives
bitwise the same results (tiles keep their K order at any minibatch size)."""

import numpy as np
import pytest
import torch

from _helpers import assert_bf16_close, assert_mxfp8_close, require_gpu, poisoned_outputs
from oracle import moe

pytestmark = pytest.mark.gpu


def f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def setup(workload, seed=1000):
    from mixture_experts_layer_side_gb300.inputs import WORKLOADS, make_inputs
    from mixture_experts_layer_side_gb300.layer import MoKLayer
    shape, routing, prec = WORKLOADS[workload]
    inp = make_inputs(shape, routing, seed=seed, device="cuda")
    wq = None
    if prec == "mxfp8":
        wq = MoKLayer(shape, precision=prec).quantize_weights(inp["W1"], inp["W3"], inp["W2"])
    return shape, prec, inp, wq


def run(shape, prec, inp, wq, minibatch_rows=0):
    from mixture_experts_layer_side_gb300.layer import MoKLayer
    layer = MoKLayer(shape, precision=prec, minibatch_rows=minibatch_rows)
    wf, wb = (wq["fwd"], wq["bwd"]) if wq else ((inp["W1"], inp["W3"], inp["W2"]),) * 2
    layer.build_schedule(inp["idx"])
    out, grads = poisoned_outputs(layer)
    layer.forward(inp["x"], inp["s"], *wf, out=out)
    layer.backward(inp["x"], inp["s"], *wb, inp["dout"], grads=grads)
    layer.check()
    return out, grads


def sampled_checks(shape, prec, inp, out, grads):
    quant = "mxfp8" if prec == "mxfp8" else None
    close = assert_mxfp8_close if quant else assert_bf16_close
    idx = inp["idx"].cpu().numpy()
    # one token through its k experts
    t = shape.T - 1
    experts = sorted(set(idx[t].tolist()))
    remap = {e: i for i, e in enumerate(experts)}
    sub_idx = np.array([[remap[e] for e in idx[t]]])
    sel = torch.tensor(experts, device=inp["W1"].device)
    W1, W3, W2 = (f64(inp[n].index_select(0, sel)) for n in ("W1", "W3", "W2"))
    x_t, s_t, d_t = f64(inp["x"][t:t + 1]), f64(inp["s"][t:t + 1]), f64(inp["dout"][t:t + 1])
    ref_out, _ = moe.forward(x_t, sub_idx, s_t, W1, W3, W2, quant=quant)
    dX, _, _, _, ds = moe.backward(x_t, sub_idx, s_t, W1, W3, W2, d_t, quant=quant)
    close(f64(out[t:t + 1]), ref_out, "out[t]")
    close(f64(grads["dX"][t:t + 1]), dX, "dX[t]")
    close(f64(grads["ds"][t:t + 1]), ds, "ds[t]")
    # the smallest and the largest non-empty expert: all tokens routed to it, k = 1
    counts = np.bincount(idx.reshape(-1), minlength=shape.E)
    nz = np.nonzero(counts)[0]
    for e in sorted({int(nz[np.argmin(counts[nz])]), int(nz[np.argmax(counts[nz])])}):
        rows = np.argwhere(idx == e)  # (t, j), ascending t = ascending flat index
        toks = torch.tensor(rows[:, 0], device=inp["x"].device)
        s_e = inp["s"][toks, torch.tensor(rows[:, 1], device=inp["x"].device)].reshape(-1, 1)
        sel = torch.tensor([e], device=inp["W1"].device)
        W1, W3, W2 = (f64(inp[n].index_select(0, sel)) for n in ("W1", "W3", "W2"))
        _, dW1, dW3, dW2, _ = moe.backward(f64(inp["x"].index_select(0, toks)),
                                           np.zeros((len(rows), 1), dtype=np.int64), f64(s_e), W1, W3, W2,
                                           f64(inp["dout"].index_select(0, toks)), quant=quant)
        close(f64(grads["dW1"][e]), dW1[0], f"dW1[{e}] ({counts[e]} rows)")
        close(f64(grads["dW3"][e]), dW3[0], f"dW3[{e}] ({counts[e]} rows)")
        close(f64(grads["dW2"][e]), dW2[0], f"dW2[{e}] ({counts[e]} rows)")
        del dW1, dW3, dW2
    # every element written (the buffers started as NaN), and the experts
    # without routed rows have exact-zero gradients
    for name, t in [("out", out)] + list(grads.items()):
        assert not torch.isnan(t).any().item(), name
    empty = torch.tensor(np.nonzero(counts == 0)[0], device=inp["W1"].device, dtype=torch.long)
    for k in ("dW1", "dW3", "dW2"):
        assert torch.count_nonzero(grads[k].index_select(0, empty)).item() == 0, k


@pytest.mark.parametrize("workload", ["dsv3", "mid", "mid_mxfp8_zipf", "mid_mxfp8_hot", "long_k"])
def test_full_size_sampled_parity(workload):
    require_gpu()
    shape, prec, inp, wq = setup(workload)
    out, grads = run(shape, prec, inp, wq)
    sampled_checks(shape, prec, inp, out, grads)


@pytest.mark.parametrize("workload", ["kimi", "kimi_mxfp8"])
def test_kimi_minibatch_sweep(workload):
    """Minibatch sizes 1024, 2368 (run as 2432 rows), 4096, 8192: bitwise equal
    outputs and gradients, and sampled oracle parity."""
    require_gpu()
    shape, prec, inp, wq = setup(workload)
    out0, g0 = run(shape, prec, inp, wq, minibatch_rows=1024)
    for mb in (2368, 4096, 8192):
        out, g = run(shape, prec, inp, wq, minibatch_rows=mb)
        assert torch.equal(out, out0), mb
        for k in g0:
            assert torch.equal(g[k], g0[k]), (mb, k)
        del out, g
    sampled_checks(shape, prec, inp, out0, g0)
