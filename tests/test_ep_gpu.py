"""Expert parallelism through the C ABI on one GPU: G ranks run as threads of
one process, each with its own ``EPMoELayer``; the exchange between them is a
host barrier plus device copies (every kernel a rank launches reads only data
that is complete before the launch; no kernel waits on another rank).  The
ranks' outputs and gradients, put together, must be BITWISE those of one
``MoKLayer`` holding all tokens and all experts (rows reach each expert in
ascending global flat index, the order one GPU uses)."""

import threading

import numpy as np
import pytest
import torch

from _helpers import require_gpu

pytestmark = pytest.mark.gpu


class ThreadHub:
    """Counts and rows between G in-process ranks: each exchange is a host
    barrier after a device synchronise, then device copies."""

    def __init__(self, G):
        self.G = G
        self.bar = threading.Barrier(G, timeout=120)
        self.slots = [None] * G

    def gather(self, rank, obj):
        self.slots[rank] = obj
        self.bar.wait()
        got = list(self.slots)
        self.bar.wait()
        return got


class ThreadExchange:
    def __init__(self, hub, rank):
        self.hub, self.rank = hub, rank

    def counts(self, part, rank, local_counts):
        torch.cuda.synchronize()
        allc = self.hub.gather(rank, local_counts.cpu().numpy())
        e0, El = part.first(rank), part.count(rank)
        return np.stack([c[e0:e0 + El] for c in allc]).astype(np.int32)

    def rows(self, send, send_rows, recv_rows, out):
        torch.cuda.synchronize()  # the send buffer is complete
        offs = np.concatenate([[0], np.cumsum(send_rows)]).astype(np.int64)
        every = self.hub.gather(self.rank, (send, offs))
        pos = 0
        for src, (buf, o) in enumerate(every):
            n = int(o[self.rank + 1] - o[self.rank])
            assert n == recv_rows[src]
            if n:
                out[pos:pos + n].copy_(buf[int(o[self.rank]):int(o[self.rank]) + n])
            pos += n
        torch.cuda.synchronize()  # copies done before any sender reuses its buffer
        self.hub.bar.wait()
        return out[:pos]


def run_ep(G, shape, inp, precision, wq=None):
    from mixture_experts_layer_side_gb300.ep import EPMoELayer, ExpertPartition
    from mixture_experts_layer_side_gb300.inputs import Shape
    from mixture_experts_layer_side_gb300.layer import quantize_weights
    T, H, I, E, k = shape
    Tl = T // G
    hub = ThreadHub(G)
    part = ExpertPartition(E, G)
    results, errors = [None] * G, []

    def rank_main(r):
        try:
            sl = slice(r * Tl, (r + 1) * Tl)
            e0, El = part.first(r), part.count(r)
            W = [inp[n][e0:e0 + El].contiguous() for n in ("W1", "W3", "W2")]
            if precision == "mxfp8":
                q = quantize_weights(*W)
                wf, wb = q["fwd"], q["bwd"]
            else:
                wf = wb = tuple(W)
            layer = EPMoELayer(Shape(Tl, H, I, E, k), G, r, ThreadExchange(hub, r), precision=precision)
            out = layer.forward(inp["x"][sl].contiguous(), inp["idx"][sl].contiguous(), inp["s"][sl].contiguous(),
                                *wf)
            grads = layer.backward(inp["s"][sl].contiguous(), *wb, inp["dout"][sl].contiguous())
            torch.cuda.synchronize()
            layer.check()
            results[r] = (out, grads, layer.plan.n_recv)
        except BaseException as e:  # noqa: BLE001
            errors.append(e)
            hub.bar.abort()

    threads = [threading.Thread(target=rank_main, args=(r,)) for r in range(G)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    if errors:
        raise errors[0]
    return results


def run_single(shape, inp, precision):
    from mixture_experts_layer_side_gb300.inputs import Shape
    from mixture_experts_layer_side_gb300.layer import MoKLayer
    layer = MoKLayer(Shape(*shape), precision=precision)
    if precision == "mxfp8":
        q = layer.quantize_weights(inp["W1"], inp["W3"], inp["W2"])
        wf, wb = q["fwd"], q["bwd"]
    else:
        wf = wb = (inp["W1"], inp["W3"], inp["W2"])
    layer.build_schedule(inp["idx"])
    out = layer.forward(inp["x"], inp["s"], *wf)
    grads = layer.backward(inp["x"], inp["s"], *wb, inp["dout"])
    layer.check()
    return out, grads


CASES = [
    # (G, (T total, H, I, E, k), routing, precision)
    (2, (512, 256, 128, 8, 2), "zipf", "bf16"),
    (4, (1024, 256, 256, 12, 4), "zipf", "bf16"),
    (3, (768, 384, 128, 7, 2), "uniform", "bf16"),
    (2, (512, 256, 128, 8, 2), "zipf", "mxfp8"),
    (4, (512, 256, 128, 10, 3), "uniform", "mxfp8"),
]


@pytest.mark.parametrize("G,shape,routing,precision", CASES)
def test_ep_ranks_bitwise_equal_one_gpu(G, shape, routing, precision):
    require_gpu()
    from mixture_experts_layer_side_gb300.inputs import Shape, make_inputs
    inp = {k: v.cuda() for k, v in make_inputs(Shape(*shape), routing, seed=60 + G, device="cpu").items()}
    ref_out, ref_g = run_single(shape, inp, precision)
    res = run_ep(G, shape, inp, precision)
    assert torch.equal(torch.cat([r[0] for r in res]), ref_out)
    for name in ("dX", "ds"):
        assert torch.equal(torch.cat([r[1][name] for r in res]), ref_g[name]), name
    for name in ("dW1", "dW3", "dW2"):
        assert torch.equal(torch.cat([r[1][name] for r in res]), ref_g[name]), name


def test_ep_rank_that_receives_nothing():
    """Every token routes to experts 0..5 of 8: the last of four ranks
    (experts 6, 7) receives no row; its weight gradients are exact zeros and
    everything else still matches one GPU bitwise."""
    require_gpu()
    from mixture_experts_layer_side_gb300.inputs import Shape, make_inputs
    shape = (512, 256, 128, 8, 2)
    inp = {k: v.cuda() for k, v in make_inputs(Shape(*shape), "uniform", seed=71, device="cpu").items()}
    inp["idx"] = torch.remainder(inp["idx"], 6).to(torch.int32)
    dup = inp["idx"][:, 0] == inp["idx"][:, 1]
    inp["idx"][dup, 1] = (inp["idx"][dup, 0] + 1) % 6
    ref_out, ref_g = run_single(shape, inp, "bf16")
    res = run_ep(4, shape, inp, "bf16")
    assert res[3][2] == 0
    assert torch.equal(torch.cat([r[0] for r in res]), ref_out)
    for name in ("dX", "ds", "dW1", "dW3", "dW2"):
        assert torch.equal(torch.cat([r[1][name] for r in res]), ref_g[name]), name
    assert torch.count_nonzero(res[3][1]["dW1"]).item() == 0
