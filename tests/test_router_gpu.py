"""The top-k softmax router through the C ABI against the float64 router
oracle: logits, selection (bit-exact on the GPU's own f32 keys, as the kernel
decides, and against the oracle on its own float64 logits with near ties
exempt), scores, the logit / weight / input gradients, the router composed
with the layer, and a full-size DeepSeek-V3-shaped case."""

import numpy as np
import pytest
import torch

from _helpers import assert_bf16_close, np64, require_gpu, rel_errors
from oracle import moe, router

pytestmark = pytest.mark.gpu


def make(T, H, E, k, seed, biased):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn((T, H), generator=g).to(torch.bfloat16)
    Wr = (0.05 * torch.randn((H, E), generator=g)).to(torch.bfloat16)
    bias = (0.5 * torch.randn(E, generator=g)).float() if biased else None
    ds = torch.randn((T, k), generator=g).float()
    return x, Wr, bias, ds


def selection_on(logits32, bias, k):
    """The oracle's selection on the kernel's keys: f32 logit + f32 bias."""
    key = logits32 if bias is None else (logits32 + bias.numpy().astype(np.float32)[None, :]).astype(np.float32)
    return router.topk_softmax(key.astype(np.float64), None, k)[0]


def check_against_oracle_logits(x, Wr, bias, k, idx, s, logits_gpu):
    """Selection and scores against the oracle on its OWN float64 logits.

    A token whose sorted keys (logit + bias) hold two neighbours among the
    first k + 1 closer than the logits' error cannot be decided the same way
    by both sides; it is exempt from the exact comparison, its selection is
    only checked to be a valid top-k within that margin, and such tokens must
    be rare (at most 5%: 149 of 8,192 at the DeepSeek-V3 shape with twice
    this margin).  Every other token: the same experts in the same column order,
    and scores within float32 rounding of the float64 softmax."""
    L64 = np64(x) @ np64(Wr)
    b64 = np.zeros(L64.shape[1]) if bias is None else bias.double().numpy()
    idx_ref, s_ref = router.topk_softmax(L64, None if bias is None else b64, k)
    # two keys can be ordered differently by the two sides only if their gap
    # is below the sum of their errors: twice the largest logit error, plus
    # the float32 rounding of the biased key
    margin = 2.0 * float(np.abs(logits_gpu.astype(np.float64) - L64).max()) + 1e-6
    key = L64 + b64[None, :]
    T, E = key.shape
    srt = -np.sort(-key, axis=1)[:, :min(k + 1, E)]
    near = (np.diff(-srt, axis=1) < margin).any(axis=1) if srt.shape[1] > 1 else np.zeros(T, bool)
    ok = ~near
    np.testing.assert_array_equal(idx[ok], idx_ref[ok])
    np.testing.assert_allclose(s[ok], s_ref[ok], rtol=1e-4, atol=1e-6)
    assert near.sum() <= max(2, T // 20), f"{near.sum()} of {T} tokens with near-tied keys"
    for t in np.nonzero(near)[0]:
        kth = srt[t, k - 1]
        assert (key[t, idx[t]] >= kth - margin).all(), t
        assert len(set(idx[t].tolist())) == k, t
        ch = L64[t, idx[t]]
        ez = np.exp(ch - ch.max())
        np.testing.assert_allclose(s[t], ez / ez.sum(), rtol=1e-4, atol=1e-6)
    return int(near.sum())


def run_router(T, H, E, k, seed, biased):
    from mixture_experts_layer_side_gb300.inputs import Shape
    from mixture_experts_layer_side_gb300.layer import MoKRouter
    x, Wr, bias, ds = make(T, H, E, k, seed, biased)
    r = MoKRouter(Shape(T, H, 128, E, k))
    xd, Wd, dsd = x.cuda(), Wr.cuda(), ds.cuda()
    bd = bias.cuda() if bias is not None else None
    idx, s, logits = r.forward(xd, Wd, bd, with_logits=True)
    dWr, dx = r.backward(xd, Wd, idx, s, dsd)
    r.check()
    return (x, Wr, bias, ds), (idx.cpu().numpy(), s.cpu().numpy(), logits.cpu().numpy(), dWr.cpu().numpy(),
                                dx.float().cpu().numpy())


CASES = [(300, 256, 24, 4, False), (300, 256, 24, 4, True), (1, 128, 5, 1, False), (1000, 512, 256, 8, True),
         (257, 384, 1024, 32, False), (129, 128, 130, 3, True)]


@pytest.mark.parametrize("T,H,E,k,biased", CASES)
def test_router_matches_oracle(T, H, E, k, biased):
    require_gpu()
    (x, Wr, bias, ds), (idx, s, logits, dWr, dx) = run_router(T, H, E, k, T + E + k, biased)
    L_ref = np64(x) @ np64(Wr)
    fro = rel_errors(logits, L_ref)[1]
    assert fro < 1e-5, fro
    # selection: bit-exact, decided on the kernel's own keys
    np.testing.assert_array_equal(idx, selection_on(logits, bias, k))
    # and against the oracle's own float64 logits, near ties exempt
    check_against_oracle_logits(x, Wr, bias, k, idx, s, logits)
    # scores: softmax of the chosen logits
    ch = np.take_along_axis(logits.astype(np.float64), idx.astype(np.int64), axis=1)
    ez = np.exp(ch - ch.max(axis=1, keepdims=True))
    np.testing.assert_allclose(s, ez / ez.sum(axis=1, keepdims=True), rtol=2e-6, atol=1e-7)
    # gradients (dL is rounded to bf16 for the tensor-core GEMMs)
    _, dWr_ref, dx_ref = router.router_backward(np64(x), np64(Wr), idx, s, np64(ds))
    assert_bf16_close(dWr, dWr_ref, "dWr")
    assert_bf16_close(dx, dx_ref, "dx_router")


def test_router_reruns_are_bitwise_identical():
    require_gpu()
    _, a = run_router(1000, 512, 256, 8, 3, True)
    for _ in range(2):
        _, b = run_router(1000, 512, 256, 8, 3, True)
        for u, v in zip(a, b):
            np.testing.assert_array_equal(u, v)


def test_router_weight_gradient_through_the_layer():
    """Router forward -> layer forward / backward -> router backward, against
    the oracle chain (layer score gradient composed with the router
    backward) on the same routing."""
    require_gpu()
    from mixture_experts_layer_side_gb300.inputs import Shape
    from mixture_experts_layer_side_gb300.layer import MoKLayer, MoKRouter
    T, H, I, E, k = 384, 256, 128, 12, 3
    g = torch.Generator().manual_seed(21)
    x = torch.randn((T, H), generator=g).to(torch.bfloat16)
    Wr = (0.05 * torch.randn((H, E), generator=g)).to(torch.bfloat16)
    W1 = (0.02 * torch.randn((E, H, I), generator=g)).to(torch.bfloat16)
    W3 = (0.02 * torch.randn((E, H, I), generator=g)).to(torch.bfloat16)
    W2 = (0.02 * torch.randn((E, I, H), generator=g)).to(torch.bfloat16)
    dout = torch.randn((T, H), generator=g).to(torch.bfloat16)
    S = Shape(T, H, I, E, k)
    r, layer = MoKRouter(S), MoKLayer(S)
    d = {n: t.cuda() for n, t in dict(x=x, Wr=Wr, W1=W1, W3=W3, W2=W2, dout=dout).items()}
    idx, s = r.forward(d["x"], d["Wr"])
    layer.build_schedule(idx)
    layer.forward(d["x"], s, d["W1"], d["W3"], d["W2"])
    grads = layer.backward(d["x"], s, d["W1"], d["W3"], d["W2"], d["dout"])
    dWr, _ = r.backward(d["x"], d["Wr"], idx, s, grads["ds"])
    layer.check()
    r.check()
    idx_n, s_n = idx.cpu().numpy(), s.cpu().numpy()
    _, _, _, _, ds_ref = moe.backward(np64(x), idx_n, s_n, np64(W1), np64(W3), np64(W2), np64(dout))
    _, dWr_ref, _ = router.router_backward(np64(x), np64(Wr), idx_n, s_n, ds_ref)
    assert_bf16_close(dWr.cpu().numpy(), dWr_ref, "dWr through the layer")


def test_router_full_size_dsv3_shape():
    """T=8192, H=7168, E=256, top-8 with a selection bias: selection exact on
    the kernel's keys, logits and scores on every token, dWr in full, dx on
    sampled rows."""
    require_gpu()
    T, H, E, k = 8192, 7168, 256, 8
    (x, Wr, bias, ds), (idx, s, logits, dWr, dx) = run_router(T, H, E, k, 5, True)
    rows = np.arange(0, T, 97)
    L_ref = np64(x[rows]) @ np64(Wr)
    assert rel_errors(logits[rows], L_ref)[1] < 1e-5
    np.testing.assert_array_equal(idx, selection_on(logits, bias, k))
    check_against_oracle_logits(x, Wr, bias, k, idx, s, logits)
    ch = np.take_along_axis(logits.astype(np.float64), idx.astype(np.int64), axis=1)
    ez = np.exp(ch - ch.max(axis=1, keepdims=True))
    np.testing.assert_allclose(s, ez / ez.sum(axis=1, keepdims=True), rtol=2e-6, atol=1e-7)
    dL = router.logit_grad(idx, s, np64(ds), E)
    assert_bf16_close(dWr, np64(x).T @ dL, "dWr")
    assert_bf16_close(dx[rows], dL[rows] @ np64(Wr).T, "dx_router rows")
