"""Pins of the router oracle (CPU): brute-force selection, softmax special
cases, float64 autograd, finite differences, and the score gradient of the
layer oracle composed with the router backward against autograd of the
whole routed network."""

import numpy as np
import pytest
import torch

from oracle import moe, router


def test_selection_matches_brute_force_with_ties():
    rng = np.random.default_rng(0)
    for _ in range(20):
        T, E = 5, 7
        k = int(rng.integers(1, E + 1))
        # small integer keys force ties; the bias moves some of them
        L = rng.integers(-2, 3, size=(T, E)).astype(np.float64)
        b = rng.integers(-1, 2, size=E).astype(np.float64)
        idx, _ = router.topk_softmax(L, b, k)
        for t in range(T):
            key = L[t] + b
            want = sorted(range(E), key=lambda e: (-key[e], e))[:k]
            assert idx[t].tolist() == want


def test_scores_are_softmax_of_unbiased_chosen_logits():
    rng = np.random.default_rng(1)
    L = rng.normal(size=(4, 6))
    b = rng.normal(size=6) * 5
    idx, s = router.topk_softmax(L, b, 3)
    chosen = np.take_along_axis(L, idx, axis=1)
    want = np.exp(chosen) / np.exp(chosen).sum(axis=1, keepdims=True)
    np.testing.assert_allclose(s, want, rtol=1e-14)
    # k = E: every expert, softmax over the whole row
    idx, s = router.topk_softmax(L, None, 6)
    full = np.exp(L) / np.exp(L).sum(axis=1, keepdims=True)
    np.testing.assert_allclose(np.take_along_axis(full, idx, axis=1), s, rtol=1e-14)
    np.testing.assert_allclose(s.sum(axis=1), 1.0, rtol=1e-14)


def test_uniform_score_gradient_has_no_logit_gradient():
    # the scores sum to one, so a gradient equal across the k chosen is void
    rng = np.random.default_rng(2)
    L = rng.normal(size=(5, 9))
    idx, s = router.topk_softmax(L, None, 4)
    ds = np.repeat(rng.normal(size=(5, 1)), 4, axis=1)
    assert np.abs(router.logit_grad(idx, s, ds, 9)).max() < 1e-15


def test_backward_matches_autograd():
    rng = np.random.default_rng(3)
    T, H, E, k = 6, 8, 5, 2
    x = rng.normal(size=(T, H))
    Wr = rng.normal(size=(H, E))
    ds = rng.normal(size=(T, k))
    _, idx, s = router.router_forward(x, Wr, None, k)
    xt = torch.tensor(x, requires_grad=True)
    Wt = torch.tensor(Wr, requires_grad=True)
    chosen = torch.gather(xt @ Wt, 1, torch.tensor(idx))
    loss = (torch.softmax(chosen, dim=1) * torch.tensor(ds)).sum()
    loss.backward()
    dL, dWr, dx = router.router_backward(x, Wr, idx, s, ds)
    np.testing.assert_allclose(dWr, Wt.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dx, xt.grad.numpy(), rtol=1e-10, atol=1e-12)


def test_finite_differences_of_the_scores():
    rng = np.random.default_rng(4)
    T, H, E, k = 3, 4, 6, 3
    x = rng.normal(size=(T, H))
    Wr = rng.normal(size=(H, E))
    ds = rng.normal(size=(T, k))
    _, idx, s = router.router_forward(x, Wr, None, k)
    _, dWr, _ = router.router_backward(x, Wr, idx, s, ds)
    h = 1e-6
    for i in range(H):
        for e in range(E):
            Wp, Wm = Wr.copy(), Wr.copy()
            Wp[i, e] += h
            Wm[i, e] -= h
            # the selection is held fixed (it is piecewise constant)
            sp = _scores(x @ Wp, idx)
            sm = _scores(x @ Wm, idx)
            fd = ((sp - sm) * ds).sum() / (2 * h)
            assert abs(fd - dWr[i, e]) < 1e-7 * max(1.0, abs(fd))


def _scores(L, idx):
    c = np.take_along_axis(L, idx, axis=1)
    c = c - c.max(axis=1, keepdims=True)
    return np.exp(c) / np.exp(c).sum(axis=1, keepdims=True)


def test_layer_score_gradient_composes_to_router_weight_gradient():
    """d<dout, out>/dWr of the whole routed network (router + dense-form MoE,
    float64 autograd, selection fixed) equals router_backward applied to the
    layer oracle's score gradient."""
    rng = np.random.default_rng(5)
    T, H, I, E, k = 6, 8, 4, 5, 2
    x = rng.normal(size=(T, H))
    Wr = rng.normal(size=(H, E))
    W1, W3 = rng.normal(size=(E, H, I)), rng.normal(size=(E, H, I))
    W2 = rng.normal(size=(E, I, H))
    dout = rng.normal(size=(T, H))
    _, idx, s = router.router_forward(x, Wr, None, k)
    _, _, _, _, ds = moe.backward(x, idx, s, W1, W3, W2, dout)
    _, dWr, _ = router.router_backward(x, Wr, idx, s, ds)

    Wt = torch.tensor(Wr, requires_grad=True)
    xt = torch.tensor(x)
    st = torch.softmax(torch.gather(xt @ Wt, 1, torch.tensor(idx)), dim=1)
    out = torch.zeros(T, H, dtype=torch.float64)
    for t in range(T):
        for j in range(k):
            e = int(idx[t, j])
            h = xt[t] @ torch.tensor(W1[e])
            u = xt[t] @ torch.tensor(W3[e])
            out[t] = out[t] + st[t, j] * ((h * torch.sigmoid(h) * u) @ torch.tensor(W2[e]))
    (out * torch.tensor(dout)).sum().backward()
    np.testing.assert_allclose(dWr, Wt.grad.numpy(), rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("k", [1, 4])
def test_k_one_gives_unit_scores_and_zero_gradient(k):
    rng = np.random.default_rng(6)
    L = rng.normal(size=(4, 5))
    idx, s = router.topk_softmax(L, None, k)
    if k == 1:
        np.testing.assert_array_equal(s, 1.0)
        assert np.abs(router.logit_grad(idx, s, rng.normal(size=(4, 1)), 5)).max() == 0.0
    else:
        assert (np.diff(np.take_along_axis(L, idx, axis=1), axis=1) <= 0).all()
