"""Top-k softmax router on either side of the layer, float64 reference (test
infrastructure only).

The pages take the routing as an input (``topk_experts`` of the schedule
call, *Mixture-of-Kittens (MoK)*, "Use the functional API") and say that the
router's weight gradients are computed with the SonicMoE-style score
gradient fused into the SwiGLU backward (*Cursor Open-Sources
Mixture-of-Kittens (MoK)*, the paragraph after "Three design decisions that
matter").  They do not print the router itself.  The plain reading, the one
the layer's inputs follow, is the DeepSeek-V3-style top-k softmax router:

    L = x Wr                    logits [T, E]  (Wr: [H, E])
    idx[t] = top-k of L[t] + b  selection only; b is a per-expert bias
                                (zero for a plain top-k router); ties go to
                                the lower expert id, columns in descending
                                key order
    s[t, j] = softmax_j L[t, idx[t, j]]   over the k chosen, unbiased logits

Backward, for the score gradient ds [T, k] of the layer (the selection is
piecewise constant, so it passes no gradient):

    dL[t, idx[t, j]] = s_j (ds_j - sum_i s_i ds_i),  dL = 0 elsewhere
    dWr = x^T dL,   dx = dL Wr^T   (the router's share of the input gradient)
"""

from __future__ import annotations

import numpy as np


def topk_softmax(logits, bias, k):
    """Selection and scores from given logits (float64 math on the values as
    given).  Returns (idx int64 [T, k], s float64 [T, k])."""
    L = np.asarray(logits, dtype=np.float64)
    T, E = L.shape
    key = L + (np.zeros(E) if bias is None else np.asarray(bias, dtype=np.float64))[None, :]
    # descending key, ascending expert id on ties: a stable sort of -key
    order = np.argsort(-key, axis=1, kind="stable")
    idx = order[:, :k].astype(np.int64)
    chosen = np.take_along_axis(L, idx, axis=1)
    z = chosen - chosen.max(axis=1, keepdims=True)
    ez = np.exp(z)
    s = ez / ez.sum(axis=1, keepdims=True)
    return idx, s


def router_forward(x, Wr, bias, k):
    """Logits, selection and scores.  Returns (logits [T, E], idx, s)."""
    L = np.asarray(x, dtype=np.float64) @ np.asarray(Wr, dtype=np.float64)
    idx, s = topk_softmax(L, bias, k)
    return L, idx, s


def logit_grad(idx, s, ds, E):
    """dL [T, E] from the score gradient (softmax over the chosen k)."""
    idx = np.asarray(idx, dtype=np.int64)
    s = np.asarray(s, dtype=np.float64)
    ds = np.asarray(ds, dtype=np.float64)
    T = idx.shape[0]
    g = s * (ds - (s * ds).sum(axis=1, keepdims=True))
    dL = np.zeros((T, E))
    np.put_along_axis(dL, idx, g, axis=1)
    return dL


def router_backward(x, Wr, idx, s, ds):
    """Returns (dL [T, E], dWr [H, E], dx [T, H])."""
    x = np.asarray(x, dtype=np.float64)
    Wr = np.asarray(Wr, dtype=np.float64)
    dL = logit_grad(idx, s, ds, Wr.shape[1])
    return dL, x.T @ dL, dL @ Wr.T
