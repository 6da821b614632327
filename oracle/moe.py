"""Routed SwiGLU MoE layer, float64 reference (test infrastructure only).

What the layer computes.  The pages describe the method's *system* design
(how tokens move and how work overlaps) but print none of the layer's
algebra.  The plain reading, which the rest of the pages supports, is the
standard routed SwiGLU mixture-of-experts layer:

* "expert-grouped GEMM" and "SwiGLU backward" (*Cursor Open-Sources
  Mixture-of-Kittens (MoK)*, "Three design decisions that matter",
  overlap-granularity paragraph, and the paragraph after that list);
* dispatch sends each token to its top-k experts, combine brings the k
  expert outputs back to the token and sums them (same section,
  communication-direction paragraph);
* the router-score gradient is computed inside the SwiGLU backward
  (the "SonicMoE-style" sentence of the paragraph after the list).

Notation: T tokens, H hidden, I expert intermediate, E experts, k top-k,
R = T*k routed rows; flat routed index f = t*k + j; W1 is the gate
projection (SiLU applied), W3 the up projection, W2 the down projection;
router scores s[t, j] weight the combine and are not applied inside the
expert.  Everything is float64 on inputs that are already bf16 values; no
intermediate is rounded (the GPU's bf16 intermediates are inside the parity
tolerance).  MXFP8 mode applies the block quantisation of ``oracle.mxfp8``
to every GEMM operand along that GEMM's K axis, then computes in float64.
"""

from __future__ import annotations

import numpy as np

from . import mxfp8

TILE_ROWS = 128  # rows per padded expert segment (one tensor-core M tile)


# ---------------------------------------------------------------------------
# schedule
# ---------------------------------------------------------------------------

def build_schedule(idx, num_experts, tile_rows=TILE_ROWS):
    """The one schedule table that serves dispatch, combine and both reverse
    directions (*Cursor Open-Sources Mixture-of-Kittens (MoK)*, "Three design
    decisions that matter", communication-direction paragraph).

    Sorted routed rows group the flat indices f by expert; within an expert
    the order is ascending f (a stable sort), which makes the permutation
    unique.  Each expert's segment is padded to a multiple of ``tile_rows``.

    Returns a dict of int64 arrays:
      counts[E], offsets[E+1]          rows per expert, exclusive scan
      perm[R]  (sorted r -> f),  inv_perm[R] (f -> r)
      padded_offsets[E+1]              exclusive scan of ceil(counts/P)*P
      pad_perm[padded_offsets[E]]      padded row -> f, or -1 for padding
      pad_inv[R]                       f -> padded row
      tile_expert[padded_offsets[E]/P] expert of each P-row tile
    """
    flat = np.asarray(idx, dtype=np.int64).reshape(-1)
    E = int(num_experts)
    if flat.size and (flat.min() < 0 or flat.max() >= E):
        raise ValueError("expert index out of range")
    R = flat.size
    counts = np.bincount(flat, minlength=E).astype(np.int64)
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    perm = np.argsort(flat, kind="stable").astype(np.int64)
    inv_perm = np.empty(R, dtype=np.int64)
    inv_perm[perm] = np.arange(R, dtype=np.int64)
    padded_counts = -(-counts // tile_rows) * tile_rows
    padded_offsets = np.zeros(E + 1, dtype=np.int64)
    padded_offsets[1:] = np.cumsum(padded_counts)
    pad_perm = np.full(int(padded_offsets[E]), -1, dtype=np.int64)
    pad_inv = np.empty(R, dtype=np.int64)
    for e in range(E):
        seg = perm[offsets[e]:offsets[e + 1]]
        rows = padded_offsets[e] + np.arange(seg.size)
        pad_perm[rows] = seg
        pad_inv[seg] = rows
    tile_expert = np.repeat(np.arange(E, dtype=np.int64), padded_counts // tile_rows)
    return dict(counts=counts, offsets=offsets, perm=perm, inv_perm=inv_perm,
                padded_offsets=padded_offsets, pad_perm=pad_perm, pad_inv=pad_inv,
                tile_expert=tile_expert)


# ---------------------------------------------------------------------------
# forward / backward
# ---------------------------------------------------------------------------

def sigmoid(h):
    return 1.0 / (1.0 + np.exp(-h))


def silu(h):
    return h * sigmoid(h)


def _f64(*arrays):
    return [np.asarray(a, dtype=np.float64) for a in arrays]


def forward(x, idx, s, W1, W3, W2, quant=None):
    """MoE layer forward.

    For each routed row f = (t, j) with e = idx[t, j]:
      h = x_t W1_e,  u = x_t W3_e,  a = silu(h) * u,  y_f = a W2_e
    and the combine  out_t = sum_j s[t, j] * y_(t, j).

    quant=None is the BF16 mode (inputs are bf16 values, math in float64);
    quant="mxfp8" quantises x and W1/W3 along H, a and W2 along I.
    Returns (out[T, H], cache) where cache holds h, u, a, y per routed row f.
    """
    x, s, W1, W3, W2 = _f64(x, s, W1, W3, W2)
    idx = np.asarray(idx, dtype=np.int64)
    T, H = x.shape
    k = idx.shape[1]
    E, _, I = W1.shape
    R = T * k
    flat = idx.reshape(-1)
    tok = np.repeat(np.arange(T), k)
    if quant == "mxfp8":
        xq = mxfp8.qdq(x, axis=1)
        W1q, W3q = mxfp8.qdq(W1, axis=1), mxfp8.qdq(W3, axis=1)
        W2q = mxfp8.qdq(W2, axis=1)
    elif quant is None:
        xq, W1q, W3q, W2q = x, W1, W3, W2
    else:
        raise ValueError(quant)
    h = np.zeros((R, I))
    u = np.zeros((R, I))
    a = np.zeros((R, I))
    y = np.zeros((R, H))
    for e in range(E):
        rows = np.nonzero(flat == e)[0]
        if rows.size == 0:
            continue
        Xe = xq[tok[rows]]
        h[rows] = Xe @ W1q[e]
        u[rows] = Xe @ W3q[e]
        a[rows] = silu(h[rows]) * u[rows]
        Ae = mxfp8.qdq(a[rows], axis=1) if quant else a[rows]
        y[rows] = Ae @ W2q[e]
    out = (s.reshape(R, 1) * y).reshape(T, k, H).sum(axis=1)
    return out, dict(h=h, u=u, a=a, y=y)


def backward(x, idx, s, W1, W3, W2, dout, quant=None):
    """MoE layer backward for the upstream gradient ``dout`` = dL/d out.

    Per routed row f = (t, j), e = idx[t, j]:
      dA'  = dout_t W2_e^T            (gradient w.r.t. a, before scaling by s)
      ds_f = <dA', a>                 router-score gradient, taken inside the
                                      SwiGLU backward (= <dout_t, y_f>)
      dA   = s_f dA'
      dh   = dA * u * sig(h) * (1 + h (1 - sig(h))),   du = dA * silu(h)
      dX_t += dh W1_e^T + du W3_e^T
      dW1_e += x_t^T dh,  dW3_e += x_t^T du,  dW2_e += (s_f a)^T dout_t

    MXFP8 mode quantises dout and W2 along H (dA'), dh|du and W1/W3 along I
    (dX), and every weight-gradient operand along its K axis, the expert's
    routed rows (zero-padded to a multiple of 32 per expert).
    Returns (dX[T,H], dW1[E,H,I], dW3[E,H,I], dW2[E,I,H], ds[T,k]).
    """
    x, s, W1, W3, W2, dout = _f64(x, s, W1, W3, W2, dout)
    idx = np.asarray(idx, dtype=np.int64)
    T, H = x.shape
    k = idx.shape[1]
    E, _, I = W1.shape
    R = T * k
    _, cache = forward(x, idx, s, W1, W3, W2, quant=quant)
    h, u, a = cache["h"], cache["u"], cache["a"]
    flat = idx.reshape(-1)
    tok = np.repeat(np.arange(T), k)
    sflat = s.reshape(R)
    if quant == "mxfp8":
        dOq = mxfp8.qdq(dout, axis=1)
        W2qH = mxfp8.qdq(W2, axis=2)
        W1qI, W3qI = mxfp8.qdq(W1, axis=2), mxfp8.qdq(W3, axis=2)
        rq = mxfp8.qdq_rows_padded
    else:
        dOq, W2qH, W1qI, W3qI = dout, W2, W1, W3
        rq = None
    dX = np.zeros((T, H))
    dW1 = np.zeros((E, H, I))
    dW3 = np.zeros((E, H, I))
    dW2 = np.zeros((E, I, H))
    ds = np.zeros(R)
    for e in range(E):
        rows = np.nonzero(flat == e)[0]
        if rows.size == 0:
            continue
        te = tok[rows]
        he, ue, ae = h[rows], u[rows], a[rows]
        dAp = dOq[te] @ W2qH[e].T
        ds[rows] = (dAp * ae).sum(axis=1)
        dA = sflat[rows, None] * dAp
        sg = sigmoid(he)
        dh = dA * ue * sg * (1.0 + he * (1.0 - sg))
        du = dA * he * sg
        if quant:
            dxr = mxfp8.qdq(dh, axis=1) @ W1qI[e].T + mxfp8.qdq(du, axis=1) @ W3qI[e].T
            Xg, dOg = x[te], dout[te]
            As = sflat[rows, None] * ae
            dW1[e] = rq(Xg).T @ rq(dh)
            dW3[e] = rq(Xg).T @ rq(du)
            dW2[e] = rq(As).T @ rq(dOg)
        else:
            dxr = dh @ W1[e].T + du @ W3[e].T
            dW1[e] = x[te].T @ dh
            dW3[e] = x[te].T @ du
            dW2[e] = (sflat[rows, None] * ae).T @ dout[te]
        np.add.at(dX, te, dxr)
    return dX, dW1, dW3, dW2, ds.reshape(T, k)
