"""Pins of the CPU oracle to things other than itself (no GPU needed).

Each test checks the oracle against a different formulation, a closed form,
a library routine, a brute-force search, or a value printed on the pages, so
that a dropped term, a wrong sign or index, or a transposed operand in the
oracle fails at least one of them.
"""

import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import heuristics, moe, mxfp8

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rand_layer(rng, T, H, I, E, k, allow_dup=False, empty=()):
    x = rng.standard_normal((T, H))
    W1 = rng.standard_normal((E, H, I)) * 0.3
    W3 = rng.standard_normal((E, H, I)) * 0.3
    W2 = rng.standard_normal((E, I, H)) * 0.3
    allowed = [e for e in range(E) if e not in empty]
    if allow_dup:
        idx = rng.choice(allowed, size=(T, k))
    else:
        idx = np.stack([rng.choice(allowed, size=k, replace=False) for _ in range(T)])
    s = rng.random((T, k)) + 0.1
    dout = rng.standard_normal((T, H))
    return x, idx, s, W1, W3, W2, dout


# ---------------------------------------------------------------------------
# schedule
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("T,k,E,case", [(37, 3, 7, "random"), (50, 2, 5, "one_hot"),
                                        (64, 4, 9, "empty"), (1, 1, 1, "single"),
                                        (300, 2, 4, "ragged")])
def test_schedule_brute_force(T, k, E, case):
    rng = np.random.default_rng(T * 1000 + E)
    if case == "one_hot":
        idx = np.full((T, k), 3)
    elif case == "empty":
        idx = rng.choice([0, 4, 8], size=(T, k))
    else:
        idx = rng.integers(0, E, size=(T, k))
    sch = moe.build_schedule(idx, E)
    flat = idx.reshape(-1).tolist()
    R = len(flat)
    brute = sorted(range(R), key=lambda f: (flat[f], f))
    assert sch["perm"].tolist() == brute
    for e in range(E):
        assert sch["counts"][e] == flat.count(e)
    assert sch["counts"].sum() == R and sch["offsets"][E] == R
    assert sorted(sch["perm"].tolist()) == list(range(R))
    assert all(sch["inv_perm"][sch["perm"][r]] == r for r in range(R))
    keys = [flat[f] for f in sch["perm"]]
    assert keys == sorted(keys)
    po = sch["padded_offsets"]
    assert all(v % 128 == 0 for v in po)
    for e in range(E):
        c = flat.count(e)
        assert po[e + 1] - po[e] == math.ceil(c / 128) * 128
        seg = sch["pad_perm"][po[e]:po[e + 1]].tolist()
        assert seg[:c] == [f for f in brute if flat[f] == e]
        assert all(v == -1 for v in seg[c:])
    for f in range(R):
        assert sch["pad_perm"][sch["pad_inv"][f]] == f
    te = sch["tile_expert"].tolist()
    assert len(te) == po[E] // 128
    for i, e in enumerate(te):
        assert po[e] <= i * 128 < po[e + 1]


def test_schedule_rejects_bad_index():
    with pytest.raises(ValueError):
        moe.build_schedule(np.array([[0, 5]]), 5)


# ---------------------------------------------------------------------------
# forward: brute-force dense routing
# ---------------------------------------------------------------------------

def dense_forward_loops(x, idx, s, W1, W3, W2):
    """Every token through every expert, weighted by the routing mask."""
    T, H = x.shape
    E = W1.shape[0]
    out = np.zeros((T, H))
    for t in range(T):
        for e in range(E):
            m = sum(s[t, j] for j in range(idx.shape[1]) if idx[t, j] == e)
            g = x[t] @ W1[e]
            up = x[t] @ W3[e]
            act = np.array([gi / (1.0 + math.exp(-gi)) for gi in g]) * up
            out[t] += m * (act @ W2[e])
    return out


@pytest.mark.parametrize("dup", [False, True])
def test_forward_matches_dense_brute_force(dup):
    rng = np.random.default_rng(7)
    x, idx, s, W1, W3, W2, _ = rand_layer(rng, 9, 16, 8, 5, 3, allow_dup=dup)
    out, _ = moe.forward(x, idx, s, W1, W3, W2)
    ref = dense_forward_loops(x, idx, s, W1, W3, W2)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)


def test_forward_dense_mlp_special_case():
    # E = 1, k = 1, s = 1: a dense SwiGLU MLP, written with torch ops.
    rng = np.random.default_rng(3)
    x, idx, s, W1, W3, W2, _ = rand_layer(rng, 11, 16, 8, 1, 1)
    s = np.ones_like(s)
    out, _ = moe.forward(x, idx, s, W1, W3, W2)
    X = torch.tensor(x)
    ref = (torch.nn.functional.silu(X @ torch.tensor(W1[0])) * (X @ torch.tensor(W3[0]))) @ torch.tensor(W2[0])
    np.testing.assert_allclose(out, ref.numpy(), rtol=1e-12, atol=1e-12)


def test_zero_down_projection():
    rng = np.random.default_rng(4)
    x, idx, s, W1, W3, W2, dout = rand_layer(rng, 6, 8, 4, 3, 2)
    W2 = np.zeros_like(W2)
    out, _ = moe.forward(x, idx, s, W1, W3, W2)
    assert np.all(out == 0)
    _, _, _, _, ds = moe.backward(x, idx, s, W1, W3, W2, dout)
    assert np.all(ds == 0)


# ---------------------------------------------------------------------------
# backward: float64 autograd of the dense formulation, finite differences
# ---------------------------------------------------------------------------

def dense_autograd(x, idx, s, W1, W3, W2, dout):
    X = torch.tensor(x, requires_grad=True)
    S = torch.tensor(s, requires_grad=True)
    A1 = torch.tensor(W1, requires_grad=True)
    A3 = torch.tensor(W3, requires_grad=True)
    A2 = torch.tensor(W2, requires_grad=True)
    E = W1.shape[0]
    onehot = torch.nn.functional.one_hot(torch.tensor(idx), E).to(torch.float64)  # [T,k,E]
    gate = torch.einsum("th,ehi->tei", X, A1)
    up = torch.einsum("th,ehi->tei", X, A3)
    y = torch.einsum("tei,eih->teh", torch.nn.functional.silu(gate) * up, A2)  # [T,E,H]
    out = torch.einsum("tj,tje,teh->th", S, onehot, y)
    (out * torch.tensor(dout)).sum().backward()
    return [t.grad.numpy() for t in (X, A1, A3, A2, S)]


@pytest.mark.parametrize("dup", [False, True])
def test_backward_matches_dense_autograd(dup):
    rng = np.random.default_rng(11)
    x, idx, s, W1, W3, W2, dout = rand_layer(rng, 10, 16, 8, 6, 3, allow_dup=dup, empty=(2,))
    got = moe.backward(x, idx, s, W1, W3, W2, dout)
    ref = dense_autograd(x, idx, s, W1, W3, W2, dout)
    for g, r in zip(got, ref):
        np.testing.assert_allclose(g, r, rtol=1e-10, atol=1e-12)


def test_backward_finite_differences():
    rng = np.random.default_rng(5)
    x, idx, s, W1, W3, W2, dout = rand_layer(rng, 4, 8, 4, 3, 2)
    grads = dict(zip(["x", "W1", "W3", "W2", "s"], moe.backward(x, idx, s, W1, W3, W2, dout)[:4] + (None,)))
    grads["s"] = moe.backward(x, idx, s, W1, W3, W2, dout)[4]
    params = dict(x=x, W1=W1, W3=W3, W2=W2, s=s)

    def loss(p):
        out, _ = moe.forward(p["x"], idx, p["s"], p["W1"], p["W3"], p["W2"])
        return float((out * dout).sum())

    eps = 1e-6
    for name, arr in params.items():
        fd = np.zeros_like(arr)
        for pos in itertools.product(*[range(n) for n in arr.shape]):
            plus = {kk: vv.copy() for kk, vv in params.items()}
            minus = {kk: vv.copy() for kk, vv in params.items()}
            plus[name][pos] += eps
            minus[name][pos] -= eps
            fd[pos] = (loss(plus) - loss(minus)) / (2 * eps)
        err = np.linalg.norm(fd - grads[name]) / np.linalg.norm(grads[name])
        assert err <= 1e-6, (name, err)


def test_permutation_invariance():
    rng = np.random.default_rng(9)
    x, idx, s, W1, W3, W2, dout = rand_layer(rng, 12, 16, 8, 5, 2)
    p = rng.permutation(12)
    out, _ = moe.forward(x, idx, s, W1, W3, W2)
    outp, _ = moe.forward(x[p], idx[p], s[p], W1, W3, W2)
    np.testing.assert_allclose(outp, out[p], rtol=1e-12, atol=1e-13)
    g = moe.backward(x, idx, s, W1, W3, W2, dout)
    gp = moe.backward(x[p], idx[p], s[p], W1, W3, W2, dout[p])
    np.testing.assert_allclose(gp[0], g[0][p], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(gp[4], g[4][p], rtol=1e-12, atol=1e-13)
    for a, b in zip(gp[1:4], g[1:4]):
        np.testing.assert_allclose(a, b, rtol=1e-11, atol=1e-12)


def test_empty_expert_gradients_are_exact_zero():
    rng = np.random.default_rng(12)
    x, idx, s, W1, W3, W2, dout = rand_layer(rng, 8, 8, 4, 4, 2, empty=(1, 3))
    _, dW1, dW3, dW2, _ = moe.backward(x, idx, s, W1, W3, W2, dout)
    for e in (1, 3):
        assert np.all(dW1[e] == 0) and np.all(dW3[e] == 0) and np.all(dW2[e] == 0)


def test_router_gradient_is_output_projection():
    # ds_f = <dout_t, y_f>: the gradient of the combine w.r.t. each score.
    rng = np.random.default_rng(13)
    x, idx, s, W1, W3, W2, dout = rand_layer(rng, 7, 8, 4, 3, 2)
    _, cache = moe.forward(x, idx, s, W1, W3, W2)
    ds = moe.backward(x, idx, s, W1, W3, W2, dout)[4].reshape(-1)
    tok = np.repeat(np.arange(7), 2)
    np.testing.assert_allclose(ds, np.einsum("fh,fh->f", dout[tok], cache["y"]), rtol=1e-12)


# ---------------------------------------------------------------------------
# MXFP8
# ---------------------------------------------------------------------------

def e4m3_table():
    vals = {}
    for c in range(256):
        sign = -1.0 if c & 0x80 else 1.0
        e, m = (c >> 3) & 0xF, c & 7
        if e == 15 and m == 7:
            continue
        v = (m / 8) * 2.0 ** -6 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7)
        vals[c] = sign * v
    return vals


def nearest_code_search(v, table):
    """Nearest finite E4M3 value by exhaustive search; ties to the even code."""
    if abs(v) > 448:
        return math.copysign(448.0, v)
    best = None
    for c, val in table.items():
        d = abs(val - v)
        key = (d, c & 1)
        if best is None or key < best[0]:
            best = (key, val)
    return best[1]


def test_e4m3_round_matches_exhaustive_search():
    table = e4m3_table()
    rng = np.random.default_rng(0)
    finite = sorted(set(table.values()))
    mids = [(a + b) / 2 for a, b in zip(finite[:-1], finite[1:])]
    samples = np.concatenate([rng.standard_normal(400) * 50, rng.standard_normal(200) * 0.01,
                              np.array(mids), np.array([500.0, -1000.0, 448.0, 464.0, 463.9, 0.0])])
    got = mxfp8.e4m3_round(samples)
    for v, g in zip(samples, got):
        assert g == nearest_code_search(float(v), table), v


def test_e4m3_codes_round_trip():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    vals = mxfp8.e4m3_decode(codes)
    table = e4m3_table()
    assert all(vals[i] == table[int(c)] for i, c in enumerate(codes))
    enc = mxfp8.e4m3_encode(vals)
    np.testing.assert_array_equal(enc, codes)
    assert np.isnan(mxfp8.e4m3_decode([0x7F, 0xFF])).all()
    assert mxfp8.e4m3_decode([0x7E])[0] == 448.0


def test_mx_scale_rule():
    rng = np.random.default_rng(1)
    a = rng.standard_normal((64, 96)) * np.exp2(rng.integers(-20, 20, size=(64, 1)))
    a[3, 32:64] = 0.0
    codes, sc, deq = mxfp8.quantize(a, axis=1)
    assert sc.shape == (64, 3)
    for r in range(64):
        for b in range(3):
            blk = a[r, 32 * b:32 * b + 32]
            amax = float(np.abs(blk).max())
            if amax == 0:
                assert sc[r, b] == 0 and np.all(codes[r, 32 * b:32 * b + 32] & 0x7F == 0)
                continue
            X = int(sc[r, b]) - 127
            # independent floor(log2) via math.frexp
            assert X == math.frexp(amax)[1] - 1 - 8
            assert 256 <= amax / 2.0 ** X < 512
    np.testing.assert_array_equal(mxfp8.e4m3_decode(codes) * np.exp2(np.repeat(sc.astype(float) - 127, 32, axis=1)), deq)


def test_exactly_representable_blocks_round_trip():
    rng = np.random.default_rng(2)
    codes = rng.integers(0, 0x7E, size=(8, 64)).astype(np.uint8)
    codes |= (rng.integers(0, 2, size=codes.shape) << 7).astype(np.uint8)
    codes[:, 0] = 0x79  # exponent field 15 (288): every block's amax lies in [256, 448]
    codes[:, 32] = 0x7A
    X = rng.integers(-20, 20, size=(8, 2))
    vals = mxfp8.e4m3_decode(codes) * np.exp2(np.repeat(X.astype(float), 32, axis=1))
    c2, s2, d2 = mxfp8.quantize(vals, axis=1)
    np.testing.assert_array_equal(s2.astype(int) - 127, X)
    np.testing.assert_array_equal(d2, vals)
    np.testing.assert_array_equal(mxfp8.e4m3_decode(c2), mxfp8.e4m3_decode(codes))


def test_quantize_axis_and_padding():
    rng = np.random.default_rng(6)
    a = rng.standard_normal((40, 64))
    d0 = mxfp8.qdq_rows_padded(a, axis=0)
    manual = mxfp8.qdq(np.vstack([a, np.zeros((24, 64))]), axis=0)[:40]
    np.testing.assert_array_equal(d0, manual)
    # along axis 0 differs from along axis 1 for generic data
    assert not np.array_equal(mxfp8.qdq(a[:32, :32], 0), mxfp8.qdq(a[:32, :32], 1))


def loop_qdq(a, axis, table):
    """Per-element loop quantiser: block amax, power-of-two scale by repeated
    halving/doubling, nearest code by exhaustive search."""
    a = np.moveaxis(np.array(a, dtype=np.float64), axis, -1).copy()
    flat = a.reshape(-1, a.shape[-1])
    for row in flat:
        for b0 in range(0, row.size, 32):
            blk = row[b0:b0 + 32]
            amax = max(abs(v) for v in blk)
            if amax == 0:
                continue
            X = 0
            while 2.0 ** (X + 1) <= amax:
                X += 1
            while 2.0 ** X > amax:
                X -= 1
            X -= 8
            for i in range(blk.size):
                blk[i] = nearest_code_search(blk[i] / 2.0 ** X, table) * 2.0 ** X
    return np.moveaxis(flat.reshape(a.shape), -1, axis)


def test_mxfp8_forward_matches_loop_quantiser():
    table = e4m3_table()
    rng = np.random.default_rng(21)
    T, H, I, E, k = 5, 64, 32, 3, 2
    x, idx, s, W1, W3, W2, _ = rand_layer(rng, T, H, I, E, k)
    out, _ = moe.forward(x, idx, s, W1, W3, W2, quant="mxfp8")
    xq = loop_qdq(x, 1, table)
    W1q, W3q, W2q = loop_qdq(W1, 1, table), loop_qdq(W3, 1, table), loop_qdq(W2, 1, table)
    ref = np.zeros((T, H))
    for t in range(T):
        for j in range(k):
            e = idx[t, j]
            g, up = xq[t] @ W1q[e], xq[t] @ W3q[e]
            act = g / (1 + np.exp(-g)) * up
            ref[t] += s[t, j] * (loop_qdq(act[None, :], 1, table)[0] @ W2q[e])
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)


def block_search_qdq(a, axis, table):
    """Quantise-dequantise along ``axis`` in blocks of 32 consecutive elements
    (a shorter last block stands for a zero-padded one: padding zeros never
    raise a block's amax).  The block exponent comes from repeated doubling or
    halving, and each element from an exhaustive search over the finite E4M3
    codes (nearest value, ties to the even code, saturating at 448).  Shares
    nothing with ``oracle.mxfp8`` but the format's definition."""
    codes = np.array(sorted(table), dtype=np.int64)
    vals = np.array([table[c] for c in codes])
    a = np.moveaxis(np.array(a, dtype=np.float64), axis, -1).copy()
    flat = a.reshape(-1, a.shape[-1])
    for row in flat:
        for b0 in range(0, row.size, 32):
            blk = row[b0:b0 + 32]
            amax = float(np.abs(blk).max())
            if amax == 0:
                continue
            X = 0
            while 2.0 ** (X + 1) <= amax:
                X += 1
            while 2.0 ** X > amax:
                X -= 1
            X -= 8
            v = np.clip(blk / 2.0 ** X, -448.0, 448.0)
            dist = np.abs(vals[None, :] - v[:, None])
            tie = dist == dist.min(axis=1, keepdims=True)
            pick = np.argmin(np.where(tie, codes[None, :] & 1, 2), axis=1)
            blk[:] = vals[pick] * 2.0 ** X
    return np.moveaxis(flat.reshape(a.shape), -1, axis)


def mxfp8_backward_per_row(x, idx, s, W1, W3, W2, dout, table):
    """The MXFP8 backward written per routed row, with every quantisation
    point spelled out (the points the GPU quantises at):
      forward   x, W1, W3 along H; a and W2 along I;
      dA'       dout and W2 along H;
      dX        dh, du and W1, W3 along I;
      dW        x, dh, du, s*a and dout along the expert's routed rows, in
                ascending flat-index order, in blocks of 32 per expert."""
    q = lambda arr, ax: block_search_qdq(arr, ax, table)
    T, H = x.shape
    k = idx.shape[1]
    E, _, I = W1.shape
    xH, W1H, W3H, W2I = q(x, 1), q(W1, 1), q(W3, 1), q(W2, 1)
    dOH, W2H, W1I, W3I = q(dout, 1), q(W2, 2), q(W1, 2), q(W3, 2)
    dX = np.zeros((T, H))
    ds = np.zeros((T, k))
    dW1, dW3, dW2 = np.zeros((E, H, I)), np.zeros((E, H, I)), np.zeros((E, I, H))
    rows_of = {e: [] for e in range(E)}
    for t in range(T):
        for j in range(k):
            e = int(idx[t, j])
            g, up = xH[t] @ W1H[e], xH[t] @ W3H[e]
            sig = 1.0 / (1.0 + np.exp(-g))
            act = g * sig * up
            dAp = dOH[t] @ W2H[e].T
            ds[t, j] = float(np.dot(dAp, act))
            dA = s[t, j] * dAp
            dh = dA * up * sig * (1.0 + g * (1.0 - sig))
            du = dA * g * sig
            dX[t] += q(dh[None, :], 1)[0] @ W1I[e].T + q(du[None, :], 1)[0] @ W3I[e].T
            rows_of[e].append((t, dh, du, s[t, j] * act))
    for e, rows in rows_of.items():
        if not rows:
            continue
        tt = [r[0] for r in rows]
        Xe, dOe = q(x[tt], 0), q(dout[tt], 0)
        dHe, dUe = q(np.array([r[1] for r in rows]), 0), q(np.array([r[2] for r in rows]), 0)
        Ase = q(np.array([r[3] for r in rows]), 0)
        for n in range(len(rows)):
            dW1[e] += np.outer(Xe[n], dHe[n])
            dW3[e] += np.outer(Xe[n], dUe[n])
            dW2[e] += np.outer(Ase[n], dOe[n])
    return dX, dW1, dW3, dW2, ds


def test_mxfp8_backward_matches_per_row_quantiser():
    # Expert 0 takes 36 routed rows (one full 32-row block and a ragged one),
    # experts 1 and 2 share the rest, so weight-gradient blocks that ran over
    # an expert's end, or that were taken along the wrong axis, would change
    # the result.
    table = e4m3_table()
    rng = np.random.default_rng(23)
    T, H, I, E, k = 40, 64, 32, 3, 2
    x, _, s, W1, W3, W2, dout = rand_layer(rng, T, H, I, E, k)
    idx = np.zeros((T, k), dtype=np.int64)
    idx[:36, 0] = 0
    idx[:36, 1] = rng.integers(1, 3, size=36)
    idx[36:] = [[1, 2], [2, 1], [2, 1], [1, 2]]
    got = moe.backward(x, idx, s, W1, W3, W2, dout, quant="mxfp8")
    ref = mxfp8_backward_per_row(x, idx, s, W1, W3, W2, dout, table)
    for name, g, r in zip(("dX", "dW1", "dW3", "dW2", "ds"), got, ref):
        np.testing.assert_allclose(g, r, rtol=1e-12, atol=1e-12 * float(np.abs(r).max()), err_msg=name)


def test_mxfp8_identity_on_prequantised_inputs():
    # Inputs already on the MXFP8 grid along every axis they are quantised
    # along (powers of two with a common exponent per block): the first GEMM
    # operands are unchanged, so h and u equal the BF16-mode values.
    rng = np.random.default_rng(22)
    T, H, I, E, k = 4, 64, 32, 2, 2
    x = np.exp2(rng.integers(-3, 3, size=(T, H))) * rng.choice([-1, 1], size=(T, H))
    W1 = np.exp2(rng.integers(-3, 3, size=(E, H, I))) * rng.choice([-1, 1], size=(E, H, I))
    W3 = np.exp2(rng.integers(-3, 3, size=(E, H, I))) * rng.choice([-1, 1], size=(E, H, I))
    W2 = np.zeros((E, I, H))
    idx = np.array([[0, 1]] * T)
    s = np.ones((T, k))
    _, c_b = moe.forward(x, idx, s, W1, W3, W2)
    _, c_q = moe.forward(x, idx, s, W1, W3, W2, quant="mxfp8")
    np.testing.assert_array_equal(c_b["h"], c_q["h"])
    np.testing.assert_array_equal(c_b["u"], c_q["u"])


# ---------------------------------------------------------------------------
# minibatch heuristic
# ---------------------------------------------------------------------------

def test_minibatch_floor_golden():
    with open(os.path.join(GOLDEN, "minibatch_floor.json")) as f:
        g = json.load(f)
    assert heuristics.minibatch_floor(g["H"], g["I"], g["num_sms"]) == g["expected_tokens"]
