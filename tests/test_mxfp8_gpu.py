"""MXFP8: the quantiser bit-exact against the oracle, the block-scaled GEMM
core against an f32 matmul of the dequantised operands, and the layer's
MXFP8 forward + backward against the oracle that applies the same
quantisation (relative Frobenius error <= 3e-2)."""

import numpy as np
import pytest
import torch

from _helpers import assert_mxfp8_close, np64, require_gpu, poisoned_outputs
from oracle import moe, mxfp8

pytestmark = pytest.mark.gpu


def dequant(q, sf, axis):
    """E4M3 codes and E8M0 scales -> float32 (torch, on the device)."""
    v = q.view(torch.float8_e4m3fn).to(torch.float32)
    scale = torch.exp2(sf.to(torch.float32) - 127.0)
    return v * torch.repeat_interleave(scale, 32, dim=axis)


@pytest.mark.parametrize("axis", [0, 1])
def test_quantiser_bit_exact(axis):
    require_gpu()
    from mixture_experts_layer_side_gb300 import _lib
    g = torch.Generator().manual_seed(3 + axis)
    a = torch.randn((3, 64, 96), generator=g) * torch.exp2(torch.randint(-12, 12, (3, 64, 1), generator=g).float())
    a[0, :32, :] = 0.0          # an all-zero block
    a[1, 5, 7] = 3.0e4          # far above the block's other values (saturation of the rest)
    a = a.to(torch.bfloat16)
    q = torch.empty(a.shape, dtype=torch.uint8, device="cuda")
    sf_shape = (3, 64 // 32, 96) if axis == 0 else (3, 64, 96 // 32)
    sf = torch.empty(sf_shape, dtype=torch.uint8, device="cuda")
    _lib.mok_mxfp8_quantize(a.cuda(), axis, q, sf)
    torch.cuda.synchronize()
    codes, scales, _ = mxfp8.quantize(a.double().numpy(), axis=axis + 1)
    np.testing.assert_array_equal(sf.cpu().numpy(), scales)
    np.testing.assert_array_equal(q.cpu().numpy(), codes)


@pytest.mark.parametrize("a_mn,b_mn", [(0, 0), (0, 1), (1, 0), (1, 1)])
# K = 16384: a 128-row run of scale blocks (64 KB) exceeds the shared memory
# the scale-tiling kernels stage, so they take their one-word-per-thread forms
@pytest.mark.parametrize("M,N,K", [(256, 512, 384), (128, 384, 128), (128, 256, 16384)])
def test_mxfp8_gemm_core(a_mn, b_mn, M, N, K):
    require_gpu()
    from mixture_experts_layer_side_gb300 import _lib
    g = torch.Generator(device="cuda").manual_seed(M + N + K + 3 * a_mn + b_mn)
    A = torch.randn((M, K), generator=g, device="cuda").to(torch.bfloat16)
    B = torch.randn((K, N), generator=g, device="cuda").to(torch.bfloat16)

    def quant(X, axis):
        q = torch.empty(X.shape, dtype=torch.uint8, device="cuda")
        shape = (X.shape[0] // 32, X.shape[1]) if axis == 0 else (X.shape[0], X.shape[1] // 32)
        sf = torch.empty(shape, dtype=torch.uint8, device="cuda")
        _lib.mok_mxfp8_quantize(X.contiguous(), axis, q, sf)
        return q, sf

    # A blocks run along K: K-major A = [M, K] blocks along columns; M/N-major A = [K, M] blocks along rows
    Aq, Asf = quant(A.t(), 0) if a_mn else quant(A, 1)
    Bq, Bsf = quant(B, 0) if b_mn else quant(B.t(), 1)
    C = torch.full((M, N), float("nan"), device="cuda")
    scratch = torch.zeros(256 + M * K // 32 + N * K // 32, dtype=torch.uint8, device="cuda")
    _lib.mok_gemm_mxfp8(Aq, Asf, a_mn, Bq, Bsf, b_mn, C, scratch)
    torch.cuda.synchronize()
    Ad = dequant(Aq, Asf, 0).t() if a_mn else dequant(Aq, Asf, 1)
    Bd = dequant(Bq, Bsf, 0) if b_mn else dequant(Bq, Bsf, 1).t()
    ref = Ad @ Bd
    err = (C - ref).abs().max().item()
    assert err <= 1e-3 * ref.abs().max().item(), (a_mn, b_mn, err)


CASES = [
    ("tiny", (256, 256, 128, 8, 2), "uniform", 1),
    ("ragged_zipf", (300, 256, 256, 6, 3), "zipf", 2),
    ("hot_empty", (512, 384, 128, 24, 4), "hot", 3),
    # no expert empty and H = 384 (128-column dW2 tiles)
    ("uniform_h384", (512, 384, 128, 6, 2), "uniform", 4),
    # degenerate and limit cases: one token and one expert; the largest
    # expert count (most experts empty); the largest top-k; every token on
    # one expert (top-1, one long weight-gradient K loop, seven empty experts)
    ("single_token", (1, 128, 128, 1, 1), "uniform", 11),
    ("max_experts", (512, 128, 128, 1024, 4), "uniform", 12),
    ("max_topk", (64, 256, 128, 40, 32), "uniform", 13),
    ("one_expert", (2048, 256, 128, 8, 1), "all_on_5", 14),
]


def run_mx(shape, routing, seed, **kw):
    from mixture_experts_layer_side_gb300.inputs import Shape, make_inputs
    from mixture_experts_layer_side_gb300.layer import MoKLayer
    S = Shape(*shape)
    if routing == "all_on_5":
        inp = make_inputs(S, "uniform", seed=seed, device="cpu")
        inp["idx"] = torch.full((S.T, S.k), 5, dtype=torch.int32)
        inp["s"] = torch.ones((S.T, S.k), dtype=torch.float32)
    else:
        inp = make_inputs(S, routing, seed=seed, device="cpu")
    g = {k: v.cuda() for k, v in inp.items()}
    layer = MoKLayer(S, precision="mxfp8", **kw)
    wq = layer.quantize_weights(g["W1"], g["W3"], g["W2"])
    layer.build_schedule(g["idx"])
    out, grads = poisoned_outputs(layer)
    layer.forward(g["x"], g["s"], *wq["fwd"], out=out)
    layer.backward(g["x"], g["s"], *wq["bwd"], g["dout"], grads=grads)
    layer.check()
    return inp, out, grads


@pytest.mark.parametrize("name,shape,routing,seed", CASES)
def test_mxfp8_layer_matches_quantised_oracle(name, shape, routing, seed):
    require_gpu()
    inp, out, grads = run_mx(shape, routing, seed)
    a = {k: np64(v) if v.dtype != torch.int32 else v.numpy() for k, v in inp.items()}
    ref_out, _ = moe.forward(a["x"], a["idx"], a["s"], a["W1"], a["W3"], a["W2"], quant="mxfp8")
    ref = dict(zip(["dX", "dW1", "dW3", "dW2", "ds"],
                   moe.backward(a["x"], a["idx"], a["s"], a["W1"], a["W3"], a["W2"], a["dout"], quant="mxfp8")))
    assert_mxfp8_close(np64(out), ref_out, "out")
    for k in ref:
        assert_mxfp8_close(np64(grads[k]), ref[k], k)
    # experts with no routed rows: exact zeros
    counts = np.bincount(a["idx"].reshape(-1), minlength=shape[3])
    for e in np.nonzero(counts == 0)[0]:
        for k in ("dW1", "dW3", "dW2"):
            assert torch.count_nonzero(grads[k][e]).item() == 0


@pytest.mark.parametrize("shape,routing", [((512, 256, 256, 24, 4), "hot"), ((1000, 512, 256, 6, 3), "zipf")])
def test_mxfp8_sorted_and_gathered_code_rows_are_bitwise_equal(shape, routing):
    """GEMM1 and dA' reading x's / dout's E4M3 rows from token-sorted copies
    by plain TMA (default) against gathering them in the load path
    (MOK_DEBUG_GATHER_X_RING | MOK_DEBUG_FUSED_WGRAD_GATHER)."""
    require_gpu()
    _, out_s, g_s = run_mx(shape, routing, 7)
    _, out_g, g_g = run_mx(shape, routing, 7, debug_flags=64 | 4)
    assert torch.equal(out_s, out_g)
    for k in g_s:
        assert torch.equal(g_s[k], g_g[k]), k


def test_mxfp8_reruns_are_bitwise_identical():
    require_gpu()
    shape, routing = (512, 256, 256, 24, 4), "hot"
    _, out0, g0 = run_mx(shape, routing, 5)
    _, out1, g1 = run_mx(shape, routing, 5)
    assert torch.equal(out0, out1)
    for k in g0:
        assert torch.equal(g0[k], g1[k]), k
