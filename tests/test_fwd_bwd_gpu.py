"""BF16 forward and backward through the C ABI against the float64 oracle on
the same seeded inputs (sizes the oracle finishes in seconds, spanning several
tiles, ragged expert segments, empty experts and skewed routing)."""

import numpy as np
import pytest
import torch

from _helpers import assert_bf16_close, np64, require_gpu, poisoned_outputs
from oracle import moe

pytestmark = pytest.mark.gpu

# (name, shape (T, H, I, E, k), routing)
CASES = [
    ("tiny", (256, 256, 128, 8, 2), "uniform", 1),
    ("ragged_zipf", (300, 256, 256, 6, 3), "zipf", 2),
    ("hot_empty", (512, 384, 128, 24, 4), "hot", 3),
    ("wide", (200, 512, 384, 5, 2), "uniform", 4),
    # experts above 1,024 routed rows: long weight-gradient K loops
    ("long_k_a", (3000, 256, 128, 20, 2), "hot", 5),
    ("long_k_b", (4096, 256, 256, 20, 2), "hot", 6),
    # at least 1,024 routed rows per expert: weight gradients on CTA pairs
    ("pair_zipf", (4096, 256, 256, 8, 2), "zipf", 7),
    ("pair_uniform", (8192, 512, 256, 8, 1), "uniform", 8),
    # degenerate and limit cases: one token and one expert; the largest
    # expert count (most experts empty); the largest top-k
    ("single_token", (1, 128, 128, 1, 1), "uniform", 11),
    ("max_experts", (512, 128, 128, 1024, 4), "uniform", 12),
    ("max_topk", (64, 256, 128, 40, 32), "uniform", 13),
    # H >= 4096: dA' on CTA pairs too
    ("long_h_pairs", (768, 4096, 256, 6, 2), "zipf", 14),
]


def run_layer(shape, routing, seed, **kw):
    from mixture_experts_layer_side_gb300.inputs import Shape, make_inputs
    from mixture_experts_layer_side_gb300.layer import MoKLayer
    S = Shape(*shape)
    inp = make_inputs(S, routing, seed=seed, device="cpu")
    g = {k: v.cuda() for k, v in inp.items()}
    layer = MoKLayer(S, **kw)
    layer.build_schedule(g["idx"])
    out, grads = poisoned_outputs(layer)
    layer.forward(g["x"], g["s"], g["W1"], g["W3"], g["W2"], out=out)
    layer.backward(g["x"], g["s"], g["W1"], g["W3"], g["W2"], g["dout"], grads=grads)
    layer.check()
    return inp, out, grads


def oracle_run(inp):
    a = {k: np64(v) if v.dtype != torch.int32 else v.numpy() for k, v in inp.items()}
    out, _ = moe.forward(a["x"], a["idx"], a["s"], a["W1"], a["W3"], a["W2"])
    dX, dW1, dW3, dW2, ds = moe.backward(a["x"], a["idx"], a["s"], a["W1"], a["W3"], a["W2"], a["dout"])
    return dict(out=out, dX=dX, dW1=dW1, dW3=dW3, dW2=dW2, ds=ds)


@pytest.mark.parametrize("name,shape,routing,seed", CASES)
def test_forward_backward_match_oracle(name, shape, routing, seed):
    require_gpu()
    inp, out, grads = run_layer(shape, routing, seed=seed)
    ref = oracle_run(inp)
    assert_bf16_close(np64(out), ref["out"], "out")
    for k in ("dX", "dW1", "dW3", "dW2", "ds"):
        assert_bf16_close(np64(grads[k]), ref[k], k)
    # experts with no routed rows: exact zeros
    counts = np.bincount(inp["idx"].numpy().reshape(-1), minlength=shape[3])
    for e in np.nonzero(counts == 0)[0]:
        for k in ("dW1", "dW3", "dW2"):
            assert torch.count_nonzero(grads[k][e]).item() == 0


@pytest.mark.parametrize("minibatch_rows,ring_slots", [(128, 2), (256, 3), (0, 0)])
def test_ring_sizes_and_serial_path_are_bitwise_equal(minibatch_rows, ring_slots):
    require_gpu()
    shape, routing = (512, 256, 256, 12, 4), "zipf"
    _, out_a, g_a = run_layer(shape, routing, 3, minibatch_rows=minibatch_rows, ring_slots=ring_slots)
    _, out_b, g_b = run_layer(shape, routing, 3, minibatch_rows=minibatch_rows, ring_slots=ring_slots,
                              debug_flags=2)
    _, out_c, _ = run_layer(shape, routing, 3)
    assert torch.equal(out_a, out_b) and torch.equal(out_a, out_c)
    for k in g_a:
        assert torch.equal(g_a[k], g_b[k]), k


@pytest.mark.parametrize("shape,routing", [((512, 256, 256, 24, 4), "hot"), ((4096, 256, 256, 20, 2), "hot")])
def test_reruns_are_bitwise_identical(shape, routing):
    require_gpu()
    _, out0, g0 = run_layer(shape, routing, 5)
    for _ in range(3):
        _, out1, g1 = run_layer(shape, routing, 5)
        assert torch.equal(out0, out1)
        for k in g0:
            assert torch.equal(g0[k], g1[k]), k


@pytest.mark.parametrize("shape,routing", [((512, 256, 256, 24, 4), "hot"), ((4096, 256, 256, 20, 2), "hot")])
def test_backward_gather_paths_are_bitwise_equal(shape, routing):
    """dA' and the weight gradients: token-sorted copies + plain TMA (dA' on
    CTA pairs) vs gathers fused in the load path (dA' on single CTAs)."""
    require_gpu()
    _, _, g_sorted = run_layer(shape, routing, 8)
    _, _, g_fused = run_layer(shape, routing, 8, debug_flags=4)
    for k in g_sorted:
        assert torch.equal(g_sorted[k], g_fused[k]), k


@pytest.mark.parametrize("shape,routing", [((4096, 256, 256, 8, 2), "zipf"), ((8192, 512, 512, 6, 1), "uniform"),
                                           ((8192, 256, 256, 4, 2), "zipf")])
def test_weight_gradient_cta_pairs_match_single_cta(shape, routing):
    """BF16 weight gradients on clusters of two CTAs (one cta_group::2 MMA per
    256 x 256 tile) against one CTA per 128 x 256 tile: bitwise equal."""
    require_gpu()
    _, _, g_pair = run_layer(shape, routing, 9)
    _, _, g_one = run_layer(shape, routing, 9, debug_flags=8)
    for k in ("dW1", "dW3", "dW2"):
        assert torch.equal(g_pair[k], g_one[k]), k


@pytest.mark.parametrize("shape,routing,kw", [
    ((4096, 256, 256, 8, 2), "zipf", {}),
    # one tile per expert: every pair is a solo pair
    ((256, 256, 256, 16, 2), "uniform", {}),
    ((2048, 256, 256, 12, 4), "hot", dict(minibatch_rows=384, ring_slots=3)),
    # I = 128: dA' on single CTAs (128-column tiles), dX on pairs
    ((3000, 256, 128, 20, 2), "hot", {}),
    ((4096, 256, 256, 16, 4), "zipf", dict(replay=True, minibatch_rows=256, ring_slots=2)),
    # H >= 4096: dA' on pairs as well
    ((2048, 4096, 256, 8, 2), "zipf", {}),
    ((1024, 4096, 256, 24, 4), "hot", {}),
])
def test_backward_row_gemm_cta_pairs_match_single_cta(shape, routing, kw):
    """dA' and dX on clusters of two CTAs (two tiles of one expert per
    cta_group::2 MMA; a solo tile's second CTA idle) against one CTA per
    128-row tile: bitwise equal."""
    require_gpu()
    _, out_p, g_p = run_layer(shape, routing, 10, **kw)
    _, out_s, g_s = run_layer(shape, routing, 10, debug_flags=16, **kw)
    assert torch.equal(out_p, out_s)
    for k in g_p:
        assert torch.equal(g_p[k], g_s[k]), k


@pytest.mark.parametrize("shape,routing,kw", [
    ((4096, 256, 256, 8, 2), "zipf", {}),
    # one tile per expert: every pair is a solo pair
    ((256, 256, 256, 16, 2), "uniform", {}),
    # three and five tiles per minibatch: pairs stop at minibatch boundaries
    ((2048, 256, 256, 12, 4), "hot", dict(minibatch_rows=384, ring_slots=3)),
    ((1000, 512, 256, 6, 3), "uniform", dict(minibatch_rows=640, ring_slots=2)),
    ((4096, 256, 256, 16, 4), "zipf", dict(replay=True, minibatch_rows=256, ring_slots=2)),
    ((1024, 4096, 256, 24, 4), "hot", {}),
    # experts of 9 tiles: pair units with a solo each, whose empty walk
    # positions a later minibatch's GEMM1 reuses (small minibatches, 2 slots)
    ((2200, 256, 128, 4, 2), "uniform", dict(minibatch_rows=640, ring_slots=2)),
    ((2200, 256, 128, 4, 2), "uniform", dict(minibatch_rows=384, ring_slots=3)),
    # one expert far above 8 tiles, the rest on single CTAs
    ((4096, 512, 256, 40, 2), "hot", dict(minibatch_rows=1024, ring_slots=2)),
])
def test_forward_ring_cta_pairs_match_single_cta(shape, routing, kw):
    """The forward ring split in two launches (each expert's tiles two at a
    time on clusters of two CTAs, one cta_group::2 MMA per pair; the odd last
    tiles on single CTAs; token-sorted x by plain TMA), all tiles on single
    CTAs reading the sorted copy, and all on single CTAs gathering x in
    their load path: bitwise equal outputs, and the backward from each
    forward (which reuses the sorted x when there is one) bitwise equal."""
    require_gpu()
    _, out_p, g_p = run_layer(shape, routing, 15, **kw)
    _, out_s, g_s = run_layer(shape, routing, 15, debug_flags=32, **kw)
    _, out_t, g_t = run_layer(shape, routing, 15, debug_flags=32 | 64, **kw)
    assert torch.equal(out_p, out_s) and torch.equal(out_t, out_s)
    for k in g_p:
        assert torch.equal(g_p[k], g_s[k]) and torch.equal(g_t[k], g_s[k]), k


@pytest.mark.parametrize("shape,routing,kw", [
    # long experts on pairs, short ones beside them, empty experts
    ((4096, 256, 256, 32, 2), "zipf", {}),
    # experts of 9 tiles (pair units with solos), small minibatches
    ((2200, 256, 128, 4, 2), "uniform", dict(minibatch_rows=640, ring_slots=2)),
    # one hot expert on pairs beside many short ones; empty experts
    ((4096, 512, 256, 40, 2), "hot", dict(minibatch_rows=1024, ring_slots=2)),
    # no expert reaches 8 tiles: the short-expert launch holds every tile
    ((1024, 256, 256, 16, 2), "uniform", {}),
    # every expert long: the short-expert launch finds no tile
    ((4096, 256, 128, 2, 1), "uniform", {}),
])
@pytest.mark.parametrize("overlap_sms", [0, 1, 7])
def test_overlapped_launches_match_one_after_another(shape, routing, kw, overlap_sms):
    """The short experts' single-CTA ring launch overlapping the CTA-pair
    ring launch on one stream (programmatic dependent launch) -- with the
    library's SM share and with 1 and 7 SMs for the first launch -- against
    the two launches one after the other (MOK_DEBUG_NO_OVERLAP): bitwise
    equal outputs, and the backward from each bitwise equal."""
    require_gpu()
    _, out_o, g_o = run_layer(shape, routing, 21, overlap_sms=overlap_sms, **kw)
    _, out_n, g_n = run_layer(shape, routing, 21, debug_flags=128, **kw)
    assert torch.equal(out_o, out_n)
    for k in g_o:
        assert torch.equal(g_o[k], g_n[k]), k


def _run_with_idx(shape, idx, seed):
    from mixture_experts_layer_side_gb300.inputs import Shape, make_inputs
    from mixture_experts_layer_side_gb300.layer import MoKLayer
    S = Shape(*shape)
    inp = make_inputs(S, "uniform", seed=seed, device="cpu")
    inp["idx"] = idx.to(torch.int32).contiguous()
    g = {k: v.cuda() for k, v in inp.items()}
    layer = MoKLayer(S)
    layer.build_schedule(g["idx"])
    out, grads = poisoned_outputs(layer)
    layer.forward(g["x"], g["s"], g["W1"], g["W3"], g["W2"], out=out)
    layer.backward(g["x"], g["s"], g["W1"], g["W3"], g["W2"], g["dout"], grads=grads)
    layer.check()
    ref = oracle_run(inp)
    assert_bf16_close(np64(out), ref["out"], "out")
    for k in ("dX", "dW1", "dW3", "dW2", "ds"):
        assert_bf16_close(np64(grads[k]), ref[k], k)
    return inp, grads


def test_every_token_on_one_expert():
    """All 2,048 tokens routed to expert 5 of 8 (top-1): one long expert on
    the CTA-pair weight-gradient path, seven exact-zero experts."""
    require_gpu()
    shape = (2048, 256, 128, 8, 1)
    _, grads = _run_with_idx(shape, torch.full((2048, 1), 5), 51)
    for e in range(8):
        if e != 5:
            for k in ("dW1", "dW3", "dW2"):
                assert torch.count_nonzero(grads[k][e]).item() == 0


def test_duplicate_experts_within_a_token():
    """Half the tokens pick the same expert twice (legal: the rows are
    independent routed rows)."""
    require_gpu()
    T, E, k = 600, 6, 2
    g = torch.Generator().manual_seed(52)
    idx = torch.randint(0, E, (T, k), generator=g)
    idx[::2, 1] = idx[::2, 0]
    _run_with_idx((T, 256, 128, E, k), idx, 52)
