"""The C-ABI library builds, loads and exports every symbol the header
declares; host-side argument checks return their status before any device
work (no GPU needed)."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mok.h")


@pytest.fixture(scope="module")
def lib():
    from mixture_experts_layer_side_gb300 import build
    if not os.path.exists(build.LIB_PATH):
        build.build()
    from mixture_experts_layer_side_gb300 import _lib
    return _lib


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+char\s*\*|mok_status|size_t|int32_t|int64_t)\s+(mok_\w+)\s*\(",
                                 text, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("mok_build_schedule", "mok_forward", "mok_backward", "mok_mxfp8_quantize"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert set(names) == set(lib.EXPORTS)
    raw = ctypes.CDLL(lib.LIB_PATH)
    for n in names:
        assert hasattr(raw, n), n


def test_version_and_status_strings(lib):
    assert "sm_103a" in lib.mok_version()
    assert lib.mok_status_string(0) == "MOK_OK"
    assert lib.mok_status_string(6) == "MOK_ERR_TIMEOUT"


def test_host_argument_checks(lib):
    L = lib.LIB
    good = lib.shape_of(256, 256, 128, 8, 2)
    cfg = lib.config()
    assert lib.mok_workspace_size(good, cfg) > 0
    # a minibatch that is not a whole number of tiles is rounded up
    assert lib.mok_workspace_size(good, lib.config(minibatch_rows=2368, ring_slots=2)) == \
        lib.mok_workspace_size(good, lib.config(minibatch_rows=2432, ring_slots=2))
    # unsupported sizes
    for bad in (lib.shape_of(256, 100, 128, 8, 2), lib.shape_of(256, 256, 96, 8, 2),
                lib.shape_of(256, 256, 128, 2000, 2), lib.shape_of(0, 256, 128, 8, 2)):
        assert lib.mok_workspace_size(bad, cfg) == 0
    # comm_sms must be 0, minibatch >= 0, ring >= 2
    for badcfg in (lib.config(comm_sms=4), lib.config(minibatch_rows=-128), lib.config(ring_slots=1),
                   lib.config(capacity_mult=0.5)):
        assert lib.mok_workspace_size(good, badcfg) == 0
    fake = ctypes.c_void_p(256)
    S, C = ctypes.byref(good), ctypes.byref(cfg)
    # null pointers
    assert L.mok_forward(S, C, 0, None, 1 << 30, fake, fake, fake, fake, fake, fake, fake, None) == 1
    assert L.mok_build_schedule(S, C, fake, 1 << 30, None, None) == 1
    # workspace too small
    assert L.mok_forward(S, C, 0, fake, 16, fake, fake, fake, fake, fake, fake, fake, None) == 3
    assert L.mok_backward(S, C, 0, fake, 16, fake, fake, fake, fake, fake, fake, fake, fake, fake, fake, fake,
                          fake, None) == 3
    # bad config on a compute call
    bad = lib.config(comm_sms=1)
    assert L.mok_forward(S, ctypes.byref(bad), 0, fake, 1 << 30, fake, fake, fake, fake, fake, fake, fake,
                         None) == 1
    # quantiser argument checks
    assert L.mok_mxfp8_quantize(fake, 1, 64, 64, 2, fake, fake, None) == 1
    # the single-launch forward: null pointers, workspace too small, bad
    # config, unsupported shape
    F = L.mok_forward_fused
    assert F(S, C, 0, None, 1 << 30, fake, fake, fake, fake, fake, fake, fake, fake, None) == 1
    assert F(S, C, 0, fake, 1 << 30, None, fake, fake, fake, fake, fake, fake, fake, None) == 1
    assert F(S, C, 0, fake, 16, fake, fake, fake, fake, fake, fake, fake, fake, None) == 3
    assert F(S, ctypes.byref(bad), 0, fake, 1 << 30, fake, fake, fake, fake, fake, fake, fake, fake, None) == 1
    odd = lib.shape_of(256, 100, 128, 8, 2)
    assert F(ctypes.byref(odd), C, 0, fake, 1 << 30, fake, fake, fake, fake, fake, fake, fake, fake, None) == 2
    # an unknown precision; MXFP8 weights whose descriptors hold null pointers
    assert F(S, C, 7, fake, 1 << 30, fake, fake, fake, fake, fake, fake, fake, fake, None) == 1
    null_mx = lib.MokMx()
    px = ctypes.cast(ctypes.pointer(null_mx), ctypes.c_void_p)
    assert F(S, C, 1, fake, 1 << 30, fake, fake, fake, px, px, px, fake, fake, None) == 1
    assert L.mok_mxfp8_quantize(fake, 1, 48, 64, 0, fake, fake, None) == 2
    assert L.mok_mxfp8_quantize(fake, 1, 64, 48, 1, fake, fake, None) == 2
    # dense GEMM diagnostic: unsupported sizes
    assert L.mok_gemm_bf16(100, 128, 64, fake, 0, fake, 0, fake, fake, None) == 2


def test_workspace_layout_is_consistent(lib):
    shape = lib.shape_of(300, 256, 256, 6, 3)
    lay = lib.mok_workspace_layout(shape, lib.config())
    R, E = 900, 6
    assert lay["pad_capacity"] == (R + E * 127) // 128 * 128
    assert lay["tile_capacity"] == lay["pad_capacity"] // 128
    offs = [lay[k] for k in ("header", "counts", "offsets", "padded_offsets", "perm", "inv_perm", "pad_perm",
                             "pad_inv", "tile_expert")]
    assert offs == sorted(offs) and all(o % 256 == 0 for o in offs)
    assert lib.mok_workspace_size(shape, lib.config()) > lay["tile_expert"]


def test_bounded_context_size_and_checks(lib):
    """replay = 1: the forward context holds ring_slots minibatches of [h|u]
    (bf16, 2I columns) in both precisions; an MXFP8 backward with it needs
    W1 and W3 in both orientations and is refused on the host without."""
    L = lib.LIB
    shape = lib.shape_of(4096, 256, 128, 16, 4)
    plain = lib.config(minibatch_rows=128, ring_slots=2)
    bounded = lib.config(minibatch_rows=128, ring_slots=2, replay=1)
    pad = lib.mok_workspace_layout(shape, plain)["pad_capacity"]
    assert lib.mok_ctx_size(shape, plain) == pad * 2 * 128 * 2
    assert lib.mok_ctx_size(shape, bounded) == 2 * 128 * 2 * 128 * 2
    # a ring larger than the padded rows: no more than the padded rows
    big = lib.config(minibatch_rows=8192, ring_slots=4, replay=1)
    assert lib.mok_ctx_size(shape, big) == pad * 2 * 128 * 2
    assert lib.mok_ctx_size(shape, bounded, lib.MOK_MXFP8) == 2 * 128 * 2 * 128 * 2
    assert lib.mok_ctx_size(shape, lib.config(replay=2)) == 0
    fake = ctypes.c_void_p(256)
    S, C = ctypes.byref(shape), ctypes.byref(bounded)
    # the second (forward-orientation) descriptor of W1 / W3 missing: refused
    # before anything is enqueued
    pair = (lib.MokMx * 2)(lib.MokMx(256, 256), lib.MokMx(0, 0))
    one = lib.MokMx(256, 256)
    P = lambda t: ctypes.cast(t, ctypes.c_void_p)
    assert L.mok_backward(S, C, lib.MOK_MXFP8, fake, 1 << 30, fake, fake, fake, P(pair), P(pair),
                          P(ctypes.pointer(one)), fake, fake, fake, fake, fake, fake, None) == 1
