"""mok_build_schedule_noalloc: the schedule built without any device
allocation by the library, checked against mok_build_schedule.

Some callers cannot allocate device memory: their device memory is all owned
by another allocator (a pool reserved once at start-up), or they must not
call cudaMalloc because it synchronises the whole device.  The no-allocation
entry point takes its scratch from a static array inside the library; the
caller passes only its routing and the output buffers.  This file is
collected last, so a run that stops at the first failure has already run
every other test.
"""

import pytest
import torch

from _helpers import require_gpu

pytestmark = pytest.mark.gpu

NAMES = ("header", "counts", "offsets", "padded_offsets", "perm", "inv_perm", "pad_perm", "pad_inv", "tile_expert")


def _buffers_for(arr):
    lens = {n: a.numel() for n, a in arr.items()}
    lens["header"] = 64
    return {n: torch.full((lens[n],), -7, dtype=torch.int32, device="cuda") for n in NAMES}


def _buffers(layer):
    return _buffers_for(layer.schedule_arrays())


def test_noalloc_schedule_matches_workspace_schedule_twice():
    require_gpu()
    from mixture_experts_layer_side_gb300 import _lib
    from mixture_experts_layer_side_gb300.inputs import Shape, make_routing
    from mixture_experts_layer_side_gb300.layer import MoKLayer

    for call, (kind, T, k, E, seed) in enumerate([("zipf", 4096, 8, 64, 1), ("hot", 2048, 4, 40, 2)]):
        g = torch.Generator().manual_seed(seed)
        idx, _ = make_routing(T, E, k, kind, g, "cpu")
        idx = idx.cuda()
        layer = MoKLayer(Shape(T, 128, 128, E, k))
        layer.build_schedule(idx)
        ref = {n: a.clone() for n, a in layer.schedule_arrays().items()}
        bufs = _buffers(layer)
        _lib.mok_build_schedule_noalloc(layer.cshape, idx, bufs)
        torch.cuda.synchronize()
        _compare(bufs, ref, call)


def _compare(bufs, ref, what):
    for n in ("counts", "offsets", "padded_offsets", "inv_perm", "pad_inv"):
        assert torch.equal(bufs[n], ref[n]), (what, n)
    # perm holds the routed rows only (an id outside [0, E) is routed nowhere)
    routed = int(ref["offsets"][-1])
    assert torch.equal(bufs["perm"][:routed], ref["perm"][:routed]), (what, "perm")
    used = int(ref["header"][1])
    assert torch.equal(bufs["header"][:3], ref["header"][:3]), what
    assert torch.equal(bufs["pad_perm"][:used], ref["pad_perm"][:used]), what
    assert torch.equal(bufs["tile_expert"][:used // 128], ref["tile_expert"][:used // 128]), what


def test_noalloc_schedule_at_its_scratch_limit():
    # ceil(T*k / 1024) * E = 2048 * 64 = 131072: the static scratch exactly
    # full, where an off-by-one would overrun it.  One expert more is refused.
    require_gpu()
    from mixture_experts_layer_side_gb300 import _lib
    from mixture_experts_layer_side_gb300.inputs import Shape, make_routing
    from mixture_experts_layer_side_gb300.layer import MoKLayer

    T, k, E = 262144, 8, 64
    g = torch.Generator().manual_seed(5)
    idx, _ = make_routing(T, E, k, "zipf", g, "cpu")
    idx = idx.cuda()
    layer = MoKLayer(Shape(T, 128, 128, E, k))
    layer.build_schedule(idx)
    ref = {n: a.clone() for n, a in layer.schedule_arrays().items()}
    del layer
    bufs = _buffers_for(ref)
    _lib.mok_build_schedule_noalloc(_lib.shape_of(T, 128, 128, E, k), idx, bufs)
    torch.cuda.synchronize()
    _compare(bufs, ref, "limit")
    with pytest.raises(_lib.MokError) as e:
        _lib.mok_build_schedule_noalloc(_lib.shape_of(T, 128, 128, E + 1, k), idx, bufs)
    assert e.value.status == 2  # MOK_ERR_UNSUPPORTED, nothing enqueued


def test_noalloc_schedule_reports_a_bad_expert_id():
    require_gpu()
    from mixture_experts_layer_side_gb300 import _lib
    from mixture_experts_layer_side_gb300.inputs import Shape, make_routing
    from mixture_experts_layer_side_gb300.layer import MoKLayer

    T, k, E = 1000, 4, 12
    g = torch.Generator().manual_seed(9)
    idx, _ = make_routing(T, E, k, "uniform", g, "cpu")
    idx[17, 2] = E       # one past the last expert
    idx[503, 0] = -1
    idx = idx.cuda()
    layer = MoKLayer(Shape(T, 128, 128, E, k))
    layer.build_schedule(idx)
    ref = {n: a.clone() for n, a in layer.schedule_arrays().items()}
    assert _lib.mok_check(layer.ws) == 5  # MOK_ERR_BAD_INDEX from the workspace path
    bufs = _buffers_for(ref)
    _lib.mok_build_schedule_noalloc(layer.cshape, idx, bufs)
    torch.cuda.synchronize()
    assert int(bufs["header"][0]) & 1, "the error bit of an id outside [0, E)"
    _compare(bufs, ref, "bad id")


def test_noalloc_schedule_rejects_a_stream_of_another_device():
    require_gpu()
    if torch.cuda.device_count() < 2:
        pytest.skip("needs a second GPU")
    from mixture_experts_layer_side_gb300 import _lib
    s1 = torch.cuda.Stream(device=1)
    tiny = {n: torch.zeros(64, dtype=torch.int32, device="cuda:0") for n in NAMES}
    with torch.cuda.device(0):
        with pytest.raises(_lib.MokError) as e:
            _lib.mok_build_schedule_noalloc(_lib.shape_of(8, 128, 128, 4, 2),
                                            torch.zeros(16, dtype=torch.int32, device="cuda:0"), tiny, s1)
    assert e.value.status == 1  # MOK_ERR_INVALID_ARG


def test_noalloc_schedule_rejects_sizes_beyond_its_scratch():
    require_gpu()
    from mixture_experts_layer_side_gb300 import _lib
    # ceil(T*k / 1024) * E = 16384 * 16 > 131072 int32 pairs of the 1 MiB scratch
    shape = _lib.shape_of(1 << 21, 128, 128, 16, 8)
    tiny = {n: torch.zeros(64, dtype=torch.int32, device="cuda") for n in NAMES}
    with pytest.raises(_lib.MokError) as e:
        _lib.mok_build_schedule_noalloc(shape, torch.zeros(8, dtype=torch.int32, device="cuda"), tiny)
    assert e.value.status == 2  # MOK_ERR_UNSUPPORTED, nothing enqueued
