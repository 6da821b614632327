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


def _buffers(layer):
    arr = layer.schedule_arrays()
    lens = {n: a.numel() for n, a in arr.items()}
    lens["header"] = 64
    return {n: torch.full((lens[n],), -7, dtype=torch.int32, device="cuda") for n in NAMES}


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
        for n in ("counts", "offsets", "padded_offsets", "perm", "inv_perm", "pad_inv"):
            assert torch.equal(bufs[n], ref[n]), (call, n)
        used = int(ref["header"][1])
        assert torch.equal(bufs["header"][:3], ref["header"][:3]), call
        assert torch.equal(bufs["pad_perm"][:used], ref["pad_perm"][:used]), call
        assert torch.equal(bufs["tile_expert"][:used // 128], ref["tile_expert"][:used // 128]), call


def test_noalloc_schedule_rejects_sizes_beyond_its_scratch():
    require_gpu()
    from mixture_experts_layer_side_gb300 import _lib
    # ceil(T*k / 1024) * E = 16384 * 16 > 131072 int32 pairs of the 1 MiB scratch
    shape = _lib.shape_of(1 << 21, 128, 128, 16, 8)
    tiny = {n: torch.zeros(64, dtype=torch.int32, device="cuda") for n in NAMES}
    with pytest.raises(_lib.MokError) as e:
        _lib.mok_build_schedule_noalloc(shape, torch.zeros(8, dtype=torch.int32, device="cuda"), tiny)
    assert e.value.status == 2  # MOK_ERR_UNSUPPORTED, nothing enqueued
