"""Device schedule, bit-exact against the oracle (integer work)."""

import numpy as np
import pytest
import torch

from _helpers import require_gpu
from oracle import moe

pytestmark = pytest.mark.gpu


def routing(case, T, k, E, seed):
    from mixture_experts_layer_side_gb300.inputs import make_routing
    g = torch.Generator().manual_seed(seed)
    if case in ("uniform", "zipf", "hot"):
        idx, _ = make_routing(T, E, k, case, g, "cpu")
        return idx
    rng = np.random.default_rng(seed)
    if case == "one_expert":
        return torch.full((T, k), E // 2, dtype=torch.int32)
    if case == "empty":
        return torch.tensor(rng.choice([0, E - 1], size=(T, k)), dtype=torch.int32)
    return torch.tensor(rng.integers(0, E, size=(T, k)), dtype=torch.int32)


CASES = [("uniform", 256, 2, 8), ("zipf", 4096, 8, 64), ("hot", 4096, 8, 64), ("one_expert", 700, 1, 9),
         ("empty", 333, 3, 17), ("random", 1000, 3, 5), ("random", 1, 1, 1), ("zipf", 8192, 8, 256),
         ("uniform", 16384, 8, 384)]


@pytest.mark.parametrize("case,T,k,E", CASES)
def test_schedule_bit_exact(case, T, k, E):
    require_gpu()
    from mixture_experts_layer_side_gb300.inputs import Shape
    from mixture_experts_layer_side_gb300.layer import MoKLayer
    idx = routing(case, T, k, E, seed=T + E)
    layer = MoKLayer(Shape(T, 128, 128, E, k))
    layer.build_schedule(idx.cuda())
    layer.check()
    got = {n: a.cpu().numpy().astype(np.int64) for n, a in layer.schedule_arrays().items()}
    ref = moe.build_schedule(idx.numpy(), E)
    for name in ("counts", "offsets", "padded_offsets", "perm", "inv_perm", "pad_inv"):
        np.testing.assert_array_equal(got[name], ref[name], err_msg=name)
    used = int(ref["padded_offsets"][-1])
    assert got["header"][1] == used and got["header"][2] == used // 128
    np.testing.assert_array_equal(got["pad_perm"][:used], ref["pad_perm"])
    np.testing.assert_array_equal(got["tile_expert"][:used // 128], ref["tile_expert"])


def test_bad_expert_index_is_reported():
    require_gpu()
    from mixture_experts_layer_side_gb300 import _lib
    from mixture_experts_layer_side_gb300.inputs import Shape
    from mixture_experts_layer_side_gb300.layer import MoKLayer
    idx = torch.zeros((64, 2), dtype=torch.int32)
    idx[5, 1] = 8  # E = 8
    layer = MoKLayer(Shape(64, 128, 128, 8, 2))
    layer.build_schedule(idx.cuda())
    assert _lib.mok_check(layer.ws) == 5  # MOK_ERR_BAD_INDEX
    arr = layer.schedule_arrays()
    assert int(arr["pad_inv"][11]) == -1 and int(arr["counts"].sum()) == 127
    assert _lib.mok_check(layer.ws) == 0  # cleared
