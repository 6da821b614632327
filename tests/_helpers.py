"""Shared test helpers: tolerances, oracle runs on seeded inputs."""

import numpy as np
import pytest
import torch

# Parity bar for BF16 outputs and gradients: max |err| <= 2e-2 * max |ref| and
# relative Frobenius error <= 1e-2; MXFP8 against the quantisation-applying
# oracle: relative Frobenius error <= 3e-2.
BF16_MAX_REL = 2e-2
BF16_FRO = 1e-2
MXFP8_FRO = 3e-2


def np64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def rel_errors(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(got - ref)
    ref_max = float(np.abs(ref).max()) if ref.size else 0.0
    ref_fro = float(np.linalg.norm(ref))
    max_rel = float(err.max()) / ref_max if ref_max > 0 else float(err.max())
    fro = float(np.linalg.norm(got - ref)) / ref_fro if ref_fro > 0 else float(np.linalg.norm(got - ref))
    return max_rel, fro


def assert_bf16_close(got, ref, name):
    max_rel, fro = rel_errors(got, ref)
    assert max_rel <= BF16_MAX_REL and fro <= BF16_FRO, f"{name}: max_rel={max_rel:.3e} fro={fro:.3e}"


def assert_mxfp8_close(got, ref, name):
    _, fro = rel_errors(got, ref)
    assert fro <= MXFP8_FRO, f"{name}: fro={fro:.3e}"


def require_gpu():
    if not torch.cuda.is_available():
        pytest.fail("this test needs a CUDA GPU")


def poisoned_outputs(layer):
    """Output and gradient buffers pre-filled with NaN, so that any element a
    call fails to write shows up in the comparison."""
    import torch
    grads = layer.alloc_grads()
    for t in grads.values():
        t.fill_(float("nan"))
    out = torch.full((layer.shape.T, layer.shape.H), float("nan"), dtype=torch.bfloat16, device=layer.device)
    return out, grads
