"""The tcgen05 GEMM core on dense problems, every operand major-ness, against
a plain fp32 PyTorch matmul of the same bf16 operands."""

import pytest
import torch

from _helpers import require_gpu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("a_mn,b_mn", [(0, 0), (0, 1), (1, 0), (1, 1)])
@pytest.mark.parametrize("M,N,K", [(256, 512, 320), (128, 384, 64), (384, 256, 1024)])
def test_dense_gemm(a_mn, b_mn, M, N, K):
    require_gpu()
    from mixture_experts_layer_side_gb300 import _lib
    g = torch.Generator(device="cuda").manual_seed(M * 7 + N * 3 + K + 11 * a_mn + 5 * b_mn)
    A_mk = torch.randn((M, K), generator=g, device="cuda").to(torch.bfloat16)
    B_kn = torch.randn((K, N), generator=g, device="cuda").to(torch.bfloat16)
    A = A_mk.t().contiguous() if a_mn else A_mk.contiguous()
    B = B_kn.contiguous() if b_mn else B_kn.t().contiguous()
    C = torch.full((M, N), float("nan"), device="cuda")
    scratch = torch.zeros(256, dtype=torch.uint8, device="cuda")
    _lib.mok_gemm_bf16(A, a_mn, B, b_mn, C, scratch)
    torch.cuda.synchronize()
    assert _lib.mok_check(scratch) == 0
    ref = A_mk.float() @ B_kn.float()
    err = (C - ref).abs().max().item()
    assert err <= 1e-3 * ref.abs().max().item(), (a_mn, b_mn, err)
