"""The tcgen05 dense GEMM (C = A B^T, bf16 in, fp32 out) against fp64 matmul on the host."""
import numpy as np
import pytest
import torch

import latent_sparse_moe_router_b300 as ext

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (300, 512, 128), (1, 256, 2560), (4096, 1792, 2560),
                                   (777, 2560, 1792), (256, 300, 192)])
def test_gemm_bf16_tn_matches_fp64(M, N, K):
    g = torch.Generator().manual_seed(M * 7 + N * 3 + K)
    A = torch.randn(M, K, generator=g).to(torch.bfloat16)
    B = (torch.randn(N, K, generator=g) / K ** 0.5).to(torch.bfloat16)
    C = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ext.edge0_gemm_bf16_tn(A.cuda(), B.cuda(), C, M, N, K, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = A.double() @ B.double().T
    got = C.cpu().double()
    assert torch.isfinite(got).all()
    scale = ref.abs().max().item()
    assert (got - ref).abs().max().item() <= 1e-5 * scale * max(1.0, K / 256) + 1e-6
