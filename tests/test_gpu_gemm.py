"""The tcgen05 grouped-GEMM kernels as plain dense GEMMs, against an FP64 CPU
matmul: K-major x K-major, K-major x MN-major, and MN-major x MN-major with fp32
accumulation into an existing buffer (the three operand layouts the routed path
uses), and the CTA-pair kernel (256 x 256 tiles) in both B layouts."""

import numpy as np
import pytest
import torch

from parity import compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    from routed_mixture_experts_gb300 import build

    build.build()
    import routed_mixture_experts_gb300 as m

    return m


@pytest.mark.parametrize("mode,M,N,K", [
    (0, 128, 64, 64), (0, 256, 256, 128), (0, 384, 512, 320), (0, 128, 128, 2048),
    (1, 128, 64, 64), (1, 256, 384, 192), (1, 512, 256, 1536),
    (2, 128, 64, 128), (2, 256, 512, 384), (2, 128, 256, 1024),
    (3, 256, 256, 64), (3, 512, 768, 320), (3, 768, 512, 2048),
    (4, 256, 256, 64), (4, 512, 512, 1536), (4, 1024, 256, 768),
])
def test_dense_gemm(moe, mode, M, N, K):
    g = torch.Generator().manual_seed(mode * 1000 + M + N + K)
    if mode in (0, 3):
        A = torch.randn(M, K, generator=g).bfloat16()
        B = torch.randn(N, K, generator=g).bfloat16()
        ref = A.double() @ B.double().T
    elif mode in (1, 4):
        A = torch.randn(M, K, generator=g).bfloat16()
        B = torch.randn(K, N, generator=g).bfloat16()
        ref = A.double() @ B.double()
    else:
        A = torch.randn(K, M, generator=g).bfloat16()
        B = torch.randn(K, N, generator=g).bfloat16()
        C0 = torch.randn(M, N, generator=g)
        ref = C0.double() + A.double().T @ B.double()
    Ad, Bd = A.cuda(), B.cuda()
    if mode == 2:
        C = C0.cuda()
    else:
        C = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    moe.gemm_bf16(mode, Ad, Bd, C, M, N, K)
    torch.cuda.synchronize()
    got = C.float().cpu().numpy()
    if mode == 2:
        assert np.max(np.abs(got - ref.numpy())) <= 1e-4 * np.abs(ref.numpy()).max()
    else:
        compare(got, ref.numpy(), bf16_out=True, what="gemm mode %d" % mode)
