"""The library's tcgen05/TMA GEMM core against a plain torch reference of the
same op (fp64 matmul of the same bf16 operands), for every operand layout the
loss uses (K-major and MN-major A and B), with ragged M, N, K tails, in both
forms: one CTA per 128 x 256 tile and a two-CTA cluster per 256 x 256 tile."""
import math

import pytest
import torch

from lm_head_top_tma_b300 import api

pytestmark = pytest.mark.gpu

SHAPES = [(128, 256, 64), (256, 512, 128), (296, 520, 200), (320, 448, 192), (384, 512, 2560), (1024, 768, 3072)]


@pytest.mark.parametrize("pair", [0, 1])
@pytest.mark.parametrize("a_mn,b_mn", [(0, 0), (0, 1), (1, 0), (1, 1)])
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_gemm_matches_torch(cuda_device, a_mn, b_mn, M, N, K, pair):
    g = torch.Generator(device=cuda_device).manual_seed(M * 7 + N * 3 + K)
    A = torch.randn(M, K, generator=g, device=cuda_device).to(torch.bfloat16)
    B = torch.randn(N, K, generator=g, device=cuda_device).to(torch.bfloat16)
    ref = (A.double() @ B.double().T).float()
    Aop = A.t().contiguous() if a_mn else A
    Bop = B.t().contiguous() if b_mn else B
    D = api.gemm_bf16(Aop, Bop, M, N, K, a_mn=bool(a_mn), b_mn=bool(b_mn), cta_pair=bool(pair))
    torch.cuda.synchronize()
    err = (D - ref).abs().max().item()
    assert err <= 2e-5 * math.sqrt(K) * ref.abs().max().item() + 1e-4, err


@pytest.mark.parametrize("pair", [0, 1])
def test_gemm_twice_same_bits(cuda_device, pair):
    g = torch.Generator(device=cuda_device).manual_seed(1)
    A = torch.randn(512, 1024, generator=g, device=cuda_device).to(torch.bfloat16)
    B = torch.randn(768, 1024, generator=g, device=cuda_device).to(torch.bfloat16)
    d1 = api.gemm_bf16(A, B, 512, 768, 1024, cta_pair=bool(pair))
    d2 = api.gemm_bf16(A, B, 512, 768, 1024, cta_pair=bool(pair))
    assert torch.equal(d1, d2)


def test_pair_and_single_forms_agree(cuda_device):
    """Both forms accumulate each output element over K in the same order."""
    g = torch.Generator(device=cuda_device).manual_seed(2)
    A = torch.randn(1024, 2048, generator=g, device=cuda_device).to(torch.bfloat16)
    B = torch.randn(1280, 2048, generator=g, device=cuda_device).to(torch.bfloat16)
    d1 = api.gemm_bf16(A, B, 1024, 1280, 2048, cta_pair=False)
    d2 = api.gemm_bf16(A, B, 1024, 1280, 2048, cta_pair=True)
    torch.cuda.synchronize()
    err = (d1 - d2).abs().max().item()
    assert err <= 1e-5 * d1.abs().max().item(), err
