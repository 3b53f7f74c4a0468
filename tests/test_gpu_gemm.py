"""The tensor-core projection kernel (tcgen05 + TMA + TMEM) against a plain
PyTorch fp32 reference of the same contraction, through the C ABI hook."""
import pytest
import torch

from tests import qwtest as Q

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def bd():
    from transformer_decode_qwen3_gb300 import binding
    binding.load()
    return binding


def _operands(M, N, K, seed):
    g = torch.Generator(device="cpu").manual_seed(seed)
    A = (torch.randn(M, K, generator=g) * 0.5).to(torch.bfloat16).cuda()
    B = (torch.randn(N, K, generator=g) * 0.02).to(torch.bfloat16).cuda()
    return A, B, A.float() @ B.float().T


@pytest.mark.parametrize("M,N,K,bn", [(128, 256, 64, 256), (1, 4096, 1024, 256), (5, 1024, 2048, 128),
                                      (300, 6144, 1024, 256), (64, 1024, 3072, 128), (257, 384, 1024, 256),
                                      (130, 151936, 1024, 256)])
def test_gemm_store(bd, M, N, K, bn):
    A, B, ref = _operands(M, N, K, M * 7 + N)
    C = torch.full((M, N), float("nan"), device="cuda")
    bd.debug_gemm(A, B, C, epi=0, bn=bn)
    torch.cuda.synchronize()
    err = (C - ref).norm() / ref.norm()
    assert torch.isfinite(C).all() and err < 1e-5, f"rel err {err:.3e}"


@pytest.mark.parametrize("M,N,K,bn", [(200, 1024, 2048, 128), (200, 1024, 2048, 256), (1, 1024, 3072, 256),
                                      (513, 1024, 3072, 256), (300, 192, 1024, 256)])
def test_gemm_residual_add(bd, M, N, K, bn):
    A, B, ref = _operands(M, N, K, 3 + M)
    X = torch.randn(M, N, device="cuda")
    C = X.clone()
    bd.debug_gemm(A, B, C, epi=1, bn=bn)
    torch.cuda.synchronize()
    torch.testing.assert_close(C, X + ref, rtol=1e-4, atol=1e-4)


def test_gemm_swiglu_pairs(bd):
    A, B, ref = _operands(130, 768, 256, 4)
    C = torch.zeros(130, 384, dtype=torch.bfloat16, device="cuda")
    bd.debug_gemm(A, B, C, epi=2, bn=256)
    torch.cuda.synchronize()
    g, u = ref[:, 0::2], ref[:, 1::2]
    expect = g * torch.sigmoid(g) * u
    torch.testing.assert_close(C.float(), expect, rtol=1e-2, atol=1e-3)


@pytest.mark.parametrize("M,N,K,bn,epi", [(1, 4096, 1024, 256, 0), (64, 1024, 2048, 128, 1), (65, 6144, 1024, 256, 2),
                                          (200, 1024, 3072, 128, 1), (16, 151936, 1024, 256, 0),
                                          (64, 4096, 1024, 32, 0), (3, 4096, 1024, 32, 0), (129, 4096, 1024, 32, 0),
                                          (64, 6144, 1024, 64, 2), (70, 6144, 1024, 64, 2), (64, 1024, 1024, 64, 0)])
def test_gemm_split_operand(bd, M, N, K, bn, epi):
    """Small-M mode: activations as bf16 hi/lo row pairs, summed in the epilogue (~16-bit mantissa)."""
    g = torch.Generator(device="cpu").manual_seed(M + N)
    a = (torch.randn(M, K, generator=g) * 0.5).cuda()
    B = (torch.randn(N, K, generator=g) * 0.02).to(torch.bfloat16).cuda()
    ref = a @ B.float().T
    A = Q.split_rows(a)
    if epi == 2:
        C = torch.zeros(A.shape[0], N // 2, dtype=torch.bfloat16, device="cuda")
        bd.debug_gemm(A, B, C, epi=2, bn=bn, split=True, M=M)
        torch.cuda.synchronize()
        idx = torch.arange(M, device="cuda")
        dst = (idx // 64) * 128 + idx % 64
        got = C[dst].float() + C[dst + 64].float()
        gt, up = ref[:, 0::2], ref[:, 1::2]
        expect = gt * torch.sigmoid(gt) * up
        err = (got - expect).norm() / expect.norm()
        assert err < 1e-4, f"rel err {err:.3e}"
        return
    X = torch.randn(M, N, device="cuda") if epi == 1 else torch.zeros(M, N, device="cuda")
    C = X.clone()
    bd.debug_gemm(A, B, C, epi=epi, bn=bn, split=True, M=M)
    torch.cuda.synchronize()
    err = (C - X - ref).norm() / ref.norm()
    assert err < 2e-5, f"rel err {err:.3e}"           # plain bf16 activations would give ~2e-3


@pytest.mark.parametrize("M,N,K,bn", [(1, 4096, 1024, 256), (64, 1024, 3072, 128), (64, 6144, 1024, 256),
                                      (200, 1024, 2048, 128), (64, 1024, 2048, 32), (64, 1024, 3072, 32),
                                      (5, 1024, 3072, 32), (130, 1024, 2048, 64)])
def test_gemm_split_k_atomic(bd, M, N, K, bn):
    """Small-M split-K: every SM takes a K slice and adds its partial product atomically."""
    g = torch.Generator(device="cpu").manual_seed(M * 3 + N)
    a = (torch.randn(M, K, generator=g) * 0.5).cuda()
    B = (torch.randn(N, K, generator=g) * 0.02).to(torch.bfloat16).cuda()
    X = torch.randn(M, N, device="cuda")
    C = X.clone()
    bd.debug_gemm(Q.split_rows(a), B, C, epi=3, bn=bn, split=True, M=M)
    torch.cuda.synchronize()
    ref = a @ B.float().T
    err = (C - X - ref).norm() / ref.norm()
    assert err < 2e-5, f"rel err {err:.3e}"


@pytest.mark.parametrize("M,N,K,epi", [(300, 6144, 1024, 0), (257, 384, 1024, 0), (384, 256, 64, 0),
                                       (129, 512, 128, 0), (513, 1024, 3072, 1), (300, 256, 1024, 1),
                                       (1000, 768, 256, 2), (2048, 4096, 1024, 0)])
def test_gemm_cta_pairs(bd, M, N, K, epi):
    """Large-M mode: CTA pairs multicast the shared weight tile (odd tile counts included)."""
    A, B, ref = _operands(M, N, K, 11 * M + N)
    if epi == 2:
        C = torch.zeros(M, N // 2, dtype=torch.bfloat16, device="cuda")
        bd.debug_gemm(A, B, C, epi=2, bn=256, split=2)
        torch.cuda.synchronize()
        g, u = ref[:, 0::2], ref[:, 1::2]
        torch.testing.assert_close(C.float(), g * torch.sigmoid(g) * u, rtol=1e-2, atol=1e-3)
        return
    X = torch.randn(M, N, device="cuda") if epi == 1 else torch.full((M, N), float("nan"), device="cuda")
    C = X.clone()
    bd.debug_gemm(A, B, C, epi=epi, bn=256, split=2)
    torch.cuda.synchronize()
    expect = X + ref if epi == 1 else ref
    err = (C - expect).norm() / expect.norm()
    assert torch.isfinite(C).all() and err < 1e-5, f"rel err {err:.3e}"
