"""The unfused comparator (tg_bias_gelu): the epilogue as its own pass over an
fp16 matrix, against the oracle. epi(C + bias) is the oracle's product with an
identity matrix, so the pass is checked against the same fp64 definition,
rounded once. A GEMM without epilogue followed by the pass must agree with the
oracle within the parity tolerance (it rounds the product to fp16 once more,
which the tolerance covers)."""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

RTOL = 1e-2
ATOL = 1e-2


@pytest.fixture(scope="module")
def tg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import tiled_tensor_core_tcgen05_gb300 as m
    torch.cuda.set_device(0)
    return m


def _tol(got, ref, what):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    bad = np.abs(got - ref) > ATOL + RTOL * np.abs(ref)
    assert np.isfinite(got).all() and not bad.any(), f"{what}: {int(bad.sum())} elements out of tolerance"


@pytest.mark.parametrize("M,N", [(64, 256), (33, 1030), (7, 13), (300, 2048)])
@pytest.mark.parametrize("gelu", [False, True])
def test_pass_matches_oracle(tg, M, N, gelu):
    g = torch.Generator().manual_seed(M * 1000 + N)
    Cin = (torch.rand((M, N), generator=g) * 6 - 3).to(torch.float16)
    bias = (torch.rand((N,), generator=g) * 0.2 - 0.1).to(torch.float16)
    ref = oracle.gemm(Cin, np.eye(N, dtype=np.float16), bias, gelu=gelu)   # epi(C + bias), rounded once
    C = Cin.cuda()
    tg.bias_gelu_(C, bias.cuda(), gelu=gelu)
    torch.cuda.synchronize()
    _tol(C.cpu().float().numpy(), ref.astype(np.float64), f"pass {M}x{N} gelu={gelu}")


def test_bias_only_is_exact_on_integers(tg):
    g = torch.Generator().manual_seed(7)
    Cin = torch.randint(-8, 9, (96, 520), generator=g).to(torch.float16)
    bias = torch.randint(-8, 9, (520,), generator=g).to(torch.float16)
    ref = oracle.gemm(Cin, np.eye(520, dtype=np.float16), bias).view(np.uint16)
    C = Cin.cuda()
    tg.bias_gelu_(C, bias.cuda(), gelu=False)
    assert np.array_equal(C.cpu().numpy().view(np.uint16), ref)


def test_unaligned_matrix_uses_the_element_path(tg):
    M, N = 40, 136
    g = torch.Generator().manual_seed(3)
    Cin = (torch.rand((M, N), generator=g) * 4 - 2).to(torch.float16)
    bias = (torch.rand((N,), generator=g) * 0.2 - 0.1).to(torch.float16)
    ref = oracle.gemm(Cin, np.eye(N, dtype=np.float16), bias, gelu=True)
    buf = torch.zeros(M * N + 1, dtype=torch.float16, device="cuda")
    C = buf[1:].view(M, N)   # 2-byte aligned only
    C.copy_(Cin)
    tg.bias_gelu_(C, bias.cuda(), gelu=True)
    _tol(C.cpu().float().numpy(), ref.astype(np.float64), "unaligned pass")


@pytest.mark.parametrize("w", [workloads.custom(512, 1024, 768, seed=61, dist=workloads.Dist("normal", 0, 0.05),
                                                bias=workloads.Dist("normal", 0, 0.02), gelu=True),
                               workloads.RAGGED_GELU], ids=lambda w: w.name)
def test_unfused_pipeline_matches_oracle(tg, w):
    A, B, bias = w.inputs()
    ref = oracle.gemm(A, B, bias, gelu=True).astype(np.float64)
    C = tg.gemm(A.cuda(), B.cuda(), None, gelu=False)
    tg.bias_gelu_(C, bias.cuda(), gelu=True)
    _tol(C.cpu().float().numpy(), ref, f"unfused {w.name}")
    fused = tg.gemm(A.cuda(), B.cuda(), bias.cuda(), gelu=True)
    _tol(fused.cpu().float().numpy(), ref, f"fused {w.name}")
