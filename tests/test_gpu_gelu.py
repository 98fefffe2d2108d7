"""The GELU epilogue on every finite fp16 input, through each kernel that has it.

A @ I with an identity B is exact in fp32 (one product of 1, the rest zeros), so
each kernel's epilogue sees the fp16 input itself; the oracle's product with the
same identity applies GELU in fp64 and rounds once, i.e. it is the correctly
rounded fp16 GELU ("Designing high-performance GPU kernels with TileLang",
section 3, the GELU(MatMul + Bias) epilogue). Every kernel is held to one ulp of
it (the fp32 evaluation may land on the other side of a rounding boundary) on at
most 1% of the inputs; and since all kernels share one epilogue routine, they
must agree with one another bit for bit. The 4-bit kernels see the same inputs
through an INT4 identity with unit scales.
"""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

MAX_ULP = 1
MAX_MISMATCH_FRACTION = 0.01


@pytest.fixture(scope="module")
def tg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import tiled_tensor_core_tcgen05_gb300 as m
    torch.cuda.set_device(0)
    return m


def _all_finite_fp16(rows, cols):
    x = np.arange(65536, dtype=np.uint32).astype(np.uint16).view(np.float16)
    x = x[np.isfinite(x)]
    assert x.size == 63488 and x.size <= rows * cols
    out = np.zeros(rows * cols, dtype=np.float16)
    out[:x.size] = x
    return out.reshape(rows, cols)


def _ulps(got, ref):
    """Distance in fp16 ulps, on the sign-magnitude order (+0 and -0 coincide)."""
    def lin(a):
        b = np.asarray(a, dtype=np.float16).view(np.uint16).astype(np.int32)
        mag = b & 0x7FFF
        return np.where(b & 0x8000, -mag, mag)
    return np.abs(lin(got) - lin(ref))


def _check(got, ref, what):
    got = np.asarray(got)
    assert not np.isnan(got.astype(np.float64)).any(), f"{what}: NaN output on a finite input"
    d = _ulps(got, ref)
    assert d.max() <= MAX_ULP, f"{what}: {int(d.max())} ulps at {tuple(np.argwhere(d == d.max())[0])}"
    frac = (d != 0).mean()
    assert frac <= MAX_MISMATCH_FRACTION, f"{what}: {frac:.4f} of inputs off by one ulp"


def _status_ok(tg):
    st, where = tg.tg_device_status(None)
    assert st == tg.OK, f"device watchdog reported status {st} at wait site {where}"


def test_gemm_kernels_and_unfused_pass(tg):
    M, K = 124, 512
    A = _all_finite_fp16(M, K)
    eye = np.eye(K, dtype=np.float16)
    ref = oracle.gemm(A, eye, None, gelu=True)
    dA, dI = torch.from_numpy(A).cuda(), torch.from_numpy(eye).cuda()
    first = None
    for kernel in (tg.KERNEL_AUTO, tg.KERNEL_TILED_LSU, tg.KERNEL_TILED_TMA, tg.KERNEL_TILED_PAIR,
                   tg.KERNEL_SPLITK):
        C = tg.gemm(dA, dI, None, gelu=True, kernel=kernel).cpu().numpy()
        _check(C, ref, f"kernel {kernel}")
        if first is None:
            first = C
        assert np.array_equal(C.view(np.uint16), first.view(np.uint16)), f"kernel {kernel} differs from kernel 0"
    C = dA.clone()
    tg.bias_gelu_(C, None, gelu=True)
    C = C.cpu().numpy()
    _check(C, ref, "unfused pass")
    assert np.array_equal(C.view(np.uint16), first.view(np.uint16)), "unfused pass differs from the fused epilogue"
    _status_ok(tg)


def test_4bit_kernels(tg):
    M, K = 16, 4096
    N = K
    A = _all_finite_fp16(M, K)
    # INT4 identity: q[n][k] = 1 where n == k (low nibble = even k); unit scales, one per 128 rows of K
    q = np.zeros((N, K), dtype=np.uint8)
    q[np.arange(N), np.arange(K)] = 1
    Bq = (q[:, 0::2] | (q[:, 1::2] << 4)).astype(np.uint8)
    s = np.ones((K // 128, N), dtype=np.float16)
    ref = oracle.gemm_w4(A, Bq, s, None, gelu=True, fmt=0)
    dA, dBq, ds = (torch.from_numpy(t).cuda() for t in (A, Bq, s))
    outs = []
    for kernel in (tg.W4_KERNEL_TMEM, tg.W4_KERNEL_REG):
        C = tg.gemm_w4(dA, dBq, ds, None, gelu=True, fmt=0, kernel=kernel).cpu().numpy()
        _check(C, ref, f"4-bit kernel {kernel}")
        outs.append(C)
    assert np.array_equal(outs[0].view(np.uint16), outs[1].view(np.uint16))
    _status_ok(tg)
