"""GPU parity of the 4-bit GEMM's register-dequant kernel (TG_W4_KERNEL_REG:
weights decoded in registers into warp-level 16-row MMAs), through the C ABI,
against the fp64 CPU oracle on the same seeded inputs, and against the
tensor-memory kernel (TG_W4_KERNEL_TMEM).

Integer activations with power-of-two scales make every product and partial
sum exact in fp32: both kernels must then match the oracle bit for bit, INT4
and FP4, with and without bias, for M from 1 to 16 and ragged N and K (a K
that ends half-way through a 256-k chunk, N not a multiple of the 64-column
block). Float inputs use the GEMM tolerance |gpu - ref| <= 1e-2 + 1e-2 |ref|,
element by element, up to the full decode shape; repeated launches must be
bit-identical (the kernel's ring has no race that timing could expose).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

RTOL = 1e-2
ATOL = 1e-2
INT2 = workloads.Dist("int", -2, 2)


@pytest.fixture(scope="module")
def tg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import tiled_tensor_core_tcgen05_gb300 as m
    torch.cuda.set_device(0)
    return m


def _dev(*ts):
    return [t.cuda() if t is not None else None for t in ts]


def _status_ok(tg):
    st, where = tg.tg_device_status(None)
    assert st == tg.OK, f"device watchdog reported status {st} at wait site {where}"


def _check_tol(got, ref, what):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - ref)
    bad = err > ATOL + RTOL * np.abs(ref)
    if bad.any():
        idx = tuple(np.argwhere(bad)[0])
        pytest.fail(f"{what}: {int(bad.sum())}/{bad.size} elements out of tolerance; first {idx}: "
                    f"gpu={got[idx]} ref={ref[idx]} (max err {err.max():.4g})")


def _bitwise(got, ref, what):
    got = np.asarray(got).view(np.uint16)
    ref = np.asarray(ref).view(np.uint16)
    mism = np.argwhere(got != ref)
    assert mism.size == 0, (f"{what}: {len(mism)} mismatches, first {tuple(mism[0])}: "
                            f"gpu={got[tuple(mism[0])]:#06x} ref={ref[tuple(mism[0])]:#06x}")


# (M, N, K): one row; a full 16-row MMA; N below, at and past a 64-column block;
# K = 128 and 384 end half-way through a 256-k chunk; K = 8192 runs 32 chunks
EXACT = [
    (1, 8, 128), (16, 64, 256), (5, 136, 384), (16, 200, 640), (3, 1032, 1152), (16, 72, 128),
    (8, 520, 8192), (12, 9728, 256), (16, 4160, 1024),
]
FMTS = [("int4", 0), ("fp4", 1)]


@pytest.mark.parametrize("fmt,code", FMTS, ids=[f for f, _ in FMTS])
@pytest.mark.parametrize("M,N,K", EXACT, ids=[f"{m}x{n}x{k}" for m, n, k in EXACT])
def test_exact_inputs_bitwise_both_kernels(tg, M, N, K, fmt, code):
    w = workloads.W4Workload(f"reg_exact_{M}x{N}x{K}", M, N, K, seed=M * 7 + N + 3 * K, a_dist=INT2,
                             bias_dist=INT2, scale_kind="pow2", fmt=fmt)
    A, Bq, s, bias = w.inputs()
    dA, dBq, ds, dbias = _dev(A, Bq, s, bias)
    for with_bias in (True, False):
        b = bias if with_bias else None
        db = dbias if with_bias else None
        ref = oracle.gemm_w4(A, Bq, s, b, fmt=code)
        reg = tg.gemm_w4(dA, dBq, ds, db, fmt=code, kernel=tg.W4_KERNEL_REG).cpu().numpy()
        _bitwise(reg, ref, f"register kernel, bias={with_bias}")
        tmem = tg.gemm_w4(dA, dBq, ds, db, fmt=code, kernel=tg.W4_KERNEL_TMEM, split_k=1).cpu().numpy()
        _bitwise(reg, tmem, f"register vs tensor-memory kernel, bias={with_bias}")
    # the GELU epilogue: the two kernels share it, so they agree bit for bit; the oracle within tolerance
    ref = oracle.gemm_w4(A, Bq, s, bias, gelu=True, fmt=code)
    reg = tg.gemm_w4(dA, dBq, ds, dbias, gelu=True, fmt=code, kernel=tg.W4_KERNEL_REG).cpu().numpy()
    tmem = tg.gemm_w4(dA, dBq, ds, dbias, gelu=True, fmt=code, kernel=tg.W4_KERNEL_TMEM, split_k=1).cpu().numpy()
    _bitwise(reg, tmem, "register vs tensor-memory kernel, GELU")
    _check_tol(reg, ref, "register kernel, GELU")
    _status_ok(tg)


@pytest.mark.parametrize("fmt,code", FMTS, ids=[f for f, _ in FMTS])
@pytest.mark.parametrize("M,N,K,gelu", [
    (16, 4096, 4096, True), (1, 1024, 2048, False), (7, 1000, 1152, True), (16, 9728, 8192, False),
])
def test_random_inputs(tg, M, N, K, gelu, fmt, code):
    w = workloads.W4Workload(f"reg_rand_{M}x{N}x{K}", M, N, K, seed=M + N + K + code,
                             bias_dist=workloads.Dist("normal", 0.0, 0.02), gelu=gelu, fmt=fmt)
    A, Bq, s, bias = w.inputs()
    ref = oracle.gemm_w4(A, Bq, s, bias, gelu=gelu, fmt=code)
    C = tg.gemm_w4(*_dev(A, Bq, s, bias), gelu=gelu, fmt=code, kernel=tg.W4_KERNEL_REG)
    _check_tol(C.cpu().numpy(), ref, f"{fmt} {M}x{N}x{K}")
    _status_ok(tg)


@pytest.mark.parametrize("w", [workloads.DECODE_W4, workloads.DECODE_FP4], ids=["int4", "fp4"])
def test_decode_shape_every_element_and_repeatable(tg, w):
    """The full decode shape (16 x 28672 x 8192), which the automatic choice
    sends to this kernel: every element within tolerance of the oracle, eight
    launches bit-identical, and the same bits as asking for the kernel by name."""
    A, Bq, s, bias = w.inputs()
    ref = oracle.gemm_w4(A, Bq, s, bias, gelu=w.gelu, fmt=w.fmt_code)
    dA, dBq, ds, dbias = _dev(A, Bq, s, bias)
    first = tg.gemm_w4(dA, dBq, ds, dbias, gelu=w.gelu, fmt=w.fmt_code, kernel=tg.W4_KERNEL_REG).cpu().numpy()
    _check_tol(first, ref, f"{w.name}")
    for _ in range(7):
        again = tg.gemm_w4(dA, dBq, ds, dbias, gelu=w.gelu, fmt=w.fmt_code, kernel=tg.W4_KERNEL_REG)
        _bitwise(again.cpu().numpy(), first, "repeated launch")
    auto = tg.gemm_w4(dA, dBq, ds, dbias, gelu=w.gelu, fmt=w.fmt_code).cpu().numpy()
    _bitwise(auto, first, "automatic choice")
    _status_ok(tg)


def test_unaligned_output_uses_single_stores(tg):
    """C at a 2-byte offset (not 4-byte aligned): the epilogue stores halves."""
    w = workloads.W4Workload("reg_unaligned_c", 4, 136, 256, seed=11, a_dist=INT2, bias_dist=INT2,
                             scale_kind="pow2")
    A, Bq, s, bias = w.inputs()
    ref = oracle.gemm_w4(A, Bq, s, bias)
    dA, dBq, ds, dbias = _dev(A, Bq, s, bias)
    buf = torch.full((4 * 136 + 1,), float("nan"), dtype=torch.float16, device="cuda")
    tg.tg_gemm_w4_kernel(dA.data_ptr(), dBq.data_ptr(), ds.data_ptr(), dbias.data_ptr(), buf.data_ptr() + 2,
                         4, 136, 256, tg.EPI_NONE, tg.W4_INT4, tg.W4_KERNEL_REG, 0, None)
    torch.cuda.synchronize()
    got = buf[1:].view(4, 136).cpu().numpy()
    _bitwise(got, ref, "unaligned C")
    assert torch.isnan(buf[0]).item(), "the element before C was written"
    _status_ok(tg)


def test_rejected_arguments(tg):
    A = torch.zeros((17, 256), dtype=torch.float16, device="cuda")
    Bq = torch.zeros((64, 128), dtype=torch.uint8, device="cuda")
    s = torch.zeros((2, 64), dtype=torch.float16, device="cuda")
    with pytest.raises(tg.TgError) as e:
        tg.gemm_w4(A, Bq, s, kernel=tg.W4_KERNEL_REG)
    assert e.value.status == tg.ERR_INVALID_ARG
    with pytest.raises(tg.TgError) as e:
        tg.gemm_w4(A[:16], Bq, s, kernel=tg.W4_KERNEL_REG, split_k=2)
    assert e.value.status == tg.ERR_INVALID_ARG
    with pytest.raises(tg.TgError) as e:
        tg.gemm_w4(A[:16], Bq, s, kernel=3)
    assert e.value.status == tg.ERR_INVALID_ARG
    # 17 rows on the tensor-memory kernel, and the automatic choice, are fine
    C = tg.gemm_w4(A, Bq, s, kernel=tg.W4_KERNEL_TMEM)
    assert torch.count_nonzero(C).item() == 0
    _status_ok(tg)
