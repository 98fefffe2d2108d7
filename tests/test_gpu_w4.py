"""GPU parity of the weight-only 4-bit GEMM (tg_gemm_w4), through the C ABI,
against the fp64 CPU oracle's dequantize-then-multiply on the same seeded
inputs.

Integer activations with power-of-two scales make every product and partial
sum exact in fp32, so those cases must match bit for bit for every split
count. Float inputs use the GEMM tolerance |gpu - ref| <= 1e-2 + 1e-2 |ref|,
element by element, up to the full decode shape 16 x 28672 x 8192.
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


EXACT = [
    (1, 8, 128), (16, 128, 256), (5, 136, 384), (17, 264, 128), (64, 1024, 1024), (128, 256, 512),
    (100, 520, 640), (33, 16, 896), (16, 3584, 1024), (112, 200, 256), (48, 392, 2048),
]


@pytest.mark.parametrize("M,N,K", EXACT, ids=[f"{m}x{n}x{k}" for m, n, k in EXACT])
def test_exact_inputs_bitwise_every_split(tg, M, N, K):
    w = workloads.W4Workload(f"exact_{M}x{N}x{K}", M, N, K, seed=M * 31 + N + K, a_dist=INT2,
                             bias_dist=INT2, scale_kind="pow2")
    A, Bq, s, bias = w.inputs()
    dA, dBq, ds, dbias = _dev(A, Bq, s, bias)
    for with_bias in (True, False):
        ref = oracle.gemm_w4(A, Bq, s, bias if with_bias else None).view(np.uint16)
        kb = (K + 255) // 256
        for split_k in sorted({0, 1, 2, 3, kb}):
            if split_k > kb:
                continue
            C = tg.gemm_w4(dA, dBq, ds, dbias if with_bias else None, split_k=split_k)
            got = C.cpu().numpy().view(np.uint16)
            mism = np.argwhere(got != ref)
            assert mism.size == 0, (f"split_k={split_k} bias={with_bias}: {len(mism)} mismatches, first "
                                    f"{tuple(mism[0])}: gpu={got[tuple(mism[0])]:#06x} ref={ref[tuple(mism[0])]:#06x}")
    _status_ok(tg)


@pytest.mark.parametrize("M,N,K,gelu", [
    (16, 4096, 4096, True), (1, 1024, 2048, False), (64, 2048, 1024, True), (128, 512, 512, True),
    (7, 1000, 1152, True), (16, 28672, 8192, False),
])
def test_random_inputs(tg, M, N, K, gelu):
    w = workloads.W4Workload(f"rand_{M}x{N}x{K}", M, N, K, seed=M + N + K,
                             bias_dist=workloads.Dist("normal", 0.0, 0.02), gelu=gelu)
    A, Bq, s, bias = w.inputs()
    ref = oracle.gemm_w4(A, Bq, s, bias, gelu=gelu)
    dA, dBq, ds, dbias = _dev(A, Bq, s, bias)
    C = tg.gemm_w4(dA, dBq, ds, dbias, gelu=gelu)
    _check_tol(C.cpu().numpy(), ref, f"{M}x{N}x{K}")
    _status_ok(tg)


def test_decode_workload_every_split_and_deterministic(tg):
    w = workloads.DECODE_W4
    A, Bq, s, bias = w.inputs()
    ref = oracle.gemm_w4(A, Bq, s, bias, gelu=w.gelu)
    dA, dBq, ds, dbias = _dev(A, Bq, s, bias)
    first = None
    for split_k in (0, 1, 2, 4, 8, 32):
        C = tg.gemm_w4(dA, dBq, ds, dbias, gelu=w.gelu, split_k=split_k)
        got = C.cpu().numpy()
        _check_tol(got, ref, f"decode split_k={split_k}")
        if split_k == 0:
            first = got.view(np.uint16).copy()
    again = tg.gemm_w4(dA, dBq, ds, dbias, gelu=w.gelu).cpu().numpy().view(np.uint16)
    assert np.array_equal(first, again), "repeated launches differ"
    _status_ok(tg)


def test_zero_k_and_empty(tg):
    bias = torch.linspace(-1, 1, 64, dtype=torch.float16)
    dbias = bias.cuda()
    A = torch.empty((4, 0), dtype=torch.float16, device="cuda")
    Bq = torch.empty((64, 0), dtype=torch.uint8, device="cuda")
    s = torch.empty((0, 64), dtype=torch.float16, device="cuda")
    C = tg.gemm_w4(A, Bq, s, dbias, gelu=True)
    ref = oracle.gemm(np.zeros((4, 0), np.float16), np.zeros((0, 64), np.float16), bias.numpy(), gelu=True)
    assert np.array_equal(C.cpu().numpy().view(np.uint16), ref.view(np.uint16))
    E = tg.gemm_w4(torch.empty((0, 256), dtype=torch.float16, device="cuda"),
                   torch.zeros((64, 128), dtype=torch.uint8, device="cuda"),
                   torch.ones((2, 64), dtype=torch.float16, device="cuda"))
    assert E.shape == (0, 64)
    _status_ok(tg)


def test_extreme_nibbles_and_scales(tg):
    # every weight -8 or 7, scales at the ends of the fp16 range that keep the
    # sums finite, including subnormal scales (the products round to binary16)
    M, N, K = 16, 256, 512
    g = torch.Generator().manual_seed(7)
    A = torch.randint(-1, 2, (M, K), generator=g).to(torch.float16)
    q = torch.where(torch.rand((N, K), generator=g) < 0.5, -8, 7).to(torch.int16)
    u = (q & 0xF).to(torch.uint8)
    Bq = (u[:, 0::2] | (u[:, 1::2] << 4)).contiguous()
    choices = torch.tensor([2.0 ** -24, 2.0 ** -15, 3.0 * 2.0 ** -14, 0.1, 1.0], dtype=torch.float32)
    s = choices[torch.randint(0, 5, (K // 128, N), generator=g)].to(torch.float16)
    ref = oracle.gemm_w4(A, Bq, s)
    C = tg.gemm_w4(*_dev(A, Bq, s))
    _check_tol(C.cpu().numpy(), ref, "extreme nibbles")
    _status_ok(tg)


# ---------------------------------------------------------------- FP4 (E2M1) weights

FP4_EXACT = [(1, 8, 128), (16, 128, 256), (5, 136, 384), (17, 264, 128), (64, 1024, 1024), (128, 256, 512),
             (33, 16, 896), (48, 392, 2048)]


@pytest.mark.parametrize("M,N,K", FP4_EXACT, ids=[f"{m}x{n}x{k}" for m, n, k in FP4_EXACT])
def test_fp4_exact_inputs_bitwise_every_split(tg, M, N, K):
    # integer activations, power-of-two scales, E2M1 values (multiples of 1/2 up to 6):
    # every product and partial sum is exact in fp32, so the result is the oracle's bit for bit
    w = workloads.W4Workload(f"fp4_exact_{M}x{N}x{K}", M, N, K, seed=M * 37 + N + K, a_dist=INT2,
                             bias_dist=INT2, scale_kind="pow2", fmt="fp4")
    A, Bq, s, bias = w.inputs()
    dA, dBq, ds, dbias = _dev(A, Bq, s, bias)
    ref = oracle.gemm_w4(A, Bq, s, bias, fmt=1).view(np.uint16)
    kb = (K + 255) // 256
    for split_k in sorted({0, 1, 2, kb}):
        C = tg.gemm_w4(dA, dBq, ds, dbias, split_k=split_k, fmt=tg.W4_FP4_E2M1)
        got = C.cpu().numpy().view(np.uint16)
        mism = np.argwhere(got != ref)
        assert mism.size == 0, (f"split_k={split_k}: {len(mism)} mismatches, first {tuple(mism[0])}: "
                                f"gpu={got[tuple(mism[0])]:#06x} ref={ref[tuple(mism[0])]:#06x}")
    _status_ok(tg)


def test_fp4_every_code_through_an_identity_product(tg):
    # A = [I | 0] picks rows of W: C[m, n] = W[m, n] = value(q[m, n]) * scale[0, n], so every
    # one of the 16 codes in both nibble positions and every column is read back exactly
    M, N, K = 64, 256, 256
    codes = (np.arange(K)[:, None] + 3 * np.arange(N)[None, :]) % 16  # every code in every column
    u = codes.T.astype(np.uint8)
    Bq = torch.from_numpy(np.ascontiguousarray(u[:, 0::2] | (u[:, 1::2] << 4)))
    s = torch.from_numpy(np.where(np.arange(N) % 2 == 0, 1.0, 0.25).astype(np.float16)[None, :].repeat(2, 0))
    A = torch.zeros((M, K), dtype=torch.float16)
    A[torch.arange(M), torch.arange(M)] = 1.0
    # values compared as numbers: a sum of zeros may come out as +0 or -0 (the sign of an
    # exact zero is not fixed by the definition, and differs between compilers of the oracle)
    ref = oracle.gemm_w4(A, Bq, s, fmt=1).astype(np.float64)
    W = oracle.dequant_w4(Bq, s, fmt=1).astype(np.float64)
    assert np.array_equal(ref, W[:M])
    C = tg.gemm_w4(*_dev(A, Bq, s), fmt=tg.W4_FP4_E2M1)
    assert np.array_equal(C.cpu().numpy().astype(np.float64), ref)
    _status_ok(tg)


@pytest.mark.parametrize("M,N,K,gelu", [(16, 4096, 4096, True), (3, 1000, 1152, False), (64, 2048, 1024, True)])
def test_fp4_random_inputs(tg, M, N, K, gelu):
    w = workloads.W4Workload(f"fp4_rand_{M}x{N}x{K}", M, N, K, seed=M + N + K + 1,
                             bias_dist=workloads.Dist("normal", 0.0, 0.02), gelu=gelu, fmt="fp4")
    A, Bq, s, bias = w.inputs()
    ref = oracle.gemm_w4(A, Bq, s, bias, gelu=gelu, fmt=1)
    C = tg.gemm_w4(*_dev(A, Bq, s, bias), gelu=gelu, fmt=tg.W4_FP4_E2M1)
    _check_tol(C.cpu().numpy(), ref, f"fp4 {M}x{N}x{K}")
    _status_ok(tg)


def test_fp4_decode_workload_every_element(tg):
    w = workloads.DECODE_FP4
    A, Bq, s, bias = w.inputs()
    ref = oracle.gemm_w4(A, Bq, s, bias, fmt=1)
    dA, dBq, ds, dbias = _dev(A, Bq, s, bias)
    for split_k in (0, 1, 4):
        C = tg.gemm_w4(dA, dBq, ds, dbias, split_k=split_k, fmt=tg.W4_FP4_E2M1)
        _check_tol(C.cpu().numpy(), ref, f"fp4 decode split_k={split_k}")
    _status_ok(tg)


def test_unaligned_32_byte_weight_base(tg):
    # packed weights at a base that is 16- but not 32-byte aligned (the documented minimum)
    w = workloads.W4Workload("w4_off16", 16, 512, 1024, seed=77, a_dist=INT2, scale_kind="pow2")
    A, Bq, s, _ = w.inputs()
    buf = torch.zeros(Bq.numel() + 16, dtype=torch.uint8, device="cuda")
    dBq = buf[16:16 + Bq.numel()].view(Bq.shape)
    dBq.copy_(Bq.cuda())
    assert dBq.data_ptr() % 32 == 16
    C = tg.gemm_w4(A.cuda(), dBq, s.cuda())
    assert np.array_equal(C.cpu().numpy().view(np.uint16), oracle.gemm_w4(A, Bq, s).view(np.uint16))
    _status_ok(tg)
