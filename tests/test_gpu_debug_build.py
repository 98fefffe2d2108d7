"""The debug build (TG_DEBUG=1, libtg_gemm_debug.so): device-side bounds checks
that record a failure in the status word instead of trapping, so no GPU is
faulted.

With the checks live, small shapes that cross every tile boundary go through
each kernel family (CTA pair with TMA stores, single CTA, ordinary loads, both
single-CTA variants with K split, skinny split-K at several slice counts, the
4-bit GEMM with split K, the attention forward with a split last round) and
must match the fp64 oracle bit for bit on exact-arithmetic inputs, twice in a
row, with no check failing. Then the test hook that shrinks the scratch size
the checks allow makes a split call's partial sums reach past it: the call
must end with TG_ERR_BOUNDS (the skipped accesses fault nothing), and the next
call, with the real size, must be exact again. The normal build compiles the
checks away: the same hook has no effect there."""
import ctypes
import os

import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

INT1 = workloads.Dist("int", -1, 1)
INT2 = workloads.Dist("int", -2, 2)
KERNELS = {"pair": 4, "tiled": 1, "lsu": 2, "splitk": 3}


@pytest.fixture(scope="module")
def libs():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    path = __graft_entry__._build_module().build(debug=True)
    import tiled_tensor_core_tcgen05_gb300 as tg
    torch.cuda.set_device(0)
    return tg, tg.bind(path)


def _status(lib):
    where = ctypes.c_int(0)
    return lib.tg_device_status(None, ctypes.byref(where)), where.value


def _gemm(lib, A, B, bias, M, N, K, kernel, split_k=0):
    C = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
    rc = lib.tg_gemm_ex(A.data_ptr(), B.data_ptr(), bias.data_ptr() if bias is not None else None, C.data_ptr(),
                        M, N, K, 0, kernel, split_k, None)
    assert rc == 0, lib.tg_last_error()
    return C


def test_the_debug_library_has_its_checks_and_the_normal_one_does_not(libs):
    tg, dbg = libs
    assert dbg.tg_debug_build() == 1
    assert tg.tg_debug_build() == 0


GEMM_SHAPES = [(1, 8, 8), (17, 24, 64), (65, 136, 136), (129, 264, 200), (255, 520, 64), (300, 1000, 256),
               (512, 11008, 64), (16, 28672 // 16, 256), (128, 512, 1024)]


@pytest.mark.parametrize("M,N,K", GEMM_SHAPES, ids=[f"{m}x{n}x{k}" for m, n, k in GEMM_SHAPES])
def test_every_kernel_exact_with_the_checks_on(libs, M, N, K):
    _, dbg = libs
    dist = INT1 if K > 256 else INT2
    w = workloads.custom(M, N, K, seed=M * 11 + N + K, dist=dist, bias=dist)
    A, B, bias = w.inputs()
    ref = oracle.gemm(A, B, bias).view(np.uint16)
    dA, dB, db = A.cuda(), B.cuda(), bias.cuda()
    runs = [("pair", 0), ("tiled", 0), ("lsu", 0)]
    if K >= 128:  # the single-CTA kernels with K split over slices
        runs += [("tiled", 2), ("lsu", 3)]
    if M <= 128:
        runs += [("splitk", s) for s in (0, 1, 3, max(1, min(16, (K + 63) // 64)))]
    for name, split in runs:
        first = _gemm(dbg, dA, dB, db, M, N, K, KERNELS[name], split).cpu().numpy().view(np.uint16)
        again = _gemm(dbg, dA, dB, db, M, N, K, KERNELS[name], split).cpu().numpy().view(np.uint16)
        assert np.array_equal(first, ref), f"{name} split_k={split}"
        assert np.array_equal(first, again), f"{name} split_k={split}: runs differ"
        assert _status(dbg) == (0, 0), f"{name} split_k={split}: a check failed"


def test_w4_and_attention_with_the_checks_on(libs):
    _, dbg = libs
    w = workloads.W4Workload("dbg_w4", 33, 392, 2048, seed=5, a_dist=INT2, bias_dist=INT2, scale_kind="pow2",
                             fmt="fp4")
    A, Bq, s, bias = w.inputs()
    ref = oracle.gemm_w4(A, Bq, s, bias, fmt=1).view(np.uint16)
    dA, dBq, ds, db = A.cuda(), Bq.cuda(), s.cuda(), bias.cuda()
    for split in (1, 3, 8):
        C = torch.empty((w.M, w.N), dtype=torch.float16, device="cuda")
        assert dbg.tg_gemm_w4_ex(dA.data_ptr(), dBq.data_ptr(), ds.data_ptr(), db.data_ptr(), C.data_ptr(), w.M, w.N,
                                 w.K, 0, 1, split, None) == 0
        assert np.array_equal(C.cpu().numpy().view(np.uint16), ref), f"split_k={split}"
    assert _status(dbg) == (0, 0)
    # the register-dequant kernel (M <= 16), ragged N and K
    w = workloads.W4Workload("dbg_w4r", 13, 200, 1152, seed=7, a_dist=INT2, bias_dist=INT2, scale_kind="pow2")
    A, Bq, s, bias = w.inputs()
    ref = oracle.gemm_w4(A, Bq, s, bias).view(np.uint16)
    dA, dBq, ds, db = A.cuda(), Bq.cuda(), s.cuda(), bias.cuda()
    C = torch.empty((w.M, w.N), dtype=torch.float16, device="cuda")
    assert dbg.tg_gemm_w4_kernel(dA.data_ptr(), dBq.data_ptr(), ds.data_ptr(), db.data_ptr(), C.data_ptr(), w.M,
                                 w.N, w.K, 0, 0, 2, 0, None) == 0
    assert np.array_equal(C.cpu().numpy().view(np.uint16), ref), "register kernel"
    assert _status(dbg) == (0, 0)
    # a shape whose last round of query blocks is split into key halves (uses the scratch)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    H = (2 * sms + 16) // 8
    a = workloads.AttnWorkload("dbg_attn", 1, 1000, H, 128, seed=6)
    Q, K, V = a.inputs()
    O = torch.empty((1, 1000, H, 128), dtype=torch.float16, device="cuda")
    dQ, dK, dV = Q.cuda(), K.cuda(), V.cuda()
    assert dbg.tg_attention_fwd(dQ.data_ptr(), dK.data_ptr(), dV.data_ptr(), O.data_ptr(), 1, 1000, H, 128, 0,
                                None) == 0
    assert _status(dbg) == (0, 0)
    rows = np.array([(s * H + h) for s in (0, 500, 999) for h in range(H)])
    ref = oracle.attention(Q, K, V, rows=rows).astype(np.float64)
    got = O.cpu().numpy().reshape(-1, 128)[rows].astype(np.float64)
    assert (np.abs(got - ref) <= 1e-2 + 1e-2 * np.abs(ref)).all()


def test_a_failed_check_is_reported_not_faulted(libs):
    tg, dbg = libs
    M, N, K = 16, 2048, 4096
    w = workloads.custom(M, N, K, seed=77, dist=INT1)
    A, B, _ = w.inputs()
    ref = oracle.gemm(A, B).view(np.uint16)
    dA, dB = A.cuda(), B.cuda()
    assert _status(dbg) == (0, 0)
    # sixteen K slices (more than a cluster sums on chip) write 16 x 16 x 2048 floats of
    # partials to scratch; allow the checks only 1024 of them
    assert dbg.tg_debug_bounds_limit(1024) == 0
    try:
        _gemm(dbg, dA, dB, None, M, N, K, KERNELS["splitk"], 16)
        st, where = _status(dbg)
    finally:
        dbg.tg_debug_bounds_limit(0)
    assert st == tg.ERR_BOUNDS and where == 8
    assert _status(dbg) == (0, 0)  # cleared, and the next call is exact again
    C = _gemm(dbg, dA, dB, None, M, N, K, KERNELS["splitk"], 16)
    assert np.array_equal(C.cpu().numpy().view(np.uint16), ref)
    assert _status(dbg) == (0, 0)


def test_a_failed_check_in_a_tiled_split_is_reported_not_faulted(libs):
    tg, dbg = libs
    M, N, K = 256, 512, 1024
    w = workloads.custom(M, N, K, seed=79, dist=INT1)
    A, B, _ = w.inputs()
    dA, dB = A.cuda(), B.cuda()
    assert _status(dbg) == (0, 0)
    # three K slices of 256 x 512 fp32 partials in scratch (the ordinary-load variant; the TMA
    # variant sums up to 8 slices on chip); allow the checks only 4096 floats of them
    assert dbg.tg_debug_bounds_limit(4096) == 0
    try:
        _gemm(dbg, dA, dB, None, M, N, K, KERNELS["lsu"], 3)
        st, where = _status(dbg)
    finally:
        dbg.tg_debug_bounds_limit(0)
    assert st == tg.ERR_BOUNDS and where == 8
    assert _status(dbg) == (0, 0)
    C = _gemm(dbg, dA, dB, None, M, N, K, KERNELS["lsu"], 3)
    assert np.array_equal(C.cpu().numpy().view(np.uint16), oracle.gemm(A, B).view(np.uint16))
    assert _status(dbg) == (0, 0)


def test_the_normal_build_ignores_the_hook(libs):
    tg, _ = libs
    M, N, K = 16, 2048, 4096
    w = workloads.custom(M, N, K, seed=78, dist=INT1)
    A, B, _ = w.inputs()
    tg.tg_debug_bounds_limit(1024)
    try:
        C = tg.gemm(A.cuda(), B.cuda(), kernel=tg.KERNEL_SPLITK, split_k=4)
        st = tg.tg_device_status(None)
    finally:
        tg.tg_debug_bounds_limit(0)
    assert st == (tg.OK, 0)
    assert np.array_equal(C.cpu().numpy().view(np.uint16), oracle.gemm(A, B).view(np.uint16))
