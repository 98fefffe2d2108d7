"""tg_gemm_splitk_noalloc: the split-K GEMM for callers that cannot let the
library allocate device memory during a call (a process whose device memory is
all handed to its own pool allocator, where a library cudaMalloc would fail,
or a latency-bound loop that cannot absorb cudaMalloc/cudaFree's device-wide
synchronisation). Its scratch is a fixed array in the library's device image.

Checked through the C ABI against the fp64 CPU oracle: bit for bit on inputs
whose products and partial sums are exact in fp32, at explicit K-slice counts
2, 3, 5 (summed on chip, in thread-block clusters) and 16 (summed through the
array), and within the tolerance of the other GPU tests
(|gpu - ref| <= 1e-2 + 1e-2 |ref|) on float inputs, over two calls in a row of
different shapes that share the one array; also against the ordinary split-K
entry point. Free device memory does not change across the calls; an automatic
call on a shape whose unconstrained slice count would not fit the array takes
fewer slices instead of failing; an explicit slice count that does not fit is
refused; and a call made right after another kernel's watchdog timeout still
computes correctly. This file is collected last."""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

RTOL = 1e-2
ATOL = 1e-2
INT1 = workloads.Dist("int", -1, 1)


@pytest.fixture(scope="module")
def tg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import tiled_tensor_core_tcgen05_gb300 as m
    torch.cuda.set_device(0)
    return m


def _close(got, ref, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    bad = np.abs(got - ref) > ATOL + RTOL * np.abs(ref)
    assert not bad.any(), f"{what}: {int(bad.sum())} elements out of tolerance"


def _noalloc(tg, A, B, bias, C, M, N, K, epi, split_k):
    tg.tg_gemm_splitk_noalloc(A.data_ptr(), B.data_ptr(), bias.data_ptr() if bias is not None else None,
                              C.data_ptr(), M, N, K, epi, split_k, torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("splits", [2, 3, 5, 16])
@pytest.mark.parametrize("M,N", [(16, 1032), (40, 512), (128, 264)])
def test_exact_inputs_bitwise_against_the_oracle(tg, M, N, splits):
    # entries in [-1, 1], K = 1024: every product and partial sum is an integer of magnitude
    # <= 1024, exact in fp32 and fp16, whatever the slice boundaries and summation order
    K = 1024
    w = workloads.custom(M, N, K, seed=500 + M + splits, dist=INT1, bias=INT1)
    A, B, bias = w.inputs()
    dA, dB, db = A.cuda(), B.cuda(), bias.cuda()
    ref = oracle.gemm(A, B, bias).view(np.uint16)
    for _ in range(2):
        C = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
        _noalloc(tg, dA, dB, db, C, M, N, K, tg.EPI_NONE, splits)
        torch.cuda.synchronize()
        assert np.array_equal(C.cpu().numpy().view(np.uint16), ref)
    assert tg.tg_device_status(None) == (tg.OK, 0)


def test_two_calls_match_the_oracle_and_the_allocating_entry_point(tg):
    dist = workloads.Dist("normal", 0.0, 0.02)
    splits = 4
    sh = torch.cuda.current_stream().cuda_stream
    cases = []
    for seed, (M, N, K) in enumerate([(16, 4096, 8192), (40, 1032, 2048)]):
        w = workloads.custom(M, N, K, seed=400 + seed, dist=dist, bias=dist, gelu=True)
        A, B, bias = w.inputs()
        dA, dB, db = A.cuda(), B.cuda(), bias.cuda()
        via_ex = torch.empty((M, N), dtype=torch.float16, device="cuda")
        tg.tg_gemm_ex(dA.data_ptr(), dB.data_ptr(), db.data_ptr(), via_ex.data_ptr(), M, N, K, tg.EPI_GELU,
                      tg.KERNEL_SPLITK, splits, sh)
        cases.append((w, (A, B, bias), (dA, dB, db), via_ex))
    outs = [torch.full((w.M, w.N), float("nan"), dtype=torch.float16, device="cuda") for w, *_ in cases]
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    for (w, _, (dA, dB, db), _), C in zip(cases, outs):  # two calls in a row, different shapes, one array
        _noalloc(tg, dA, dB, db, C, w.M, w.N, w.K, tg.EPI_GELU, splits)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free_before
    assert tg.tg_device_status(None) == (tg.OK, 0)
    for (w, (A, B, bias), _, via_ex), C in zip(cases, outs):
        got = C.cpu().numpy()
        _close(got, oracle.gemm(A, B, bias, gelu=True), w.name)
        _close(got, via_ex.cpu().numpy(), w.name + " vs tg_gemm_ex")


def test_repeat_call_reuses_the_array(tg):
    w = workloads.custom(16, 2048, 4096, seed=420, dist=workloads.Dist("normal", 0.0, 0.02))
    A, B, _ = w.inputs()
    dA, dB = A.cuda(), B.cuda()
    ref = oracle.gemm(A, B)
    for _ in range(2):
        C = torch.empty((w.M, w.N), dtype=torch.float16, device="cuda")
        _noalloc(tg, dA, dB, None, C, w.M, w.N, w.K, tg.EPI_NONE, 8)
        torch.cuda.synchronize()
        _close(C.cpu().numpy(), ref, w.name)


def test_automatic_slices_stay_within_the_array(tg):
    # 64 x 8192 x 8192: the cost model alone picks more K slices than the array holds (each
    # slice's partials are 64 x 8192 x 4 bytes = 2 MiB, at most 3 fit in 8 MiB beside the
    # reserved head of the array), so the automatic choice is capped and the call succeeds
    M, N, K = 64, 8192, 8192
    w = workloads.custom(M, N, K, seed=430, dist=workloads.Dist("normal", 0.0, 0.02))
    A, B, _ = w.inputs()
    dA, dB = A.cuda(), B.cuda()
    C = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
    # sixteen explicit slices are summed through the array (more than a cluster holds) and
    # need 32 MiB of partials
    with pytest.raises(tg.TgError) as ei:
        _noalloc(tg, dA, dB, None, C, M, N, K, tg.EPI_NONE, 16)
    assert ei.value.status == tg.ERR_INVALID_ARG
    _noalloc(tg, dA, dB, None, C, M, N, K, tg.EPI_NONE, 0)
    torch.cuda.synchronize()
    assert tg.tg_device_status(None) == (tg.OK, 0)
    rows = (0, 8)
    _close(C.cpu().numpy()[:8], oracle.gemm(A, B, rows=rows), "automatic slices")
    _close(C.cpu().numpy()[56:], oracle.gemm(A, B, rows=(56, 8)), "automatic slices")


def test_too_large_for_the_fixed_array_is_refused(tg):
    # 64 rows x 28672 columns x 4 slices of fp32 partials = 29 MB > 8 MiB
    M, N, K = 64, 28672, 1024
    A = torch.zeros((M, K), dtype=torch.float16, device="cuda")
    B = torch.zeros((K, N), dtype=torch.float16, device="cuda")
    C = torch.zeros((M, N), dtype=torch.float16, device="cuda")
    with pytest.raises(tg.TgError) as ei:
        _noalloc(tg, A, B, None, C, M, N, K, tg.EPI_NONE, 4)
    assert ei.value.status == tg.ERR_INVALID_ARG
    assert "static scratch" in str(ei.value)


def test_call_after_a_watchdog_timeout(tg):
    # the tiled kernel's test hook withholds one producer arrival, so that launch ends with a
    # bounded-wait timeout (nothing faults); the fixed array's next use must still be correct
    w = workloads.custom(256, 512, 256, seed=440, dist=workloads.Dist("int", -2, 2))
    A, B, _ = w.inputs()
    tg.tg_set_watchdog_ns(20_000_000)
    tg.tg_debug_skip_first_arrive(True)
    try:
        tg.gemm(A.cuda(), B.cuda(), kernel=tg.KERNEL_TILED_TMA)
        st, _ = tg.tg_device_status(None)
    finally:
        tg.tg_debug_skip_first_arrive(False)
        tg.tg_set_watchdog_ns(0)
    assert st == tg.ERR_TIMEOUT
    K = 1024
    x = workloads.custom(32, 1032, K, seed=441, dist=INT1)
    A, B, _ = x.inputs()
    dA, dB = A.cuda(), B.cuda()
    ref = oracle.gemm(A, B).view(np.uint16)
    for splits in (5, 16):  # on chip, then through the array
        C = torch.full((x.M, x.N), float("nan"), dtype=torch.float16, device="cuda")
        _noalloc(tg, dA, dB, None, C, x.M, x.N, K, tg.EPI_NONE, splits)
        torch.cuda.synchronize()
        assert np.array_equal(C.cpu().numpy().view(np.uint16), ref)
    assert tg.tg_device_status(None) == (tg.OK, 0)
