"""tg_gemm_splitk_noalloc: the split-K GEMM for callers that cannot let the
library allocate device memory during a call (a process whose device memory is
all handed to its own pool allocator, where a library cudaMalloc would fail,
or a latency-bound loop that cannot absorb cudaMalloc/cudaFree's device-wide
synchronisation). Its scratch is a fixed array in the library's device image.

Checked through the C ABI: two calls in a row agree with the ordinary split-K
entry point (tg_gemm_ex with the same slice count) within the tolerance the
other GPU tests use, free device memory does not change across the calls, and
a problem whose partial sums would not fit the fixed array is refused."""
import numpy as np
import pytest
import torch

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


def _close(got, ref):
    got = got.float().cpu().numpy().astype(np.float64)
    ref = ref.float().cpu().numpy().astype(np.float64)
    assert np.isfinite(got).all()
    bad = np.abs(got - ref) > ATOL + RTOL * np.abs(ref)
    assert not bad.any(), f"{int(bad.sum())} elements out of tolerance"


def test_two_calls_match_the_allocating_entry_point(tg):
    dist = workloads.Dist("normal", 0.0, 0.02)
    splits = 4
    stream = torch.cuda.current_stream()
    sh = stream.cuda_stream
    cases = []
    for seed, (M, N, K) in enumerate([(16, 4096, 8192), (40, 1032, 2048)]):
        w = workloads.custom(M, N, K, seed=400 + seed, dist=dist, bias=dist, gelu=True)
        A, B, bias = [t.cuda() for t in w.inputs()]
        ref = torch.empty((M, N), dtype=torch.float16, device="cuda")
        tg.tg_gemm_ex(A.data_ptr(), B.data_ptr(), bias.data_ptr(), ref.data_ptr(), M, N, K, tg.EPI_GELU,
                      tg.KERNEL_SPLITK, splits, sh)
        cases.append((w, A, B, bias, ref))
    outs = [torch.full((w.M, w.N), float("nan"), dtype=torch.float16, device="cuda") for w, *_ in cases]
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    for (w, A, B, bias, ref), C in zip(cases, outs):  # two calls in a row, different shapes, one array
        tg.tg_gemm_splitk_noalloc(A.data_ptr(), B.data_ptr(), bias.data_ptr(), C.data_ptr(), w.M, w.N, w.K,
                                  tg.EPI_GELU, splits, sh)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free_before
    assert tg.tg_device_status(None) == (tg.OK, 0)
    for (w, A, B, bias, ref), C in zip(cases, outs):
        _close(C, ref)


def test_repeat_call_reuses_the_array(tg):
    w = workloads.custom(16, 2048, 4096, seed=420, dist=workloads.Dist("normal", 0.0, 0.02))
    A, B, _ = [t.cuda() if t is not None else None for t in w.inputs()]
    sh = torch.cuda.current_stream().cuda_stream
    ref = torch.empty((w.M, w.N), dtype=torch.float16, device="cuda")
    tg.tg_gemm_ex(A.data_ptr(), B.data_ptr(), None, ref.data_ptr(), w.M, w.N, w.K, tg.EPI_NONE,
                  tg.KERNEL_SPLITK, 8, sh)
    for _ in range(2):
        C = torch.empty_like(ref)
        tg.tg_gemm_splitk_noalloc(A.data_ptr(), B.data_ptr(), None, C.data_ptr(), w.M, w.N, w.K, tg.EPI_NONE, 8, sh)
        torch.cuda.synchronize()
        _close(C, ref)


def test_too_large_for_the_fixed_array_is_refused(tg):
    # 64 rows x 28672 columns x 4 slices of fp32 partials = 29 MB > 8 MiB
    M, N, K = 64, 28672, 1024
    A = torch.zeros((M, K), dtype=torch.float16, device="cuda")
    B = torch.zeros((K, N), dtype=torch.float16, device="cuda")
    C = torch.zeros((M, N), dtype=torch.float16, device="cuda")
    with pytest.raises(tg.TgError) as ei:
        tg.tg_gemm_splitk_noalloc(A.data_ptr(), B.data_ptr(), None, C.data_ptr(), M, N, K, tg.EPI_NONE, 4,
                                  torch.cuda.current_stream().cuda_stream)
    assert ei.value.status == tg.ERR_INVALID_ARG
    assert "static scratch" in str(ei.value)
