"""GPU parity of the single-CTA tiled kernel with K split over slices.

When a problem's 128 x 256 tiles leave SMs idle (few rows, long K), a work unit
of the tiled kernel is one K slice of one tile. With TMA loads and up to 8
slices, the slices of a tile run as one thread-block cluster and are summed in
distributed shared memory; otherwise each unit writes its fp32 tile to scratch
and a second kernel sums the slices. Either way the slices are added in order,
then bias, GELU and one rounding follow (the epilogue of "Designing
high-performance GPU kernels with TileLang ...", section 3, applied once to the
full sum). The product is still the tile program of "TileLang: writing LLM GPU
kernels by thinking in tiles", section 3: only the K loop is divided.

Integer inputs keep every partial sum exact in fp32, so every split count must
reproduce the oracle bit for bit; float inputs are held to the parity
tolerance |gpu - ref| <= 1e-2 + 1e-2 |ref|.
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


def _status_ok(tg):
    st, where = tg.tg_device_status(None)
    assert st == tg.OK, f"device watchdog reported status {st} at wait site {where}"


def _check_tol(got, ref, what):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    bad = np.abs(got - ref) > ATOL + RTOL * np.abs(ref)
    if bad.any():
        idx = tuple(np.argwhere(bad)[0])
        pytest.fail(f"{what}: {int(bad.sum())}/{bad.size} out of tolerance; first {idx}: "
                    f"gpu={got[idx]} ref={ref[idx]}")


# Shapes: several 128-row blocks with a ragged last one, N not a multiple of the 256-column
# tile, K not a multiple of the 64-deep K block; split counts that divide the K blocks
# evenly, unevenly, and one slice per K block.
SPLIT_SHAPES = [(300, 520, 1000), (129, 264, 2056), (512, 1024, 2048), (16, 384, 1024)]
_refs = {}


def _exact_case(M, N, K, gelu):
    """Integer inputs of one shape and the oracle's result for them (computed once)."""
    w = workloads.custom(M, N, K, seed=7000 + M + N + K, dist=INT2, bias=INT2)
    A, B, bias = w.inputs()
    key = (M, N, K, gelu)
    if key not in _refs:
        _refs[key] = oracle.gemm(A, B, bias, gelu=gelu).view(np.uint16)
    return A, B, bias, _refs[key]


@pytest.mark.parametrize("M,N,K", SPLIT_SHAPES, ids=[f"{m}x{n}x{k}" for m, n, k in SPLIT_SHAPES])
@pytest.mark.parametrize("split_k", [1, 2, 3, 5, 16])
def test_explicit_splits_bitwise(tg, M, N, K, split_k):
    for gelu in (False, True):
        A, B, bias, ref = _exact_case(M, N, K, gelu)
        dA, dB, dbias = A.cuda(), B.cuda(), bias.cuda()
        for kernel in (tg.KERNEL_TILED_TMA, tg.KERNEL_TILED_LSU):
            C = tg.gemm(dA, dB, dbias, gelu=gelu, kernel=kernel, split_k=split_k)
            got = C.cpu().numpy().view(np.uint16)
            mism = np.argwhere(got != ref)
            assert mism.size == 0, (f"kernel {kernel} split_k={split_k} gelu={gelu}: {len(mism)} mismatches, "
                                    f"first {tuple(mism[0])}")
    _status_ok(tg)


def test_split_without_bias_and_unaligned_operands(tg):
    # K and N not multiples of 8: only the ordinary-load variant applies
    M, N, K = 200, 131, 1003
    w = workloads.custom(M, N, K, seed=7101, dist=INT2)
    A, B, _ = w.inputs()
    ref = oracle.gemm(A, B, None).view(np.uint16)
    C = tg.gemm(A.cuda(), B.cuda(), None, kernel=tg.KERNEL_TILED_LSU, split_k=4)
    assert np.array_equal(C.cpu().numpy().view(np.uint16), ref)
    _status_ok(tg)


@pytest.mark.parametrize("M,N,K,gelu", [(256, 2048, 8192, True), (130, 1032, 4104, False), (384, 768, 6144, True)])
def test_random_inputs_split(tg, M, N, K, gelu):
    w = workloads.custom(M, N, K, seed=7200 + M, bias=workloads.Dist("uniform", -0.1, 0.1), gelu=gelu)
    A, B, bias = w.inputs()
    ref = oracle.gemm(A, B, bias, gelu=gelu)
    dA, dB, dbias = A.cuda(), B.cuda(), bias.cuda()
    for split_k in (0, 4, 7):
        C = tg.gemm(dA, dB, dbias, gelu=gelu, kernel=tg.KERNEL_TILED_TMA, split_k=split_k)
        _check_tol(C.cpu().float().numpy(), ref, f"{M}x{N}x{K} split_k={split_k}")
    _status_ok(tg)


def test_automatic_choice_splits_a_mid_size_long_k_product(tg):
    # 256 x 4096: 32 tiles of 128 x 256 on 152 SMs, with 224 K blocks each. The automatic choice
    # is the single-CTA kernel with K split; it must be bit-identical to that kernel pinned with
    # the same split count, and sampled rows must meet the oracle.
    M, N, K = 256, 4096, 14336
    w = workloads.custom(M, N, K, seed=7300, dist=workloads.Dist("normal", 0.0, 0.5),
                         bias=workloads.Dist("uniform", -0.1, 0.1), gelu=True)
    A, B, bias = w.inputs()
    dA, dB, dbias = A.cuda(), B.cuda(), bias.cuda()
    kernel, splits, copy = tg.tg_gemm_plan(dA.data_ptr(), dB.data_ptr(), M, N, K)
    assert (kernel, copy) == (tg.KERNEL_TILED_TMA, 0) and splits > 1, (kernel, splits, copy)
    C = tg.gemm(dA, dB, dbias, gelu=True)
    pinned = tg.gemm(dA, dB, dbias, gelu=True, kernel=tg.KERNEL_TILED_TMA, split_k=splits)
    assert torch.equal(C.view(torch.int16), pinned.view(torch.int16))
    C = C.cpu().float().numpy()
    for r0 in (0, 127, 128, 255):
        ref = oracle.gemm(A, B, bias, gelu=True, rows=(r0, 1))
        _check_tol(C[r0:r0 + 1], ref, f"row {r0}")
    _status_ok(tg)


def test_pair_kernel_refuses_a_split(tg):
    A = torch.zeros((256, 64), dtype=torch.float16, device="cuda")
    B = torch.zeros((64, 256), dtype=torch.float16, device="cuda")
    with pytest.raises(tg.TgError) as ei:
        tg.gemm(A, B, kernel=tg.KERNEL_TILED_PAIR, split_k=2)
    assert ei.value.status == tg.ERR_INVALID_ARG


def test_on_chip_and_scratch_reductions_agree_bit_for_bit(tg):
    # The TMA variant sums up to 8 slices inside a cluster (distributed shared memory); the
    # ordinary-load variant sums them in scratch with the reduction kernel. Both add the
    # slices in order 0, 1, ... to the same fp32 partials, so on float inputs their outputs
    # must be the same bits, and both within the oracle's tolerance.
    M, N, K = 200, 1032, 4104
    w = workloads.custom(M, N, K, seed=7400, bias=workloads.Dist("uniform", -0.1, 0.1), gelu=True)
    A, B, bias = w.inputs()
    dA, dB, dbias = A.cuda(), B.cuda(), bias.cuda()
    ref = oracle.gemm(A, B, bias, gelu=True)
    for split_k in (2, 3, 7):
        on_chip = tg.gemm(dA, dB, dbias, gelu=True, kernel=tg.KERNEL_TILED_TMA, split_k=split_k)
        scratch = tg.gemm(dA, dB, dbias, gelu=True, kernel=tg.KERNEL_TILED_LSU, split_k=split_k)
        assert torch.equal(on_chip.view(torch.int16), scratch.view(torch.int16)), f"split_k={split_k}"
        _check_tol(on_chip.cpu().float().numpy(), ref, f"split_k={split_k}")
    _status_ok(tg)


def test_whole_waves_then_a_split_last_wave(tg):
    # 1280 x 4096 with K = 8192: 160 tiles of 128 x 256, a wave on 152 SMs plus 8. The whole
    # wave runs unsplit, then the last 8 tiles (column block 15, rows 256..1279 in the grouped
    # order) run K-split as clusters summed on chip. Exact integer inputs: sampled whole rows,
    # inside and outside the split tiles, must match the oracle bit for bit.
    M, N, K = 1280, 4096, 8192
    w = workloads.custom(M, N, K, seed=7500, dist=workloads.Dist("int", -1, 1), bias=INT2)
    A, B, bias = w.inputs()
    dA, dB, dbias = A.cuda(), B.cuda(), bias.cuda()
    kernel, splits, _ = tg.tg_gemm_plan(dA.data_ptr(), dB.data_ptr(), M, N, K)
    if kernel != tg.KERNEL_TILED_TMA or splits < 2:
        pytest.skip(f"no split last wave chosen on this device (kernel {kernel}, {splits} slices)")
    for k in (tg.KERNEL_AUTO, tg.KERNEL_TILED_TMA):
        C = tg.gemm(dA, dB, dbias, gelu=True, kernel=k).cpu().numpy().view(np.uint16)
        for r0 in (0, 130, 256, 700, 1279):
            ref = oracle.gemm(A, B, bias, gelu=True, rows=(r0, 1)).view(np.uint16)
            mism = np.argwhere(C[r0:r0 + 1] != ref)
            assert mism.size == 0, f"kernel {k} row {r0}: {len(mism)} mismatches, first {tuple(mism[0])}"
    _status_ok(tg)
