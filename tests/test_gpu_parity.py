"""GPU parity: the CUDA kernels, called through the C ABI, against the fp64 CPU
oracle on the same seeded inputs.

Tolerance for floating-point inputs, per element: |gpu - ref| <= 1e-2 + 1e-2 |ref|
(ref = the oracle's binary16 result). Inputs whose products and partial sums are
exact in fp32 (small integers) must match bit for bit, for every kernel.
Full-size workloads are checked on sampled outputs covering every output tile
(the oracle evaluates each sampled element from the definition), plus whole
rows; the smaller ones element by element.
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


def _to_dev(*ts):
    return [t.cuda() if t is not None else None for t in ts]


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
    return float(err.max())


def _status_ok(tg):
    st, where = tg.tg_device_status(None)
    assert st == tg.OK, f"device watchdog reported status {st} at wait site {where}"


def _kernels_for(tg, M, N, K):
    ks = [tg.KERNEL_AUTO, tg.KERNEL_TILED_LSU]
    if K % 8 == 0 and N % 8 == 0:
        ks.append(tg.KERNEL_TILED_TMA)
        ks.append(tg.KERNEL_TILED_PAIR)
        if M <= 128:
            ks.append(tg.KERNEL_SPLITK)
    return ks


# --------------------------------------------------------------- exact cases

EXACT_SHAPES = [
    (1, 8, 8), (1, 1, 1), (16, 16, 16), (17, 24, 64), (63, 64, 72), (64, 128, 128), (65, 136, 136),
    (127, 248, 192), (128, 256, 256), (129, 264, 200), (255, 512, 64), (257, 520, 128),
    (300, 1000, 256), (33, 40, 8), (128, 8, 256), (7, 13, 29), (129, 257, 31), (200, 3, 5),
    (5, 200, 3), (100, 96, 256), (16, 28672 // 16, 256),
    # 2 x 43 = 86 tiles of 256 x 256: one wave of 76 CTA pairs plus 10 tiles that
    # the pair kernel runs as 20 half-width units (whole, ragged, and an empty half)
    (512, 11008, 64), (512, 10992, 72), (500, 10816, 64),
    # neither K nor N a multiple of 8, at least 2^32 flops and enough tiles for CTA pairs: the
    # automatic choice copies A and B to aligned strides and runs the pair kernel on the copies
    (2048, 10990, 103),
]


@pytest.mark.parametrize("M,N,K", EXACT_SHAPES, ids=[f"{m}x{n}x{k}" for m, n, k in EXACT_SHAPES])
def test_exact_integer_inputs_bitwise(tg, M, N, K):
    w = workloads.custom(M, N, K, seed=M * 7 + N * 3 + K, dist=INT2, bias=INT2)
    A, B, bias = w.inputs()
    ref = oracle.gemm(A, B, bias).view(np.uint16)
    dA, dB, dbias = _to_dev(A, B, bias)
    for kernel in _kernels_for(tg, M, N, K):
        for with_bias in (True, False):
            r = ref if with_bias else oracle.gemm(A, B, None).view(np.uint16)
            C = tg.gemm(dA, dB, dbias if with_bias else None, kernel=kernel)
            got = C.cpu().numpy().view(np.uint16)
            mism = np.argwhere(got != r)
            assert mism.size == 0, (f"kernel {kernel} bias={with_bias}: {len(mism)} mismatches, first "
                                    f"{tuple(mism[0])}: gpu={got[tuple(mism[0])]:#06x} ref={r[tuple(mism[0])]:#06x}")
    _status_ok(tg)


@pytest.mark.parametrize("split_k", [1, 2, 3, 5, 16])
def test_splitk_explicit_splits_bitwise(tg, split_k):
    w = workloads.custom(16, 384, 1024, seed=100 + split_k, dist=INT1, bias=INT1)
    A, B, bias = w.inputs()
    ref = oracle.gemm(A, B, bias).view(np.uint16)
    dA, dB, dbias = _to_dev(A, B, bias)
    C = tg.gemm(dA, dB, dbias, kernel=tg.KERNEL_SPLITK, split_k=split_k)
    assert np.array_equal(C.cpu().numpy().view(np.uint16), ref)
    _status_ok(tg)


# --------------------------------------------------------------- float cases

@pytest.mark.parametrize("M,N,K,gelu", [
    (200, 264, 136, True), (70, 131, 67, True), (129, 257, 520, False), (512, 512, 512, True),
    (16, 1024, 4096, True), (100, 136, 1000, True), (1, 4096, 4096, False), (128, 2048, 8192, False),
    # both sides of the automatic skinny / tiled choice for 16 < M <= 128: few 64-column tiles
    # with a long K loop (split-K up to M = 48 here, tiled at 64), and a short K loop (tiled)
    (24, 2048, 4096, True), (48, 1024, 8192, False), (64, 1024, 8192, True), (96, 3072, 2048, True),
])
def test_random_inputs_all_kernels(tg, M, N, K, gelu):
    w = workloads.custom(M, N, K, seed=M + N + K, bias=workloads.Dist("uniform", -0.1, 0.1), gelu=gelu)
    A, B, bias = w.inputs()
    ref = oracle.gemm(A, B, bias, gelu=gelu).astype(np.float64)
    dA, dB, dbias = _to_dev(A, B, bias)
    for kernel in _kernels_for(tg, M, N, K):
        C = tg.gemm(dA, dB, dbias, gelu=gelu, kernel=kernel)
        _check_tol(C.cpu().float().numpy(), ref, f"{M}x{N}x{K} gelu={gelu} kernel={kernel}")
    _status_ok(tg)


def test_square_256(tg):
    w = workloads.SQUARE_256
    A, B, bias = w.inputs()
    ref = oracle.gemm(A, B, bias, gelu=w.gelu)
    C = tg.gemm(*_to_dev(A, B), None, gelu=w.gelu)
    _check_tol(C.cpu().float().numpy(), ref.astype(np.float64), w.name)
    _status_ok(tg)


def test_ragged_bias_gelu_full(tg):
    w = workloads.RAGGED_GELU
    A, B, bias = w.inputs()
    ref = oracle.gemm(A, B, bias, gelu=True)
    dA, dB, dbias = _to_dev(A, B, bias)
    # N = 1030 gives B a stride TMA cannot describe: at this size the automatic choice is the
    # ordinary-load kernel, reading B in place
    for kernel in (tg.KERNEL_AUTO, tg.KERNEL_TILED_LSU):
        C = tg.gemm(dA, dB, dbias, gelu=True, kernel=kernel)
        _check_tol(C.cpu().float().numpy(), ref.astype(np.float64), f"{w.name} kernel {kernel}")
    _status_ok(tg)


def _tile_samples(M, N, bm, bn, per_tile, seed):
    rng = np.random.default_rng(seed)
    rows, cols = [], []
    for m0 in range(0, M, bm):
        for n0 in range(0, N, bn):
            hm, hn = min(bm, M - m0), min(bn, N - n0)
            rows.extend(m0 + rng.integers(0, hm, per_tile))
            cols.extend(n0 + rng.integers(0, hn, per_tile))
            rows.extend([m0, m0 + hm - 1])
            cols.extend([n0 + hn - 1, n0])
    return np.array(rows, dtype=np.int64), np.array(cols, dtype=np.int64)


def _check_full_size(tg, w, full_rows):
    A, B, bias = w.inputs()
    dA, dB, dbias = _to_dev(A, B, bias)
    C = tg.gemm(dA, dB, dbias, gelu=w.gelu)       # the call the benchmark times (automatic kernel)
    torch.cuda.synchronize()
    _status_ok(tg)
    rows, cols = _tile_samples(w.M, w.N, 128, 128, 3, seed=w.seed)
    got = C[torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()].cpu().float().numpy()
    ref = oracle.gemm_sampled(A, B, bias, w.gelu, rows, cols)
    _check_tol(got, ref.astype(np.float64), f"{w.name} sampled ({rows.size} points)")
    for r0 in full_rows:
        ref_rows = oracle.gemm(A, B, bias, gelu=w.gelu, rows=(r0, 1))
        _check_tol(C[r0:r0 + 1].cpu().float().numpy(), ref_rows.astype(np.float64), f"{w.name} row {r0}")
    assert bool(torch.isfinite(C).all())


def test_square_8192_sampled(tg):
    _check_full_size(tg, workloads.SQUARE_8192, full_rows=[0, 4097, 8191])


def test_ffn_up_bias_gelu_sampled(tg):
    _check_full_size(tg, workloads.FFN_UP, full_rows=[0, 2049, 4095])


def test_decode_full(tg):
    w = workloads.DECODE
    A, B, bias = w.inputs()
    dA, dB, dbias = _to_dev(A, B, bias)
    C = tg.gemm(dA, dB, dbias, gelu=w.gelu)
    got = C.cpu().float().numpy()
    _status_ok(tg)
    ref = oracle.gemm(A, B, bias, gelu=w.gelu)
    _check_tol(got, ref.astype(np.float64), w.name)
    # the tiled kernel agrees too (it is not the automatic choice for M = 16)
    C2 = tg.gemm(dA, dB, dbias, gelu=w.gelu, kernel=tg.KERNEL_TILED_TMA)
    _check_tol(C2.cpu().float().numpy(), ref.astype(np.float64), w.name + " tiled")


# --------------------------------------------------------------- edge cases

def test_empty_m_n_leave_output_untouched(tg):
    C = torch.full((4, 3), 7.0, dtype=torch.float16, device="cuda")
    tg.tg_gemm(None, None, None, C.data_ptr(), 0, 3, 5, 0, None)
    tg.tg_gemm(None, None, None, C.data_ptr(), 4, 0, 5, 0, None)
    torch.cuda.synchronize()
    assert bool((C == 7).all())


@pytest.mark.parametrize("gelu", [False, True])
def test_k_zero_is_epilogue_of_bias(tg, gelu):
    bias = torch.tensor([0.5, -1.0, 2.0, 0.0, -3.0], dtype=torch.float16)
    A = torch.zeros((3, 0), dtype=torch.float16)
    B = torch.zeros((0, 5), dtype=torch.float16)
    ref = oracle.gemm(A, B, bias, gelu=gelu).astype(np.float64)
    C = torch.empty((3, 5), dtype=torch.float16, device="cuda")
    tg.tg_gemm(None, None, bias.cuda().data_ptr(), C.data_ptr(), 3, 5, 0, int(gelu), None)
    _check_tol(C.cpu().float().numpy(), ref, "K=0")
    C0 = torch.full((3, 5), 9.0, dtype=torch.float16, device="cuda")
    tg.tg_gemm(None, None, None, C0.data_ptr(), 3, 5, 0, int(gelu), None)
    torch.cuda.synchronize()
    assert bool((C0 == 0).all())


def test_unaligned_pointers_take_the_load_path(tg):
    M, N, K = 96, 136, 200
    w = workloads.custom(M, N, K, seed=77, bias=workloads.Dist("uniform", -0.1, 0.1), gelu=True)
    A, B, bias = w.inputs()
    ref = oracle.gemm(A, B, bias, gelu=True).astype(np.float64)
    # views starting one element into a buffer: 2-byte aligned only
    bufA = torch.zeros(M * K + 1, dtype=torch.float16, device="cuda")
    bufB = torch.zeros(K * N + 1, dtype=torch.float16, device="cuda")
    bufb = torch.zeros(N + 1, dtype=torch.float16, device="cuda")
    bufC = torch.zeros(M * N + 1, dtype=torch.float16, device="cuda")
    dA = bufA[1:].view(M, K); dA.copy_(A)
    dB = bufB[1:].view(K, N); dB.copy_(B)
    db = bufb[1:]; db.copy_(bias)
    dC = bufC[1:].view(M, N)
    with pytest.raises(tg.TgError):
        tg.gemm(dA, dB, db, gelu=True, out=dC, kernel=tg.KERNEL_TILED_TMA)
    tg.gemm(dA, dB, db, gelu=True, out=dC)
    _check_tol(dC.cpu().float().numpy(), ref, "unaligned")
    _status_ok(tg)


def test_unaligned_large_products_take_the_copy_path(tg):
    # 2 M N K >= 2^32 with 2-byte-aligned A, B, bias and C (and odd strides): A and B are
    # copied to aligned strides and the TMA kernels run on the copies; bias and C are used
    # in place. Checked on sampled rows and columns of every tile.
    for M, N, K in ((1536, 1400, 1008), (1040, 2050, 1031)):
        w = workloads.custom(M, N, K, seed=78 + K, bias=workloads.Dist("uniform", -0.1, 0.1), gelu=True)
        A, B, bias = w.inputs()
        bufA = torch.zeros(M * K + 1, dtype=torch.float16, device="cuda")
        bufB = torch.zeros(K * N + 1, dtype=torch.float16, device="cuda")
        bufb = torch.zeros(N + 1, dtype=torch.float16, device="cuda")
        bufC = torch.zeros(M * N + 1, dtype=torch.float16, device="cuda")
        dA = bufA[1:].view(M, K); dA.copy_(A)
        dB = bufB[1:].view(K, N); dB.copy_(B)
        db = bufb[1:]; db.copy_(bias)
        dC = bufC[1:].view(M, N)
        tg.gemm(dA, dB, db, gelu=True, out=dC)
        rows, cols = _tile_samples(M, N, 128, 128, 4, seed=M + N)
        got = dC[torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()].cpu().float().numpy()
        _check_tol(got, oracle.gemm_sampled(A, B, bias, True, rows, cols).astype(np.float64),
                   f"unaligned {M}x{N}x{K}")
        # the inputs are untouched and nothing is written outside C
        assert torch.equal(dA.cpu(), A) and torch.equal(dB.cpu(), B)
        assert bufC[0].item() == 0
    _status_ok(tg)


def test_copy_path_pads_only_the_operand_that_needs_it(tg):
    # K = 519: A's rows are not 16-byte multiples (A is copied), B (519 x 2048) is used in place;
    # no bias, no GELU
    M, N, K = 2048, 2048, 519
    w = workloads.custom(M, N, K, seed=91)
    A, B, _ = w.inputs()
    dA, dB, _ = _to_dev(A, B, None)
    C = tg.gemm(dA, dB)
    rows, cols = _tile_samples(M, N, 128, 128, 2, seed=91)
    got = C[torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()].cpu().float().numpy()
    _check_tol(got, oracle.gemm_sampled(A, B, None, False, rows, cols).astype(np.float64), "pad A only")
    _status_ok(tg)


@pytest.mark.parametrize("M,N,K", [(3, 24, 1 << 22), (5, 7, (1 << 20) + 3)], ids=["splitk_K4M", "loads_K1M_odd"])
def test_very_long_k(tg, M, N, K):
    # K in the millions: the skinny path's K slices and the ordinary-load path's 64-bit offsets;
    # inputs uniform[-1/4, 1/4] keep |C| moderate for the fp16 output
    w = workloads.custom(M, N, K, seed=K % 1000, dist=workloads.Dist("uniform", -0.25, 0.25))
    A, B, _ = w.inputs()
    dA, dB, _ = _to_dev(A, B, None)
    C = tg.gemm(dA, dB)
    _check_tol(C.cpu().float().numpy(), oracle.gemm(A, B, None).astype(np.float64), f"{M}x{N}x{K}")
    _status_ok(tg)


def test_repeatable_bit_for_bit(tg):
    for M, N, K, kernel in [(300, 520, 1000, 1), (16, 2048, 4096, 3), (70, 131, 67, 2)]:
        w = workloads.custom(M, N, K, seed=5, bias=workloads.Dist("uniform", -0.1, 0.1), gelu=True)
        A, B, bias = _to_dev(*w.inputs())
        c1 = tg.gemm(A, B, bias, gelu=True, kernel=kernel)
        c2 = tg.gemm(A, B, bias, gelu=True, kernel=kernel)
        assert torch.equal(c1.view(torch.int16), c2.view(torch.int16))


def test_non_default_stream(tg):
    w = workloads.custom(256, 512, 512, seed=9, bias=workloads.Dist("uniform", -0.1, 0.1), gelu=True)
    A, B, bias = w.inputs()
    ref = oracle.gemm(A, B, bias, gelu=True).astype(np.float64)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        dA, dB, db = _to_dev(A, B, bias)
        C = tg.gemm(dA, dB, db, gelu=True)
    s.synchronize()
    _check_tol(C.cpu().float().numpy(), ref, "side stream")


def test_staged_host_buffers(tg):
    w = workloads.custom(300, 264, 520, seed=21, bias=workloads.Dist("uniform", -0.1, 0.1), gelu=True)
    A, B, bias = w.inputs()
    ref = oracle.gemm(A, B, bias, gelu=True).astype(np.float64)
    hA, hB, hb = A.pin_memory(), B.pin_memory(), bias.pin_memory()
    hC = torch.empty((w.M, w.N), dtype=torch.float16).pin_memory()
    dA = torch.empty_like(A, device="cuda"); dB = torch.empty_like(B, device="cuda")
    db = torch.empty_like(bias, device="cuda"); dC = torch.empty((w.M, w.N), dtype=torch.float16, device="cuda")
    tg.gemm_staged(hA, hB, hb, hC, dA, dB, db, dC, gelu=True)
    torch.cuda.current_stream().synchronize()
    _check_tol(hC.float().numpy(), ref, "staged")
