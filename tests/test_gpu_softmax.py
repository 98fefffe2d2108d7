"""GPU parity of the row softmax (tg_softmax_rows), through the C ABI, against
the fp64 CPU oracle on the same inputs.

Tolerance per element, from the arithmetic: fp32 exponentials (hardware
exp2, relative error ~1e-7 for the arguments that matter), an fp32 sum and one
final binary16 rounding (relative 2^-11): |gpu - ref| <= 2e-3 |ref| + 1e-6."""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

RTOL = 2e-3
ATOL = 1e-6


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


def _check(got, ref, what):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan), f"{what}: NaN positions differ"
    err = np.abs(got - ref)[~nan]
    bad = err > ATOL + RTOL * np.abs(ref[~nan])
    if bad.any():
        pytest.fail(f"{what}: {int(bad.sum())}/{bad.size} out of tolerance (max err {err.max():.3g})")


# one size per path: warp per row (1, 2, 4, 8 chunks), 64..512-thread groups, three passes
SIZES = [(37, 1), (37, 8), (37, 64), (37, 256), (37, 264), (37, 512), (37, 1000), (37, 1024), (37, 2048), (37, 2056),
         (37, 4096), (9, 8192), (9, 16384), (5, 32768), (5, 32776), (3, 65536), (301, 7), (3, 100003)]


@pytest.mark.parametrize("M,N", SIZES, ids=[f"{m}x{n}" for m, n in SIZES])
def test_sizes_every_element(tg, M, N):
    w = workloads.SoftmaxWorkload(f"s_{M}x{N}", M, N, seed=M * 7 + N)
    (X,) = w.inputs()
    got = tg.softmax(X.cuda()).cpu().numpy()
    _check(got, oracle.softmax(X), w.name)
    _status_ok(tg)


def test_ragged_workload_every_element(tg):
    (X,) = workloads.SOFTMAX_RAGGED.inputs()
    _check(tg.softmax(X.cuda()).cpu().numpy(), oracle.softmax(X), "ragged")


@pytest.mark.parametrize("w", [workloads.SOFTMAX_4096, workloads.SOFTMAX_VOCAB], ids=lambda w: w.name)
def test_full_size_row_ranges(tg, w):
    (X,) = w.inputs()
    got = tg.softmax(X.cuda()).cpu().numpy()
    for r0 in (0, w.M // 2 - 17, w.M - 40):
        _check(got[r0:r0 + 40], oracle.softmax(X, rows=(r0, 40)), f"{w.name} rows {r0}")
    _status_ok(tg)


def test_infinities_and_extremes(tg):
    X = np.random.default_rng(5).normal(0, 2, size=(6, 4096)).astype(np.float16)
    X[0, ::3] = -np.inf
    X[1, :] = -np.inf          # no defined softmax: NaN like the arithmetic
    X[2, 17] = 60000.0
    X[3, :] = 60000.0
    X[4, -1] = 65504.0
    X[4, 0] = -65504.0
    Xt = torch.from_numpy(X)
    _check(tg.softmax(Xt.cuda()).cpu().numpy(), oracle.softmax(Xt), "extremes")
    Xs = torch.from_numpy(X[:, :4093].copy())  # the three-pass path too
    _check(tg.softmax(Xs.cuda()).cpu().numpy(), oracle.softmax(Xs), "extremes, ragged")


def test_in_place_and_unaligned(tg):
    w = workloads.SoftmaxWorkload("s_inplace", 33, 2048, seed=9)
    (X,) = w.inputs()
    ref = oracle.softmax(X)
    d = X.cuda()
    tg.softmax(d, out=d)
    _check(d.cpu().numpy(), ref, "in place")
    buf = torch.empty(33 * 2048 + 1, dtype=torch.float16, device="cuda")
    xs = buf[1:].view(33, 2048)              # 2-byte offset: not 16-byte aligned
    xs.copy_(X.cuda())
    _check(tg.softmax(xs).cpu().numpy(), ref, "unaligned")
    _status_ok(tg)
