"""The kernels' bounded waits: a withheld producer arrival must end the call
with TG_ERR_TIMEOUT (reported by tg_device_status) instead of hanging, and the
device must stay usable for the next call.

The test hook makes the tiled kernel's TMA producer skip its arrival on the
first pipeline stage of every CTA, so the MMA thread's wait on that stage can
never complete; its bounded wait expires, the CTA's other roles see the abort
flag, in-flight copies are drained, tensor memory is freed and the kernel
returns. Nothing faults or traps."""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import tiled_tensor_core_tcgen05_gb300 as m
    torch.cuda.set_device(0)
    return m


def test_withheld_arrival_times_out_and_recovers(tg):
    w = workloads.custom(256, 512, 256, seed=31, dist=workloads.Dist("int", -2, 2))
    A, B, _ = w.inputs()
    dA, dB = A.cuda(), B.cuda()
    assert tg.tg_device_status(None) == (tg.OK, 0)
    tg.tg_set_watchdog_ns(20_000_000)  # 20 ms
    tg.tg_debug_skip_first_arrive(True)
    try:
        tg.gemm(dA, dB, kernel=tg.KERNEL_TILED_TMA)
        st, where = tg.tg_device_status(None)
    finally:
        tg.tg_debug_skip_first_arrive(False)
        tg.tg_set_watchdog_ns(0)
    assert st == tg.ERR_TIMEOUT
    assert where == 2  # the MMA thread's wait on a full stage expired first
    # the status word was cleared and the device still computes correctly
    assert tg.tg_device_status(None) == (tg.OK, 0)
    C = tg.gemm(dA, dB, kernel=tg.KERNEL_TILED_TMA)
    ref = oracle.gemm(A, B).view(np.uint16)
    assert np.array_equal(C.cpu().numpy().view(np.uint16), ref)
    assert tg.tg_device_status(None) == (tg.OK, 0)


def test_withheld_arrival_in_a_split_launch_times_out_and_recovers(tg):
    """The tiled kernel with K split over slices: the first unit of every CTA never gets its
    first stage, so that launch times out; the reduction that follows sums whatever the
    partials hold (the result is void, the status says so), and the next call is exact."""
    w = workloads.custom(256, 1024, 2048, seed=35, dist=workloads.Dist("int", -2, 2))
    A, B, _ = w.inputs()
    dA, dB = A.cuda(), B.cuda()
    assert tg.tg_device_status(None) == (tg.OK, 0)
    tg.tg_set_watchdog_ns(20_000_000)
    tg.tg_debug_skip_first_arrive(True)
    try:
        tg.gemm(dA, dB, kernel=tg.KERNEL_TILED_TMA, split_k=4)
        st, where = tg.tg_device_status(None)
    finally:
        tg.tg_debug_skip_first_arrive(False)
        tg.tg_set_watchdog_ns(0)
    assert st == tg.ERR_TIMEOUT
    assert where == 2
    assert tg.tg_device_status(None) == (tg.OK, 0)
    C = tg.gemm(dA, dB, kernel=tg.KERNEL_TILED_TMA, split_k=4)
    assert np.array_equal(C.cpu().numpy().view(np.uint16), oracle.gemm(A, B).view(np.uint16))
    assert tg.tg_device_status(None) == (tg.OK, 0)


def test_withheld_stage_in_the_pair_kernel_times_out_and_recovers(tg):
    """The CTA-pair kernel, with its epilogue hand-off warp: a withheld first stage
    makes the MMA thread's wait expire; every other wait (the odd CTA's, the
    epilogue's, the hand-off's) is bounded too, so the launch ends, and the next
    call is exact."""
    w = workloads.custom(512, 768, 1024, seed=34, dist=workloads.Dist("int", -2, 2), bias=workloads.Dist("int", -2, 2))
    A, B, bias = w.inputs()
    dA, dB, db = A.cuda(), B.cuda(), bias.cuda()
    assert tg.tg_device_status(None) == (tg.OK, 0)
    tg.tg_set_watchdog_ns(20_000_000)  # 20 ms
    tg.tg_debug_skip_first_arrive(True)
    try:
        tg.gemm(dA, dB, db, kernel=tg.KERNEL_TILED_PAIR)
        st, where = tg.tg_device_status(None)
    finally:
        tg.tg_debug_skip_first_arrive(False)
        tg.tg_set_watchdog_ns(0)
    assert st == tg.ERR_TIMEOUT
    assert where in (1, 2, 4, 5), where  # producer, MMA, epilogue or drain wait
    assert tg.tg_device_status(None) == (tg.OK, 0)
    C = tg.gemm(dA, dB, db, kernel=tg.KERNEL_TILED_PAIR)
    ref = oracle.gemm(A, B, bias).view(np.uint16)
    assert np.array_equal(C.cpu().numpy().view(np.uint16), ref)
    assert tg.tg_device_status(None) == (tg.OK, 0)


def test_hook_off_by_default(tg):
    w = workloads.custom(128, 256, 128, seed=32, dist=workloads.Dist("int", -2, 2))
    A, B, _ = w.inputs()
    C = tg.gemm(A.cuda(), B.cuda(), kernel=tg.KERNEL_TILED_TMA)
    assert np.array_equal(C.cpu().numpy().view(np.uint16), oracle.gemm(A, B).view(np.uint16))
    assert tg.tg_device_status(None) == (tg.OK, 0)


def test_withheld_stage_in_the_register_4bit_kernel_times_out_and_recovers(tg):
    """The same hook in the register-dequant 4-bit kernel: its producer never fills the
    first stage of each CTA, so those consumers' bounded wait expires (or, a moment later,
    the producer's wait for that stage to be freed)."""
    w = workloads.W4Workload("wd_w4r", 16, 1024, 2048, seed=33, a_dist=workloads.Dist("int", -2, 2),
                             scale_kind="pow2")
    A, Bq, s, _ = w.inputs()
    dA, dBq, ds = A.cuda(), Bq.cuda(), s.cuda()
    assert tg.tg_device_status(None) == (tg.OK, 0)
    tg.tg_set_watchdog_ns(20_000_000)  # 20 ms
    tg.tg_debug_skip_first_arrive(True)
    try:
        tg.gemm_w4(dA, dBq, ds, kernel=tg.W4_KERNEL_REG)
        st, where = tg.tg_device_status(None)
    finally:
        tg.tg_debug_skip_first_arrive(False)
        tg.tg_set_watchdog_ns(0)
    assert st == tg.ERR_TIMEOUT
    assert where in (6, 1)  # a consumer's wait for the stage, or the producer's wait to refill it
    assert tg.tg_device_status(None) == (tg.OK, 0)
    C = tg.gemm_w4(dA, dBq, ds, kernel=tg.W4_KERNEL_REG)
    assert np.array_equal(C.cpu().numpy().view(np.uint16), oracle.gemm_w4(A, Bq, s).view(np.uint16))
    assert tg.tg_device_status(None) == (tg.OK, 0)
