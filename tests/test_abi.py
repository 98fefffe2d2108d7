"""CPU checks of the C-ABI library: it loads without a GPU, exports every
function include/tg_gemm.h declares, and rejects bad arguments on the host
before touching a device (no compute call is made here)."""
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def tg():
    import __graft_entry__
    __graft_entry__.build()
    import tiled_tensor_core_tcgen05_gb300 as m
    return m


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "tg_gemm.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*[A-Za-z_][\w\s\*]*?\b(tg_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_documented_entry_points():
    names = _declared_functions()
    assert "tg_gemm" in names and "tg_gemm_ex" in names and "tg_gemm_staged" in names
    assert len(names) >= 11


def test_library_exports_every_declared_function(tg):
    lib = tg.library()
    for name in _declared_functions():
        assert hasattr(lib, name), name
    assert set(_declared_functions()) == set(tg.EXPORTS)


def test_status_strings_and_version(tg):
    assert tg.tg_status_string(0) == "TG_OK"
    for s in range(1, 6):
        assert tg.tg_status_string(s).startswith("TG_ERR_")
    assert "unknown" in tg.tg_status_string(99)
    assert tg.tg_version() >= 10000


def test_ring_bytes_follow_the_tile_footprint_formula(tg):
    # tiled kernels: 4 stages of a 128x64 A tile and a 64x256 B tile, fp16
    assert tg.tg_ring_bytes(tg.KERNEL_TILED_TMA) == tg.ring_bytes(128, 256, 64, 4) == 196608
    assert tg.tg_ring_bytes(tg.KERNEL_TILED_LSU) == tg.ring_bytes(128, 256, 64, 4)
    assert tg.tg_ring_bytes(tg.KERNEL_SPLITK) % tg.ring_bytes(16, 256, 64, 1) == 0
    assert tg.tg_ring_bytes(tg.KERNEL_SPLITK) <= 227 * 1024
    assert tg.tg_ring_bytes(tg.KERNEL_TILED_PAIR) == tg.ring_bytes(128, 128, 64, 6)
    assert tg.tg_ring_bytes(42) == -1


def test_footprint_worked_example(tg):
    # "TileLang: you write the dataflow, the compiler owns the schedule", section
    # "What a tile costs, exactly": 128/128/32, 3 stages, fp16 -> 16 KB per stage, 48 KB
    g = {}
    for line in open(os.path.join(ROOT, "tests", "golden", "smem_footprint.txt")):
        line = line.split("#", 1)[0].strip()
        if line:
            k, v = line.split()
            g[k] = int(v)
    bm, bn, bk, st, b = g["block_M"], g["block_N"], g["block_K"], g["num_stages"], g["bytes_per_elem"]
    assert tg.ring_bytes(bm, bn, bk, 1, b) == g["stage_kb"] * 1024
    assert tg.ring_bytes(bm, bn, bk, st, b) == g["total_kb"] * 1024
    assert bm * bn * 4 == g["accum_kb"] * 1024
    assert bm * bn * 4 // 4 // g["threads"] == g["regs_per_thread"]


@pytest.mark.parametrize("args,msg", [
    (dict(epilogue=2), "epilogue"),
    (dict(M=-1), "sizes"),
    (dict(K=2 ** 31), "sizes"),
    (dict(kernel=9), "kernel"),
    (dict(kernel=4, N=20), "TG_KERNEL_TILED_PAIR"),
    (dict(split_k=65), "split_k"),
    (dict(split_k=-1), "split_k"),
    (dict(C=0), "C is NULL"),
    (dict(A=0), "A or B"),
    (dict(C=0x10000 + 10), "overlaps"),
    (dict(kernel=1, K=12), "TG_KERNEL_TILED_TMA"),
    (dict(kernel=1, A=0x10002), "TG_KERNEL_TILED_TMA"),
    (dict(kernel=3, M=129), "TG_KERNEL_SPLITK"),
    (dict(kernel=3, N=20), "TG_KERNEL_SPLITK"),
    (dict(kernel=4, split_k=2), "split_k does not apply"),
])
def test_invalid_arguments_rejected_on_host(tg, args, msg):
    base = dict(A=0x10000, B=0x20000000, bias=None, C=0x40000000, M=64, N=64, K=64, epilogue=0,
                kernel=0, split_k=0)
    base.update(args)
    with pytest.raises(tg.TgError) as ei:
        tg.tg_gemm_ex(base["A"] or None, base["B"] or None, base["bias"], base["C"] or None, base["M"],
                      base["N"], base["K"], base["epilogue"], base["kernel"], base["split_k"], None)
    assert ei.value.status == tg.ERR_INVALID_ARG
    assert msg in str(ei.value)


def test_empty_products_need_no_device(tg):
    # M == 0 or N == 0: nothing to do, so success without any CUDA call
    tg.tg_gemm(None, None, None, None, 0, 5, 7, 0, None)
    tg.tg_gemm(None, None, None, None, 5, 0, 7, 1, None)


def test_staged_argument_checks(tg):
    with pytest.raises(tg.TgError):
        tg.tg_gemm_staged(1, 2, 3, 4, 5, 6, None, 8, 4, 4, 4, 0, None)   # hbias without dbias
    with pytest.raises(tg.TgError):
        tg.tg_gemm_staged(1, 2, None, 4, 5, 6, None, 8, -1, 4, 4, 0, None)


def test_product_package_never_touches_the_oracle():
    pkg = os.path.join(ROOT, "tiled_tensor_core_tcgen05_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "oracle." not in text.replace("oracle.c", ""), f
                assert "liboracle" not in text, f


@pytest.mark.parametrize("args,msg", [
    (dict(epilogue=3), "epilogue"),
    (dict(M=129), "M <= 128"),
    (dict(K=192), "K % 128"),
    (dict(N=20), "N % 8"),
    (dict(split_k=65), "split_k"),
    (dict(C=0), "C is NULL"),
    (dict(S=0), "A, Bq or scales"),
    (dict(Bq=0x20000008), "16-byte aligned"),
    (dict(C=0x20000000 + 64), "overlaps"),
])
def test_w4_invalid_arguments_rejected_on_host(tg, args, msg):
    base = dict(A=0x10000, Bq=0x20000000, S=0x30000000, bias=None, C=0x40000000, M=16, N=64, K=256, epilogue=0,
                split_k=0)
    base.update(args)
    with pytest.raises(tg.TgError) as ei:
        tg.tg_gemm_w4(base["A"] or None, base["Bq"] or None, base["S"] or None, base["bias"], base["C"] or None,
                      base["M"], base["N"], base["K"], base["epilogue"], base["split_k"], None)
    assert ei.value.status == tg.ERR_INVALID_ARG
    assert msg in str(ei.value)


def test_w4_empty_products_need_no_device(tg):
    tg.tg_gemm_w4(None, None, None, None, None, 0, 64, 256, 0, 0, None)
    tg.tg_gemm_w4(None, None, None, None, None, 4, 0, 256, 1, 0, None)


@pytest.mark.parametrize("args,msg", [
    (dict(D=64), "head dimension"),
    (dict(causal=2), "causal"),
    (dict(S=-1), "out of range"),
    (dict(Q=0), "NULL"),
    (dict(K=0x20000008), "16-byte aligned"),
    (dict(O=0x10000 + 256), "overlaps"),
])
def test_attention_invalid_arguments_rejected_on_host(tg, args, msg):
    base = dict(Q=0x10000, K=0x20000000, V=0x30000000, O=0x40000000, B=1, S=64, H=2, D=128, causal=0)
    base.update(args)
    with pytest.raises(tg.TgError) as ei:
        tg.library().tg_attention_fwd and tg._check(tg.library().tg_attention_fwd(
            base["Q"] or None, base["K"] or None, base["V"] or None, base["O"] or None, base["B"], base["S"],
            base["H"], base["D"], base["causal"], None))
    assert ei.value.status == tg.ERR_INVALID_ARG
    assert msg in str(ei.value)


def test_attention_empty_needs_no_device(tg):
    tg.tg_attention_fwd(None, None, None, None, 0, 64, 2, 128, False, None)
    tg.tg_attention_fwd(None, None, None, None, 1, 0, 2, 128, True, None)


def test_softmax_argument_checks(tg):
    tg.tg_softmax_rows(None, None, 0, 10, None)
    tg.tg_softmax_rows(None, None, 10, 0, None)
    for args, msg in [((0x1000, 0x2000, -1, 4), "sizes"), ((None, 0x2000, 4, 4), "NULL"),
                      ((0x1000, 0x1004, 4, 4), "overlaps")]:
        with pytest.raises(tg.TgError) as ei:
            tg.tg_softmax_rows(*args, None)
        assert ei.value.status == tg.ERR_INVALID_ARG and msg in str(ei.value)


def test_w4_ex_rejects_an_unknown_format_and_shares_the_checks(tg):
    with pytest.raises(tg.TgError) as ei:
        tg.tg_gemm_w4_ex(0x10000, 0x20000000, 0x30000000, None, 0x40000000, 16, 64, 256, 0, 2, 0, None)
    assert ei.value.status == tg.ERR_INVALID_ARG and "weight_format" in str(ei.value)
    with pytest.raises(tg.TgError) as ei:
        tg.tg_gemm_w4_ex(0x10000, 0x20000000, 0x30000000, None, 0x40000000, 16, 64, 192, 0, tg.W4_FP4_E2M1, 0, None)
    assert ei.value.status == tg.ERR_INVALID_ARG and "K % 128" in str(ei.value)
    tg.tg_gemm_w4_ex(None, None, None, None, None, 0, 64, 256, 0, tg.W4_FP4_E2M1, 0, None)


def test_release_build_has_no_device_checks_and_the_hook_validates(tg):
    assert tg.tg_debug_build() == 0
    tg.tg_debug_bounds_limit(0)
    with pytest.raises(tg.TgError) as ei:
        tg.tg_debug_bounds_limit(-1)
    assert ei.value.status == tg.ERR_INVALID_ARG
    assert "BOUNDS" in tg.tg_status_string(tg.ERR_BOUNDS)


def test_gemm_plan_argument_checks(tg):
    with pytest.raises(tg.TgError) as ei:
        tg.tg_gemm_plan(None, None, -1, 8, 8)
    assert ei.value.status == tg.ERR_INVALID_ARG
    lib = tg.library()
    assert lib.tg_gemm_plan(None, None, 8, 8, 8, None, None, None) == tg.ERR_INVALID_ARG
