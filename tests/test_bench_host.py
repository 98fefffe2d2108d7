"""Host-side logic of bench.py, on CPU: max-over-ranks timing across a
world_size-2 gloo group (the N>1 replicas path), roofline arithmetic, the
staleness rule for recorded DRAM traffic, and the reference arm (the CPU
oracle) producing its JSON line."""
import importlib.util
import io
import json
import os
import socket
import sys
from contextlib import redirect_stdout
from types import SimpleNamespace

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    m = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(m)
    return m


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    b = _bench()
    w, r, local, pg = b.dist_setup(world)
    assert (w, r, local) == (world, rank, rank)
    b.barrier(pg)
    m = b.max_over_ranks(pg, 10.0 + rank)   # each rank times a different region
    out[rank] = m
    pg.destroy_process_group()


def test_max_over_ranks_gloo_world_2():
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank_main, args=(2, port, out), nprocs=2, join=True)
        assert dict(out) == {0: 11.0, 1: 11.0}


def test_roofline_entry_math():
    b = _bench()
    import workloads
    pk = {"hbm_gbs": 6000.0, "bf16_tflops": 2000.0, "bf16_tflops_sustained": 1600.0}
    w = workloads.SQUARE_8192
    e = b.roofline_entry(w, 0.55, pk, "measured", "tensor", traffic=123)
    assert e["achieved"] == pytest.approx(w.flops() / 0.55e-3 / 1e12, rel=1e-4)
    assert e["frac"] == pytest.approx(e["achieved"] / 2000.0, abs=1e-4)
    assert e["frac_of_sustained"] == pytest.approx(e["achieved"] / 1600.0, abs=1e-4)
    assert e["traffic"] == 123 and e["unit"] == "TFLOP/s"
    d = workloads.DECODE
    e = b.roofline_entry(d, 0.0785, pk, "measured", "hbm")
    assert e["unit"] == "GB/s" and e["achieved"] == pytest.approx(d.bytes() / 0.0785e-3 / 1e9, rel=1e-4)


def test_recorded_traffic_is_dropped_when_kernels_change(tmp_path, monkeypatch):
    b = _bench()
    (tmp_path / "profiles").mkdir()
    rec = {"square_8192": {"dram_bytes_per_launch": 42, "kernel_hash": "not-the-current-hash"}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(b, "ROOT", str(tmp_path))
    monkeypatch.setattr(b, "kernel_source_hash", lambda kernel=None: "current")
    assert b.recorded_traffic("square_8192") is None
    rec["square_8192"]["kernel_hash"] = "current"
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    assert b.recorded_traffic("square_8192") == 42
    assert b.recorded_traffic("decode_16x28672x8192") is None


def test_kernel_hash_follows_only_that_kernels_sources():
    b = _bench()
    assert set(b.KERNEL_SOURCES) >= {"tiled_pair_kernel", "tiled_gemm_kernel", "splitk_gemm_kernel",
                                     "w4_gemm_kernel", "attn_fwd_kernel", "softmax_rows"}
    csrc = os.path.join(b.ROOT, "tiled_tensor_core_tcgen05_gb300", "csrc")
    for files in b.KERNEL_SOURCES.values():
        for f in files + b._COMMON_SOURCES:
            assert os.path.exists(os.path.join(csrc, f)), f
    # a template instance name maps to its kernel's sources, and kernels differ
    assert b.kernel_source_hash("softmax_rows_reg<32, 16>") == b.kernel_source_hash("softmax_rows")
    assert b.kernel_source_hash("attn_fwd_kernel") != b.kernel_source_hash("softmax_rows")


def test_reference_arm_prints_its_line(monkeypatch):
    b = _bench()
    monkeypatch.delenv("RANK", raising=False)
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    args = SimpleNamespace(workload="square_256", steps=2, warmup=1, ref_budget_s=0.5)
    buf = io.StringIO()
    with redirect_stdout(buf):
        b.run_reference(args)
    line = json.loads(buf.getvalue().strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "TFLOP/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]


def test_reference_arm_other_ranks_do_nothing(monkeypatch):
    b = _bench()
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    buf = io.StringIO()
    with redirect_stdout(buf):
        b.run_reference(SimpleNamespace(workload="square_256", steps=1, warmup=1, ref_budget_s=0.1))
    assert buf.getvalue() == ""


def test_roofline_entry_reports_the_sku_fractions():
    b = _bench()
    import workloads
    pk = {"hbm_gbs": 6000.0, "bf16_tflops": 2000.0, "bf16_tflops_sustained": 1600.0}
    e = b.roofline_entry(workloads.SQUARE_8192, 0.55, pk, "measured", "tensor")
    assert e["sku_peak"] == 2250.0 and e["frac_of_sku"] == pytest.approx(e["achieved"] / 2250.0, abs=1e-4)
    e = b.roofline_entry(workloads.DECODE, 0.0785, pk, "measured", "hbm")
    assert e["sku_peak"] == 8000.0 and e["frac_of_sku"] == pytest.approx(e["achieved"] / 8000.0, abs=1e-4)


def _small_cases():
    import workloads
    return [workloads.custom(40, 72, 64, seed=3, bias=workloads.Dist("uniform", -0.1, 0.1), gelu=True),
            workloads.W4Workload("w4_small", 3, 64, 256, seed=4),
            workloads.AttnWorkload("attn_small", 1, 40, 2, 128, seed=5, causal=True),
            workloads.SoftmaxWorkload("softmax_small", 5, 24, seed=6)]


def _oracle_output(w, inputs):
    import oracle
    import workloads
    if isinstance(w, workloads.Workload):
        A, B, bias = inputs
        return oracle.gemm(A, B, bias, gelu=w.gelu)
    if isinstance(w, workloads.W4Workload):
        return oracle.gemm_w4(*inputs, gelu=w.gelu)
    if isinstance(w, workloads.AttnWorkload):
        return oracle.attention(*inputs, causal=w.causal)
    return oracle.softmax(*inputs)


@pytest.mark.parametrize("k", range(4), ids=["gemm", "w4", "attention", "softmax"])
def test_parity_check_passes_the_oracle_and_counts_a_planted_error(k):
    b = _bench()
    w = _small_cases()[k]
    inputs = w.inputs()
    out = torch.from_numpy(_oracle_output(w, inputs).copy())
    p = b.parity_check(w, inputs, out, n_samples=64)
    assert p["violations"] == 0 and p["max_abs_err"] == 0.0 and p["checked"] > 0
    bad = out.clone().view(-1)
    bad[:] = bad + 0.5  # every element off by 0.5: well outside the tolerance everywhere
    p = b.parity_check(w, inputs, bad.view(out.shape), n_samples=64)
    assert p["violations"] == p["checked"]


@pytest.mark.parametrize("k", range(4), ids=["gemm", "w4", "attention", "softmax"])
def test_cpu_baseline_leg_for_every_workload_kind(k):
    b = _bench()
    w = _small_cases()[k]
    unit = "GB/s" if k in (1, 3) else "TFLOP/s"
    e = b.cpu_baseline(w, 0.05, unit)
    assert e["kind"] == "oracle" and e["unit"] == unit and e["value"] > 0 and e["cores"] >= 1


def test_one_thread_oracle_timing_and_host_cpu():
    b = _bench()
    import workloads
    e = b.cpu_baseline_one_thread(workloads.custom(32, 64, 48, seed=7), row_budget=8)
    assert e["threads"] == 1 and e["rows"] == "0..7 of 32" and e["seconds_whole_product"] >= e["seconds"]
    c = b.host_cpu()
    assert c["logical_cpus"] >= 1 and isinstance(c["model"], str)


def test_smi_timestamps_parse():
    b = _bench()
    t = b._smi_time("2026/12/03 05:30:36.250")
    assert t is not None and abs((t % 1) - 0.25) < 1e-6
    assert b._smi_time("not a time") is None


def test_all_core_baselines_survive_a_one_thread_timing():
    b = _bench()
    import oracle
    import workloads
    n = b.oracle_threads()
    assert n == max(1, oracle.max_threads()) or n >= 1
    b.cpu_baseline_one_thread(workloads.custom(8, 16, 16, seed=8))  # leaves the oracle at one thread
    e = b.cpu_baseline(workloads.custom(32, 64, 48, seed=9), 0.05, "TFLOP/s")
    assert e["cores"] == n


def test_kernel_pinning_maps_to_each_entry_points_codes():
    """--kernel takes GEMM kernel names for GEMM workloads and w4tmem / w4reg for
    4-bit ones, and refuses a name that does not apply to the workload."""
    b = _bench()
    import workloads
    gemm = workloads.BY_NAME["square_8192"]
    w4 = workloads.DECODE_W4
    assert b.kernel_code(gemm, "auto") == 0 and b.kernel_code(gemm, "pair") == 4
    assert b.kernel_code(w4, "auto") == 0 and b.kernel_code(w4, "w4tmem") == 1 and b.kernel_code(w4, "w4reg") == 2
    with pytest.raises(SystemExit):
        b.kernel_code(gemm, "w4reg")
    with pytest.raises(SystemExit):
        b.kernel_code(w4, "pair")
