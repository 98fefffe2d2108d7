#!/usr/bin/env python3
"""Benchmark of the fp16 tiled tensor-core GEMM (+ fused bias/GELU) on GB300.

A step is one call of the GEMM through the C ABI (tg_gemm) on one batch of
synthetic seeded input already resident in HBM. The headline workload is the
square 8192^3 fp16 GEMM (TFLOP/s against the dense fp16 tensor roofline); the
other workloads of the suite are reported in the same JSON line (the decode
GEMM as HBM GB/s). Prints exactly one JSON line on rank 0.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl tg|reference]

--impl reference times the CPU oracle (fp64, all host cores) on a bounded
sample of the same workload, in the same unit, as the reference arm.
Multi-GPU (under torchrun): N independent replicas, one per GPU, no data
exchange (the work is independent per problem); value = all ranks' flops over
the slowest rank's time.
"""
from __future__ import annotations

import argparse
import glob
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "fp16 GEMM TFLOP/s & % of GB300 tensor peak; decode-GEMM HBM GB/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# fp16 and bf16 share the same dense tensor-core rate on this part (2.25 PFLOP/s nominal each)
FP16_PER_BF16 = 1.0


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            d = json.load(fh)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# The sources each kernel is built from (its translation unit and the headers it
# includes); recorded traffic stays valid while these files are unchanged.
_COMMON_SOURCES = ("tg_ptx.cuh", "tg_device.cuh", "tg_internal.h")
KERNEL_SOURCES = {
    "tiled_pair_kernel": ("k_tiled2.cu",),
    "tiled_gemm_kernel": ("k_tiled.cu",),
    "splitk_gemm_kernel": ("k_splitk.cu", "tg_skinny.cuh"),
    "w4_gemm_kernel": ("k_w4.cu",),
    "attn_fwd_kernel": ("k_attn.cu",),
    "softmax_rows": ("k_softmax.cu",),
}


def kernel_source_hash(kernel: str | None = None) -> str:
    """Hash of the sources of `kernel` (a key of KERNEL_SOURCES or a name starting
    with one), or of every source file when kernel is None or unknown."""
    csrc = os.path.join(ROOT, "tiled_tensor_core_tcgen05_gb300", "csrc")
    files = None
    if kernel is not None:
        for k, own in KERNEL_SOURCES.items():
            if kernel.startswith(k):
                files = [os.path.join(csrc, f) for f in own + _COMMON_SOURCES]
                break
    if files is None:
        files = glob.glob(os.path.join(csrc, "*"))
    h = hashlib.sha256()
    for f in sorted(files):
        with open(f, "rb") as fh:
            h.update(os.path.basename(f).encode())
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on the
    current kernel sources (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as fh:
        d = json.load(fh)
    e = d.get(workload)
    if not e or e.get("kernel_hash") != kernel_source_hash(e.get("kernel")):
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as fh:
            for line in fh:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        pw = [num(r[3]) for r in rows if num(r[3]) is not None]
        # "under load": samples drawing well above idle power
        loaded = [s for s, p in zip(sm, pw) if p is not None and pw and p > 0.5 * max(pw)] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows),
                "power_w_max": max(pw) if pw else None}


def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
        pg = dist
    return world, rank, local, pg


def max_over_ranks(pg, x: float) -> float:
    if pg is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def barrier(pg):
    if pg is not None:
        pg.barrier()


# ------------------------------------------------------------------ GPU arm

KERNELS = {"auto": 0, "tiled": 1, "lsu": 2, "splitk": 3, "pair": 4}


def time_workload(tg, w, steps: int, warmup: int, flush_bytes: int, pg=None, sampler=None, kernel: int = 0):
    """Time `steps` calls of tg_gemm on device-resident inputs. Returns the timed
    region (ms, max over ranks) and per-launch kernel durations."""
    import torch
    import workloads
    stream = torch.cuda.current_stream()
    sh = stream.cuda_stream
    dC = torch.empty((w.M, w.N), dtype=torch.float16, device="cuda") if hasattr(w, "M") else None
    if isinstance(w, workloads.SoftmaxWorkload):
        (X,) = w.inputs()
        dA = X.cuda()
        dB = ds = None
        db = torch.empty_like(dA)
        args = (dA.data_ptr(), db.data_ptr(), w.M, w.N, sh)

        def call():
            tg.tg_softmax_rows(*args)
    elif isinstance(w, workloads.AttnWorkload):
        dC = None
        Q, K, V = w.inputs()
        dA, dB, ds = Q.cuda(), K.cuda(), V.cuda()
        db = torch.empty_like(dA)
        args = (dA.data_ptr(), dB.data_ptr(), ds.data_ptr(), db.data_ptr(), w.B, w.S, w.H, w.D, bool(w.causal), sh)

        def call():
            tg.tg_attention_fwd(*args)
    elif isinstance(w, workloads.W4Workload):
        A, Bq, sc, bias = w.inputs()
        dA, dB, ds = A.cuda(), Bq.cuda(), sc.cuda()
        db = bias.cuda() if bias is not None else None
        args = (dA.data_ptr(), dB.data_ptr(), ds.data_ptr(), db.data_ptr() if db is not None else None,
                dC.data_ptr(), w.M, w.N, w.K, int(w.gelu), 0, sh)

        def call():
            tg.tg_gemm_w4(*args)
    else:
        A, B, bias = w.inputs()
        dA, dB = A.cuda(), B.cuda()
        db = bias.cuda() if bias is not None else None
        args = (dA.data_ptr(), dB.data_ptr(), db.data_ptr() if db is not None else None, dC.data_ptr(),
                w.M, w.N, w.K, int(w.gelu))

        def call():
            if kernel:
                tg.tg_gemm_ex(*args, kernel, 0, sh)
            else:
                tg.tg_gemm(*args, sh)
    flush = torch.empty(flush_bytes, dtype=torch.uint8, device="cuda") if flush_bytes else None

    for _ in range(warmup):
        call()
    torch.cuda.synchronize()
    st, where = tg.tg_device_status(None)
    if st != tg.OK:
        raise RuntimeError(f"watchdog status {st} (site {where}) during warm-up of {w.name}")
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    barrier(pg)
    torch.cuda.synchronize()
    if sampler:
        sampler.start()
    t_start.record(stream)
    for i in range(steps):
        if flush is not None:
            flush.zero_()  # evict the (L2-sized) inputs between steps
        starts[i].record(stream)
        call()
        ends[i].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop() if sampler else None
    barrier(pg)
    launch_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    region_ms = t_start.elapsed_time(t_end)
    kernel_ms = sum(launch_ms)
    st, where = tg.tg_device_status(None)
    if st != tg.OK:
        raise RuntimeError(f"watchdog status {st} (site {where}) during timing of {w.name}")
    del dA, dB, db, dC, flush
    return {"region_ms": max_over_ranks(pg, region_ms), "kernel_ms": max_over_ranks(pg, kernel_ms),
            "launch_ms": launch_ms, "clocks": clocks}


def time_e2e(tg, w, steps: int, warmup: int, n_streams: int = 2):
    """Same metric through the host-buffer entry point: every step copies the
    step's inputs from pinned host memory, runs the GEMM and copies C back
    (tg_gemm_staged). Steps alternate between `n_streams` streams, each with its
    own device buffers, so one step's copies overlap another step's kernel."""
    import torch
    A, B, bias = w.inputs()
    hA, hB = A.pin_memory(), B.pin_memory()
    hb = bias.pin_memory() if bias is not None else None
    hC = [torch.empty((w.M, w.N), dtype=torch.float16).pin_memory() for _ in range(n_streams)]
    dev = [(torch.empty_like(A, device="cuda"), torch.empty_like(B, device="cuda"),
            torch.empty_like(bias, device="cuda") if bias is not None else None,
            torch.empty((w.M, w.N), dtype=torch.float16, device="cuda")) for _ in range(n_streams)]
    streams = [torch.cuda.Stream() for _ in range(n_streams)]
    main = torch.cuda.current_stream()

    def run(n):
        start = torch.cuda.Event()
        start.record(main)
        for s in streams:
            s.wait_event(start)
        for i in range(n):
            j = i % n_streams
            dA, dB, db, dC = dev[j]
            tg.gemm_staged(hA, hB, hb, hC[j], dA, dB, db, dC, gelu=w.gelu, stream=streams[j])
        for s in streams:
            done = torch.cuda.Event()
            done.record(s)
            main.wait_event(done)

    run(warmup)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(main)
    run(steps)
    e1.record(main)
    e1.synchronize()
    ms = e0.elapsed_time(e1)
    h2d = 2 * (w.M * w.K + w.K * w.N) + (2 * w.N if bias is not None else 0)
    d2h = 2 * w.M * w.N
    return ms, h2d, d2h


def time_unfused(tg, w, steps: int, warmup: int):
    """The unfused comparator for a workload with an epilogue: the GEMM with no
    epilogue and no bias (C written to HBM), then tg_bias_gelu reading C back,
    adding the bias, applying GELU and writing C again. Returns ms per step."""
    import torch
    A, B, bias = w.inputs()
    dA, dB = A.cuda(), B.cuda()
    db = bias.cuda() if bias is not None else None
    dC = torch.empty((w.M, w.N), dtype=torch.float16, device="cuda")
    sh = torch.cuda.current_stream().cuda_stream

    def step():
        tg.tg_gemm(dA.data_ptr(), dB.data_ptr(), None, dC.data_ptr(), w.M, w.N, w.K, tg.EPI_NONE, sh)
        tg.tg_bias_gelu(dC.data_ptr(), db.data_ptr() if db is not None else None, w.M, w.N, int(w.gelu), sh)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        step()
    e1.record()
    e1.synchronize()
    return e0.elapsed_time(e1) / steps


def roofline_entry(w, avg_launch_ms, pk, pk_kind, bound, traffic=None):
    t = avg_launch_ms / 1e3
    if bound == "tensor":
        achieved = w.flops() / t / 1e12
        peak = pk["bf16_tflops"] * FP16_PER_BF16
        unit = "TFLOP/s"
        peak_note = f"bf16_tflops (burst) of {pk_kind}; fp16 dense rate = bf16 dense rate"
    else:
        achieved = w.bytes() / t / 1e9
        peak = pk["hbm_gbs"]
        unit = "GB/s"
        peak_note = f"hbm_gbs of {pk_kind}"
    e = {"bound": bound, "achieved": round(achieved, 2), "peak": peak, "unit": unit,
         "frac": round(achieved / peak, 4), "traffic": traffic, "peak_source": peak_note}
    if bound == "tensor" and "bf16_tflops_sustained" in pk:
        e["frac_of_sustained"] = round(achieved / (pk["bf16_tflops_sustained"] * FP16_PER_BF16), 4)
    return e


def cpu_baseline(w, budget_s: float, metric_unit: str):
    """The oracle as it stands, on the host cores, on whole rows of C."""
    import oracle
    A, B, bias = w.inputs()
    threads = oracle.max_threads()
    # calibrate on one row per thread (the oracle spreads rows over its threads)
    cal = max(1, min(w.M, threads))
    t0 = time.perf_counter()
    oracle.gemm(A, B, bias, gelu=w.gelu, rows=(0, cal))
    t_cal = time.perf_counter() - t0
    rows = max(1, min(w.M, int(budget_s / max(t_cal, 1e-4)) * cal))
    t0 = time.perf_counter()
    oracle.gemm(A, B, bias, gelu=w.gelu, rows=(0, rows))
    dt = time.perf_counter() - t0
    flops = 2.0 * rows * w.N * w.K
    if metric_unit == "GB/s":
        value = (2.0 * rows * w.K + 2.0 * w.K * w.N + 2.0 * rows * w.N) / dt / 1e9
    else:
        value = flops / dt / 1e12
    return {"value": value, "unit": metric_unit, "cores": threads, "kind": "oracle",
            "sample": f"rows 0..{rows - 1} of {w.M} of the {w.name} product ({rows * w.N * w.K:.3g} fp64 FMAs, "
                      f"{dt:.2f} s)"}


def run_gpu(args):
    import torch
    world, rank, local, pg = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    import workloads
    import tiled_tensor_core_tcgen05_gb300 as tg

    pk, pk_kind = peaks()
    l2 = torch.cuda.get_device_properties(local).L2_cache_size
    main = workloads.BY_NAME[args.workload]
    sampler = ClockSampler(local) if rank == 0 else None
    res = time_workload(tg, main, args.steps, args.warmup, 0 if main.bytes() > 2 * l2 else 2 * l2 + (1 << 20),
                        pg=pg, sampler=sampler, kernel=KERNELS[args.kernel])
    ms_per_step = res["region_ms"] / args.steps
    avg_launch = res["kernel_ms"] / args.steps
    gemm_main = isinstance(main, workloads.Workload)
    if hasattr(main, "flops") and not isinstance(main, workloads.SoftmaxWorkload):
        value, unit, main_bound = world * main.flops() / (ms_per_step / 1e3) / 1e12, "TFLOP/s", "tensor"
    else:  # a bandwidth kernel timed as the main line (profiling runs)
        value, unit, main_bound = world * main.bytes() / (ms_per_step / 1e3) / 1e9, "GB/s", "hbm"
    config = {"workload": main.describe(),
              "l2": (f"inputs larger than L2 ({main.bytes() / 1e6:.0f} MB vs {l2 / 1e6:.0f} MB)"
                     if main.bytes() > 2 * l2 else "L2 flushed between steps"),
              "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}
    if gemm_main:
        config.update({"M": main.M, "N": main.N, "K": main.K,
                       "epilogue": ("bias+" if main.has_bias else "") + ("gelu" if main.gelu else "none"),
                       "kernel": args.kernel})
    out = {
        "metric": METRIC, "value": round(value, 2), "unit": unit, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16 in, f32 accumulate, f16 out",
        "data": "synthetic (seeded uniform/normal fp16, see workloads/)",
        "config": config,
        "gpu_launches": args.steps,
    }
    out["roofline"] = roofline_entry(main, avg_launch, pk, pk_kind, main_bound, recorded_traffic(main.name))
    out["clocks"] = res["clocks"]
    # the rest of the suite, same rules, fewer steps
    extra = []
    if not args.only_main:
        for w in (workloads.ALL + workloads.W4_ALL + (workloads.ATTN_4096, workloads.ATTN_4096_CAUSAL) +
                  (workloads.SOFTMAX_4096, workloads.SOFTMAX_VOCAB)):
            if w.name == main.name:
                continue
            steps = max(5, min(args.steps, 50))  # secondary workloads: at most 50 timed launches
            r = time_workload(tg, w, steps, max(3, args.warmup), 0 if w.bytes() > 2 * l2 else 2 * l2 + (1 << 20),
                              pg=pg)
            avg = r["kernel_ms"] / steps
            # the skinny (decode) shapes stream their weights; attention and the big GEMMs are contractions
            bound = ("hbm" if getattr(w, "M", 1 << 30) <= 128 or isinstance(w, workloads.SoftmaxWorkload)
                     else "tensor")
            e = {"workload": w.describe(), "ms_per_launch": round(avg, 5),
                 "GB/s": round(w.bytes() / (avg / 1e3) / 1e9, 1),
                 "roofline": roofline_entry(w, avg, pk, pk_kind, bound, recorded_traffic(w.name))}
            if hasattr(w, "flops"):
                e["TFLOP/s"] = round(w.flops() / (avg / 1e3) / 1e12, 2)
            if getattr(w, "gelu", False) or getattr(w, "has_bias", False):
                # unfused comparator, back to back (the fused figure above is per launch)
                un_ms = time_unfused(tg, w, steps, max(3, args.warmup))
                e["unfused_ms_per_step"] = round(un_ms, 5)
                e["fusion_speedup"] = round(un_ms / avg, 3)
                out["gpu_launches"] += 2 * steps
            extra.append(e)
            out["gpu_launches"] += steps
    out["workloads"] = extra
    if rank == 0:
        if gemm_main:
            e2e_steps = max(3, min(args.steps, 20))
            ms, h2d, d2h = time_e2e(tg, main, e2e_steps, 2)
            out["e2e"] = {"value": round(main.flops() * e2e_steps / (ms / 1e3) / 1e12, 2), "unit": "TFLOP/s",
                          "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                          "ms_per_step": round(ms / e2e_steps, 4),
                          "api": "tg_gemm_staged, pinned host buffers, steps alternating over 2 streams"}
            if world == 1 and not args.no_cpu_baseline:
                out["cpu_baseline"] = cpu_baseline(main, args.cpu_budget_s, "TFLOP/s")
        print(json.dumps(out), flush=True)
    if pg is not None:
        pg.destroy_process_group()


# ------------------------------------------------------------------ reference arm (the oracle)

def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    import workloads
    w = workloads.BY_NAME[args.workload]
    A, B, bias = w.inputs()
    threads = oracle.max_threads()
    # calibrate on one row per thread (the oracle spreads rows over its threads)
    cal = max(1, min(w.M, threads))
    t0 = time.perf_counter()
    oracle.gemm(A, B, bias, gelu=w.gelu, rows=(0, cal))
    t_cal = time.perf_counter() - t0
    total_budget = args.ref_budget_s
    rows = max(1, min(w.M, int(total_budget / max(1, args.steps + args.warmup) / max(t_cal, 1e-4)) * cal))
    for i in range(args.warmup):
        oracle.gemm(A, B, bias, gelu=w.gelu, rows=((i * rows) % w.M, min(rows, w.M - (i * rows) % w.M)))
    t0 = time.perf_counter()
    done_rows = 0
    for i in range(args.steps):
        r0 = (i * rows) % w.M
        n = min(rows, w.M - r0)
        oracle.gemm(A, B, bias, gelu=w.gelu, rows=(r0, n))
        done_rows += n
    dt = time.perf_counter() - t0
    value = 2.0 * done_rows * w.N * w.K / dt / 1e12
    sample = f"{rows} rows of C per step ({rows * w.N * w.K:.3g} fp64 FMAs) of the {w.name} product"
    out = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64 (fp16 inputs)",
           "data": "synthetic (seeded uniform/normal fp16, see workloads/)",
           "config": {"workload": w.describe(), "M": w.M, "N": w.N, "K": w.K, "sample": sample},
           "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle", "sample": sample},
           "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
           "gpu_launches": 0}
    print(json.dumps(out), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["tg", "reference"], default="tg")
    ap.add_argument("--workload", default="square_8192")
    ap.add_argument("--only-main", action="store_true", help="time the headline workload only")
    ap.add_argument("--kernel", choices=sorted(KERNELS), default="auto",
                    help="pin the kernel of the headline workload (profiling); default: the library's choice")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget-s", type=float, default=10.0)
    ap.add_argument("--ref-budget-s", type=float, default=60.0)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
