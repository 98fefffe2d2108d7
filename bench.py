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
# the GB300's datasheet dense fp16 tensor rate (without sparsity), TFLOP/s
SKU_FP16_DENSE_TFLOPS = 2250.0
# nominal HBM3e bandwidth of the part, GB/s
SKU_HBM_GBS = 8000.0


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
    "w4r_gemm_kernel": ("k_w4r.cu",),
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
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,timestamp")

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
        self.timed = []  # (host time of the sample, SM MHz)
        for r in rows:
            if len(r) >= 10 and num(r[1]) is not None:
                t = _smi_time(r[9])
                if t is not None:
                    self.timed.append((t, num(r[1])))
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows),
                "samples_under_load": len(loaded), "power_w_max": max(pw) if pw else None}


def _smi_time(text: str):
    """nvidia-smi's timestamp ("2026/12/03 05:30:36.123", local time) as seconds since the epoch."""
    import datetime
    try:
        return datetime.datetime.strptime(text.strip(), "%Y/%m/%d %H:%M:%S.%f").timestamp()
    except ValueError:
        return None


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
# the 4-bit GEMM's kernels (tg_gemm_w4_kernel), for --kernel with a 4-bit workload
W4_KERNELS = {"auto": 0, "w4tmem": 1, "w4reg": 2}
# one-thread oracle timings: the whole product (None) or its first rows
ONE_THREAD_ROWS = {"square_256": None, "ragged_1000x1030x520_bias_gelu": None, "decode_16x28672x8192": 2}


def kernel_code(w, name: str) -> int:
    """The --kernel choice as the code the workload's entry point takes."""
    import workloads
    table = W4_KERNELS if isinstance(w, workloads.W4Workload) else KERNELS
    if name not in table:
        raise SystemExit(f"--kernel {name} does not apply to {w.name}")
    return table[name]


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
        host_inputs = (X,)
        dC = None
        dA = X.cuda()
        dB = ds = None
        db = torch.empty_like(dA)
        args = (dA.data_ptr(), db.data_ptr(), w.M, w.N, sh)

        def call():
            tg.tg_softmax_rows(*args)
    elif isinstance(w, workloads.AttnWorkload):
        dC = None
        Q, K, V = w.inputs()
        host_inputs = (Q, K, V)
        dA, dB, ds = Q.cuda(), K.cuda(), V.cuda()
        db = torch.empty_like(dA)
        args = (dA.data_ptr(), dB.data_ptr(), ds.data_ptr(), db.data_ptr(), w.B, w.S, w.H, w.D, bool(w.causal), sh)

        def call():
            tg.tg_attention_fwd(*args)
    elif isinstance(w, workloads.W4Workload):
        A, Bq, sc, bias = w.inputs()
        host_inputs = (A, Bq, sc, bias)
        dA, dB, ds = A.cuda(), Bq.cuda(), sc.cuda()
        db = bias.cuda() if bias is not None else None
        args = (dA.data_ptr(), dB.data_ptr(), ds.data_ptr(), db.data_ptr() if db is not None else None,
                dC.data_ptr(), w.M, w.N, w.K, int(w.gelu), w.fmt_code, kernel, 0, sh)

        def call():
            tg.tg_gemm_w4_kernel(*args)
    else:
        A, B, bias = w.inputs()
        host_inputs = (A, B, bias)
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
    # the last timed launch's output, for the parity check against the oracle
    out = (dC if dC is not None else db).cpu()
    del dA, dB, db, dC, flush
    return {"region_ms": max_over_ranks(pg, region_ms), "kernel_ms": max_over_ranks(pg, kernel_ms),
            "launch_ms": launch_ms, "clocks": clocks, "output": out, "inputs": host_inputs, "call": None}


def time_sustained(tg, w, seconds: float, sampler, chunk: int = 50):
    """Back-to-back launches of `w` for about `seconds`, in chunks of `chunk`
    launches each timed with CUDA events between two host timestamps, while
    nvidia-smi samples the SM clock. Each chunk gets the median clock of the
    samples inside its host window; chunks are binned by that clock (50 MHz
    bins), so the rate can be read against the clock the power limit allowed."""
    import torch
    A, B, bias = w.inputs()
    dA, dB = A.cuda(), B.cuda()
    db = bias.cuda() if bias is not None else None
    dC = torch.empty((w.M, w.N), dtype=torch.float16, device="cuda")
    stream = torch.cuda.current_stream()
    args = (dA.data_ptr(), dB.data_ptr(), db.data_ptr() if db is not None else None, dC.data_ptr(),
            w.M, w.N, w.K, int(w.gelu), stream.cuda_stream)
    for _ in range(10):
        tg.tg_gemm(*args)
    torch.cuda.synchronize()
    sampler.start()
    chunks = []
    t_stop = time.time() + seconds
    while time.time() < t_stop:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        h0 = time.time()
        e0.record(stream)
        for _ in range(chunk):
            tg.tg_gemm(*args)
        e1.record(stream)
        e1.synchronize()
        chunks.append((h0, time.time(), e0.elapsed_time(e1)))
    clocks = sampler.stop()
    st, where = tg.tg_device_status(None)
    if st != tg.OK:
        raise RuntimeError(f"watchdog status {st} (site {where}) during the sustained run of {w.name}")
    total_ms = sum(c[2] for c in chunks)
    launches = chunk * len(chunks)
    bins = {}
    for h0, h1, ms in chunks:
        mhz = [m for t, m in getattr(sampler, "timed", []) if h0 <= t <= h1]
        if not mhz:
            continue
        b = int(round(statistics.median(mhz) / 50.0) * 50)
        n, t = bins.get(b, (0, 0.0))
        bins[b] = (n + 1, t + ms)
    by_clock = [{"sm_mhz": b, "chunks": n, "TFLOP/s": round(w.flops() * chunk * n / (t / 1e3) / 1e12, 1)}
                for b, (n, t) in sorted(bins.items())]
    return {"seconds": round(total_ms / 1e3, 3), "launches": launches, "chunk": chunk,
            "ms_per_launch": round(total_ms / launches, 5),
            "TFLOP/s": round(w.flops() * launches / (total_ms / 1e3) / 1e12, 2),
            "by_clock": by_clock, "clocks": clocks}


def host_call_us(tg, w, calls: int = 200):
    """Host time to enqueue one tg_gemm call (argument checks, kernel choice,
    tensor maps, launch), averaged over `calls` back-to-back calls."""
    import torch
    A, B, bias = w.inputs()
    dA, dB = A.cuda(), B.cuda()
    db = bias.cuda() if bias is not None else None
    dC = torch.empty((w.M, w.N), dtype=torch.float16, device="cuda")
    args = (dA.data_ptr(), dB.data_ptr(), db.data_ptr() if db is not None else None, dC.data_ptr(),
            w.M, w.N, w.K, int(w.gelu), torch.cuda.current_stream().cuda_stream)
    tg.tg_gemm(*args)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(calls):
        tg.tg_gemm(*args)
    dt = time.perf_counter() - t0
    torch.cuda.synchronize()
    return round(dt / calls * 1e6, 2)


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
    if bound == "tensor":
        if "bf16_tflops_sustained" in pk:
            e["frac_of_sustained"] = round(achieved / (pk["bf16_tflops_sustained"] * FP16_PER_BF16), 4)
        e["frac_of_sku"] = round(achieved / SKU_FP16_DENSE_TFLOPS, 4)
        e["sku_peak"] = SKU_FP16_DENSE_TFLOPS
    else:
        e["frac_of_sku"] = round(achieved / SKU_HBM_GBS, 4)
        e["sku_peak"] = SKU_HBM_GBS
    return e


_ALL_THREADS = []


def oracle_threads() -> int:
    """Threads of the oracle's parallel regions on this host: taken once, before
    any one-thread timing (the oracle's thread setting persists in the process),
    and passed explicitly to every all-core call."""
    if not _ALL_THREADS:
        import oracle
        _ALL_THREADS.append(max(1, oracle.max_threads()))
    return _ALL_THREADS[0]


def _oracle_unit(w, inputs, n: int, first: int = 0, threads: int = 0, rng=None):
    """Run the oracle on `n` units of workload `w` (rows of C, or query rows for
    attention) and return (flops, algorithmic bytes) of that sample."""
    import numpy as np
    import oracle
    import workloads
    if isinstance(w, workloads.Workload):
        A, B, bias = inputs
        oracle.gemm(A, B, bias, gelu=w.gelu, rows=(first, n), threads=threads)
        return 2.0 * n * w.N * w.K, 2.0 * (n * w.K + w.K * w.N + n * w.N)
    if isinstance(w, workloads.W4Workload):
        A, Bq, sc, bias = inputs
        oracle.gemm_w4(A, Bq, sc, bias, gelu=w.gelu, rows=(first, n), threads=threads, fmt=w.fmt_code)
        groups = (w.K + w.group - 1) // w.group
        return 2.0 * n * w.N * w.K, 2.0 * n * w.K + w.K * w.N / 2 + 2.0 * groups * w.N + 2.0 * n * w.N
    if isinstance(w, workloads.AttnWorkload):
        Q, K, V = inputs
        rng = rng or np.random.default_rng(0)
        rows = rng.integers(0, w.B * w.S * w.H, n)
        oracle.attention(Q, K, V, causal=w.causal, rows=rows, threads=threads)
        pos = (rows // w.H) % w.S
        keys = (pos + 1).sum() if w.causal else n * w.S
        return 4.0 * w.D * float(keys), 8.0 * w.D * n  # this query's q, o; its share of k, v
    (X,) = inputs
    oracle.softmax(X, rows=(first, n), threads=threads)
    return 0.0, 4.0 * n * w.N


def cpu_baseline(w, budget_s: float, metric_unit: str, inputs=None):
    """The oracle as it stands, on all host cores, on a bounded sample of the
    workload's units (whole rows of C, or query rows), about `budget_s` of work."""
    import oracle
    import workloads
    if inputs is None:
        inputs = w.inputs()
    threads = oracle_threads()
    total = w.B * w.S * w.H if isinstance(w, workloads.AttnWorkload) else w.M
    # calibrate on one unit per thread (the oracle spreads units over its threads)
    cal = max(1, min(total, threads))
    t0 = time.perf_counter()
    _oracle_unit(w, inputs, cal, threads=threads)
    t_cal = time.perf_counter() - t0
    n = max(1, min(total, int(budget_s / max(t_cal, 1e-4)) * cal))
    t0 = time.perf_counter()
    flops, nbytes = _oracle_unit(w, inputs, n, threads=threads)
    dt = time.perf_counter() - t0
    value = nbytes / dt / 1e9 if metric_unit == "GB/s" else flops / dt / 1e12
    unit_name = "query rows" if isinstance(w, workloads.AttnWorkload) else "rows"
    return {"value": value, "unit": metric_unit, "cores": threads, "kind": "oracle",
            "sample": f"{n} of {total} {unit_name} of {w.name} ({flops / 2:.3g} fp64 FMAs, {dt:.2f} s)"}


PARITY_TOL = {"default": (1e-2, 1e-2), "softmax": (1e-6, 2e-3)}  # (abs, rel) per element


def parity_check(w, inputs, out, n_samples: int = 4096, seed: int = 12345):
    """The timed launch's output against the oracle, on sampled outputs the
    oracle evaluates one by one from the definition (GEMMs: single elements;
    4-bit GEMM, attention and softmax: whole rows). Returns the element count,
    the largest absolute and relative errors and the number of elements outside
    |gpu - ref| <= atol + rtol |ref|."""
    import numpy as np
    import oracle
    import workloads
    rng = np.random.default_rng(seed)
    got_all = out.numpy()
    if isinstance(w, workloads.Workload):
        A, B, bias = inputs
        if w.M * w.N <= n_samples:
            rows, cols = np.divmod(np.arange(w.M * w.N), w.N)
        else:
            rows = np.concatenate([[0, w.M - 1, 0, w.M - 1], rng.integers(0, w.M, n_samples - 4)])
            cols = np.concatenate([[0, 0, w.N - 1, w.N - 1], rng.integers(0, w.N, n_samples - 4)])
        ref = oracle.gemm_sampled(A, B, bias, w.gelu, rows, cols, threads=oracle_threads())
        got = got_all[rows, cols]
        what = "sampled elements (first and last rows and columns included)"
    elif isinstance(w, workloads.W4Workload):
        A, Bq, sc, bias = inputs
        picks = sorted({0, w.M - 1})
        ref = np.concatenate([oracle.gemm_w4(A, Bq, sc, bias, gelu=w.gelu, rows=(r, 1), threads=oracle_threads(),
                                              fmt=w.fmt_code)
                              for r in picks])
        got = got_all[picks]
        what = f"rows {picks} (every column)"
    elif isinstance(w, workloads.AttnWorkload):
        Q, K, V = inputs
        pos = np.concatenate([[0, w.S - 1], rng.integers(0, w.S, 14)])
        rows = np.array([(b * w.S + s) * w.H + h for b in range(w.B) for s in pos for h in (0, w.H - 1)])
        ref = oracle.attention(Q, K, V, causal=w.causal, rows=rows, threads=oracle_threads())
        got = got_all.reshape(-1, w.D)[rows]
        what = f"{len(rows)} query rows (first and last positions, first and last heads)"
    else:
        (X,) = inputs
        picks = sorted({0, w.M - 1, *rng.integers(0, w.M, 6).tolist()})
        ref = np.concatenate([oracle.softmax(X, rows=(r, 1), threads=oracle_threads()) for r in picks])
        got = got_all[picks]
        what = f"{len(picks)} rows"
    atol, rtol = PARITY_TOL["softmax" if isinstance(w, workloads.SoftmaxWorkload) else "default"]
    got = np.asarray(got, dtype=np.float64).ravel()
    ref = np.asarray(ref, dtype=np.float64).ravel()
    err = np.abs(got - ref)
    bad = ~(err <= atol + rtol * np.abs(ref))  # NaN counts as a violation
    rel = err / np.maximum(np.abs(ref), 1e-30)
    return {"checked": int(got.size), "what": what, "max_abs_err": float(np.nanmax(err)),
            "max_rel_err": float(np.nanmax(rel)), "violations": int(bad.sum()),
            "tolerance": f"|gpu - ref| <= {atol:g} + {rtol:g} |ref|", "oracle": "fp64 CPU oracle"}


def host_cpu():
    """Host CPU model and logical core count (for the oracle timings)."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if model is None:
        try:
            with open("/proc/cpuinfo") as fh:
                for line in fh:
                    if line.lower().startswith(("model name", "cpu part")):
                        model = line.split(":", 1)[1].strip()
                        break
        except OSError:
            pass
    return {"model": model or "unknown", "logical_cpus": os.cpu_count()}


def cpu_baseline_one_thread(w, row_budget: int | None = None):
    """The oracle on one host thread: the whole product when `row_budget` is None,
    else its first `row_budget` rows, with the time scaled to the whole product."""
    import oracle
    A, B, bias = w.inputs()
    rows = w.M if row_budget is None else max(1, min(w.M, row_budget))
    t0 = time.perf_counter()
    oracle.gemm(A, B, bias, gelu=w.gelu, rows=(0, rows), threads=1)
    dt = time.perf_counter() - t0
    full_s = dt * w.M / rows
    return {"threads": 1, "seconds": round(dt, 4), "rows": f"0..{rows - 1} of {w.M}",
            "seconds_whole_product": round(full_s, 4), "fp64_fmas": rows * w.N * w.K,
            "GFLOP/s": round(2.0 * rows * w.N * w.K / dt / 1e9, 3)}


def run_gpu(args):
    import torch
    world, rank, local, pg = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    import workloads
    import tiled_tensor_core_tcgen05_gb300 as tg

    pk, pk_kind = peaks()
    l2 = torch.cuda.get_device_properties(local).L2_cache_size
    main = workloads.BY_NAME[args.workload]
    oracle_threads()
    sampler = ClockSampler(local) if rank == 0 else None
    res = time_workload(tg, main, args.steps, args.warmup, 0 if main.bytes() > 2 * l2 else 2 * l2 + (1 << 20),
                        pg=pg, sampler=sampler, kernel=kernel_code(main, args.kernel))
    ms_per_step = res["region_ms"] / args.steps
    avg_launch = res["kernel_ms"] / args.steps
    gemm_main = isinstance(main, workloads.Workload)
    skinny = getattr(main, "M", 1 << 30) <= 128  # decode shapes stream their weights from HBM
    if hasattr(main, "flops") and not isinstance(main, workloads.SoftmaxWorkload) and not skinny:
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
    cpu_ok = rank == 0 and world == 1 and not args.no_cpu_baseline
    if rank == 0:
        out["parity"] = parity_check(main, res["inputs"], res["output"])
    if cpu_ok:
        out["host_cpu"] = host_cpu()
    if rank == 0 and gemm_main and args.sustained_s > 0:
        s = time_sustained(tg, main, args.sustained_s, ClockSampler(local))
        s["frac_of_sustained_peak"] = round(s["TFLOP/s"] / (pk["bf16_tflops_sustained"] * FP16_PER_BF16), 4)
        s["peak_source"] = f"bf16_tflops_sustained of {pk_kind}; fp16 dense rate = bf16 dense rate"
        out["sustained"] = s
        out["gpu_launches"] += s["launches"]
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
            if rank == 0:
                e["parity"] = parity_check(w, r["inputs"], r["output"])
            if cpu_ok:
                e["cpu_baseline"] = cpu_baseline(w, args.cpu_budget_other_s, e["roofline"]["unit"], r["inputs"])
                if w.name in ONE_THREAD_ROWS:
                    e["cpu_one_thread"] = cpu_baseline_one_thread(w, ONE_THREAD_ROWS[w.name])
            if rank == 0 and isinstance(w, workloads.Workload) and w.M <= 256:
                e["host_us_per_call"] = host_call_us(tg, w)
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
            e2e_value = (main.flops() * e2e_steps / (ms / 1e3) / 1e12 if unit == "TFLOP/s"
                         else main.bytes() * e2e_steps / (ms / 1e3) / 1e9)
            out["e2e"] = {"value": round(e2e_value, 2), "unit": unit,
                          "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                          "ms_per_step": round(ms / e2e_steps, 4),
                          "api": "tg_gemm_staged, pinned host buffers, steps alternating over 2 streams"}
            if cpu_ok:
                out["cpu_baseline"] = cpu_baseline(main, args.cpu_budget_s, unit, res["inputs"])
                out["cpu_baseline"]["cpu_model"] = out["host_cpu"]["model"]
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
    ap.add_argument("--kernel", choices=sorted(set(KERNELS) | set(W4_KERNELS)), default="auto",
                    help="pin the kernel of the headline workload (profiling): GEMM kernels for GEMM workloads, "
                         "w4tmem / w4reg for 4-bit ones; default: the library's choice")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget-s", type=float, default=10.0, help="oracle seconds for the headline workload")
    ap.add_argument("--cpu-budget-other-s", type=float, default=2.0, help="oracle seconds for each other workload")
    ap.add_argument("--sustained-s", type=float, default=2.0,
                    help="seconds of back-to-back headline launches with binned clocks (0: skip)")
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
