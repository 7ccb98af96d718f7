#!/usr/bin/env python
"""Benchmark of the ONNX matrix-product kernels on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints ONE JSON line on stdout.  The headline workload is the bf16 Gemm
M=N=K=8192, transB=1, alpha=0.5, beta=2.0, C[1,8192] (one step = one mm_gemm
call = one tcgen05 kernel launch); the metric is achieved TFLOP/s (2*M*N*K per
step) and its fraction of the measured dense bf16 peak.  The line's
"per_config" object holds the same metric for each of the five workloads (f32
MatMul, the Gemm, batched broadcast bf16 MatMul, int8 QLinearMatMul, bf16
GroupedMatMul) and for their type variants, each with its roofline fraction and,
for the five, the C++ oracle's throughput on a stated sample of the same
workload timed on this host's cores.  The full per-workload detail goes to
stderr as one JSON line.

Timing: W untimed warm-up steps, then K steps bracketed by a barrier and
torch.cuda.synchronize(), timed with CUDA events on the stream the library
launches on; the max over ranks is reported.  The Gemm inputs (A and B,
256 MiB) are larger than L2 (129 MB); the small f32 workload flushes L2
(reads a 258 MB buffer) between timed iterations.  nvidia-smi samples the SM
clock and throttle reasons every 20 ms while the timed loop runs.

Under torchrun (N > 1) every rank runs the same workload on its own GPU
(independent problems, no data-path collective: weak scaling); the
process group is used only for barriers and the max of the timings.
"""

import os

os.environ.setdefault("OPENBLAS_NUM_THREADS", str(os.cpu_count() or 1))

import argparse  # noqa: E402
import hashlib  # noqa: E402
import json  # noqa: E402
import math  # noqa: E402
import re  # noqa: E402
import statistics  # noqa: E402
import subprocess  # noqa: E402
import sys  # noqa: E402
import threading  # noqa: E402
import time  # noqa: E402

import numpy as np  # noqa: E402
import torch  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "achieved TFLOPS/TOPS and % of GB300 dense tensor peak, per config"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# CUDA-core peak probes (mm_alu_probe op, dependent steps per chain): int32
# multiply-add for the int32 GEMM, fp64 FMA for the f64 one.  The fp64 probe
# reads below what the f64 GEMM itself sustains (about 1.06 against 1.24
# TFLOP/s), so the f64 GEMM is compared with the part's nominal fp64 rate
# (1.25 TFLOP/s) and the probe is reported beside it.
ALU_PROBES = {"gemm_i32_simt": (0, 100000), "gemm_f64_simt": (1, 4000)}
NOMINAL_FP64_TFLOPS = 1.25
L2_BYTES = 129 * 10 ** 6
# The other workloads' short loops (compared with the burst peak, itself a
# short best-of-10 measurement) each start after this much idle time, so
# that none inherits the heat of the one before.
EXTRA_IDLE_S = 1.0


# ------------------------------------------------------------------ distributed plumbing

def dist_init(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if torch.cuda.is_available() else torch.device("cpu")
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ measurement helpers

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi SM clock / throttle-reason samples, 20 ms apart, for one GPU."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, device):
        self.samples = []
        self.proc = None
        self.window = None
        try:
            uuid = str(torch.cuda.get_device_properties(device).uuid)
            sel = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", sel, "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.time(), parts))

    def mark(self, t0, t1):
        self.window = (t0, t1)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = self.samples
        if self.window:
            inside = [s for s in rows if self.window[0] - 0.05 <= s[0] <= self.window[1] + 0.05]
            rows = inside or rows
        mhz, maxes, reasons = [], [], set()
        for _, p in rows:
            try:
                mhz.append(float(p[1]))
                maxes.append(float(p[2]))
            except ValueError:
                continue
            for name, val in zip(self.REASONS, p[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not mhz:
            return None
        return {"sm_mhz": statistics.median(mhz), "sm_max_mhz": max(maxes), "reasons": sorted(reasons),
                "samples": len(mhz)}


def l2_flusher(device):
    """Evicts L2 by reading a buffer twice its size.  The buffer is written
    once here; the flush itself only reads, so it leaves no dirty lines whose
    write-back the next timed kernel would pay."""
    buf = torch.ones(2 * L2_BYTES // 4, dtype=torch.float32, device=device)
    sink = torch.empty((), dtype=torch.float32, device=device)
    torch.cuda.synchronize(device)

    def flush():
        sink.copy_(buf.sum())
    return flush


def time_loop(step, steps, warmup, world, stream, flush=None, sampler=None, idle_s=0.0):
    """Average ms per step (max over ranks).  Back-to-back when flush is None,
    else each step timed alone after an L2 flush.  With idle_s the GPU first
    idles that long, so that short loops start from the same state."""
    if idle_s > 0:
        torch.cuda.synchronize()
        time.sleep(idle_s)
    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    t_wall0 = time.time()
    if flush is None:
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            step()
        e1.record(stream)
        e1.synchronize()
        ms = e0.elapsed_time(e1) / steps
    else:
        total = 0.0
        for _ in range(steps):
            flush()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            step()
            e1.record(stream)
            e1.synchronize()
            total += e0.elapsed_time(e1)
        ms = total / steps
    torch.cuda.synchronize()
    t_wall1 = time.time()
    if sampler is not None:
        sampler.mark(t_wall0, t_wall1)
    barrier(world)
    return max_over_ranks(ms, world), t_wall1 - t_wall0


KERNEL_SOURCES = ("common.cuh", "tc_internal.h", "tc_ptx.cuh", "tc_gemm.cu")


def _code_only(text):
    """C++ source with comments and blank space removed (string literals in the
    kernel sources hold no comment markers)."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def source_hash():
    """Hash of the tensor-core GEMM's code (comments and spacing ignored): a
    stored ncu traffic figure is valid only while this hash is unchanged."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "quantized_gemm_gb300", "csrc")
    for f in KERNEL_SOURCES:
        with open(os.path.join(csrc, f)) as fh:
            h.update((f + "\n" + _code_only(fh.read())).encode())
    return h.hexdigest()[:16]


def stored_traffic(name):
    """dram bytes per launch recorded from an ncu capture in profiles/<name>.md, if current."""
    path = os.path.join(ROOT, "profiles", name + ".md")
    try:
        text = open(path).read()
    except OSError:
        return None
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    h = re.search(r"source_hash:\s*([0-9a-f]+)", text)
    if not m or not h or h.group(1) != source_hash():
        return None
    return float(m.group(1))


# ------------------------------------------------------------------ workloads

def gemm_case(dev, M=8192, N=8192, K=8192):
    import quantized_gemm_gb300 as qg
    d = workloads.gemm_bf16(device=dev, M=M, N=N, K=K)
    Y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)

    def step():
        qg.mm_gemm(d["A"], d["B"], d["C"], d["alpha"], d["beta"], d["transA"], d["transB"], out=Y)
    return d, Y, step


def stream_peaks(dev, world, stream):
    """Write-only and copy bandwidth of the library's streaming kernels over
    2 GiB (best of 10 calls, CUDA events): the HBM roofline of a product whose
    traffic is nearly all output (the batched MatMul writes 2.15 GB and reads
    0.15 GB)."""
    import quantized_gemm_gb300 as qg
    nbytes = 2 << 30
    dst = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    src = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    src.fill_(1)
    out = {}
    for name, mode, traffic in (("write", 0, nbytes), ("write_bulk", 2, nbytes), ("copy", 1, 2 * nbytes)):
        best = None
        for _ in range(3):
            qg.mm_stream_probe(dst, src if mode == 1 else None, mode)
        for _ in range(10):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            qg.mm_stream_probe(dst, src if mode == 1 else None, mode)
            e1.record(stream)
            e1.synchronize()
            ms = e0.elapsed_time(e1)
            best = ms if best is None else min(best, ms)
        out[name + "_gbs"] = traffic / best / 1e6
    del dst, src
    torch.cuda.empty_cache()
    return out


def alu_peak(dev, stream, op, iters):
    """Peak multiply-add rate of one CUDA-core instruction (2 ops each), in
    T ops/s: best of 3 launches of the library's arithmetic-rate probe."""
    import quantized_gemm_gb300 as qg
    macs = qg.mm_alu_probe(op, iters)
    out = torch.empty(macs // (qg.MM_ALU_CHAINS * iters), dtype=torch.float64, device=dev)
    qg.mm_alu_probe(op, iters, out=out)
    best = None
    for _ in range(3):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        qg.mm_alu_probe(op, iters, out=out)
        e1.record(stream)
        e1.synchronize()
        ms = e0.elapsed_time(e1)
        best = ms if best is None else min(best, ms)
    return 2.0 * macs / best / 1e9


def bench_extra_workloads(dev, world, stream, peaks, peak_kind, cpu=True):
    """The four other workloads and their type variants: one call of the public API per step.
    With cpu, the C++ oracle is also timed on a sample of each of the four."""
    import quantized_gemm_gb300 as qg
    import oracle.native as orc
    out = {}
    bf16_peak = peaks["bf16_tflops"]
    hbm = peaks["hbm_gbs"]

    # 1. f32 MatMul [4,128,64] @ [64,96] and [64] @ [4,64,96]: latency-bound.
    d = workloads.matmul_f32(device=dev)
    Y1 = torch.empty((4, 128, 96), dtype=torch.float32, device=dev)
    Y2 = torch.empty((4, 96), dtype=torch.float32, device=dev)

    def s1():
        qg.mm_matmul(d["A"], d["B"], out=Y1)
        qg.mm_matmul(d["A1"], d["B1"], out=Y2)
    flush = l2_flusher(dev)
    ms, _ = time_loop(s1, 50, 5, world, stream, flush=flush, idle_s=EXTRA_IDLE_S)
    paths = []
    for a, b, y in ((d["A"], d["B"], Y1), (d["A1"], d["B1"], Y2)):
        qg.mm_matmul(a, b, out=y)
        paths.append({qg.MM_PATH_SIMT: "simt", qg.MM_PATH_VECTOR: "vector", qg.MM_PATH_TENSOR: "tensor"}.get(
            qg.mm_last_path(), "?"))
    # The same two calls captured once in a CUDA graph and replayed: the
    # GPU-side latency without the per-call host work of the binding.
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        s1()
    torch.cuda.synchronize()
    ms_graph, _ = time_loop(graph.replay, 50, 5, world, torch.cuda.current_stream(dev), flush=flush,
                            idle_s=EXTRA_IDLE_S)
    flops = 2 * 4 * 128 * 64 * 96 + 2 * 4 * 64 * 96
    nbytes = 4 * (4 * 128 * 64 + 64 * 96 + 4 * 128 * 96 + 64 + 4 * 64 * 96 + 4 * 96)
    out["matmul_f32"] = {"value": flops / ms / 1e9, "unit": "TFLOP/s", "us_per_call": ms * 1e3,
                         "us_per_graph_replay": ms_graph * 1e3, "bound": "latency", "paths": "+".join(paths),
                         "hbm_gbs": nbytes / ms / 1e6, "kernels_per_call": 2, "l2": "flushed between iterations"}
    if cpu:
        h = {k: d[k].cpu().numpy() for k in ("A", "B", "A1", "B1")}
        rate, _ = oracle_rate(lambda: (orc.matmul(h["A"], h["B"]), orc.matmul(h["A1"], h["B1"])), flops)
        out["matmul_f32"]["cpu_baseline"] = cpu_entry(rate, "whole")
    del d, Y1, Y2, graph

    # 2a. Skinny products of the headline Gemm's B (stored [N, K], transB = 1):
    # one row (a vector-matrix product), 4 and 16 rows against 8192 x 8192 bf16.
    # One stream over B (134 MB): bound by HBM bandwidth.  1 and 4 rows run the
    # few-row CUDA-core kernel, 16 rows the tensor cores.  A call takes about as
    # long as the binding's host work, so the value is taken from a CUDA graph
    # of 10 calls that alternate between two copies of B (each call reads the B
    # the previous call did not: nothing of it is left in L2); us_per_call is
    # the same call made directly, back to back.
    Bs = workloads.gemm_bf16(device=dev)["B"]
    Bs2 = Bs.clone()
    reps = 10
    for rows in (1, 4, 16, 64):
        As = (torch.randn((rows, 8192), generator=torch.Generator(device=dev).manual_seed(rows), device=dev)
              / math.sqrt(8192)).to(torch.bfloat16)
        Ys = torch.empty((rows, 8192), dtype=torch.bfloat16, device=dev)
        ms_call, _ = time_loop(lambda: qg.mm_gemm(As, Bs, None, 1.0, 1.0, 0, 1, out=Ys), 50, 5, world, stream,
                               idle_s=EXTRA_IDLE_S)
        path = qg.mm_last_path()
        assert path == (qg.MM_PATH_VECTOR if rows <= 4 else qg.MM_PATH_TENSOR)

        def calls():
            for i in range(reps):
                qg.mm_gemm(As, (Bs, Bs2)[i % 2], None, 1.0, 1.0, 0, 1, out=Ys)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            calls()
        torch.cuda.synchronize()
        ms_graph, _ = time_loop(graph.replay, 10, 3, world, torch.cuda.current_stream(dev))
        ms = ms_graph / reps
        nbytes = 2 * (rows * 8192 + 8192 * 8192 + rows * 8192)
        out["gemm_bf16_skinny_m%d" % rows] = {
            "value": nbytes / ms / 1e6, "unit": "GB/s", "us_per_call_in_graph": ms * 1e3,
            "us_per_call": ms_call * 1e3, "bound": "hbm", "peak_gbs": hbm,
            "frac": nbytes / ms / 1e6 / hbm, "tflops": 2 * rows * 8192 * 8192 / ms / 1e9, "kernels_per_call": 1,
            "kernel": "vec_gemm_kernel" if path == qg.MM_PATH_VECTOR else "tc_gemm_kernel<kSkinny>",
            "shape": "[%d, 8192] @ B^T, B [8192, 8192] bf16" % rows,
            "l2": "each call in the graph reads the copy of B the previous call did not"}
        del As, Ys, graph
    del Bs, Bs2
    torch.cuda.empty_cache()

    # 2b. The headline Gemm in fp32 (three tf32 tensor-core products per step).
    d = workloads.gemm_bf16(device=dev, dtype=torch.float32)
    Yf = torch.empty((8192, 8192), dtype=torch.float32, device=dev)
    ms, _ = time_loop(lambda: qg.mm_gemm(d["A"], d["B"], d["C"], d["alpha"], d["beta"], 0, 1, out=Yf), 10, 3, world,
                      stream, idle_s=EXTRA_IDLE_S)
    assert qg.mm_last_path() == qg.MM_PATH_TENSOR
    tf = 2 * 8192 ** 3 / ms / 1e9
    tf32_peak = bf16_peak * 1.1 / 2.25      # measured bf16 peak x nominal dense tf32/bf16 (1.1 / 2.25 PFLOP/s)
    out["gemm_f32"] = {"value": tf, "unit": "TFLOP/s", "ms_per_call": ms, "bound": "tensor",
                       "pipe": "tf32 x3 (hi*hi + hi*lo + lo*hi)", "peak_tflops": tf32_peak / 3,
                       "frac": tf / (tf32_peak / 3), "kernels_per_call": 1,
                       "peak_note": "measured bf16 peak x nominal tf32/bf16 ratio (1.1/2.25), / 3 products"}
    del d, Yf
    torch.cuda.empty_cache()

    # 2c. The CUDA-core kernel on the types without a tensor-core path:
    # f64 and int32 Gemm, 4096^3 (FFMA/DFMA/IMAD throughput).
    for name, dt in (("gemm_f64_simt", torch.float64), ("gemm_i32_simt", torch.int32)):
        g = torch.Generator(device=dev).manual_seed(5)
        if dt.is_floating_point:
            A = torch.randn((4096, 4096), generator=g, device=dev, dtype=dt)
            B = torch.randn((4096, 4096), generator=g, device=dev, dtype=dt)
        else:
            A = torch.randint(-100, 100, (4096, 4096), generator=g, device=dev, dtype=dt)
            B = torch.randint(-100, 100, (4096, 4096), generator=g, device=dev, dtype=dt)
        Yx = torch.empty((4096, 4096), dtype=dt, device=dev)
        ms, _ = time_loop(lambda: qg.mm_gemm(A, B, None, 1.0, 0.0, 0, 0, out=Yx), 5, 2, world, stream,
                          idle_s=EXTRA_IDLE_S)
        assert qg.mm_last_path() == qg.MM_PATH_SIMT
        val = 2 * 4096 ** 3 / ms / 1e9
        probe = alu_peak(dev, stream, *ALU_PROBES[name])
        apeak = NOMINAL_FP64_TFLOPS if dt == torch.float64 else probe
        out[name] = {"value": val, "unit": "TFLOP/s" if dt.is_floating_point else "TOP/s",
                     "ms_per_call": ms, "bound": "alu", "kernel": "simt_gemm_kernel", "shape": "4096^3",
                     "peak": apeak, "frac": val / apeak, "probe": probe,
                     "peak_note": ("nominal GB300 fp64 (the mm_alu_probe fp64 reading is lower)" if dt == torch.float64
                                   else "measured: mm_alu_probe int32 multiply-add chains")}
        del A, B, Yx
    torch.cuda.empty_cache()

    # 3. bf16 batched MatMul A[8,32,2048,128] @ B[1,32,128,2048]: HBM-bound
    #    (2.15 GB output), compared with the copy bandwidth and with the
    #    write-only stream measured here.
    sp = stream_peaks(dev, world, stream)
    d = workloads.matmul_bf16_bcast(device=dev)
    Y = torch.empty((8, 32, 2048, 2048), dtype=torch.bfloat16, device=dev)
    ms, _ = time_loop(lambda: qg.mm_matmul(d["A"], d["B"], out=Y), 20, 3, world, stream, idle_s=EXTRA_IDLE_S)
    flops = 2 * 256 * 2048 * 2048 * 128
    nbytes = (d["A"].numel() + d["B"].numel() + Y.numel()) * 2
    gbs = nbytes / ms / 1e6
    wpeak = max(sp["write_gbs"], sp["write_bulk_gbs"])
    out["matmul_bf16_bcast"] = {"value": flops / ms / 1e9, "unit": "TFLOP/s", "ms_per_call": ms,
                                "bound": "hbm", "achieved_gbs": gbs, "peak_gbs": hbm, "frac": gbs / hbm,
                                "write_gbs": Y.numel() * 2 / ms / 1e6, "write_peak_gbs": wpeak,
                                "frac_of_write_peak": Y.numel() * 2 / ms / 1e6 / wpeak, "stream_probe": sp,
                                "kernels_per_call": 1, "l2": "inputs+output larger than L2"}
    if cpu:
        A = d["A"][0, :8].double().cpu().numpy()
        B = d["B"][0, :8].double().cpu().numpy()
        rate, _ = oracle_rate(lambda: orc.matmul(A, B), 2 * 8 * 2048 * 2048 * 128)
        out["matmul_bf16_bcast"]["cpu_baseline"] = cpu_entry(rate, "8 of 256 batches")
        del A, B
    del d, Y
    torch.cuda.empty_cache()

    # 4. int8 QLinearMatMul 16384 x 4096 x 4096 (runs on the f16 tensor pipe),
    #    then the same product with uint8 / mixed operands, float16 scales and
    #    batch-indexed quantisation parameters.
    out["qlinear_s8"] = bench_qlinear(workloads.qlinear_s8(device=dev), world, stream, bf16_peak, cpu=cpu)
    for name, kw in sorted(workloads.QLINEAR_VARIANTS.items()):
        out[name] = bench_qlinear(workloads.qlinear(device=dev, **kw), world, stream, bf16_peak)

    # 5. GroupedMatMul M=16384, S=2, G=64, K=4096, N=14336: bf16 with int32
    #    indices, then float16 with int64 indices.
    out["grouped_bf16"] = bench_grouped(workloads.grouped_bf16(device=dev), world, stream, bf16_peak, cpu=cpu)
    out["grouped_f16_i64"] = bench_grouped(
        workloads.grouped_bf16(device=dev, dtype=torch.float16, index_dtype=torch.int64), world, stream, bf16_peak)
    # The same sizes with 8 groups (4096 rows each on average): CTA-pair tiles.
    out["grouped_bf16_g8"] = bench_grouped(workloads.grouped_bf16(device=dev, G=8), world, stream, bf16_peak)
    # Weight-only int8 experts at the same sizes (dequantization fused into the
    # mainloop): one scale per group and column, and per 128 rows of K.
    for block in (0, 128):
        out["grouped_qweights_b%d" % block] = bench_grouped_q(workloads.grouped_qweights(device=dev, block=block),
                                                              world, stream, bf16_peak)
    # The same with int4 experts (two weights per byte, 1.9 GB), one scale per
    # group and column.
    out["grouped_qweights4_b0"] = bench_grouped_q(workloads.grouped_qweights(device=dev, bits=4), world, stream,
                                                  bf16_peak)
    return out


def bench_qlinear(d, world, stream, peak, cpu=False):
    import quantized_gemm_gb300 as qg
    keys = ("a", "a_scale", "a_zero_point", "b", "b_scale", "b_zero_point", "y_scale", "y_zero_point")
    a, b = d["a"], d["b"]
    ydims = tuple(a.shape[:-1]) + (b.shape[-1],)
    y = torch.empty(ydims, dtype=d["y_zero_point"].dtype, device=a.device)
    ws = torch.empty(qg.mm_qlinear_matmul_workspace_size(a, b), dtype=torch.uint8, device=a.device)
    ms, _ = time_loop(lambda: qg.mm_qlinear_matmul(*[d[k] for k in keys], out=y, workspace=ws), 20, 3, world,
                      stream, idle_s=EXTRA_IDLE_S)
    assert qg.mm_last_path() == qg.MM_PATH_TENSOR
    ops = 2 * y.numel() * a.shape[-1]
    tops = ops / ms / 1e9
    info = torch.iinfo(y.dtype)
    sat = float(((y == info.max) | (y == info.min)).float().mean().item())
    res = {"value": tops, "unit": "TOP/s", "ms_per_call": ms, "bound": "tensor",
           "pipe": "f16 (no int8 tensor-core instruction on sm_103a)", "peak_tflops": peak, "frac": tops / peak,
           "kernels_per_call": 3, "saturated_fraction": sat, "l2": "inputs+workspace larger than L2",
           "types": "a %s, b %s, y %s, scales %s" % (a.dtype, b.dtype, y.dtype, d["a_scale"].dtype),
           "shape": "a %s, b %s" % (list(a.shape), list(b.shape))}
    if cpu:
        import oracle.native as orc
        rows = 256
        h = {k: d[k].cpu().numpy() for k in keys}
        for k in ("a", "a_scale", "a_zero_point"):
            h[k] = h[k][:rows]
        rate, _ = oracle_rate(lambda: orc.qlinear_matmul(*[h[k] for k in keys]), 2 * rows * b.shape[-1] * a.shape[-1])
        res["cpu_baseline"] = cpu_entry(rate, "%d of %d rows" % (rows, a.shape[0]))
        res["cpu_baseline"]["unit"] = "TOP/s"
    del d, y, ws
    torch.cuda.empty_cache()
    return res


def bench_grouped(d, world, stream, peak, cpu=False):
    import quantized_gemm_gb300 as qg
    x, w, gi = d["input"], d["weights"], d["group_indices"]
    M, K = x.shape
    S, N = gi.shape[1], w.shape[2]
    yo = torch.empty((M, S, N), dtype=x.dtype, device=x.device)
    ws = torch.empty(qg.mm_grouped_matmul_workspace_size(x, w, gi), dtype=torch.uint8, device=x.device)
    ms, _ = time_loop(lambda: qg.mm_grouped_matmul(x, w, gi, d["bias"], out=yo, workspace=ws), 10, 3, world,
                      stream, idle_s=EXTRA_IDLE_S)
    assert qg.mm_last_path() == qg.MM_PATH_TENSOR
    tf = 2 * M * S * K * N / ms / 1e9
    res = {"value": tf, "unit": "TFLOP/s", "ms_per_call": ms, "bound": "tensor", "peak_tflops": peak,
           "frac": tf / peak, "kernels_per_call": 4, "l2": "weights (7.5 GB) larger than L2",
           "types": "%s, indices %s" % (x.dtype, gi.dtype)}
    if cpu:
        import oracle.native as orc
        toks, cols = 512, 512
        hx = x[:toks].double().cpu().numpy()
        hw = w[:, :, :cols].double().cpu().numpy()
        hb = d["bias"][:, :cols].double().cpu().numpy()
        hg = gi[:toks].cpu().numpy()
        rate, _ = oracle_rate(lambda: orc.grouped_matmul(hx, hw, hg, hb), 2 * toks * S * K * cols)
        res["cpu_baseline"] = cpu_entry(rate, "%d tokens x %d cols" % (toks, cols))
        del hx, hw
    del d, x, w, gi, yo, ws
    torch.cuda.empty_cache()
    return res


def bench_grouped_q(d, world, stream, peak):
    import quantized_gemm_gb300 as qg
    x, wq, gi = d["input"], d["weights_q"], d["group_indices"]
    p4 = d.get("packed4")
    M, K = x.shape
    S, N = gi.shape[1], wq.shape[2] * (2 if p4 else 1)
    yo = torch.empty((M, S, N), dtype=x.dtype, device=x.device)
    args = (x, wq, d["w_scale"], d["w_zero_point"], d["block_size"], gi)
    ws = torch.empty(qg.mm_grouped_matmul_qweights_workspace_size(*args, packed4=p4), dtype=torch.uint8,
                     device=x.device)
    ms, _ = time_loop(lambda: qg.mm_grouped_matmul_qweights(*args, d["bias"], out=yo, workspace=ws, packed4=p4), 10,
                      3, world, stream, idle_s=EXTRA_IDLE_S)
    assert qg.mm_last_path() == qg.MM_PATH_TENSOR
    tf = 2 * M * S * K * N / ms / 1e9
    wdesc = p4 or "int8"
    res = {"value": tf, "unit": "TFLOP/s", "ms_per_call": ms, "bound": "tensor", "peak_tflops": peak,
           "frac": tf / peak, "kernels_per_call": 4,
           "l2": "weights (%.1f GB %s) larger than L2" % (wq.numel() / 1e9, wdesc),
           "types": "input %s, weights %s, block %s" % (x.dtype, wdesc, d["block_size"] or "K")}
    del d, x, wq, gi, yo, ws
    torch.cuda.empty_cache()
    return res


def cpu_baseline_gemm(d, rows):
    """The C++ oracle on the first `rows` rows of the Gemm workload: (TFLOP/s, seconds)."""
    import oracle.native as orc
    A = d["A"][:rows].double().cpu().numpy()
    B = d["B"].double().cpu().numpy()
    C = d["C"].double().cpu().numpy()
    flops = 2.0 * rows * B.shape[0] * B.shape[1]
    return oracle_rate(lambda: orc.gemm(A, B, C, alpha=d["alpha"], beta=d["beta"], transA=d["transA"],
                                        transB=d["transB"]), flops)


def e2e_gemm(d, flops, world, steps, warmup=3):
    import quantized_gemm_gb300 as qg
    dev = d["A"].device
    M, N = d["A"].shape[0], d["B"].shape[0]
    host = [d[k].cpu().pin_memory() for k in ("A", "B", "C")]
    bufs = [[torch.empty_like(d[k]) for k in ("A", "B", "C")] for _ in range(2)]
    outs = [torch.empty((M, N), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    hys = [torch.empty((M, N), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    s_in, s_mm, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    ev = {k: [torch.cuda.Event() for _ in range(2)] for k in ("in", "mm", "out")}

    def run(n):
        for i in range(n):
            b = i % 2
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev["mm"][b])            # step i-2 has read this input set
                for dst, src in zip(bufs[b], host):
                    dst.copy_(src, non_blocking=True)
                ev["in"][b].record(s_in)
            with torch.cuda.stream(s_mm):
                s_mm.wait_event(ev["in"][b])
                if i >= 2:
                    s_mm.wait_event(ev["out"][b])           # step i-2's result has been copied out
                A, B, C = bufs[b]
                qg.mm_gemm(A, B, C, d["alpha"], d["beta"], 0, 1, out=outs[b], stream=s_mm)
                ev["mm"][b].record(s_mm)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev["mm"][b])
                hys[b].copy_(outs[b], non_blocking=True)
                ev["out"][b].record(s_out)

    run(warmup)
    torch.cuda.synchronize()
    barrier(world)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    s_mm.wait_event(e0)
    s_out.wait_event(e0)
    run(steps)
    s_out.wait_stream(s_in)
    s_out.wait_stream(s_mm)
    e1.record(s_out)
    e1.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1) / steps, world)
    h2d = sum(h.numel() * h.element_size() for h in host)
    d2h = hys[0].numel() * hys[0].element_size()
    return {"value": _r(flops / ms / 1e9 * world), "unit": "TFLOP/s", "ms_per_step": _r(ms),
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "host_link_gbs": _r((h2d + d2h) / ms / 1e6)}


def oracle_rate(fn, ops, min_s=0.5):
    """The C++ oracle's throughput on one sample: fn (one oracle call on it)
    repeated until min_s of wall time has passed; returns (T ops/s, seconds)."""
    fn()                                     # builds/loads the library, warms the caches
    n, t0 = 0, time.perf_counter()
    while True:
        fn()
        n += 1
        dt = time.perf_counter() - t0
        if dt >= min_s:
            return ops * n / dt / 1e12, dt


def cpu_entry(rate, sample):
    import oracle.native
    return {"value": rate, "unit": "TFLOP/s", "cores": oracle.native.num_threads(), "kind": "oracle",
            "sample": sample}


# ------------------------------------------------------------------ arms

def run_reference(args, rank, world):
    """The C++ oracle as the reference arm: each step is a bounded row sample of the Gemm."""
    if rank != 0:
        return
    import oracle.native as orc
    d = workloads.gemm_bf16(device="cpu")
    A = d["A"].double().numpy()
    B = d["B"].double().numpy()
    C = d["C"].double().numpy()

    def gemm_rows(r0, rows):
        orc.gemm(A[r0:r0 + rows], B, C, alpha=d["alpha"], beta=d["beta"], transB=1)
    # Rows per step from a timed probe of 8 rows, so that the whole
    # warm-up + timed run takes about 40 s of CPU time.
    t0 = time.perf_counter()
    gemm_rows(0, 8)
    per_row = (time.perf_counter() - t0) / 8
    total_steps = args.steps + args.warmup
    rows = int(max(8, min(1024, 40.0 / max(1, total_steps) / max(per_row, 1e-6))))
    for i in range(args.warmup):
        gemm_rows(0, rows)
    t0 = time.perf_counter()
    for i in range(args.steps):
        gemm_rows((i * rows) % (A.shape[0] - rows + 1), rows)
    dt = (time.perf_counter() - t0) / max(1, args.steps)
    tflops = 2.0 * rows * 8192 * 8192 / dt / 1e12
    sample = "%d rows of the 8192^3 Gemm per step (C++ oracle: plain double loops)" % rows
    line = {
        "impl": "reference", "metric": METRIC, "value": tflops, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "gemm_bf16", "M": 8192, "N": 8192, "K": 8192, "transB": 1,
                   "alpha": 0.5, "beta": 2.0, "sample_rows_per_step": rows},
        "cpu_baseline": {"value": tflops, "unit": "TFLOP/s", "cores": orc.num_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": tflops, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def _r(x, sig=4):
    """x rounded to `sig` significant digits (None, integers and text unchanged)."""
    if not isinstance(x, float) or x == 0 or not math.isfinite(x):
        return x
    return float("%.*g" % (sig, x))


SHORT_KEYS = {"us_per_graph_replay": "us_graph", "us_per_call_in_graph": "us_graph", "achieved_gbs": "gbs",
              "frac_of_write_peak": "frac_write",
              "write_peak_gbs": "write_peak_gbs"}


def compact(entry, keys):
    """The listed keys of a workload's detail, numbers rounded, some keys
    shortened (SHORT_KEYS); a cpu_baseline keeps its value, core count and
    sample (its unit is the entry's)."""
    out = {}
    for k in keys:
        v = entry.get(k)
        if v is None:
            continue
        if isinstance(v, dict):
            v = {kk: _r(vv) for kk, vv in v.items() if kk in ("value", "cores", "sample")}
        out[SHORT_KEYS.get(k, k)] = _r(v)
    return out


# Workload name in the detail -> key in per_config: the five configurations,
# then the type variants (other operand, scale and index types, int8 and int4
# experts, fp32) at the same sizes.
PER_CONFIG = (
    ("1_matmul_f32", "matmul_f32", ("value", "unit", "us_per_call", "us_per_graph_replay", "paths",
                                    "cpu_baseline")),
    ("3_matmul_bf16_bcast", "matmul_bf16_bcast", ("value", "unit", "ms_per_call", "achieved_gbs", "frac",
                                                 "frac_of_write_peak", "cpu_baseline")),
    ("4_qlinear_s8", "qlinear_s8", ("value", "unit", "ms_per_call", "frac", "cpu_baseline")),
    ("5_grouped_bf16", "grouped_bf16", ("value", "unit", "ms_per_call", "frac", "cpu_baseline")),
    ("f1_qlinear_u8", "qlinear_u8", ("value", "frac")),
    ("f1_qlinear_u8s8_f16scales", "qlinear_u8s8_f16scales", ("value", "frac")),
    ("f1_qlinear_s8_batched4", "qlinear_s8_batched4", ("value", "frac")),
    ("f2_grouped_qweights_b0", "grouped_qweights_b0", ("value", "frac")),
    ("f2_grouped_qweights_b128", "grouped_qweights_b128", ("value", "frac")),
    ("f2_grouped_qweights_int4", "grouped_qweights4_b0", ("value", "frac")),
    ("f3_grouped_f16_i64", "grouped_f16_i64", ("value", "frac")),
    ("f4_gemm_f32", "gemm_f32", ("value", "ms_per_call", "frac")),
    ("a3_skinny_m16", "gemm_bf16_skinny_m16", ("value", "unit", "us_per_call_in_graph", "frac")),
    ("a3_skinny_m64", "gemm_bf16_skinny_m64", ("value", "us_per_call_in_graph", "frac")),
    ("a13_gemm_f64_simt", "gemm_f64_simt", ("value", "frac", "peak")),
    ("a13_gemm_i32_simt", "gemm_i32_simt", ("value", "frac", "peak")),
)


def per_config_entries(headline, extras):
    """The line's per_config object: the headline Gemm's entry and the compact
    entry (PER_CONFIG) of every other workload measured, sorted by key; an
    error of the other workloads is kept, cut to 200 characters."""
    per_config = {"2_gemm_bf16": headline}
    for key, name, keys in PER_CONFIG:
        if name in extras:
            per_config[key] = compact(extras[name], keys)
    if "error" in extras:
        per_config["error"] = extras["error"][:200]
    return dict(sorted(per_config.items()))


def run_ours(args, rank, world, local):
    import quantized_gemm_gb300 as qg
    from quantized_gemm_gb300 import build as qbuild
    qbuild.build()
    dev = torch.device("cuda", torch.cuda.current_device())
    stream = torch.cuda.current_stream(dev)
    peaks, peak_src = measured_peaks()

    M = N = K = 8192
    d, Y, step = gemm_case(dev, M, N, K)
    sampler = ClockSampler(dev)
    ms, wall = time_loop(step, args.steps, args.warmup, world, stream, sampler=sampler)
    clocks = sampler.stop()
    flops = 2.0 * M * N * K
    tflops_rank = flops / ms / 1e9
    value = tflops_rank * world
    # The denominator measured in the same regime as the timed loop: the
    # sustained (power-capped, back-to-back) cuBLAS figure when the loop ran
    # longer than a second or the power cap was active while it ran, else the
    # burst figure.  Both fractions are reported.
    capped = bool(clocks) and "sw_power_cap" in clocks.get("reasons", [])
    peak_kind = "bf16_tflops_sustained" if (wall > 1.0 or capped) else "bf16_tflops"
    peak = peaks.get(peak_kind, peaks["bf16_tflops"])
    burst_peak = peaks["bf16_tflops"]
    status = qg.mm_get_device_status()
    assert qg.mm_last_path() == qg.MM_PATH_TENSOR, "the Gemm did not run on the tensor-core kernel"

    # e2e: the same call from pinned host buffers, every step copying its inputs
    # in and its result out inside the timed region.  As a user of the API
    # would, steps are pipelined over three streams and two sets of device
    # buffers: the copies of step k+1's inputs and of step k-1's result overlap
    # step k's product.
    e2e = None
    if not args.skip_e2e:
        e2e = e2e_gemm(d, flops, world, min(max(args.steps, 3), 40))

    cpu = None
    want_cpu = rank == 0 and world == 1 and not args.skip_cpu
    if want_cpu:
        rows = 256
        cpu_tf, _ = cpu_baseline_gemm(d, rows)
        cpu = cpu_entry(_r(cpu_tf), "%d of 8192 rows, C++ oracle (plain double loops)" % rows)
    del d, Y
    torch.cuda.empty_cache()

    extras = {}
    if not args.skip_extras:
        # The headline line is printed even if one of the other workloads fails.
        try:
            extras = bench_extra_workloads(dev, world, stream, peaks, peak_kind, cpu=want_cpu)
        except Exception as exc:  # noqa: BLE001 - reported in the JSON line
            extras = {"error": "%s: %s" % (type(exc).__name__, exc)}

    # (the headline's roofline and CPU baseline are in the line itself)
    per_config = per_config_entries({"value": _r(tflops_rank), "unit": "TFLOP/s", "ms_per_call": _r(ms),
                                     "frac": _r(tflops_rank / peak)}, extras)

    traffic = stored_traffic("tc_gemm_kernel_gemm_bf16_8192")
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "per_config": per_config,
        "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic, seeded",
        "config": {"workload": "gemm_bf16", "M": M, "N": N, "K": K, "transB": 1, "alpha": 0.5,
                   "beta": 2.0, "C": [1, N], "parallelism": "replicas x%d" % world, "l2": "A+B 256 MiB > L2"},
        "roofline": {"bound": "tensor", "achieved": _r(tflops_rank), "peak": peak, "unit": "TFLOP/s",
                     "frac": _r(tflops_rank / peak), "traffic": traffic, "peak_kind": "%s %s" % (peak_src, peak_kind),
                     "frac_of_burst": _r(tflops_rank / burst_peak)},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": args.steps,
        "clocks": clocks,
        "device_status": status,
    }
    if rank == 0:
        # The detail of every workload, for the record, on stderr; stdout holds
        # only the one JSON line.
        sys.stderr.write("bench detail: " + json.dumps({"workloads": extras}) + "\n")
        sys.stderr.flush()
        print(json.dumps(line), flush=True)


def run_profile_workload(args):
    """Only one workload's public-API call, W + K times (for ncu captures)."""
    import quantized_gemm_gb300 as qg
    from quantized_gemm_gb300 import build as qbuild
    qbuild.build()
    dev = torch.device("cuda", torch.cuda.current_device())
    name = args.profile_workload
    if name == "gemm_bf16":
        _, _, step = gemm_case(dev)
    elif name == "matmul_f32":
        d = workloads.matmul_f32(device=dev)
        Y1 = torch.empty((4, 128, 96), dtype=torch.float32, device=dev)
        Y2 = torch.empty((4, 96), dtype=torch.float32, device=dev)
        step = lambda: (qg.mm_matmul(d["A"], d["B"], out=Y1), qg.mm_matmul(d["A1"], d["B1"], out=Y2))
    elif name in ("gemm_f64_simt", "gemm_i32_simt"):
        dt = torch.float64 if name == "gemm_f64_simt" else torch.int32
        A = torch.ones((4096, 4096), dtype=dt, device=dev)
        B = torch.ones((4096, 4096), dtype=dt, device=dev)
        Yx = torch.empty((4096, 4096), dtype=dt, device=dev)
        step = lambda: qg.mm_gemm(A, B, None, 1.0, 0.0, 0, 0, out=Yx)
    elif name == "gemm_f32":
        d = workloads.gemm_bf16(device=dev, dtype=torch.float32)
        Yf = torch.empty((8192, 8192), dtype=torch.float32, device=dev)
        step = lambda: qg.mm_gemm(d["A"], d["B"], d["C"], d["alpha"], d["beta"], 0, 1, out=Yf)
    elif name.startswith("gemm_bf16_skinny_m"):
        # [rows, 8192] @ B^T, B the headline's; a _tensor suffix forces the
        # tensor-core kernel where the planner would take the few-row one
        rows = int(name[len("gemm_bf16_skinny_m"):].split("_")[0])
        if name.endswith("_tensor"):
            qg.mm_set_path_policy(qg.MM_PATH_TENSOR)
        Bs = workloads.gemm_bf16(device=dev)["B"]
        As = (torch.randn((rows, 8192), device=dev) / math.sqrt(8192)).to(torch.bfloat16)
        Ys = torch.empty((rows, 8192), dtype=torch.bfloat16, device=dev)
        step = lambda: qg.mm_gemm(As, Bs, None, 1.0, 1.0, 0, 1, out=Ys)
    elif name.startswith("matmul_bf16_bcast"):
        # a _bN suffix: N leading batches instead of 8 (a smaller case of the
        # same product, for full ncu captures)
        nb = int(name.split("_b")[-1]) if name.startswith("matmul_bf16_bcast_b") else 8
        d = workloads.matmul_bf16_bcast(device=dev, batch=(nb, 32))
        Y = torch.empty((nb, 32, 2048, 2048), dtype=torch.bfloat16, device=dev)
        step = lambda: qg.mm_matmul(d["A"], d["B"], out=Y)
    elif name == "qlinear_s8" or name in workloads.QLINEAR_VARIANTS:
        d = workloads.qlinear(device=dev, **workloads.QLINEAR_VARIANTS.get(name, {}))
        keys = ("a", "a_scale", "a_zero_point", "b", "b_scale", "b_zero_point", "y_scale", "y_zero_point")
        yq = torch.empty(tuple(d["a"].shape[:-1]) + (d["b"].shape[-1],), dtype=d["y_zero_point"].dtype, device=dev)
        ws = torch.empty(qg.mm_qlinear_matmul_workspace_size(d["a"], d["b"]), dtype=torch.uint8, device=dev)
        step = lambda: qg.mm_qlinear_matmul(*[d[k] for k in keys], out=yq, workspace=ws)
    elif name.startswith("grouped_qweights"):
        # grouped_qweights_b128: blocks of 128 rows; a _gN suffix: N groups (same M, K, N);
        # grouped_qweights4_...: int4 experts
        bits = 4 if name.startswith("grouped_qweights4") else 8
        parts = dict((t[0], int(t[1:])) for t in name[len("grouped_qweights") + (bits == 4):].split("_") if t)
        d = workloads.grouped_qweights(device=dev, block=parts.get("b", 0), G=parts.get("g", 64), bits=bits)
        p4 = d.get("packed4")
        yo = torch.empty((16384, 2, 14336), dtype=torch.bfloat16, device=dev)
        qargs = (d["input"], d["weights_q"], d["w_scale"], d["w_zero_point"], d["block_size"], d["group_indices"])
        ws = torch.empty(qg.mm_grouped_matmul_qweights_workspace_size(*qargs, packed4=p4), dtype=torch.uint8,
                         device=dev)
        step = lambda: qg.mm_grouped_matmul_qweights(*qargs, d["bias"], out=yo, workspace=ws, packed4=p4)
    elif name.startswith("grouped_bf16"):
        # grouped_bf16_g8: 8 groups (same M, K, N); a _nN suffix: N output
        # columns (a smaller case of the same routing, for full ncu captures)
        parts = dict((t[0], int(t[1:])) for t in name[len("grouped_bf16"):].split("_") if t)
        N = parts.get("n", 14336)
        d = workloads.grouped_bf16(device=dev, G=parts.get("g", 64), N=N)
        yo = torch.empty((16384, 2, N), dtype=torch.bfloat16, device=dev)
        ws = torch.empty(qg.mm_grouped_matmul_workspace_size(d["input"], d["weights"], d["group_indices"]),
                         dtype=torch.uint8, device=dev)
        step = lambda: qg.mm_grouped_matmul(d["input"], d["weights"], d["group_indices"], d["bias"], out=yo,
                                            workspace=ws)
    else:
        raise SystemExit("unknown workload " + name)
    stream = torch.cuda.current_stream(dev)
    ms, _ = time_loop(step, args.steps, args.warmup, 1, stream)
    print(json.dumps({"profile_workload": name, "ms_per_call": ms, "status": qg.mm_get_device_status()}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--skip-e2e", action="store_true")
    ap.add_argument("--skip-cpu", action="store_true")
    ap.add_argument("--skip-extras", action="store_true")
    ap.add_argument("--profile-workload", default=None,
                    help="run only this workload (gemm_bf16, matmul_f32, gemm_f64_simt, gemm_i32_simt, "
                         "gemm_bf16_skinny_mR[_tensor], matmul_bf16_bcast[_bN], qlinear_s8 or a "
                         "QLinear variant, "
                         "grouped_bf16[_gG][_nN])")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    rank, world, local = dist_init(args.gpus)
    if args.profile_workload:
        run_profile_workload(args)
        return
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
