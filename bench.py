#!/usr/bin/env python3
"""Benchmark of the tcgen05 GEMM library (one JSON line on stdout, rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--no-suite] [--no-cpu] [--detail]

A step is one GEMM C <- alpha*A*B + beta*C of the chosen workload (default: the
largest one, 8192^3 bf16 -> fp32 with A row-major, B column-major and beta = 0.5
reading an fp32 C) with operands already resident in HBM.  Between
timed steps L2 is flushed by writing a buffer larger than L2 and then reading it
back (so L2 holds clean lines of the flush buffer, not dirty ones whose write-back
would be charged to the next step), and only the GEMM launch is inside each
step's CUDA-event pair (on the stream the kernel runs on).
Value = whole-job TFLOP/s (2MNK per step, logical FLOPs) over all ranks.

Besides value and ms_per_step the line carries: the roofline of the GEMM kernel
(achieved TFLOP/s or GB/s against the measured peak), the end-to-end rate through
the host-buffer entry point gemm_host (pinned host operands, copies included),
the CPU oracle timed on the host cores on a bounded sample, SM clocks sampled
during the timed region, and compact summaries of every workload (512^3,
2048^3, 4096^3, 8192^3 and the 128x8192x8192 skinny shape, each beside cuBLAS),
of the odd and tail shapes and of the FP8 shapes, placed at the end of the line
so that a reader keeping only its tail still has them (--detail adds the full
per-workload records).

--impl reference times the CPU oracle (the plain FP64 triple loop) on the same
workload, one bounded row sample per step, on the host cores.

Multi-GPU: one process per GPU (torchrun); every rank runs its own replica
of the workload (the GEMM does not shard across GPUs here: replicas only),
a barrier and synchronize bracket the timed region, the time is the max over
ranks, and value = sum of the ranks' FLOPs / that time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import seeded_inputs as si  # noqa: E402

WORKLOAD_BY_NAME = {w["name"]: k for k, w in si.WORKLOADS.items()}
DEFAULT_WORKLOAD = si.WORKLOADS[4]["name"]
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 512 << 20    # > 129 MB L2
CSRC = os.path.join(ROOT, "dense_tensor_core_tcgen05_gb300", "csrc")


# ------------------------------------------------------------------ helpers

class L2Flush:
    """Evicts everything of the timed problem from L2 between steps: writes a
    buffer larger than L2, then reads it back (a column sum), so the next step
    starts with a cold L2 holding only clean lines."""

    def __init__(self, device):
        import torch
        self.buf = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
        self.rows = self.buf.view(-1, 1 << 16)
        self.sink = torch.empty(1 << 16, dtype=torch.float32, device=device)

    def __call__(self):
        import torch
        self.buf.zero_()
        torch.sum(self.rows, dim=0, out=self.sink)


def gemm_flops(M, N, K):
    """Logical FLOPs, 2MNK (one multiply and one add per inner-loop step)."""
    return 2 * M * N * K


def algorithmic_bytes(w):
    """Compulsory HBM bytes of one GEMM: each input read once, C written once
    (and read once when beta != 0)."""
    isz = 2
    osz = 4 if w["out_dtype"] == "f32" else 2
    b = w["M"] * w["K"] * isz + w["K"] * w["N"] * isz + w["M"] * w["N"] * osz
    if w["beta"] != 0.0:
        b += w["M"] * w["N"] * osz
    return b


def panel_intensity(bm, bn, item_bytes):
    """FLOP per byte of operand loads for a BM x BN output tile: 2*BM*BN/(s*(BM+BN))."""
    return 2 * bm * bn / (item_bytes * (bm + bn))


def roofline_bound(w, peak_tflops, hbm_gbs):
    """'tensor' when the tensor-core roof is lower than HBM bandwidth x intensity."""
    intensity = gemm_flops(w["M"], w["N"], w["K"]) / algorithmic_bytes(w)
    return "tensor" if peak_tflops * 1e12 <= hbm_gbs * 1e9 * intensity else "hbm"


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_hash():
    h = hashlib.sha256()
    for f in sorted(os.listdir(CSRC)):
        with open(os.path.join(CSRC, f), "rb") as fh:
            h.update(f.encode())
            h.update(fh.read())
    return h.hexdigest()[:16]


def load_traffic(workload_name):
    """DRAM bytes per launch from a committed ncu capture, if it was taken on the
    current kernel sources (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(workload_name)
    if not e or e.get("kernel_hash") != kernel_source_hash():
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling during the timed region."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            import tempfile
            self.path = os.path.join(tempfile.gettempdir(), f"clocks_bench_{os.getpid()}.csv")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.2)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        loaded = [s for s in sm if s > 0.5 * (max(mx) if mx else 1)] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


def aggregate_ranks(local_step_ms, flops_per_step, world, device=None):
    """Whole-job result of a replicated run: the step time is the MAX over ranks
    (the slowest replica bounds the job) and the value is the FLOPs all ranks
    processed per step divided by that time, in TFLOP/s.  With world > 1 it must
    be called by every rank of the initialised process group (any backend)."""
    step_ms = float(local_step_ms)
    if world > 1:
        import torch
        import torch.distributed as dist
        dev = device if (device is not None and dist.get_backend() == "nccl") else "cpu"
        tt = torch.tensor([step_ms], dtype=torch.float64, device=dev)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        step_ms = float(tt.item())
    return step_ms, world * flops_per_step / (step_ms * 1e-3) / 1e12


# ------------------------------------------------------------------ our arm

def upload(bits, fmt, device):
    import torch
    b = np.ascontiguousarray(bits)
    if fmt == "f32":
        return torch.from_numpy(b.view(np.int32).copy()).view(torch.float32).to(device)
    dt = torch.float16 if fmt == "f16" else torch.bfloat16
    return torch.from_numpy(b.view(np.int16).copy()).view(dt).to(device)


def make_device_problem(cfg, device):
    import torch
    w = si.workload_operands(cfg)
    a = upload(w["A"], w["in_dtype"], device)
    b = upload(w["B"], w["in_dtype"], device)
    odt = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[w["out_dtype"]]
    if w["C"] is not None:
        c0 = upload(w["C"], w["out_dtype"], device)
    else:
        c0 = None
    c = torch.empty(w["M"], w["N"], dtype=odt, device=device)
    return w, a, b, c, c0


def time_gemm(g, w, a, b, c, c0, steps, warmup, stream, flush, **epilogue):
    """Per-step CUDA-event times (ms) of the GEMM launch alone, L2 flushed before
    each step outside the event pair.  C is reset from c0 before each step when
    beta != 0 (outside the event pair) so every step computes the same result."""
    import torch
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    st = stream
    with torch.cuda.stream(st):
        for i in range(warmup + steps):
            if c0 is not None:
                c.copy_(c0)
            flush()
            if i >= warmup:
                evs[i - warmup][0].record(st)
            g.matmul(a, b, c, alpha=w["alpha"], beta=w["beta"], a_col=w["a_col"],
                     b_col=w["b_col"], stream=st.cuda_stream, **epilogue)
            if i >= warmup:
                evs[i - warmup][1].record(st)
    torch.cuda.synchronize()
    return [s.elapsed_time(e) for s, e in evs]


def time_e2e(g, w, steps, warmup, device):
    """End-to-end through gemm_host: pinned host A, B (C when beta != 0) in,
    device GEMM, host C out; CUDA events around the whole enqueued sequence."""
    import torch
    hA = torch.from_numpy(w["A"].view(np.int16).copy()).pin_memory()
    hB = torch.from_numpy(w["B"].view(np.int16).copy()).pin_memory()
    osz = 4 if w["out_dtype"] == "f32" else 2
    cnp = np.zeros((w["M"], w["N"]), dtype=np.uint32 if osz == 4 else np.uint16)
    if w["C"] is not None:
        cnp[:] = w["C"]
    hC = torch.from_numpy(cnp.view(np.int32 if osz == 4 else np.int16)).pin_memory()
    dA = torch.empty(hA.numel(), dtype=torch.int16, device=device)
    dB = torch.empty(hB.numel(), dtype=torch.int16, device=device)
    dC = torch.empty(hC.numel() * osz // 2, dtype=torch.int16, device=device)
    din = g.GEMM_F16 if w["in_dtype"] == "f16" else g.GEMM_BF16
    dout = {"f32": g.GEMM_F32, "bf16": g.GEMM_BF16, "f16": g.GEMM_F16}[w["out_dtype"]]
    layout = (g.GEMM_A_COL if w["a_col"] else 0) | (g.GEMM_B_COL if w["b_col"] else 0)
    lda = w["A"].shape[1]
    ldb = w["B"].shape[1]
    st = torch.cuda.current_stream(device)
    times = []
    for i in range(warmup + steps):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(st)
        s = g.gemm_host(w["M"], w["N"], w["K"], w["alpha"], hA.data_ptr(), lda, hB.data_ptr(),
                        ldb, w["beta"], hC.data_ptr(), w["N"], din, dout, layout,
                        dA.data_ptr(), dB.data_ptr(), dC.data_ptr(), st.cuda_stream)
        if s != g.GEMM_OK:
            raise g.GemmError(s, "gemm_host")
        e1.record(st)
        st.synchronize()
        if i >= warmup:
            times.append(e0.elapsed_time(e1))
    h2d = w["A"].nbytes + w["B"].nbytes + (cnp.nbytes if w["beta"] != 0.0 else 0)
    return times, h2d, cnp.nbytes


def cpu_baseline(w, target_s=12.0):
    """The oracle, as it stands, on the host cores over a bounded row sample."""
    import oracle
    t0 = time.perf_counter()
    rows = list(range(min(8, w["M"])))
    oracle.gemm(w["A"], w["B"], M=w["M"], N=w["N"], K=w["K"], in_dtype=w["in_dtype"],
                out_dtype=w["out_dtype"], a_col=w["a_col"], b_col=w["b_col"], alpha=w["alpha"],
                beta=w["beta"], C=w["C"], rows=rows)
    dt = max(time.perf_counter() - t0, 1e-3)
    nrows = int(min(w["M"], max(8, len(rows) * target_s / dt)))
    rows = list(range(nrows))
    t0 = time.perf_counter()
    oracle.gemm(w["A"], w["B"], M=w["M"], N=w["N"], K=w["K"], in_dtype=w["in_dtype"],
                out_dtype=w["out_dtype"], a_col=w["a_col"], b_col=w["b_col"], alpha=w["alpha"],
                beta=w["beta"], C=w["C"], rows=rows)
    dt = time.perf_counter() - t0
    flops = gemm_flops(nrows, w["N"], w["K"])
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": os.cpu_count(),
            "kind": "oracle",
            "sample": f"rows 0..{nrows - 1} of the {w['M']}x{w['N']}x{w['K']} problem "
                      f"({flops / 1e9:.1f} GFLOP, {dt:.1f} s, binary64 accumulation)"}


def run_ours(args, rank, world, device):
    import torch
    import dense_tensor_core_tcgen05_gb300 as g
    cfg = WORKLOAD_BY_NAME[args.workload]
    peaks, peak_src = load_peaks()
    torch.cuda.set_device(device)
    w, a, b, c, c0 = make_device_problem(cfg, device)
    flush = L2Flush(device)
    st = torch.cuda.current_stream(device)
    # correctness launch on a NaN-poisoned output before timing
    c.fill_(float("nan"))
    if c0 is not None:
        c.copy_(c0)
    g.matmul(a, b, c, alpha=w["alpha"], beta=w["beta"], a_col=w["a_col"], b_col=w["b_col"])
    s, site = g.gemm_sync_status(st.cuda_stream)
    if s != g.GEMM_OK or not bool(torch.isfinite(c).all()):
        raise RuntimeError(f"correctness launch failed: status {s} site {site}")

    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    if sampler:
        sampler.start()
    t_wall0 = time.perf_counter()
    times = time_gemm(g, w, a, b, c, c0, args.steps, args.warmup, st, flush)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    t_wall = time.perf_counter() - t_wall0
    clocks = sampler.stop() if sampler else None

    flops = gemm_flops(w["M"], w["N"], w["K"])
    step_ms, value = aggregate_ranks(sum(times) / len(times), flops, world, device)

    # roofline of the GEMM kernel (the only kernel of a step)
    peak_t = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    hbm = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    bound = roofline_bound(w, peak_t, hbm)
    kernel_ms = step_ms
    if bound == "tensor":
        achieved = flops / (kernel_ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak_t, "unit": "TFLOP/s",
                "frac": achieved / peak_t}
    else:
        achieved = algorithmic_bytes(w) / (kernel_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                "frac": achieved / hbm}
    roof["peak_source"] = f"{peak_src} ({'bf16_tflops burst' if bound == 'tensor' else 'hbm_gbs'})"
    roof["traffic"] = load_traffic(w["name"])
    roof["algorithmic_bytes"] = algorithmic_bytes(w)

    out = {"metric": "GEMM TFLOP/s (2MNK/s) and % of dense FP16/BF16 tensor peak on 1 GB300",
           "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": w["in_dtype"] + "->f32acc->" + w["out_dtype"],
           "data": "synthetic (seeded splitmix64, see seeded_inputs)",
           "config": {"workload": w["name"], "M": w["M"], "N": w["N"], "K": w["K"],
                      "in_dtype": w["in_dtype"], "out_dtype": w["out_dtype"],
                      "layout": ("A col" if w["a_col"] else "A row") + ", " +
                                ("B col" if w["b_col"] else "B row"),
                      "alpha": w["alpha"], "beta": w["beta"],
                      "l2": "flushed between timed steps (512 MiB write, then read back; outside the events)",
                      "parallelism": f"replicas x{world}"},
           "median_ms": statistics.median(times), "min_ms": min(times),
           "wall_s_timed_region": t_wall,
           "roofline": roof, "clocks": clocks, "gpu_launches": args.steps * world}

    if rank == 0:
        # end-to-end through the host-buffer entry point
        e2e_steps = max(3, min(args.steps, 10))
        et, h2d, d2h = time_e2e(g, w, e2e_steps, 2, device)
        e_ms = sum(et) / len(et)
        out["e2e"] = {"value": flops / (e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                      "ms_per_step": e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                      "entry_point": "gemm_host (pinned host operands)"}
        if not args.no_cpu:
            out["cpu_baseline"] = cpu_baseline(w)
        out["kernel_hash"] = kernel_source_hash()
        if not args.no_suite:
            suite = run_suite(g, args, device, peaks, cfg)
            odd = run_odd_tail(g, device, peaks)
            fp8 = run_fp8(g, device, peaks)
            if args.detail:
                out.update(suite=suite, odd_tail=odd, fp8=fp8)
            # compact summaries last: a reader that keeps only the line's tail has them
            out.update(summarise(suite, odd, fp8))
    return out


def _r(x, nd=4):
    return None if x is None else float(f"{x:.{nd}g}")


def summarise(suite, odd, fp8):
    """Short per-workload records (microseconds, fractions of the measured peaks)."""
    cols = {"suite_cols": "ours_us, frac (tensor or HBM, of measured), bound, cuBLAS_us (same "
                          "output dtype and beta), ours_hot_us, cuBLAS_hot_us, bias_relu_us, "
                          "cuBLAS_us with input-dtype output and no beta",
            "suite_summary": {}, "odd_tail_cols": "ours_us, frac_hbm, cuBLAS_us (same output dtype)",
            "odd_tail_summary": {}, "fp8_cols": "ours_us, frac (of 2x measured bf16), cuBLASLt_us",
            "fp8_summary": {}}
    for name, r in suite.items():
        cols["suite_summary"][name] = [
            _r(r["median_ms"] * 1e3), _r(r["frac"], 3), r["bound"], _r(r["cublas_ms"] * 1e3),
            _r(r.get("hot_ms", 0) * 1e3) if "hot_ms" in r else None,
            _r(r.get("cublas_hot_ms", 0) * 1e3) if "cublas_hot_ms" in r else None,
            _r(r["bias_relu_median_ms"] * 1e3), _r(r["cublas_inout_ms"] * 1e3)]
    for name, r in odd.items():
        cols["odd_tail_summary"][name] = [_r(r["median_ms"] * 1e3), _r(r["frac_hbm"], 3),
                                          _r(r["cublas_ms"] * 1e3)]
    for name, r in fp8.items():
        cols["fp8_summary"][name] = [_r(r["median_ms"] * 1e3), _r(r["frac"], 3),
                                     _r(r["cublaslt_ms"] * 1e3) if r.get("cublaslt_ms") else None]
    return cols


def cublas_call(w, a, b, matched=True):
    """A torch (cuBLAS) call for the workload's GEMM (bench only, never the
    product path).  matched: the same problem as ours, i.e. the workload's output
    dtype (fp16/bf16 inputs with fp32 output through torch's out_dtype) and its
    alpha/beta (addmm reading a copy of C); when torch cannot express that, or
    matched is False, the output is in the input dtype with no beta term.
    Returns (callable, kind)."""
    import torch
    aa = a.t() if w["a_col"] else a      # [M, K] view of A
    bb = b.t() if w["b_col"] else b      # [K, N] view of B (column-major when b_col)
    if matched:
        odt = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[w["out_dtype"]]
        out = torch.empty(w["M"], w["N"], dtype=odt, device=a.device)
        kw = {} if odt == a.dtype else {"out_dtype": odt}
        if w["beta"] != 0.0:
            c_in = torch.randn(w["M"], w["N"], device=a.device).to(odt)
            fn = lambda: torch.addmm(c_in, aa, bb, beta=w["beta"], alpha=w["alpha"], out=out, **kw)
        elif w["alpha"] != 1.0:
            fn = lambda: torch.addmm(out, aa, bb, beta=0.0, alpha=w["alpha"], out=out, **kw)
        else:
            fn = lambda: torch.mm(aa, bb, out=out, **kw)
        try:
            fn()
            torch.cuda.synchronize()
            return fn, "matched (output dtype, alpha, beta)"
        except (TypeError, RuntimeError):
            pass
    return (lambda: torch.matmul(aa, bb)), "input-dtype output, no beta"


def time_cublas(w, a, b, steps, warmup, flush, matched=True):
    """cuBLAS reference point, timed like ours (L2 flushed before each step,
    outside the events).  Returns (median ms, kind) with kind from cublas_call."""
    import torch
    fn, kind = cublas_call(w, a, b, matched)
    evs = []
    for i in range(warmup + steps):
        flush()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        if i >= warmup:
            evs.append((e0, e1))
    torch.cuda.synchronize()
    return statistics.median([x.elapsed_time(y) for x, y in evs]), kind


def time_hot(launch, reps=20, warmup=3):
    """Mean ms per launch of `reps` back-to-back launches inside one CUDA-event
    pair, with no flush between them (operands warm in L2)."""
    import torch
    for _ in range(warmup):
        launch()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        launch()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps


def run_suite(g, args, device, peaks, skip_cfg):
    """Every workload timed the same way (20 steps, 5 warm-ups), with the cuBLAS
    reference point beside ours; the headline workload is included again so its
    cuBLAS time sits next to it.  Tensor-bound workloads are also timed hot
    (back-to-back launches), ours and cuBLAS's."""
    import torch
    res = {}
    flush = L2Flush(device)
    for cfg in sorted(si.WORKLOADS):
        w, a, b, c, c0 = make_device_problem(cfg, device)
        times = time_gemm(g, w, a, b, c, c0, 20, 5, torch.cuda.current_stream(device), flush)
        ms = statistics.median(times)
        flops = gemm_flops(w["M"], w["N"], w["K"])
        peak_t = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
        hbm = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
        bound = roofline_bound(w, peak_t, hbm)
        tf = flops / (ms * 1e-3) / 1e12
        gbs = algorithmic_bytes(w) / (ms * 1e-3) / 1e9
        cub_ms, cub_kind = time_cublas(w, a, b, 20, 5, flush)
        # cuBLAS writing the input dtype with no beta term (a smaller problem
        # whenever the workload's output is fp32 or beta != 0)
        cub_inout_ms, _ = time_cublas(w, a, b, 20, 5, flush, matched=False)
        # the same GEMM with the fused epilogue (per-column fp32 bias, then ReLU)
        bias = torch.from_numpy(si.normal(4000 + cfg, w["N"], 1.0)).to(device)
        ftimes = time_gemm(g, w, a, b, c, c0, 20, 5, torch.cuda.current_stream(device), flush,
                           bias=bias, relu=True)
        res[w["name"]] = {"median_ms": ms, "tflops": tf, "gbs_algorithmic": gbs, "bound": bound,
                          "frac": tf / peak_t if bound == "tensor" else gbs / hbm,
                          "cublas_ms": cub_ms, "cublas_tflops": flops / (cub_ms * 1e-3) / 1e12,
                          "cublas_kind": cub_kind, "cublas_inout_ms": cub_inout_ms,
                          "bias_relu_median_ms": statistics.median(ftimes),
                          "bias_relu_mean_over_plain_mean": statistics.mean(ftimes) / statistics.mean(times)}
        if bound == "tensor":
            # back-to-back launches ("hot": no flush in between), ours and cuBLAS's
            try:
                st = torch.cuda.current_stream(device)
                hot = time_hot(lambda: g.matmul(a, b, c, alpha=w["alpha"], beta=w["beta"],
                                                a_col=w["a_col"], b_col=w["b_col"],
                                                stream=st.cuda_stream))
                cub_hot = time_hot(cublas_call(w, a, b)[0])
                res[w["name"]].update({"hot_ms": hot, "hot_tflops": flops / (hot * 1e-3) / 1e12,
                                       "cublas_hot_ms": cub_hot})
            except Exception as e:  # reported, never fatal to the bench line
                res[w["name"]]["hot_error"] = str(e)[:200]
        del a, b, c, c0
        torch.cuda.empty_cache()
    return res


# Second workload: odd and tail shapes ("GEMM From Naive CUDA to Tensor Cores":
# its default 257 x 263 x 251 and the index-check fixtures 73 x 61 x 67,
# 31 x 29 x 37, 17 x 65 x 19; its M = N = 64 sweep over K = 32, 256, 4096) and
# decode-like shapes with a few rows against a wide, deep B (column-major), the
# split-K shapes beyond the 128-row skinny workload.  Timed like the suite; the
# inputs are seeded normal draws made on the device (their parity is covered by
# the GPU tests on the same shapes).
ODD_TAIL = [
    # name, M, N, K, in, out, B column-major
    ("lab_257x263x251", 257, 263, 251, "f16", "f32", False),
    ("lab_73x61x67", 73, 61, 67, "f16", "f32", False),
    ("lab_31x29x37", 31, 29, 37, "f16", "f32", False),
    ("lab_17x65x19", 17, 65, 19, "f16", "f32", False),
    ("ksweep_64x64x32", 64, 64, 32, "f16", "f32", False),
    ("ksweep_64x64x256", 64, 64, 256, "f16", "f32", False),
    ("ksweep_64x64x4096", 64, 64, 4096, "f16", "f32", False),
    ("decode_1x8192x8192", 1, 8192, 8192, "bf16", "bf16", True),
    ("decode_16x4096x8192", 16, 4096, 8192, "bf16", "bf16", True),
    ("decode_32x2048x8192", 32, 2048, 8192, "bf16", "bf16", True),
    ("decode_64x8192x2048", 64, 8192, 2048, "bf16", "bf16", True),
    ("decode_8x14336x4096", 8, 14336, 4096, "bf16", "bf16", True),
]


def run_odd_tail(g, device, peaks):
    import torch
    tdt = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}
    flush = L2Flush(device)
    hbm = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    gen = torch.Generator(device=device)
    res = {}
    for i, (name, M, N, K, din, dout, b_col) in enumerate(ODD_TAIL):
        gen.manual_seed(5000 + i)
        pad = lambda n: (n + 7) // 8 * 8   # noqa: E731  (16-byte row pitches)
        a = torch.randn(M, pad(K), device=device, generator=gen).to(tdt[din])[:, :K]
        b = (torch.randn(N, pad(K), device=device, generator=gen).to(tdt[din])[:, :K] if b_col
             else torch.randn(K, pad(N), device=device, generator=gen).to(tdt[din])[:, :N])
        c = torch.empty(M, pad(N), device=device, dtype=tdt[dout])[:, :N]
        w = {"alpha": 1.0, "beta": 0.0, "a_col": False, "b_col": b_col}
        times = time_gemm(g, w, a, b, c, None, 20, 5, torch.cuda.current_stream(device), flush)
        ms = statistics.median(times)
        cub_fn, _ = cublas_call(dict(w, M=M, N=N, out_dtype=dout), a, b)
        ctimes = []
        for _ in range(25):
            flush()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            cub_fn()
            e1.record()
            torch.cuda.synchronize()
            ctimes.append(e0.elapsed_time(e1))
        cub = statistics.median(ctimes[5:])
        byts = 2 * (M * K + K * N) + (4 if dout == "f32" else 2) * M * N
        res[name] = {"M": M, "N": N, "K": K, "median_ms": ms,
                     "tflops": 2 * M * N * K / (ms * 1e-3) / 1e12,
                     "gbs_algorithmic": byts / (ms * 1e-3) / 1e9,
                     "frac_hbm": byts / (ms * 1e-3) / 1e9 / hbm,
                     "cublas_ms": cub}
    return res


# FP8 operands (tcgen05.mma kind::f8f6f4, fp32 accumulation), K-major A and B.
# The roofline peak is the measured bf16 dense rate times 2, the nominal FP8/BF16
# ratio of the part (4.5 / 2.25 PFLOP/s); cuBLASLt's FP8 GEMM (torch._scaled_mm
# with unit scales) is timed beside it.
FP8_SHAPES = [
    ("fp8_2048_e4m3_f32", 2048, 2048, 2048, "e4m3", "f32"),
    ("fp8_4096_e4m3_bf16", 4096, 4096, 4096, "e4m3", "bf16"),
    ("fp8_8192_e4m3_f32", 8192, 8192, 8192, "e4m3", "f32"),
    ("fp8_8192_e5m2_bf16", 8192, 8192, 8192, "e5m2", "bf16"),
]


def run_fp8(g, device, peaks):
    import torch
    tdt = {"e4m3": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2, "f32": torch.float32,
           "bf16": torch.bfloat16}
    flush = L2Flush(device)
    peak8 = 2.0 * peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    gen = torch.Generator(device=device)
    res = {}
    for i, (name, M, N, K, din, dout) in enumerate(FP8_SHAPES):
        gen.manual_seed(6000 + i)
        a = torch.randn(M, K, device=device, generator=gen).to(tdt[din])
        b = torch.randn(N, K, device=device, generator=gen).to(tdt[din])   # B column-major
        c = torch.empty(M, N, device=device, dtype=tdt[dout])
        w = {"alpha": 1.0, "beta": 0.0, "a_col": False, "b_col": True}
        steps = 10 if M >= 8192 else 20
        times = time_gemm(g, w, a, b, c, None, steps, 5, torch.cuda.current_stream(device), flush)
        ms = statistics.median(times)
        tf = 2 * M * N * K / (ms * 1e-3) / 1e12
        entry = {"M": M, "N": N, "K": K, "in": din, "out": dout, "median_ms": ms, "tflops": tf,
                 "peak_tflops": peak8, "frac": tf / peak8}
        try:
            one = torch.ones((), device=device)
            odt = torch.float32 if dout == "f32" else torch.bfloat16
            ctimes = []
            for _ in range(steps + 5):
                flush()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                torch._scaled_mm(a, b.t(), scale_a=one, scale_b=one, out_dtype=odt)
                e1.record()
                torch.cuda.synchronize()
                ctimes.append(e0.elapsed_time(e1))
            entry["cublaslt_ms"] = statistics.median(ctimes[5:])
        except (RuntimeError, TypeError) as e:   # an FP8 format the library rejects
            entry["cublaslt_ms"] = None
            entry["cublaslt_note"] = str(e).splitlines()[0][:120]
        res[name] = entry
        del a, b, c
        torch.cuda.empty_cache()
    return res


# ------------------------------------------------------------ reference arm

def run_reference(args):
    """The CPU oracle on the host cores: each step computes a bounded row sample
    of the same workload (FP64 accumulation)."""
    import oracle
    cfg = WORKLOAD_BY_NAME[args.workload]
    w = si.workload_operands(cfg)
    rows_per_step = 256 if w["M"] >= 256 else w["M"]
    run = lambda r0: oracle.gemm(w["A"], w["B"], M=w["M"], N=w["N"], K=w["K"],  # noqa: E731
                                 in_dtype=w["in_dtype"], out_dtype=w["out_dtype"],
                                 a_col=w["a_col"], b_col=w["b_col"], alpha=w["alpha"],
                                 beta=w["beta"], C=w["C"],
                                 rows=[(r0 + i) % w["M"] for i in range(rows_per_step)])
    for i in range(args.warmup):
        run(i * rows_per_step)
    times = []
    for i in range(args.steps):
        t0 = time.perf_counter()
        run((args.warmup + i) * rows_per_step)
        times.append(time.perf_counter() - t0)
    step_s = sum(times) / len(times)
    flops = gemm_flops(rows_per_step, w["N"], w["K"])
    value = flops / step_s / 1e12
    sample = (f"{rows_per_step} rows of the {w['M']}x{w['N']}x{w['K']} problem per step "
              f"({flops / 1e9:.2f} GFLOP), binary64 accumulation")
    return {"impl": "reference", "metric": "GEMM TFLOP/s (2MNK/s) and % of dense FP16/BF16 tensor peak on 1 GB300",
            "value": value, "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": step_s * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded splitmix64, see seeded_inputs)",
            "config": {"workload": w["name"], "M": w["M"], "N": w["N"], "K": w["K"]},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": os.cpu_count(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOAD_BY_NAME))
    ap.add_argument("--no-suite", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--detail", action="store_true",
                    help="add the full per-workload suite, odd-tail and FP8 records")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return

    import torch
    if world > 1:
        torch.cuda.set_device(local)
        torch.distributed.init_process_group("nccl")
    from dense_tensor_core_tcgen05_gb300 import build as b
    if rank == 0 or world == 1:
        b.build()
    if world > 1:
        torch.distributed.barrier()
    out = run_ours(args, rank, world, torch.device("cuda", local))
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
