"""Benchmark of the absmax-quantized low-precision hot path on GB300.

One step = the whole path over one batch of the large workload (M=16384,
N=8192, K=8192, A and B bf16 Student-t(3), seeded):
  FP8:  quantize A and B to E4M3 with the amax fused in (delayed scales), then
        the scaled FP8 GEMM C = A B^T * sa * sb (bf16 out);
  INT8: per-row quantize A and B, then the exact INT8 GEMM with the per-row x
        per-row fp32 dequant epilogue.
Metric: quant+GEMM TFLOP/s = (2*M*N*K for each of the two GEMMs) / step time.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl sq|reference]

Prints one JSON line (rank 0).  Under torchrun each rank runs its own replica
(the path shards into independent problems: no collective on the data path).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

M, N, K = 16384, 8192, 8192
SEED_A, SEED_B, SEED_PA, SEED_PB = 501, 502, 601, 602
METRIC = "quant+GEMM TFLOPS & % of GB300 INT8/FP8 tensor peak; quantize GB/s vs HBM"
UNIT = "TFLOP/s"
WORKLOAD = ("large: M=16384 N=8192 K=8192, A/B bf16 Student-t(3) seeded; FP8 E4M3 per-tensor "
            "delayed-scale quantize+NT GEMM (bf16 out) and INT8 per-row quantize+GEMM "
            "(exact int32 acc, fp32 out)")
FLOPS_PER_STEP = 2 * (2.0 * M * N * K)


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="sq", choices=["sq", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--size", type=int, nargs=3, metavar=("M", "N", "K"),
                    help="override the workload sizes (small cases for profiler captures)")
    args = ap.parse_args()
    if args.size:
        global M, N, K, FLOPS_PER_STEP, WORKLOAD
        M, N, K = args.size
        FLOPS_PER_STEP = 2 * (2.0 * M * N * K)
        WORKLOAD = WORKLOAD.replace("M=16384 N=8192 K=8192", f"M={M} N={N} K={K}")
    return args


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16": p["bf16_tflops"],
                "bf16_sustained": p["bf16_tflops_sustained"], "src": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16": 1900.0, "bf16_sustained": 1700.0, "src": "fallback"}


class Clocks:
    """Samples SM clocks and throttle reasons with single-shot nvidia-smi queries
    from a background thread while the timed region runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index, period_s=0.1):
        self.index = index
        self.period = period_s
        self.lines = []
        self.errors = []

    def _loop(self):
        while not self._stop.is_set():
            try:
                r = subprocess.run(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                    "--format=csv,noheader,nounits"],
                                   capture_output=True, text=True, timeout=10)
                if r.returncode == 0:
                    self.lines += [l for l in r.stdout.splitlines() if l.strip()]
                elif len(self.errors) < 3:
                    self.errors.append(r.stderr.strip()[:200])
            except Exception as e:   # no nvidia-smi: no samples
                if len(self.errors) < 3:
                    self.errors.append(str(e)[:200])
                return
            self._stop.wait(self.period)

    def __enter__(self):
        import threading
        self._stop = threading.Event()
        self._thr = threading.Thread(target=self._loop, daemon=True)
        self._thr.start()
        return self

    def __exit__(self, *exc):
        self._stop.set()
        self._thr.join(timeout=15)

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        out = {"sm_mhz": None, "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}
        if sm:
            loaded = [x for x in sm if mx is None or x > 0.5 * mx] or sm
            out["sm_mhz"] = statistics.median(loaded)
        if self.errors:
            out["errors"] = self.errors
        return out


def make_inputs():
    import numpy as np

    import synth
    a = synth.student_t(SEED_A, (M, K), df=3, dtype=synth.BF16)
    b = synth.student_t(SEED_B, (N, K), df=3, dtype=synth.BF16)
    pa = synth.bf16_bits_to_f32(synth.student_t(SEED_PA, (M, K), df=3, dtype=synth.BF16))
    sa = np.float32(np.abs(pa).max()) / np.float32(448.0)
    del pa
    pb = synth.bf16_bits_to_f32(synth.student_t(SEED_PB, (N, K), df=3, dtype=synth.BF16))
    sb = np.float32(np.abs(pb).max()) / np.float32(448.0)
    del pb
    return a, b, sa, sb


# ---------------------------------------------------------------- CPU oracle leg
def cpu_oracle_sample(a, b, sa, sb, rows_a, b0, b1):
    """The oracle on a bounded sample of one step: FP8 and INT8 quantization of
    the sampled rows of A and of rows b0..b1 of B, then the sampled block of
    both GEMMs (full K).  Returns (seconds, GEMM flops of the block, threads)."""
    import numpy as np

    import oracle
    r = np.asarray(rows_a)
    t0 = time.perf_counter()
    a_rows = np.ascontiguousarray(a[r])
    b_rows = np.ascontiguousarray(b[b0:b1])
    a8, _ = oracle.quantize_fp8(a_rows, sa, oracle.E4M3)
    b8, _ = oracle.quantize_fp8(b_rows, sb, oracle.E4M3)
    oracle.gemm_fp8(a8, b8, oracle.E4M3, oracle.NT, sa, sb)
    qa, ssa = oracle.quantize_rowwise_i8(a_rows, oracle.BF16)
    qb, ssb = oracle.quantize_rowwise_i8(b_rows, oracle.BF16)
    oracle.gemm_i8(qa, qb, ssa, ssb)
    dt = time.perf_counter() - t0
    return dt, 2 * (2.0 * len(r) * (b1 - b0) * K), oracle.num_threads()


REF_ROWS_A, REF_ROWS_B = 2, 512          # per step of the reference arm
CPU_ROWS_A = 4096                        # the one-off CPU baseline: 4096 rows x all of B


def run_reference(args, rank, world):
    if rank != 0:
        return
    import numpy as np

    import oracle
    oracle.build()
    a, b, sa, sb = make_inputs()
    rng = np.random.default_rng(0)
    times, flops, thr = [], 0.0, 1
    for i in range(args.warmup + args.steps):
        rows = np.sort(rng.choice(M, REF_ROWS_A, replace=False))
        b0 = int(rng.integers(0, N - REF_ROWS_B + 1))
        dt, fl, thr = cpu_oracle_sample(a, b, sa, sb, rows, b0, b0 + REF_ROWS_B)
        if i >= args.warmup:
            times.append(dt)
            flops += fl
    tot = sum(times)
    value = flops / tot / 1e12
    sample = (f"per step: {REF_ROWS_A} seeded rows of A x a {REF_ROWS_B}-row block of B, full K: "
              "FP8 and INT8 quantize of those rows, then that block of both GEMMs")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "e4m3/int8",
        "data": "synthetic (seeded Student-t(3) bf16)",
        "config": {"workload": WORKLOAD, "M": M, "N": N, "K": K,
                   "l2": "inputs larger than L2 (no flush)"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": thr, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- GPU leg
def run_sq(args, rank, world, local_rank):
    import numpy as np
    import torch

    import __graft_entry__
    import absmax_quantized_precision_gb300 as sq

    __graft_entry__.build()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    dist = None
    if world > 1:
        import torch.distributed as dist_
        dist = dist_
        dist.init_process_group("nccl", device_id=dev)

    a_np, b_np, sa_np, sb_np = make_inputs()
    a_host = torch.from_numpy(a_np.view(np.int16)).view(torch.bfloat16).pin_memory()
    b_host = torch.from_numpy(b_np.view(np.int16)).view(torch.bfloat16).pin_memory()
    A = a_host.to(dev)
    B = b_host.to(dev)
    tsa = torch.tensor([sa_np], device=dev)
    tsb = torch.tensor([sb_np], device=dev)
    ws = sq.new_workspace(dev)
    a8 = torch.empty((M, K), dtype=torch.uint8, device=dev)
    b8 = torch.empty((N, K), dtype=torch.uint8, device=dev)
    amax_a = torch.empty(1, device=dev)
    amax_b = torch.empty(1, device=dev)
    C8 = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    qa = torch.empty((M, K), dtype=torch.int8, device=dev)
    qb = torch.empty((N, K), dtype=torch.int8, device=dev)
    sA = torch.empty(M, device=dev)
    sB = torch.empty(N, device=dev)
    Ci = torch.empty((M, N), dtype=torch.float32, device=dev)
    wsi = torch.empty(sq.gemm_i8_workspace_bytes(1, M, N, K), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    names = ["quant_fp8_A", "quant_fp8_B", "gemm_fp8_nt", "quant_i8_A", "quant_i8_B", "gemm_i8"]
    launches_per_step = 8   # the INT8 GEMM call stages A and B (2 launches) before its GEMM

    def step(events=None):
        def mark(i):
            if events is not None:
                events[i].record(stream)
        mark(0)
        sq.sq_quantize_fp8(A, tsa, sq.SQ_FMT_E4M3, ws, x8=a8, amax=amax_a)
        mark(1)
        sq.sq_quantize_fp8(B, tsb, sq.SQ_FMT_E4M3, ws, x8=b8, amax=amax_b)
        mark(2)
        sq.sq_gemm_fp8_scaled(a8, b8, tsa, tsb, sq.SQ_FMT_E4M3, sq.SQ_NT, C=C8)
        mark(3)
        sq.sq_quantize_rowwise_i8(A, q=qa, scales=sA)
        mark(4)
        sq.sq_quantize_rowwise_i8(B, q=qb, scales=sB)
        mark(5)
        sq.sq_gemm_i8_rowscaled(qa, sA, qb, sB, wsi, C=Ci)
        mark(6)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if sq.sq_get_last_device_error() != sq.SQ_OK:
        raise RuntimeError("device error during warm-up")

    # ------------------------------------------------ timed region (device-resident)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(7)] for _ in range(args.steps)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    with Clocks(local_rank) as clk:
        t_start.record(stream)
        for s in range(args.steps):
            step(ev[s])
        t_end.record(stream)
        torch.cuda.synchronize(dev)
    if dist:
        dist.barrier()
    elapsed_ms = t_start.elapsed_time(t_end)
    per_kernel = {n: statistics.mean(ev[s][i].elapsed_time(ev[s][i + 1]) for s in range(args.steps))
                  for i, n in enumerate(names)}
    if sq.sq_get_last_device_error() != sq.SQ_OK:
        raise RuntimeError("device error in the timed region")

    # ------------------------------------------------ e2e: host buffers, copies inside
    e2e = None
    if not args.no_e2e:
        c8_host = torch.empty((M, N), dtype=torch.bfloat16).pin_memory()
        ci_host = torch.empty((M, N), dtype=torch.float32).pin_memory()
        e_steps = max(2, min(args.steps, 5))

        def e2e_step():
            A.copy_(a_host, non_blocking=True)
            B.copy_(b_host, non_blocking=True)
            step()
            c8_host.copy_(C8, non_blocking=True)
            ci_host.copy_(Ci, non_blocking=True)

        e2e_step()
        torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        if dist:
            dist.barrier()
        e0.record(stream)
        for _ in range(e_steps):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        e_ms = e0.elapsed_time(e1) / e_steps
        h2d = (a_host.numel() + b_host.numel()) * 2
        d2h = C8.numel() * 2 + Ci.numel() * 4
        e2e = {"ms_per_step": e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "unit": UNIT, "value": FLOPS_PER_STEP / (e_ms * 1e-3) / 1e12}

    # ------------------------------------------------ max over ranks
    t = torch.tensor([elapsed_ms, e2e["ms_per_step"] if e2e else 0.0], device=dev)
    if dist:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    elapsed_ms = float(t[0])
    ms_per_step = elapsed_ms / args.steps
    value = world * FLOPS_PER_STEP / (ms_per_step * 1e-3) / 1e12
    if e2e:
        e2e["value"] = world * FLOPS_PER_STEP / (float(t[1]) * 1e-3) / 1e12

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return

    pk = peaks()
    fp8_peak = 2.0 * pk["bf16_sustained"]          # nominal fp8:bf16 dense ratio 2
    bf16_peak = pk["bf16_sustained"]
    quant_fp8_bytes = {"quant_fp8_A": M * K * 3 + 4, "quant_fp8_B": N * K * 3 + 4}
    quant_i8_bytes = {"quant_i8_A": M * K * 3 + M * 4, "quant_i8_B": N * K * 3 + N * 4}
    kernels = {}
    for n, ms in per_kernel.items():
        d = {"ms": ms}
        if n in quant_fp8_bytes or n in quant_i8_bytes:
            by = quant_fp8_bytes.get(n) or quant_i8_bytes.get(n)
            d["GB/s"] = by / (ms * 1e-3) / 1e9
            d["frac_hbm"] = d["GB/s"] / pk["hbm_gbs"]
        else:
            tf = 2.0 * M * N * K / (ms * 1e-3) / 1e12
            d["TFLOP/s"] = tf
            d["frac_peak"] = tf / (fp8_peak if n == "gemm_fp8_nt" else bf16_peak)
        kernels[n] = d
    dom = max(("gemm_fp8_nt", "gemm_i8"), key=lambda n: per_kernel[n])
    dom_peak = fp8_peak if dom == "gemm_fp8_nt" else bf16_peak
    achieved = kernels[dom]["TFLOP/s"]
    roofline = {"kernel": dom, "bound": "tensor", "achieved": achieved, "peak": dom_peak,
                "unit": "TFLOP/s", "frac": achieved / dom_peak, "traffic": None,
                "peak_src": f"{pk['src']} bf16 sustained"
                            + (" x2 (nominal fp8:bf16)" if dom == "gemm_fp8_nt" else
                               " (INT8 runs on the f16 tensor path)"),
                "algorithmic": "2*M*N*K flops per launch"}

    cpu = None
    if not args.no_cpu:
        import numpy as np
        rows = np.sort(np.random.default_rng(0).choice(M, min(CPU_ROWS_A, M), replace=False))
        dt, fl, thr = cpu_oracle_sample(a_np, b_np, sa_np, sb_np, rows, 0, N)
        cpu = {"value": fl / dt / 1e12, "unit": UNIT, "cores": thr, "kind": "oracle",
               "sample": f"{len(rows)} seeded rows of A x all of B, full K: FP8 and INT8 quantize "
                         "of those rows and of B, then those rows of both GEMMs",
               "seconds": dt}

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3/int8",
        "data": "synthetic (seeded Student-t(3) bf16)",
        "config": {"workload": WORKLOAD, "M": M, "N": N, "K": K,
                   "l2": "inputs larger than L2 (no flush)", "parallelism": f"replicas x{world}"},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk.summary(),
        "roofline": roofline,
        "kernels": kernels,
        "e2e": e2e,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def main():
    args = parse()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_sq(args, rank, world, local_rank)


if __name__ == "__main__":
    main()
