"""Benchmark of the absmax-quantized low-precision hot path on GB300.

One step = the whole path over one batch of the large workload (M=16384,
N=8192, K=8192, A and B bf16 Student-t(3), seeded):
  FP8:  quantize A and B to E4M3 with the amax fused in (delayed scales), then
        the scaled FP8 GEMM C = A B^T * sa * sb (bf16 out);
  INT8: per-row quantize A and B (each launch also stages its codes for the
        GEMM), then the exact INT8 GEMM with the per-row x per-row fp32
        dequant epilogue.
Metric: quant+GEMM TFLOP/s = (2*M*N*K for each of the two GEMMs) / step time.

The same JSON line also carries the pages' four smaller workloads under
"configs" (INT8 per-row, INT8 per-head, the FP8 linear forward and the FP8
MLP backward), each timed on the GPU after an L2 flush and run by the oracle
on the host.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl sq|reference]
  python bench.py --config {int8_per_row,int8_per_head,fp8_fwd,fp8_bwd,all,
                            fp8_linear,large_next,extra}   (one line each)

Prints one JSON line (rank 0).  Under torchrun each rank runs its own replica
(the path shards into independent problems: no collective on the data path).
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics
import subprocess
import sys
import threading
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

# Nominal dense tensor rates of a GB300 (context beside the measured peaks).
# INT8 codes run on the f16 tensor path here (sm_103a has no integer MMA
# kind), so the INT8 GEMM is set against the f16 rate.
NOMINAL_TFLOPS = {"fp8": 4500.0, "f16": 2250.0}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="sq", choices=["sq", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="leave the four smaller workloads out of the default line")
    ap.add_argument("--overlap", action="store_true",
                    help="run the INT8 quantization on a second stream during the FP8 GEMM")
    ap.add_argument("--size", type=int, nargs=3, metavar=("M", "N", "K"),
                    help="override the workload sizes (small cases for profiler captures)")
    ap.add_argument("--config", default="large",
                    choices=["large", "int8_per_row", "int8_per_head", "fp8_fwd", "fp8_bwd", "all",
                             "fp8_linear", "large_next", "extra"],
                    help="the pages' other workloads, each with its own JSON line")
    args = ap.parse_args()
    if args.size:
        global M, N, K, FLOPS_PER_STEP, WORKLOAD
        M, N, K = args.size
        FLOPS_PER_STEP = 2 * (2.0 * M * N * K)
        WORKLOAD = WORKLOAD.replace("M=16384 N=8192 K=8192", f"M={M} N={N} K={K}")
    return args


def algo_bytes(kernel):
    """Algorithmic bytes of one launch of the large workload's GEMMs (codes
    read once, output written once): FP8 A8 + B8 + bf16 C; INT8 qa + qb +
    fp32 C."""
    return {"gemm_fp8_nt": M * K + N * K + 2 * M * N,
            "gemm_i8_kernel": M * K + N * K + 4 * M * N}[kernel]


# DRAM traffic per launch (ncu dram__bytes_read.sum + dram__bytes_write.sum,
# full-size workload, 1-pass capture), valid only for the kernel sources it
# was taken from: when the sha256 of those sources no longer matches, the
# bench reports traffic as null.
PROFILED_TRAFFIC = {
    "gemm_fp8_nt": {"bytes": 783018496, "sources_sha256": "93b889f8edef3ce402fface7e53a20fd42f7301691e376ee9cbf993dead2a1f8"},
    "gemm_i8_kernel": {"bytes": 2733592320, "sources_sha256": "93b889f8edef3ce402fface7e53a20fd42f7301691e376ee9cbf993dead2a1f8"},
}
TRAFFIC_SOURCES = ["absmax_quantized_precision_gb300/csrc/gemm.cu",
                   "absmax_quantized_precision_gb300/csrc/sq_device.cuh",
                   "absmax_quantized_precision_gb300/csrc/quantize.cu"]


def sources_sha256():
    import hashlib
    h = hashlib.sha256()
    for rel in TRAFFIC_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def profiled_traffic(kernel):
    rec = PROFILED_TRAFFIC.get(kernel)
    if not rec or rec.get("sources_sha256") != sources_sha256():
        return None
    return rec["bytes"]


def peaks():
    """Roofline denominators.  Every kernel here is timed by CUDA events over a
    short region, so the burst figures apply: HBM copy GB/s and the cuBLAS
    bf16 burst rate; FP8 is twice the bf16 rate (nominal dense ratio)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16": p["bf16_tflops"],
                "bf16_sustained": p["bf16_tflops_sustained"], "src": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16": 1900.0, "bf16_sustained": 1700.0, "src": "fallback"}


def tensor_peak(pk, fp8):
    return (2.0 if fp8 else 1.0) * pk["bf16"]


# ---------------------------------------------------------------- clocks
class _Nvml:
    """Read-only NVML queries through ctypes (no Python NVML package needed)."""
    CLOCK_SM = 1
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, device):
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        ok = False
        bus = self._pci_bus_id(device)
        if bus:
            ok = self.lib.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(self.h)) == 0
        if not ok:
            idx = device.index if device.index is not None else 0
            if os.environ.get("CUDA_VISIBLE_DEVICES"):
                raise RuntimeError("no PCI bus id to map the CUDA device to NVML")
            if self.lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(idx), ctypes.byref(self.h)) != 0:
                raise RuntimeError("nvmlDeviceGetHandleByIndex failed")
        self._reasons_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons

    @staticmethod
    def _pci_bus_id(device):
        import torch
        p = torch.cuda.get_device_properties(device)
        try:
            return f"{p.pci_domain_id:08x}:{p.pci_bus_id:02x}:{p.pci_device_id:02x}.0"
        except AttributeError:
            return None

    def sm_mhz(self):
        v = ctypes.c_uint()
        return v.value if self.lib.nvmlDeviceGetClockInfo(self.h, self.CLOCK_SM, ctypes.byref(v)) == 0 else None

    def sm_max_mhz(self):
        v = ctypes.c_uint()
        return v.value if self.lib.nvmlDeviceGetMaxClockInfo(self.h, self.CLOCK_SM, ctypes.byref(v)) == 0 else None

    def reasons(self):
        v = ctypes.c_ulonglong()
        if self._reasons_fn(self.h, ctypes.byref(v)) != 0:
            return None
        return [n for bit, n in self.REASONS.items() if v.value & bit]

    def power_w(self):
        v = ctypes.c_uint()
        return v.value / 1000.0 if self.lib.nvmlDeviceGetPowerUsage(self.h, ctypes.byref(v)) == 0 else None


class Clocks:
    """Samples the SM clock, power and clock-event reasons while the timed
    region runs: in process through NVML every `period_s` from a background
    thread (read-only queries), else with nvidia-smi queries."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device, period_s=0.002):
        self.device = device
        self.period = period_s
        self.samples = []        # (sm_mhz, reasons, power_w)
        self.max_mhz = None
        self.errors = []
        self.source = None
        try:
            self.nvml = _Nvml(device)
            self.max_mhz = self.nvml.sm_max_mhz()
            self.source = "nvml"
        except Exception as e:
            self.nvml = None
            self.errors.append(f"nvml: {str(e)[:120]}")
            self.source = "nvidia-smi"

    def _loop_nvml(self):
        while not self._stop.is_set():
            self.samples.append((self.nvml.sm_mhz(), self.nvml.reasons(), self.nvml.power_w()))
            time.sleep(self.period)

    def _loop_smi(self):
        idx = self.device.index if self.device.index is not None else 0
        while not self._stop.is_set():
            try:
                r = subprocess.run(["nvidia-smi", f"--id={idx}", f"--query-gpu={self.Q}",
                                    "--format=csv,noheader,nounits"],
                                   capture_output=True, text=True, timeout=10)
            except Exception as e:
                self.errors.append(str(e)[:200])
                return
            for line in r.stdout.splitlines():
                f = [x.strip() for x in line.split(",")]
                if len(f) < 9:
                    continue
                try:
                    mhz, self.max_mhz = float(f[1]), float(f[2])
                except ValueError:
                    continue
                names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
                rs = [n for n, v in zip(names, f[5:9]) if v.lower().startswith("active")]
                try:
                    pw = float(f[3])
                except ValueError:
                    pw = None
                self.samples.append((mhz, rs, pw))
            self._stop.wait(0.1)

    def __enter__(self):
        self._stop = threading.Event()
        self._thr = threading.Thread(target=self._loop_nvml if self.nvml else self._loop_smi,
                                     daemon=True)
        self._thr.start()
        return self

    def __exit__(self, *exc):
        self._stop.set()
        self._thr.join(timeout=15)

    def summary(self):
        sm = [s[0] for s in self.samples if s[0] is not None]
        reasons = sorted({r for s in self.samples if s[1] for r in s[1]})
        out = {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": reasons, "samples": len(sm),
               "source": self.source}
        if self.nvml:
            out["period_ms"] = 1e3 * self.period
        if sm:
            loaded = [x for x in sm if self.max_mhz is None or x > 0.5 * self.max_mhz] or sm
            out["sm_mhz"] = statistics.median(loaded)
            out["sm_mhz_min"] = min(loaded)
        pw = [s[2] for s in self.samples if s[2] is not None]
        if pw:
            out["power_w_max"] = max(pw)
        if self.errors:
            out["errors"] = self.errors[:3]
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


# ---------------------------------------------------------------- multi-rank helpers
def max_over_ranks(values, dist, device):
    """Element-wise max of a list of floats over all ranks (the slowest rank
    sets the time); a single process returns the values unchanged."""
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    if dist is not None:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def whole_job_tflops(world, flops_per_step_per_rank, ms_per_step):
    """Throughput of the whole job: every rank runs its own replica of the
    workload (weak scaling), so the work is world x the per-rank work."""
    return world * flops_per_step_per_rank / (ms_per_step * 1e-3) / 1e12


def check_frac(name, frac):
    """A kernel far above its measured peak is not doing the work it claims."""
    if frac > 1.5:
        raise RuntimeError(f"{name}: {frac:.2f} of its peak; the timed region does not hold the work")
    return frac


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

    launches_per_step = 6
    shape_i8 = (0, M, N, K)

    # One stream by default.  --overlap runs the INT8 quantization (memory-
    # bound) on a second stream during the FP8 GEMM (tensor-bound); the INT8
    # GEMM call then follows the FP8 GEMM, alone.  On a power-capped GB300 the
    # overlap gained ~2% (the concurrent traffic lowers the SM clock).
    s_i8 = torch.cuda.Stream(dev) if args.overlap else stream
    q_done = torch.cuda.Event()
    g_done = torch.cuda.Event()

    def step(events=None, bufs=None):
        """One step of the path; with `events`, an event after every call."""
        xa, xb, c8, ci = bufs if bufs is not None else (A, B, C8, Ci)

        def mark(i, st):
            if events is not None:
                events[i].record(st)
        mark(0, stream)
        # One launch per FP8 operand here: each saturates the GPU, and one
        # launch of both (sq_quantize_fp8_multi, which the smaller workloads
        # use) measured the same step time on this workload.
        sq.sq_quantize_fp8(xa, tsa, sq.SQ_FMT_E4M3, ws, x8=a8, amax=amax_a, stream=stream)
        mark(1, stream)
        sq.sq_quantize_fp8(xb, tsb, sq.SQ_FMT_E4M3, ws, x8=b8, amax=amax_b, stream=stream)
        mark(2, stream)
        q_done.record(stream)
        sq.sq_gemm_fp8_scaled(a8, b8, tsa, tsb, sq.SQ_FMT_E4M3, sq.SQ_NT, C=c8, stream=stream)
        mark(3, stream)
        g_done.record(stream)
        s_i8.wait_event(q_done)
        mark(7, s_i8)
        sq.sq_quantize_rowwise_i8_staged(xa, 0, shape_i8, wsi, q=qa, scales=sA, stream=s_i8)
        mark(4, s_i8)
        sq.sq_quantize_rowwise_i8_staged(xb, 1, shape_i8, wsi, q=qb, scales=sB, stream=s_i8)
        mark(5, s_i8)
        s_i8.wait_event(g_done)
        mark(8, s_i8)
        sq.sq_gemm_i8_rowscaled_staged(sA, sB, shape_i8, wsi, C=ci, stream=s_i8)
        mark(6, s_i8)
        stream.wait_stream(s_i8)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if sq.sq_get_last_device_error() != sq.SQ_OK:
        raise RuntimeError("device error during warm-up")

    # ------------------------------------------------ timed region (device-resident)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    clk = Clocks(dev)
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    # The step time: K steps back to back with nothing between the calls (an
    # event between two kernels would turn their programmatic launch overlap
    # back into plain stream order).
    with clk:
        t_start.record(stream)
        for s in range(args.steps):
            step()
        t_end.record(stream)
        torch.cuda.synchronize(dev)
    if dist:
        dist.barrier()
    elapsed_ms = t_start.elapsed_time(t_end)
    if sq.sq_get_last_device_error() != sq.SQ_OK:
        raise RuntimeError("device error in the timed region")

    # The per-call breakdown: a second pass of the same steps with events
    # around every call.
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(9)] for _ in range(args.steps)]
    for s in range(args.steps):
        step(ev[s])
    torch.cuda.synchronize(dev)
    spans = {"quant_fp8_A": (0, 1), "quant_fp8_B": (1, 2), "gemm_fp8_nt": (2, 3),
             "quant_i8_A": (7, 4), "quant_i8_B": (4, 5), "gemm_i8_kernel": (8, 6)}
    per_kernel = {n: statistics.mean(ev[s][a].elapsed_time(ev[s][b]) for s in range(args.steps))
                  for n, (a, b) in spans.items()}
    if sq.sq_get_last_device_error() != sq.SQ_OK:
        raise RuntimeError("device error in the event pass")

    # The SM clock the GEMMs actually ran at: one more pass of the K steps in
    # which every GEMM launch records its CTAs' cycles and nanoseconds (the
    # records left are those of the last step).
    rec_fp8 = torch.zeros(4 * 1024, dtype=torch.int64, device=dev)
    rec_i8 = torch.zeros(4 * 1024, dtype=torch.int64, device=dev)
    sq.sq_set_clock_probe(rec_fp8, rec_i8)
    try:
        for s in range(args.steps):
            step()
        torch.cuda.synchronize(dev)
    finally:
        sq.sq_set_clock_probe()
    kernel_mhz = {"gemm_fp8_nt": sq.clock_probe_mhz(rec_fp8),
                  "gemm_i8_kernel": sq.clock_probe_mhz(rec_i8)}

    # What each call costs inside the step (one stream): pass j runs the
    # step's first j + 1 calls, with an event at the step's start and one after
    # call j and nothing between, so the calls keep their launch overlap; call
    # j's cost is the mean prefix time through j minus the one through j - 1.
    seq = [("quant_fp8_A", lambda: sq.sq_quantize_fp8(A, tsa, sq.SQ_FMT_E4M3, ws, x8=a8,
                                                        amax=amax_a, stream=stream)),
           ("quant_fp8_B", lambda: sq.sq_quantize_fp8(B, tsb, sq.SQ_FMT_E4M3, ws, x8=b8,
                                                        amax=amax_b, stream=stream)),
           ("gemm_fp8_nt", lambda: sq.sq_gemm_fp8_scaled(a8, b8, tsa, tsb, sq.SQ_FMT_E4M3, sq.SQ_NT,
                                                         C=C8, stream=stream)),
           ("quant_i8_A", lambda: sq.sq_quantize_rowwise_i8_staged(A, 0, shape_i8, wsi, q=qa,
                                                                    scales=sA, stream=stream)),
           ("quant_i8_B", lambda: sq.sq_quantize_rowwise_i8_staged(B, 1, shape_i8, wsi, q=qb,
                                                                    scales=sB, stream=stream)),
           ("gemm_i8_kernel", lambda: sq.sq_gemm_i8_rowscaled_staged(sA, sB, shape_i8, wsi, C=Ci,
                                                                     stream=stream))]
    in_step_ms = {}
    if not args.overlap:
        # every round runs each prefix once, so that all prefixes see the same
        # mix of clocks (the GPU may reach its power cap as the passes go on)
        nseq = len(seq)
        pe = [[[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(nseq)]
              for _ in range(args.steps)]
        for s in range(args.steps):
            for j in range(nseq):
                pe[s][j][0].record(stream)
                for _, fn in seq[:j + 1]:
                    fn()
                pe[s][j][1].record(stream)
        torch.cuda.synchronize(dev)
        pt = [[pe[s][j][0].elapsed_time(pe[s][j][1]) for j in range(nseq)] for s in range(args.steps)]
        for j, (name, _) in enumerate(seq):
            # median over rounds of the paired difference of the two prefixes
            in_step_ms[name] = statistics.median(pt[s][j] - (pt[s][j - 1] if j > 0 else 0.0)
                                                 for s in range(args.steps))
        if sq.sq_get_last_device_error() != sq.SQ_OK:
            raise RuntimeError("device error in the prefix passes")

    # Steady-state rate of each quantize call: 10 launches back to back (each
    # overlapping the tail of the one before), events only around the batch.
    # B's launches alternate between B and the first rows of A, so that no
    # launch finds its input in L2 from the one before (A alone exceeds L2).
    def steady(fn, reps=10, batches=3):
        t = []
        for _ in range(batches):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for r in range(reps):
                fn(r)
            e1.record(stream)
            torch.cuda.synchronize(dev)
            t.append(e0.elapsed_time(e1) / reps)
        return statistics.median(t)

    b_alt = A[:N] if M >= N else None
    steady_ms = {
        "quant_fp8_A": steady(lambda r: sq.sq_quantize_fp8(A, tsa, sq.SQ_FMT_E4M3, ws, x8=a8,
                                                           amax=amax_a, stream=stream)),
        "quant_fp8_B": steady(lambda r: sq.sq_quantize_fp8(B if (r % 2 == 0 or b_alt is None) else b_alt,
                                                           tsb, sq.SQ_FMT_E4M3, ws, x8=b8,
                                                           amax=amax_b, stream=stream)),
        "quant_i8_A": steady(lambda r: sq.sq_quantize_rowwise_i8_staged(A, 0, shape_i8, wsi, q=qa,
                                                                        scales=sA, stream=stream)),
        "quant_i8_B": steady(lambda r: sq.sq_quantize_rowwise_i8_staged(
            B if (r % 2 == 0 or b_alt is None) else b_alt, 1, shape_i8, wsi, q=qb, scales=sB,
            stream=stream)),
    }
    if sq.sq_get_last_device_error() != sq.SQ_OK:
        raise RuntimeError("device error in the steady-state pass")

    # ------------------------------------------------ e2e: host buffers, copies inside
    # Every step copies its own inputs in from pinned host memory and its two
    # results out to pinned host memory inside the timed region.  The copies
    # are pipelined the way a serving loop runs them: step s+1's upload and
    # step s-1's download run on their own streams (the copy engines) while
    # step s computes, with double-buffered device inputs and outputs; events
    # keep a buffer from being overwritten before its consumer is done.
    e2e = None
    if not args.no_e2e:
        c8_host = [torch.empty((M, N), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
        ci_host = [torch.empty((M, N), dtype=torch.float32).pin_memory() for _ in range(2)]
        bufs = [(A, B, C8, Ci),
                (torch.empty_like(A), torch.empty_like(B), torch.empty_like(C8), torch.empty_like(Ci))]
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        in_ready = [torch.cuda.Event() for _ in range(2)]
        in_free = [torch.cuda.Event() for _ in range(2)]
        out_ready = [torch.cuda.Event() for _ in range(2)]
        out_free = [torch.cuda.Event() for _ in range(2)]
        e_steps = max(2, min(args.steps, 20))

        def e2e_run(n):
            s_in.wait_stream(stream)
            s_out.wait_stream(stream)
            for s in range(n):
                k = s % 2
                xa, xb, c8, ci = bufs[k]
                if s >= 2:
                    s_in.wait_event(in_free[k])      # step s-2 has finished reading xa, xb
                with torch.cuda.stream(s_in):
                    xa.copy_(a_host, non_blocking=True)
                    xb.copy_(b_host, non_blocking=True)
                in_ready[k].record(s_in)
                stream.wait_event(in_ready[k])
                if s >= 2:
                    stream.wait_event(out_free[k])   # step s-2's results have been read out
                step(bufs=bufs[k])
                in_free[k].record(stream)
                out_ready[k].record(stream)
                s_out.wait_event(out_ready[k])
                with torch.cuda.stream(s_out):
                    c8_host[k].copy_(c8, non_blocking=True)
                    ci_host[k].copy_(ci, non_blocking=True)
                out_free[k].record(s_out)
            stream.wait_stream(s_in)
            stream.wait_stream(s_out)

        e2e_run(2)
        torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        if dist:
            dist.barrier()
        e0.record(stream)
        e2e_run(e_steps)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        e_ms = e0.elapsed_time(e1) / e_steps
        h2d = (a_host.numel() + b_host.numel()) * 2
        d2h = C8.numel() * 2 + Ci.numel() * 4
        e2e = {"ms_per_step": e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "unit": UNIT, "value": FLOPS_PER_STEP / (e_ms * 1e-3) / 1e12, "steps": e_steps,
               "schedule": "uploads of step s+1 and downloads of step s-1 overlap step s on two "
                           "copy streams (double-buffered device tensors, pinned host buffers)"}
        if sq.sq_get_last_device_error() != sq.SQ_OK:
            raise RuntimeError("device error in the e2e region")
        # every step has the same inputs: what reached the host must equal the
        # device-resident results of the timed region (spot rows)
        for k in range(2):
            for rows in (slice(0, 64), slice(M - 64, M)):
                if not (torch.equal(c8_host[k][rows], C8[rows].cpu()) and
                        torch.equal(ci_host[k][rows], Ci[rows].cpu())):
                    raise RuntimeError("e2e results differ from the device-resident ones")
        del c8_host, ci_host, bufs

    # ------------------------------------------------ max over ranks
    elapsed_ms, e2e_ms = max_over_ranks([elapsed_ms, e2e["ms_per_step"] if e2e else 0.0], dist, dev)
    ms_per_step = elapsed_ms / args.steps
    value = whole_job_tflops(world, FLOPS_PER_STEP, ms_per_step)
    if e2e:
        e2e["value"] = whole_job_tflops(world, FLOPS_PER_STEP, e2e_ms)

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return

    pk = peaks()
    clocks = clk.summary()
    # INT8 quantize: bf16 in, int8 codes and their exact fp16 copy out, scales
    quant_bytes = {"quant_fp8_A": M * K * 3 + 4, "quant_fp8_B": N * K * 3 + 4,
                   "quant_i8_A": M * K * 5 + M * 4, "quant_i8_B": N * K * 5 + N * 4}
    gemm_flops = {"gemm_fp8_nt": 2.0 * M * N * K, "gemm_i8_kernel": 2.0 * M * N * K}

    def rate(n, ms):
        d = {"ms": ms}
        if ms <= 0.0:
            # a difference of two replays at the timer's resolution (one
            # round of a short run): no rate
            return d
        if n in quant_bytes:
            d["GB/s"] = quant_bytes[n] / (ms * 1e-3) / 1e9
            d["frac_hbm"] = d["GB/s"] / pk["hbm_gbs"]
        elif n in gemm_flops:
            d["TFLOP/s"] = gemm_flops[n] / (ms * 1e-3) / 1e12
            d["frac_peak"] = d["TFLOP/s"] / tensor_peak(pk, n == "gemm_fp8_nt")
        return d

    kernels = {n: rate(n, ms) for n, ms in per_kernel.items()}
    kernels_in_step = {n: rate(n, ms) for n, ms in in_step_ms.items()}
    kernels_steady = {n: rate(n, ms) for n, ms in steady_ms.items()}

    # Fraction of the tensor pipe's peak at the clock the kernel ran at: dense
    # MMA rates per SM per clock of 8192 FP8 and 4096 f16 multiply-adds.
    sms = torch.cuda.get_device_properties(dev).multi_processor_count

    def at_kernel_clock(name, tflops):
        rec = kernel_mhz.get(name, {})
        mhz = rec.get("median")
        if not mhz:
            return None
        per_clk = 16384 if name == "gemm_fp8_nt" else 8192
        return {"sm_mhz": mhz, "flops_per_sm_per_clk": per_clk, "sms": sms,
                "peak_tflops": per_clk * sms * mhz * 1e6 / 1e12,
                "frac": tflops / (per_clk * sms * mhz * 1e6 / 1e12),
                # the same launches' own cycles: the flops over what the SMs could
                # have done in the cycles the CTAs lived (independent of the clock)
                "frac_of_cycles": (2.0 * M * N * K) / (per_clk * sms * rec["cycles_median"])}

    # Roofline: the dominant kernel of the step (the longest single launch).
    dom = max(("gemm_fp8_nt", "gemm_i8_kernel"), key=lambda n: per_kernel[n])
    fp8 = dom == "gemm_fp8_nt"
    dom_peak = tensor_peak(pk, fp8)
    achieved = kernels[dom]["TFLOP/s"]
    traffic = profiled_traffic(dom)
    nominal = NOMINAL_TFLOPS["fp8" if fp8 else "f16"]
    roofline = {
        "kernel": dom, "bound": "tensor", "achieved": achieved, "peak": dom_peak,
        "unit": "TFLOP/s", "frac": check_frac(dom, achieved / dom_peak), "traffic": traffic,
        "peak_src": (f"{pk['src']} bf16 burst (cuBLAS bf16 GEMM, best of 10)"
                     + (" x2, the nominal fp8:bf16 dense ratio" if fp8 else
                        "; the INT8 codes run on the f16 tensor path (sm_103a has no integer "
                        "MMA kind), whose dense rate equals bf16's")
                     + "; the kernel is timed by CUDA events over a short region, so the burst "
                       "figure applies"),
        "algorithmic": "2*M*N*K flops per launch",
        "algorithmic_bytes": algo_bytes(dom),
        "traffic_vs_algorithmic": (traffic / algo_bytes(dom)) if traffic else None,
        "timed": ("one sq_gemm_i8_rowscaled_staged launch (its operands were staged by the "
                  "quantize launches)" if not fp8 else "one sq_gemm_fp8_scaled launch"),
        "vs_nominal": {"nominal_dense_tflops": nominal, "frac": achieved / nominal,
                       "note": "nominal dense FP8 4.5 / f16 2.25 PFLOP/s"},
        "at_kernel_clock": at_kernel_clock(dom, achieved),
    }
    other = "gemm_i8_kernel" if fp8 else "gemm_fp8_nt"
    other_rec = {"kernel": other, "achieved": kernels[other]["TFLOP/s"],
                 "peak": tensor_peak(pk, other == "gemm_fp8_nt"),
                 "frac": check_frac(other, kernels[other]["frac_peak"]),
                 "traffic": profiled_traffic(other), "algorithmic_bytes": algo_bytes(other),
                 "at_kernel_clock": at_kernel_clock(other, kernels[other]["TFLOP/s"])}
    if other_rec["traffic"]:
        other_rec["traffic_vs_algorithmic"] = other_rec["traffic"] / algo_bytes(other)
    roofline["other_gemm"] = other_rec
    if clocks.get("sm_mhz"):
        clocks["step_kcycles"] = ms_per_step * clocks["sm_mhz"]

    cpu = None
    if not args.no_cpu:
        rows = np.sort(np.random.default_rng(0).choice(M, min(CPU_ROWS_A, M), replace=False))
        dt, fl, thr = cpu_oracle_sample(a_np, b_np, sa_np, sb_np, rows, 0, N)
        cpu = {"value": fl / dt / 1e12, "unit": UNIT, "cores": thr, "kind": "oracle",
               "sample": f"{len(rows)} seeded rows of A x all of B, full K: FP8 and INT8 quantize "
                         "of those rows and of B, then those rows of both GEMMs",
               "seconds": dt}

    configs = None
    if not args.no_configs and not args.size and world == 1:
        configs = {}
        for name in SMALL_CONFIGS:
            configs[name] = measure_config(name, args, with_cpu=not args.no_cpu, compact=True)

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3/int8",
        "data": "synthetic (seeded Student-t(3) bf16)",
        "config": {"workload": WORKLOAD, "M": M, "N": N, "K": K,
                   "l2": "inputs larger than L2 (no flush)", "parallelism": f"replicas x{world}",
                   "schedule": ("one stream" if not args.overlap else
                                "two streams: INT8 quantize of A and B during the FP8 GEMM; "
                                "INT8 GEMM call after it")},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
        "kernel_clocks": kernel_mhz,
        "kernel_clocks_note": ("mean SM clock of each GEMM launch's CTAs (their cycle counter over "
                               "the global timer, recorded by the kernels), median over CTAs, last "
                               "step of an extra pass; the NVML samples above miss the fast clock "
                               "reductions under the tensor cores"),
        "roofline": roofline,
        "kernels": kernels,
        "kernels_note": ("mean CUDA-event span of each call on the stream it ran on, from a second "
                         "pass of the same steps with events around every call (each call then "
                         "waits for the one before and pays its own launch); the INT8 quantize "
                         "calls (sq_quantize_rowwise_i8_staged) also stage their codes for "
                         "sq_gemm_i8_rowscaled_staged"
                         + ("; with two streams the INT8 quantize spans overlap the FP8 GEMM and "
                            "share the GPU with it" if args.overlap else "")),
        "kernels_in_step": kernels_in_step,
        "kernels_in_step_note": ("what each call costs inside the step: the median over K "
                                 "rounds of the time of the step's first j + 1 calls minus that of "
                                 "its first j calls in the same round, each prefix timed with "
                                 "events only at its two ends (the calls keep their launch "
                                 "overlap); the first call's figure includes its launch"),
        "kernels_steady": kernels_steady,
        "kernels_steady_note": ("each quantize call launched 10 times back to back with events only "
                                "around the batch; B alternates with a same-size block of A so "
                                "no launch reads its input from L2"),
        "peaks": {"hbm_gbs": pk["hbm_gbs"], "bf16_burst_tflops": pk["bf16"],
                  "fp8_tflops": 2.0 * pk["bf16"], "src": pk["src"]},
        "configs": configs,
        "e2e": e2e,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


# ---------------------------------------------------------------- the other workloads
SMALL_CONFIGS = ["int8_per_row", "int8_per_head", "fp8_fwd", "fp8_bwd"]
EXTRA_CONFIGS = ["fp8_linear", "large_next"]


def config_ops(name, dev, sq, synth, oracle, bf16_dev, prev_scale):
    """(description, [(label, kind, amount, fn)], GEMM flops per step, the
    oracle's work on the host or None) for one of the pages' workloads."""
    import numpy as np
    import torch

    if name in ("int8_per_row", "int8_per_head"):
        if name == "int8_per_row":
            a = synth.normal(11, (128, 1024))
            b = synth.normal(12, (512, 1024))
            desc = "INT8 per-row: A f32 128x1024, B f32 512x1024 ~N(0,1); C = A B^T, fp32 out"
        else:
            a = synth.normal(21, (16, 196, 64))
            b = synth.normal(22, (16, 196, 64))
            desc = "INT8 per-head: Q, K f32 (16,196,64) ~N(0,1); C[h] = Q[h] K[h]^T, fp32 out"
        A, B = torch.from_numpy(a).to(dev), torch.from_numpy(b).to(dev)
        qa = torch.empty(A.shape, dtype=torch.int8, device=dev)
        qb = torch.empty(B.shape, dtype=torch.int8, device=dev)
        sa = torch.empty(A.shape[:-1], device=dev)
        sb = torch.empty(B.shape[:-1], device=dev)
        nb = A.shape[0] if A.dim() == 3 else 1
        Mi, Kk = A.shape[-2], A.shape[-1]
        Ni = B.shape[-2]
        ws = torch.empty(sq.gemm_i8_workspace_bytes(nb, Mi, Ni, Kk), dtype=torch.uint8, device=dev)
        C = torch.empty((nb, Mi, Ni) if nb > 1 else (Mi, Ni), device=dev)
        flops = 2.0 * nb * Mi * Ni * Kk
        shape = (nb if A.dim() == 3 else 0, Mi, Ni, Kk)
        # f32 in; int8 codes, their exact fp16 copy and the scales out; both
        # operands in one call (one launch: their rows fit in registers)
        ops = [("quant_i8_AB", "bytes", (A.numel() + B.numel()) * 7 + (sa.numel() + sb.numel()) * 4,
                lambda: sq.sq_quantize_rowwise_i8_staged_pair(A, B, shape, ws, qa=qa, sa=sa, qb=qb,
                                                              sb=sb)),
               ("gemm_i8_kernel", "flops", flops,
                lambda: sq.sq_gemm_i8_rowscaled_staged(sa.reshape(-1), sb.reshape(-1), shape, ws,
                                                       C=C))]
        # the one-call form on the same codes (its own staging + the GEMM), for comparison
        call = ("gemm_i8", "flops", flops,
                lambda: sq.sq_gemm_i8_rowscaled(qa, sa.reshape(-1), qb, sb.reshape(-1), ws, C=C))

        def oracle_work():
            oqa, osa = oracle.quantize_rowwise_i8(a)
            oqb, osb = oracle.quantize_rowwise_i8(b)
            oracle.gemm_i8(oqa, oqb, osa, osb)
        return desc, ops, [call], flops, oracle_work

    if name in EXTRA_CONFIGS:
        desc, ops, flops = extra_config_ops(name, dev, bf16_dev, prev_scale)
        return desc, ops, [], flops, None

    fmt = sq.SQ_FMT_E4M3
    wsq = sq.new_workspace(dev)
    if name == "fp8_fwd":
        x = synth.normal(31, (2048, 1024), std=1.0, dtype=synth.BF16)
        w = synth.normal(32, (1024, 1024), std=0.02, dtype=synth.BF16)
        sx, sw = prev_scale(33, x.shape, 1.0), prev_scale(34, w.shape, 0.02)
        X, W = bf16_dev(x), bf16_dev(w)
        tsx, tsw = torch.tensor([sx], device=dev), torch.tensor([sw], device=dev)
        x8 = torch.empty(X.shape, dtype=torch.uint8, device=dev)
        w8 = torch.empty(W.shape, dtype=torch.uint8, device=dev)
        ax, aw = torch.empty(1, device=dev), torch.empty(1, device=dev)
        Y = torch.empty((2048, 1024), dtype=torch.bfloat16, device=dev)
        flops = 2.0 * 2048 * 1024 * 1024
        desc = ("FP8 E4M3 linear forward: X bf16 2048x1024 ~N(0,1), W bf16 1024x1024 "
                "~N(0,0.02), delayed scales; Y = X W^T (NT), bf16 out")
        # X and W in one launch, each with its own step and amax
        ops = [("quant_fp8_XW", "bytes", (X.numel() + W.numel()) * 3,
                lambda: sq.sq_quantize_fp8_multi([X, W], [tsx, tsw], fmt, wsq, x8s=[x8, w8],
                                                 amaxs=[ax, aw])),
               ("gemm_fp8_nt", "flops", flops,
                lambda: sq.sq_gemm_fp8_scaled(x8, w8, tsx, tsw, fmt, sq.SQ_NT, C=Y))]

        def oracle_work():
            ox8, _ = oracle.quantize_fp8(x, sx, 0)
            ow8, _ = oracle.quantize_fp8(w, sw, 0)
            oracle.gemm_fp8(ox8, ow8, 0, oracle.NT, sx, sw)
        return desc, ops, [], flops, oracle_work

    T, H, D = 2048, 4096, 1024
    g = synth.normal(41, (T, H), std=1e-3, dtype=synth.BF16)
    w = synth.normal(42, (H, D), std=0.02, dtype=synth.BF16)
    x = synth.normal(43, (T, D), std=1.0, dtype=synth.BF16)
    sg, sw, sx = prev_scale(44, g.shape, 1e-3), prev_scale(45, w.shape, 0.02), \
        prev_scale(46, x.shape, 1.0)
    G, W, X = bf16_dev(g), bf16_dev(w), bf16_dev(x)
    tsg, tsw, tsx = (torch.tensor([v], device=dev) for v in (sg, sw, sx))
    g8 = torch.empty(G.shape, dtype=torch.uint8, device=dev)
    w8 = torch.empty(W.shape, dtype=torch.uint8, device=dev)
    x8 = torch.empty(X.shape, dtype=torch.uint8, device=dev)
    am = [torch.empty(1, device=dev) for _ in range(3)]
    dX = torch.empty((T, D), dtype=torch.bfloat16, device=dev)
    dW = torch.empty((H, D), dtype=torch.bfloat16, device=dev)
    flops = 2 * (2.0 * T * H * D)
    desc = ("FP8 E4M3 MLP backward (dim 1024, hidden 4096, 2048 tokens): G bf16 2048x4096 "
            "~N(0,1e-3), W bf16 4096x1024 ~N(0,0.02), X bf16 2048x1024 ~N(0,1); "
            "dX = G W (NN), dW = G^T X (TN), bf16 out")
    # G, W and X in one launch, each with its own step and amax; then dX and
    # dW in one call (one launch deals both products' tiles to every SM)
    ops = [("quant_fp8_GWX", "bytes", (G.numel() + W.numel() + X.numel()) * 3,
            lambda: sq.sq_quantize_fp8_multi([G, W, X], [tsg, tsw, tsx], fmt, wsq,
                                             x8s=[g8, w8, x8], amaxs=am)),
           ("gemm_fp8_dX_nn_dW_tn", "flops", 2 * (2.0 * T * H * D),
            lambda: sq.sq_gemm_fp8_scaled_pair([g8, g8], [w8, x8], [tsg, tsg], [tsw, tsx], fmt,
                                               [sq.SQ_NN, sq.SQ_TN], Cs=[dX, dW]))]
    # each product as its own call, for comparison
    alt = [("gemm_fp8_dX_nn", "flops", 2.0 * T * H * D,
            lambda: sq.sq_gemm_fp8_scaled(g8, w8, tsg, tsw, fmt, sq.SQ_NN, C=dX)),
           ("gemm_fp8_dW_tn", "flops", 2.0 * T * H * D,
            lambda: sq.sq_gemm_fp8_scaled(g8, x8, tsg, tsx, fmt, sq.SQ_TN, C=dW))]

    def oracle_work():
        og8, _ = oracle.quantize_fp8(g, sg, 0)
        ow8, _ = oracle.quantize_fp8(w, sw, 0)
        ox8, _ = oracle.quantize_fp8(x, sx, 0)
        oracle.gemm_fp8(og8, ow8, 0, oracle.NN, sg, sw, want_bf16=False)
        oracle.gemm_fp8(og8, ox8, 0, oracle.TN, sg, sx, want_bf16=False)
    return desc, ops, alt, flops, oracle_work


def measure_config(name, args, with_cpu=True, compact=False):
    """Times one of the pages' smaller workloads on cuda:0.  Every timed pass
    runs after a 256 MiB write that evicts the inputs from L2:
      step   the whole step (its calls in order) captured as one CUDA graph;
      calls  each call alone, captured as its own graph (its device time plus
             one launch);
      in_step  what each call adds to the step: the median over rounds of the
             replay time of the step's first j + 1 calls minus that of its
             first j calls in the same round (the first call's figure
             includes the replay's own start);
    plus the oracle's time for the whole workload on the host (all cores and
    one core).  Returns a dict; compact leaves out the eager timings."""
    import numpy as np
    import torch

    import __graft_entry__
    import absmax_quantized_precision_gb300 as sq
    import oracle
    import synth

    __graft_entry__.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def bf16_dev(u16):
        return torch.from_numpy(u16.view(np.int16)).to(dev).view(torch.bfloat16)

    def prev_scale(seed, shape, std, fmax=448.0):
        p = synth.bf16_bits_to_f32(synth.normal(seed, shape, std=std, dtype=synth.BF16))
        return np.float32(np.abs(p).max()) / np.float32(fmax)

    desc, ops, alt_calls, gemm_flops, oracle_work = config_ops(name, dev, sq, synth, oracle,
                                                               bf16_dev, prev_scale)

    cpu = None
    if with_cpu and oracle_work is not None:
        cores = oracle.num_threads()
        t0 = time.perf_counter()
        oracle_work()
        cpu = {"seconds": time.perf_counter() - t0, "cores": cores}
        oracle.set_num_threads(1)
        t0 = time.perf_counter()
        oracle_work()
        cpu["seconds_1core"] = time.perf_counter() - t0
        oracle.set_num_threads(cores)
        cpu["sample"] = "the whole workload"

    iters = 200
    for _ in range(max(args.warmup, 3)):
        for _, _, _, fn in ops + alt_calls:
            fn()
    torch.cuda.synchronize(dev)

    def capture(fns):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for fn in fns:
                fn()
        g.replay()
        torch.cuda.synchronize(dev)
        return g

    def time_graphs(graphs):
        """Replay times [round][graph]: every round replays each graph once,
        after an L2-evicting write, so that all see the same drift."""
        ev = [[[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in graphs]
              for _ in range(iters)]
        for it in range(iters):
            for j, g in enumerate(graphs):
                flush.fill_((it + j) & 0xFF)   # evict the inputs from L2 before each pass
                ev[it][j][0].record(stream)
                g.replay()
                ev[it][j][1].record(stream)
        torch.cuda.synchronize(dev)
        return [[ev[i][j][0].elapsed_time(ev[i][j][1]) for j in range(len(graphs))]
                for i in range(iters)]

    with Clocks(dev) as clk:
        # the graphs of the step's first j + 1 calls, then of each call alone
        graphs = [capture([fn for _, _, _, fn in ops[:j + 1]]) for j in range(len(ops))]
        graphs += [capture([fn]) for _, _, _, fn in ops + alt_calls]
        t = time_graphs(graphs)
        med = [statistics.median(t[i][j] for i in range(iters)) for j in range(len(graphs))]
        step_ms = med[len(ops) - 1]
        call_ms = med[len(ops):]
        # a call's cost in the step: the median over rounds of the paired
        # difference between the prefixes through it and through the call before
        inc_ms = [statistics.median(t[i][j] - (t[i][j - 1] if j > 0 else 0.0) for i in range(iters))
                  for j in range(len(ops))]
    if sq.sq_get_last_device_error() != sq.SQ_OK:
        raise RuntimeError("device error in the graph passes")

    eager = None
    if not compact:
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(ops) + 1)]
               for _ in range(iters)]
        for it in range(iters):
            flush.fill_(it & 0xFF)
            evs[it][0].record(stream)
            for i, (_, _, _, fn) in enumerate(ops):
                fn()
                evs[it][i + 1].record(stream)
        torch.cuda.synchronize(dev)
        eager = statistics.median(evs[i][0].elapsed_time(evs[i][-1]) for i in range(iters))
        if sq.sq_get_last_device_error() != sq.SQ_OK:
            raise RuntimeError("device error in the eager pass")

    pk = peaks()

    def rates(label, kind, amount, ms):
        d = {"us": 1e3 * ms}
        if ms <= 0.0:
            return d
        if kind == "bytes":
            d["GB/s"] = amount / (ms * 1e-3) / 1e9
            d["frac_hbm"] = d["GB/s"] / pk["hbm_gbs"]
        else:
            tf = amount / (ms * 1e-3) / 1e12
            d["TFLOP/s"] = tf
            is_fp8 = "fp8" in label or label.startswith("linear_")
            d["frac_peak"] = tf / tensor_peak(pk, is_fp8)
        return d

    calls = {}
    for j, (label, kind, amount, _) in enumerate(ops + alt_calls):
        calls[label] = rates(label, kind, amount, call_ms[j])
    in_step = {}
    for j, (label, kind, amount, _) in enumerate(ops):
        inc = inc_ms[j]
        in_step[label] = ({"us": 1e3 * inc} if inc <= 0 else rates(label, kind, amount, inc))
    out = {"desc": desc, "value": gemm_flops / (step_ms * 1e-3) / 1e12, "unit": UNIT,
           "us_per_step": 1e3 * step_ms, "calls": calls, "in_step": in_step,
           "l2": "256 MiB write before every timed pass", "iters": iters,
           "clocks": clk.summary(), "cpu_oracle": cpu}
    if eager is not None:
        out["us_per_step_eager"] = 1e3 * eager
    return out


def run_config(name, args):
    rec = measure_config(name, args, with_cpu=not args.no_cpu)
    line = {"metric": METRIC, "config": {"workload": name, "desc": rec.pop("desc"),
                                         "l2": rec.pop("l2")}}
    line.update(rec)
    print(json.dumps(line), flush=True)


def extra_config_ops(name, dev, bf16_dev, prev_scale):
    """Workloads of the widened path: the fused FP8 linear layer, and the
    large-size ring / E4M3-output / per-tensor INT8 variants."""
    import numpy as np
    import torch

    import absmax_quantized_precision_gb300 as sq
    import synth

    if name == "fp8_linear":
        M, K, N = 2048, 1024, 1024            # forward: X W^T + b
        T, Hd, D = 2048, 4096, 1024           # backward of the MLP up-projection
        x = bf16_dev(synth.normal(301, (M, K), dtype=synth.BF16))
        w = bf16_dev(synth.normal(302, (N, K), std=0.02, dtype=synth.BF16))
        b = bf16_dev(synth.normal(303, (N,), std=0.5, dtype=synth.BF16))
        g = bf16_dev(synth.normal(304, (T, Hd), std=1e-3, dtype=synth.BF16))
        wb = bf16_dev(synth.normal(305, (Hd, D), std=0.02, dtype=synth.BF16))
        xb = bf16_dev(synth.normal(306, (T, D), dtype=synth.BF16))
        xr = sq.new_ring(16, float(prev_scale(307, (M, K), 1.0)), dev)
        wr = sq.new_ring(16, float(prev_scale(308, (N, K), 0.02)), dev)
        gr = sq.new_ring(16, float(prev_scale(309, (T, Hd), 1e-3, 57344.0)), dev)
        sw_b = torch.tensor([prev_scale(310, (Hd, D), 0.02, 57344.0)], device=dev)
        sx_b = torch.tensor([prev_scale(311, (T, D), 1.0, 57344.0)], device=dev)
        wsf = sq.linear_workspace(M, N, K, dev)
        wsb = sq.linear_workspace(T, Hd, D, dev)
        fwd_flops = 2.0 * M * N * K
        bwd_flops = 2 * (2.0 * T * Hd * D)
        ops = [("linear_forward_e4m3_rings_bias", "flops", fwd_flops,
                lambda: sq.sq_linear_forward_fp8(x, w, b, None, None, sq.SQ_FMT_E4M3, wsf,
                                                 x_ring=xr, w_ring=wr)),
               ("linear_backward_e5m2_ring", "flops", bwd_flops,
                lambda: sq.sq_linear_backward_fp8(g, xb, wb, (True, True, True), None, sw_b, sx_b,
                                                  sq.SQ_FMT_E5M2, wsb, g_ring=gr))]
        desc = ("fused FP8 linear: forward X bf16 2048x1024, W 1024x1024, bf16 bias, E4M3 with "
                "delayed-scaling rings; backward of the 1024->4096 projection over 2048 tokens, "
                "E5M2 gradient with a ring, dX + dW + bias gradient")
        return desc, ops, fwd_flops + bwd_flops

    # large_next
    M, N, K = 16384, 8192, 8192
    a = synth.student_t(SEED_A, (M, K), df=3, dtype=synth.BF16)
    b = synth.student_t(SEED_B, (N, K), df=3, dtype=synth.BF16)
    A, B = bf16_dev(a), bf16_dev(b)
    sa_v = float(np.float32(np.abs(synth.bf16_bits_to_f32(a)).max()) / np.float32(448.0))
    ring = sq.new_ring(16, sa_v, dev)
    ws = sq.new_workspace(dev)
    a8 = torch.empty((M, K), dtype=torch.uint8, device=dev)
    b8 = torch.empty((N, K), dtype=torch.uint8, device=dev)
    amax = torch.empty(1, device=dev)
    tsb = torch.tensor([sa_v], device=dev)
    out_scale = torch.tensor([2.0], device=dev)
    C8 = torch.empty((M, N), dtype=torch.uint8, device=dev)
    qa = torch.empty((M, K), dtype=torch.int8, device=dev)
    qb = torch.empty((N, K), dtype=torch.int8, device=dev)
    sqa, sqb = torch.empty(1, device=dev), torch.empty(1, device=dev)
    wga = torch.empty(sq.load_library().sq_quantize_grouped_i8_workspace_bytes(M, M),
                      dtype=torch.uint8, device=dev)
    wgb = torch.empty(sq.load_library().sq_quantize_grouped_i8_workspace_bytes(N, N),
                      dtype=torch.uint8, device=dev)
    wsi = torch.empty(sq.gemm_i8_workspace_bytes(1, M, N, K), dtype=torch.uint8, device=dev)
    Ci = torch.empty((M, N), device=dev)
    ops = [("quant_fp8_ring_A", "bytes", M * K * 3,
            lambda: sq.sq_quantize_fp8_ring(A, sq.SQ_FMT_E4M3, ring, 0, 0, ws, x8=a8, amax=amax)),
           ("quant_fp8_B", "bytes", N * K * 3,
            lambda: sq.sq_quantize_fp8(B, tsb, sq.SQ_FMT_E4M3, ws, x8=b8, amax=amax)),
           ("gemm_fp8_nt_e4m3_out", "flops", 2.0 * M * N * K,
            lambda: sq.sq_gemm_fp8_scaled_e4m3(a8, b8, tsb, tsb, sq.SQ_FMT_E4M3, sq.SQ_NT,
                                               out_scale, C=C8)),
           ("quant_i8_per_tensor_A", "bytes", M * K * 3,
            lambda: sq.sq_quantize_grouped_i8(A, M, q=qa, scales=sqa, workspace=wga)),
           ("quant_i8_per_tensor_B", "bytes", N * K * 3,
            lambda: sq.sq_quantize_grouped_i8(B, N, q=qb, scales=sqb, workspace=wgb)),
           ("gemm_i8_per_tensor", "flops", 2.0 * M * N * K,
            lambda: sq.sq_gemm_i8_grouped(qa, sqa, M, qb, sqb, N, wsi, C=Ci))]
    desc = ("large M=16384 N=8192 K=8192 bf16 Student-t(3): FP8 quantize with a ring, FP8 GEMM "
            "with E4M3 output; per-tensor INT8 quantize (two passes) and GEMM")
    return desc, ops, 2 * (2.0 * M * N * K)


def main():
    args = parse()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.config != "large" and args.impl == "sq":
        names = {"all": SMALL_CONFIGS, "extra": EXTRA_CONFIGS}.get(args.config, [args.config])
        for name in names:
            run_config(name, args)
        return
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_sq(args, rank, world, local_rank)


if __name__ == "__main__":
    main()
