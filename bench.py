"""Benchmark of relu(A·B) on GB300: GEMM+ReLU TFLOP/s (2MNK / device time) and the fraction of
the GB300 roofline, for one named workload (default: the 8192^3 compute-bound case).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step = one call of the C ABI (tg_gemm_relu_f16) on inputs already resident in HBM.
Prints ONE JSON line on rank 0.  Under torchrun each rank runs an independent replica on its
own GPU (the path needs no exchange between GPUs); ``value`` is the work of all ranks over the
slowest rank's time.  ``--impl reference`` times the CPU oracle instead (host cores only).
"""

from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from fp16_gemm_relu_gb300 import workloads  # noqa: E402

METRIC = "GEMM+ReLU TFLOP/s (2MNK/t) and % of GB300 fp16 tensor/HBM roofline, 1 GPU"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# the int4 / NF4 GEMM's default: decode the weights first from this M
DECODE_FIRST_MIN_M = {"w4": 512, "nf4": 384}
FP16_OVER_BF16 = 1.0  # dense fp16 and bf16 tensor rates are equal (nominal 2.25 PF each)


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="square8192", choices=workloads.ORDER)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--pass", dest="pass_", default="forward", choices=["forward", "backward"],
                    help="backward: one step = dZ = relu'(C) * dC, dA = dZ B^T, dB = A^T dZ "
                         "(4MNK flops), all in the library's kernels")
    ap.add_argument("--dequant", default="none", choices=["none", "w4", "nf4"],
                    help="w4 / nf4: B is int4 / NF4 weights (group 128 scales), decoded inside "
                         "the GEMM (or, for M >= 512 (int4) / 384 (NF4), once into fp16 before "
                         "the fp16 GEMM)")
    ap.add_argument("--epilogue", default="relu", choices=["relu", "bias_gelu", "bias_relu_residual"],
                    help="relu: the metric's path; the others time the fused bias/GELU/residual "
                         "epilogue on the same GEMM")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip timing the other named workloads and the backward, epilogue and "
                         "int4/NF4 variants (the 'workloads' and 'variants' blocks)")
    ap.add_argument("--workload-seconds", type=float, default=0.5,
                    help="minimum wall time of each other workload's timed region")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target seconds of oracle work for the cpu_baseline sample")
    return ap.parse_args()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# Sources of the kernels a bench line times: the fp16 GEMMs (and the host code that plans and
# launches them), plus the dequantising kernels for the int4 / NF4 lines.
DENSE_SOURCES = ["tg_api.cu", "tg_gemm_kernel.cuh", "tg_gemm_pair.cu", "tg_gemm_bn128.cu",
                 "tg_gemm_bn192.cu", "tg_gemm_bn256.cu", "tg_internal.h"]
DEQUANT_SOURCES = DENSE_SOURCES + ["tg_gemm_w4.cuh", "tg_gemm_w4.cu"]


def kernel_source_hash(dequant: bool = False) -> str:
    """Hash of the sources behind a measured kernel (the dense set, or with the dequantising
    kernels); a committed ncu summary applies while its hash matches."""
    csrc = os.path.join(ROOT, "fp16_gemm_relu_gb300", "csrc")
    h = hashlib.sha256()
    for name in sorted(DEQUANT_SOURCES if dequant else DENSE_SOURCES):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def traffic_key(workload: str, pass_: str, epilogue: str, dequant: str) -> str:
    """Row name in profiles/traffic.txt: the workload alone for the forward relu GEMM, else
    the workload with the variant (e.g. 'square8192/w4')."""
    if (pass_, epilogue, dequant) == ("forward", "relu", "none"):
        return workload
    parts = [workload] + [v for v, d in ((pass_, "forward"), (epilogue, "relu"),
                                         (dequant, "none")) if v != d]
    return "/".join(parts)


def traffic_from_profiles(workload: str):
    """DRAM bytes per launch of the GEMM kernel from the committed ncu summary, if it was
    taken on the current kernel source (its 'source_hash' line must match).  `workload` is a
    traffic_key."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    cur = kernel_source_hash(dequant=any(t in workload.split("/") for t in ("w4", "nf4")))
    for line in open(path):
        parts = line.split()
        if len(parts) >= 3 and parts[0] == workload and parts[1] == cur:
            return float(parts[2])
    return None


# ----------------------------------- clocks -----------------------------------

class ClockSampler:
    """Samples SM clock and throttle reasons of one GPU while running, through NVML
    (read-only queries), falling back to nvidia-smi."""

    REASONS = {0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x4: "sw_power_cap", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, pci_bus_id: str, period_s: float = 0.002):
        self.period = period_s
        self.samples = []  # (sm_mhz, reasons_mask)
        self.max_mhz = None
        self._stop = threading.Event()
        self._thread = None
        self._nvml = None
        self._handle = None
        self._smi = None
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                raise OSError("nvmlInit failed")
            h = ctypes.c_void_p()
            if nv.nvmlDeviceGetHandleByPciBusId_v2(pci_bus_id.encode(), ctypes.byref(h)) != 0:
                raise OSError("no NVML handle for " + pci_bus_id)
            self._nvml, self._handle = nv, h
            v = ctypes.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(v)) == 0:  # NVML_CLOCK_SM
                self.max_mhz = float(v.value)
        except OSError:
            self._nvml = None
        self.pci = pci_bus_id

    def _poll_nvml(self):
        nv, h = self._nvml, self._handle
        clk = ctypes.c_uint()
        reasons = ctypes.c_ulonglong()
        while not self._stop.is_set():
            if nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0:
                r = 0
                if nv.nvmlDeviceGetCurrentClocksEventReasons(h, ctypes.byref(reasons)) == 0:
                    r = reasons.value
                self.samples.append((float(clk.value), int(r)))
            time.sleep(self.period)

    def start(self):
        if self._nvml is not None:
            self._thread = threading.Thread(target=self._poll_nvml, daemon=True)
            self._thread.start()
        else:
            q = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
                 "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
                 "clocks_event_reasons.sw_power_cap")
            try:
                self._smi = subprocess.Popen(
                    ["nvidia-smi", f"--id={self.pci}", f"--query-gpu={q}",
                     "--format=csv,noheader,nounits", "-lms", "100"],
                    stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            except OSError:
                self._smi = None

    def stop(self):
        self._stop.set()
        if self._thread is not None:
            self._thread.join()
        if self._smi is not None:
            self._smi.terminate()
            out, _ = self._smi.communicate(timeout=10)
            names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            for line in out.splitlines():
                f = [x.strip() for x in line.split(",")]
                if len(f) < 6:
                    continue
                try:
                    sm, mx = float(f[0]), float(f[1])
                except ValueError:
                    continue
                self.max_mhz = mx
                mask = 0
                for i, n in enumerate(names):
                    if f[2 + i].lower().startswith("active"):
                        mask |= {v: k for k, v in self.REASONS.items()}[n]
                self.samples.append((sm, mask))

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": 0}
        mask = 0
        for _, r in self.samples:
            mask |= r
        reasons = sorted(n for bit, n in self.REASONS.items() if mask & bit)
        return {"sm_mhz": statistics.median(s for s, _ in self.samples),
                "sm_max_mhz": self.max_mhz, "reasons": reasons, "samples": len(self.samples)}


# ----------------------------------- helpers -----------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def slowest_rank_ms(total_ms: float, device=None) -> float:
    """The timed region's length on the slowest rank (all-reduce MAX; the identity without a
    process group)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return total_ms
    t = torch.tensor([total_ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(world: int, steps: int, flops_per_step: float, total_ms: float) -> float:
    """Work of all replicas (each rank runs the full workload) over the slowest rank's time."""
    return world * steps * flops_per_step / (total_ms * 1e-3) / 1e12


def sample_rows(wl, a, b, target_s: float, relu=True) -> int:
    """Rows of C that one oracle call computes in about target_s seconds: each call has a
    fixed cost (decoding B) plus a cost per row of C, calibrated on two small calls."""
    import oracle

    t1, _, _ = oracle.timed_rows(a, b, 8, relu=relu)
    t2, _, _ = oracle.timed_rows(a, b, 40, relu=relu)
    per_row = max((t2 - t1) / 32, 1e-6)
    fixed = max(t1 - 8 * per_row, 0.0)
    return int(max(1, min(wl.M, 0.9 * (target_s - fixed) / per_row)))


def cpu_baseline(wl, a, b, target_s: float, relu=True):
    """The oracle as it stands, on a bounded sample: the first R rows of C."""
    import oracle

    rows = sample_rows(wl, a, b, target_s, relu)
    dt, flops, threads = oracle.timed_rows(a, b, rows, relu=relu)
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"first {rows} of {wl.M} rows of C ({rows}x{wl.N}x{wl.K}), float32 "
                      f"accumulation, {dt:.1f} s"}


def run_reference(args, wl):
    """The oracle on the host cores: each step computes a bounded sample of C's rows."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle

    a, b = wl.make_a(), wl.make_b()
    steps, warm = max(args.steps, 1), max(args.warmup, 0)
    budget = 150.0 / steps  # the timed steps within a few minutes
    rows = sample_rows(wl, a, b, budget)
    for _ in range(warm):  # warm caches and threads on a shorter sample
        oracle.timed_rows(a, b, min(rows, 64))
    times = []
    flops = 0.0
    threads = oracle.max_threads()
    for _ in range(steps):
        t, f, threads = oracle.timed_rows(a, b, rows)
        times.append(t)
        flops += f
    total = sum(times)
    value = flops / total / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": 1,
        "steps": steps, "warmup": warm, "ms_per_step": 1e3 * total / steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded SplitMix64 inputs of the workload's distribution)",
        "config": {"workload": wl.name, "M": wl.M, "N": wl.N, "K": wl.K,
                   "sample_rows_per_step": rows},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": f"first {rows} rows of C per step"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def timed_steps(torch, step, stream, steps, scrub=None, sampler=None):
    """Runs `steps` calls of step() on `stream`, each bracketed by CUDA events; with `scrub`
    (a buffer larger than L2) it is rewritten between steps, outside the step's events.
    Returns (per-step ms, ms of the whole region)."""
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    if sampler is not None:
        sampler.start()
    t0.record(stream)
    for i in range(steps):
        if scrub is not None:
            scrub.fill_(1.0)  # L2 flush between timed steps, outside the step's events
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    t1.record(stream)
    stream.synchronize()
    if sampler is not None:
        sampler.stop()
    return [s.elapsed_time(e) for s, e in zip(starts, ends)], t0.elapsed_time(t1)


def clock_soak(torch, step, stream, scrub, bus, seconds):
    """Clock record of the step run back to back for about `seconds` (outside any timed
    region): what the sampler sees of the GPU under this load."""
    _, probe_ms = timed_steps(torch, step, stream, 3, scrub)
    n = int(min(max(3, seconds * 1e3 / max(probe_ms / 3, 1e-3)), 100000))
    sampler = ClockSampler(bus)
    _, region_ms = timed_steps(torch, step, stream, n, scrub, sampler)
    out = sampler.summary()
    out.update(steps=n, region_ms=region_ms)
    return out


def roofline(flops, alg_bytes, flops_per_step, kernel_ms, peaks, peak_src):
    """Bound (the slower of dense fp16 tensor time and algorithmic bytes over HBM), achieved
    rate per step and its fraction of the measured peak."""
    t_tensor = flops / (peaks["bf16_tflops"] * FP16_OVER_BF16 * 1e12)
    t_hbm = alg_bytes / (peaks["hbm_gbs"] * 1e9)
    if t_tensor >= t_hbm:
        achieved = flops_per_step / (kernel_ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved,
                "peak": peaks["bf16_tflops"] * FP16_OVER_BF16, "unit": "TFLOP/s"}
    else:
        achieved = alg_bytes / (kernel_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["peak_source"] = (f"{peak_src} (MEASURED_PEAKS.json bf16 burst x {FP16_OVER_BF16} "
                           "fp16/bf16 nominal ratio)" if roof["bound"] == "tensor"
                           else f"{peak_src} (MEASURED_PEAKS.json copy bandwidth)")
    roof["kernel_ms"] = kernel_ms
    roof["t_roof_ms"] = 1e3 * max(t_tensor, t_hbm)
    return roof


def other_workloads(args, headline, lib, binding, dev, stream, bus, peaks, peak_src):
    """The other named workloads, each timed like the headline (W warm-up steps, CUDA events
    per step on the launching stream, L2 flushed between steps when the operands fit in it)
    for at least `args.workload_seconds` of wall time, with its own clock record."""
    import torch

    import fp16_gemm_relu_gb300 as tg

    props = torch.cuda.get_device_properties(dev)
    out = {}
    for name in workloads.ORDER:
        if name == headline:
            continue
        wl = workloads.get(name)
        A = torch.from_numpy(wl.make_a()).to(dev)
        B = torch.from_numpy(wl.make_b()).to(dev)
        C = torch.empty((wl.M, wl.N), dtype=torch.float16, device=dev)
        plan = tg.plan(wl.M, wl.N, wl.K, num_sms=props.multi_processor_count,
                       a_ptr=A.data_ptr(), b_ptr=B.data_ptr(), c_ptr=C.data_ptr())
        in_bytes = wl.algorithmic_bytes - 2 * wl.M * wl.N
        scrub = (torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
                 if in_bytes <= L2_BYTES else None)

        def step():
            st = lib.tg_gemm_relu_f16(A.data_ptr(), B.data_ptr(), C.data_ptr(), wl.M, wl.N, wl.K,
                                      wl.K, wl.N, wl.N, binding.TG_EPILOGUE_RELU, stream.cuda_stream)
            if st != 0:
                raise binding.TgError(st, "tg_gemm_relu_f16")

        with torch.cuda.stream(stream):
            for _ in range(max(args.warmup, 3)):
                if scrub is not None:
                    scrub.fill_(1.0)
                step()
            _, probe_ms = timed_steps(torch, step, stream, 3, scrub)
            steps = int(min(max(args.steps, args.workload_seconds * 1e3 / max(probe_ms / 3, 1e-3)),
                            100000))
            sampler = ClockSampler(bus)
            step_ms, region_ms = timed_steps(torch, step, stream, steps, scrub, sampler)
        st, word = binding.tg_device_error_check(clear=True)
        if st != 0:
            raise RuntimeError(f"device error word {word:#x} after workload {name}")
        ms = statistics.mean(step_ms)
        roof = roofline(wl.flops, wl.algorithmic_bytes, wl.flops, ms, peaks, peak_src)
        clocks = sampler.summary()
        entry = {
            "M": wl.M, "N": wl.N, "K": wl.K, "steps": steps, "ms_per_step": ms,
            "value": wl.flops / (ms * 1e-3) / 1e12, "unit": "TFLOP/s",
            "roofline": {k: roof[k] for k in ("bound", "achieved", "unit", "peak", "frac",
                                               "t_roof_ms")},
            "kernel_ms": ms if plan["kernels"] == 1 else None,
            "step_kernels": plan["kernels"],
            "plan": {k: plan[k] for k in ("block_m", "block_n", "split_k", "tail_tiles",
                                          "repack_a", "repack_b", "workspace_epilogue", "grid",
                                          "cta_pair") if k in plan},
            "l2": "flushed between steps" if scrub is not None else "operands larger than L2",
            "clocks": clocks, "region_ms": region_ms,
        }
        if clocks.get("sm_mhz"):
            entry["sm_cycles_per_step"] = ms * 1e-3 * clocks["sm_mhz"] * 1e6
        if roof["bound"] == "tensor" and "bf16_tflops_sustained" in peaks:
            # each workload is timed for about half a second of back-to-back steps, the regime
            # of the seconds-long cuBLAS loop behind the sustained peak: reported beside frac
            sus = peaks["bf16_tflops_sustained"] * FP16_OVER_BF16
            entry["roofline"]["peak_sustained"] = sus
            entry["roofline"]["frac_of_sustained"] = roof["achieved"] / sus
        if plan["kernels"] > 1:
            entry["note"] = ("frac is the whole step (operand repack, GEMM and split-K "
                             "reduction) against the GEMM's roofline")
        out[name] = entry
        del A, B, C, scrub
        torch.cuda.empty_cache()
    return out


def other_variants(args, lib, binding, dev, stream, bus, peaks, peak_src, A, B):
    """The scope table's further rows, each timed like the workloads block (W warm-up steps,
    CUDA events per step, L2 flushed between steps when the operands fit in it, at least
    `args.workload_seconds` of steps): the backward step and the two fused epilogues on
    8192^3 (A and B are the headline's operands), and the int4 / NF4 weight GEMMs on 8192^3
    and on 64 x 28672 x 8192.  A variant that fails records its error instead of a time."""
    import torch

    from fp16_gemm_relu_gb300 import inputs as _inputs

    handle = stream.cuda_stream
    sq = workloads.get("square8192")
    sk = workloads.get("skinny64x28672x8192")

    def check(st, what):
        if st != 0:
            raise binding.TgError(st, what)

    def backward():
        C = torch.empty((sq.M, sq.N), dtype=torch.float16, device=dev)
        check(lib.tg_gemm_relu_f16(A.data_ptr(), B.data_ptr(), C.data_ptr(), sq.M, sq.N, sq.K,
                                   sq.K, sq.N, sq.N, binding.TG_EPILOGUE_RELU, handle), "forward")
        dC = torch.from_numpy(_inputs.tensor(sq.M, sq.N, sq.seed + 102, 1)).to(dev)
        dZ, dA, dB = torch.empty_like(dC), torch.empty_like(A), torch.empty_like(B)

        def step():
            st = lib.tg_relu_backward_f16(dC.data_ptr(), C.data_ptr(), dZ.data_ptr(), sq.M, sq.N,
                                          sq.N, sq.N, sq.N, handle)
            if st == 0:
                st = lib.tg_gemm_f16_t(0, 1, dZ.data_ptr(), B.data_ptr(), dA.data_ptr(), sq.M,
                                       sq.K, sq.N, sq.N, sq.N, sq.K, None, None, handle)
            if st == 0:
                st = lib.tg_gemm_f16_t(1, 0, A.data_ptr(), dZ.data_ptr(), dB.data_ptr(), sq.K,
                                       sq.N, sq.M, sq.K, sq.N, sq.N, None, None, handle)
            check(st, "backward step")
        return step, sq, 2 * sq.flops, sq.algorithmic_bytes, 3, (C, dC, dZ, dA, dB)

    def epilogue(kind):
        def make():
            C = torch.empty((sq.M, sq.N), dtype=torch.float16, device=dev)
            bias = torch.from_numpy(_inputs.tensor(1, sq.N, sq.seed + 100, 0).ravel()).to(dev)
            resid = None
            act = binding.TG_ACT_GELU
            if kind == "bias_relu_residual":
                resid = torch.from_numpy(_inputs.tensor(sq.M, sq.N, sq.seed + 101, 1)).to(dev)
                act = binding.TG_ACT_RELU
            epi = binding.tg_epilogue(act, bias.data_ptr(),
                                      resid.data_ptr() if resid is not None else None,
                                      sq.N if resid is not None else 0)

            def step():
                check(lib.tg_gemm_f16_epilogue(A.data_ptr(), B.data_ptr(), C.data_ptr(), sq.M,
                                               sq.N, sq.K, sq.K, sq.N, sq.N, ctypes.byref(epi),
                                               None, handle), "tg_gemm_f16_epilogue")
            return step, sq, sq.flops, sq.algorithmic_bytes, 1, (C, bias, resid, epi)
        return make

    def weights(w, fmt):
        def make():
            G = 128
            Aw = A if w is sq else torch.from_numpy(w.make_a()).to(dev)
            ldq = -(-(-(-w.N // 8)) // 4) * 4
            Wq = torch.from_numpy(_inputs.int4_weights(w.K, w.N, w.seed, ldq=ldq)
                                  .view(np.int32)).to(dev)
            Sc = torch.from_numpy(_inputs.int4_scales(-(-w.K // G), w.N, w.seed,
                                                      1.0 / np.sqrt(w.K))).to(dev)
            C = torch.empty((w.M, w.N), dtype=torch.float16, device=dev)
            fn = lib.tg_gemm_w4a16_f16 if fmt == "w4" else lib.tg_gemm_nf4a16_f16
            alg = 2 * w.M * w.K + w.K * w.N // 2 + 2 * w.N * (-(-w.K // G)) + 2 * w.M * w.N
            kernels = 2 if w.M >= DECODE_FIRST_MIN_M[fmt] else 1

            def step():
                check(fn(Aw.data_ptr(), Wq.data_ptr(), Sc.data_ptr(), C.data_ptr(), w.M, w.N, w.K,
                         w.K, ldq, w.N, w.N, G, None, None, handle), f"{fmt} GEMM")
            return step, w, w.flops, alg, kernels, (Aw, Wq, Sc, C)
        return make

    variants = [("square8192/backward", backward),
                ("square8192/bias_gelu", epilogue("bias_gelu")),
                ("square8192/bias_relu_residual", epilogue("bias_relu_residual")),
                ("square8192/w4", weights(sq, "w4")), ("square8192/nf4", weights(sq, "nf4")),
                ("skinny64x28672x8192/w4", weights(sk, "w4")),
                ("skinny64x28672x8192/nf4", weights(sk, "nf4"))]
    out = {}
    for name, make in variants:
        try:
            step, w, flops_step, alg, kernels, keep = make()
            in_bytes = alg - 2 * w.M * w.N
            scrub = (torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
                     if in_bytes <= L2_BYTES else None)
            with torch.cuda.stream(stream):
                for _ in range(max(args.warmup, 3)):
                    if scrub is not None:
                        scrub.fill_(1.0)
                    step()
                _, probe_ms = timed_steps(torch, step, stream, 3, scrub)
                steps = int(min(max(args.steps, args.workload_seconds * 1e3 /
                                    max(probe_ms / 3, 1e-3)), 100000))
                sampler = ClockSampler(bus)
                step_ms, region_ms = timed_steps(torch, step, stream, steps, scrub, sampler)
            st, word = binding.tg_device_error_check(clear=True)
            if st != 0:
                raise RuntimeError(f"device error word {word:#x}")
            ms = statistics.mean(step_ms)
            roof = roofline(w.flops, alg, flops_step, ms, peaks, peak_src)
            rl = {k: roof[k] for k in ("bound", "achieved", "unit", "peak", "frac")}
            if roof["bound"] == "tensor" and "bf16_tflops_sustained" in peaks:
                # about half a second of back-to-back steps: the power-capped regime of the
                # sustained peak
                rl["peak_sustained"] = peaks["bf16_tflops_sustained"] * FP16_OVER_BF16
                rl["frac_of_sustained"] = roof["achieved"] / rl["peak_sustained"]
            out[name] = {"M": w.M, "N": w.N, "K": w.K, "steps": steps, "ms_per_step": ms,
                         "value": flops_step / (ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                         "roofline": rl,
                         "step_kernels": kernels,
                         "l2": "flushed between steps" if scrub is not None
                               else "operands larger than L2",
                         "clocks": sampler.summary(), "region_ms": region_ms}
            del keep, scrub
        except Exception as e:  # recorded in the line; the other variants still run
            out[name] = {"error": f"{type(e).__name__}: {e}"}
        torch.cuda.empty_cache()
    return out


def run_ours(args, wl):
    import torch

    import fp16_gemm_relu_gb300 as tg
    from fp16_gemm_relu_gb300 import binding, build

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    build.build()
    binding.load_library()

    a_np, b_np = wl.make_a(), wl.make_b()
    props = torch.cuda.get_device_properties(dev)
    A_h = torch.from_numpy(a_np).pin_memory()
    B_h = torch.from_numpy(b_np).pin_memory()
    A = A_h.to(dev)
    B = B_h.to(dev)
    C = torch.empty((wl.M, wl.N), dtype=torch.float16, device=dev)
    plan = tg.plan(wl.M, wl.N, wl.K, num_sms=props.multi_processor_count,
                   a_ptr=A.data_ptr(), b_ptr=B.data_ptr(), c_ptr=C.data_ptr())

    stream = torch.cuda.Stream(dev)
    handle = stream.cuda_stream
    lib = binding.load_library()

    flops_per_step = wl.flops
    alg_bytes = wl.algorithmic_bytes
    if args.dequant in ("w4", "nf4"):
        from fp16_gemm_relu_gb300 import inputs as _inputs

        G = 128
        ldq = -(-(-(-wl.N // 8)) // 4) * 4
        Wq = torch.from_numpy(_inputs.int4_weights(wl.K, wl.N, wl.seed, ldq=ldq).view(np.int32)).to(dev)
        Sc = torch.from_numpy(_inputs.int4_scales(-(-wl.K // G), wl.N, wl.seed,
                                                  1.0 / np.sqrt(wl.K))).to(dev)
        del B
        alg_bytes = 2 * wl.M * wl.K + wl.K * wl.N // 2 + 2 * wl.N * (-(-wl.K // G)) + 2 * wl.M * wl.N
        # the int4 plan the library picks for the two int4 workloads: the swapped-operand
        # kernel for a few rows of A; for many (the library's default threshold per format)
        # the weights decoded once into fp16 scratch, then the fp16 GEMM
        if wl.M >= DECODE_FIRST_MIN_M[args.dequant]:
            plan = {"block_m": 256, "block_n": 256, "block_k": 64, "kernels": 2,
                    "kernel": "tg_dequant_kernel (weights to fp16 scratch), then the fp16 GEMM"}
        elif wl.M <= 128:
            # the library's rule for the swapped kernel: a last wave of at most half a grid
            # of tiles runs as two K halves
            bmt = 64 if wl.M <= 64 else 128
            tiles = -(-wl.M // bmt) * -(-wl.N // 128)
            r = tiles % props.multi_processor_count
            tail = r if (-(-wl.K // 64) >= 2 and 0 < 2 * r <= props.multi_processor_count) else 0
            plan = {"block_m": bmt, "block_n": 128, "block_k": 64, "tail_tiles": tail,
                    "kernel": "tg_gemm_w4t_kernel (C^T = W^T A^T)"}
        else:
            plan = {"block_m": 256, "block_n": 256, "block_k": 64,
                    "kernel": "tg_gemm_w4_pair_kernel"}
        plan.setdefault("kernels", 1)
        plan.update({"split_k": 1, "dequant": f"{args.dequant} g128"})
        dq_fn = lib.tg_gemm_w4a16_f16 if args.dequant == "w4" else lib.tg_gemm_nf4a16_f16

        def step():
            st = dq_fn(A.data_ptr(), Wq.data_ptr(), Sc.data_ptr(), C.data_ptr(), wl.M, wl.N, wl.K,
                       wl.K, ldq, wl.N, wl.N, G, None, None, handle)
            if st != 0:
                raise binding.TgError(st, f"dequantising GEMM ({args.dequant})")
    elif args.pass_ == "backward":
        # gradients of C = relu(A·B) for a seeded dC; the step is mask + two GEMMs
        from fp16_gemm_relu_gb300 import inputs as _inputs

        st = lib.tg_gemm_relu_f16(A.data_ptr(), B.data_ptr(), C.data_ptr(), wl.M, wl.N, wl.K,
                                  wl.K, wl.N, wl.N, binding.TG_EPILOGUE_RELU, handle)
        if st != 0:
            raise binding.TgError(st, "tg_gemm_relu_f16")
        dC = torch.from_numpy(_inputs.tensor(wl.M, wl.N, wl.seed + 102, 1)).to(dev)
        dZ = torch.empty_like(dC)
        dA = torch.empty_like(A)
        dB = torch.empty_like(B)
        flops_per_step = 2 * wl.flops
        plan = {**plan, "kernels": 3}

        def step():
            st = lib.tg_relu_backward_f16(dC.data_ptr(), C.data_ptr(), dZ.data_ptr(), wl.M, wl.N,
                                          wl.N, wl.N, wl.N, handle)
            if st == 0:
                st = lib.tg_gemm_f16_t(0, 1, dZ.data_ptr(), B.data_ptr(), dA.data_ptr(), wl.M,
                                       wl.K, wl.N, wl.N, wl.N, wl.K, None, None, handle)
            if st == 0:
                st = lib.tg_gemm_f16_t(1, 0, A.data_ptr(), dZ.data_ptr(), dB.data_ptr(), wl.K,
                                       wl.N, wl.M, wl.K, wl.N, wl.N, None, None, handle)
            if st != 0:
                raise binding.TgError(st, "backward step")
    elif args.epilogue == "relu":
        def step():
            st = lib.tg_gemm_relu_f16(A.data_ptr(), B.data_ptr(), C.data_ptr(), wl.M, wl.N, wl.K,
                                      wl.K, wl.N, wl.N, binding.TG_EPILOGUE_RELU, handle)
            if st != 0:
                raise binding.TgError(st, "tg_gemm_relu_f16")
    else:
        from fp16_gemm_relu_gb300 import inputs as _inputs

        bias = torch.from_numpy(_inputs.tensor(1, wl.N, wl.seed + 100, 0).ravel()).to(dev)
        resid = None
        act = binding.TG_ACT_GELU
        if args.epilogue == "bias_relu_residual":
            resid = torch.from_numpy(_inputs.tensor(wl.M, wl.N, wl.seed + 101, 1)).to(dev)
            act = binding.TG_ACT_RELU
        epi = binding.tg_epilogue(act, bias.data_ptr(), resid.data_ptr() if resid is not None else None,
                                  wl.N if resid is not None else 0)

        def step():
            st = lib.tg_gemm_f16_epilogue(A.data_ptr(), B.data_ptr(), C.data_ptr(), wl.M, wl.N,
                                          wl.K, wl.K, wl.N, wl.N, ctypes.byref(epi), None, handle)
            if st != 0:
                raise binding.TgError(st, "tg_gemm_f16_epilogue")

    # operand bytes the step reads; below the L2 size, L2 is flushed between timed steps
    in_bytes = alg_bytes - 2 * wl.M * wl.N
    flush = in_bytes <= L2_BYTES
    scrub = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev) if flush else None

    bus = f"{props.pci_domain_id:08x}:{props.pci_bus_id:02x}:{props.pci_device_id:02x}.0"
    sampler = ClockSampler(bus)
    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 0)):
            if flush:
                scrub.fill_(1.0)
            step()
        stream.synchronize()
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)
        step_ms, region_ms = timed_steps(torch, step, stream, args.steps, scrub, sampler)
        torch.cuda.synchronize(dev)
        if world > 1:
            torch.distributed.barrier()
    total_ms = sum(step_ms) if flush else region_ms
    total_ms = slowest_rank_ms(total_ms, device=dev)
    ms_per_step = total_ms / args.steps
    value = whole_job_tflops(world, args.steps, flops_per_step, total_ms)
    st, word = binding.tg_device_error_check(clear=True)
    if st != 0:
        raise RuntimeError(f"device error word {word:#x} after the timed region")
    clocks = sampler.summary()
    clocks["region_ms"] = region_ms
    if region_ms < 500.0:
        # the timed region is too short for the clock sampler to see the GPU under load: run the
        # same step back to back for ~0.5 s more (after the timed region, outside it) and report
        # what the sampler saw there too
        clocks["soak"] = clock_soak(torch, step, stream, scrub, bus, 0.5)
    if clocks.get("sm_mhz"):
        clocks["sm_cycles_per_step"] = ms_per_step * 1e-3 * clocks["sm_mhz"] * 1e6

    # roofline of the dominant kernel (the tcgen05 GEMM); one launch per step when the plan has
    # a single kernel, so the per-step events bracket exactly that kernel
    peaks, peak_src = load_peaks()
    kernel_ms = statistics.mean(step_ms)
    roof = roofline(wl.flops, alg_bytes, flops_per_step, kernel_ms, peaks, peak_src)
    roof["traffic"] = (traffic_from_profiles(traffic_key(wl.name, args.pass_, args.epilogue,
                                                         args.dequant))
                       if plan["kernels"] == 1 else None)
    if roof["bound"] == "tensor" and "bf16_tflops_sustained" in peaks:
        # context only: the cuBLAS rate measured in a seconds-long loop under the power cap
        # (MEASURED_PEAKS.json's sustained figure; the bench's back-to-back steps run in the
        # same regime)
        roof["peak_sustained"] = peaks["bf16_tflops_sustained"] * FP16_OVER_BF16
        roof["frac_of_sustained"] = roof["achieved"] / roof["peak_sustained"]

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic (seeded SplitMix64 inputs of the workload's distribution)",
        "config": {"workload": wl.name, "M": wl.M, "N": wl.N, "K": wl.K,
                   "accumulate": "f32", "output": "f16", "epilogue": args.epilogue,
                   "pass": args.pass_, "dequant": args.dequant,
                   "parallelism": f"replicas{world}" if world > 1 else "single",
                   "l2": "flushed between steps" if flush else
                         f"inputs ({in_bytes / 2**20:.0f} MiB) larger than L2",
                   "plan": {k: plan[k] for k in ("block_m", "block_n", "block_k", "stages",
                                                 "split_k", "tail_tiles", "units", "grid",
                                                 "kernels", "kernel") if k in plan}},
        "gpu_launches": args.steps * plan["kernels"],
        "roofline": roof,
        "clocks": clocks,
    }
    if (rank == 0 and not args.no_workloads and args.pass_ == "forward"
            and args.epilogue == "relu" and args.dequant == "none"):
        line["workloads"] = other_workloads(args, wl.name, lib, binding, dev, stream, bus, peaks,
                                            peak_src)
        if wl.name == "square8192":
            line["variants"] = other_variants(args, lib, binding, dev, stream, bus, peaks,
                                              peak_src, A, B)

    if rank == 0 and not args.no_e2e and args.pass_ == "forward" and args.dequant == "none":
        line["e2e"] = e2e(wl, A_h, B_h, dev, max(3, min(args.steps, 10)))
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, a_np, b_np, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def e2e(wl, A_h, B_h, dev, steps):
    """Same metric through the host-buffer C entry point: H2D of A and B from page-locked
    memory, the GEMM, D2H of C, all inside the timed region."""
    import torch

    from fp16_gemm_relu_gb300 import binding

    C_h = torch.empty((wl.M, wl.N), dtype=torch.float16).pin_memory()
    lib = binding.load_library()
    stream = torch.cuda.Stream(dev)

    def call():
        st = lib.tg_gemm_relu_f16_host(A_h.data_ptr(), B_h.data_ptr(), C_h.data_ptr(), wl.M,
                                       wl.N, wl.K, wl.K, wl.N, wl.N, binding.TG_EPILOGUE_RELU,
                                       stream.cuda_stream)
        if st != 0:
            raise binding.TgError(st, "tg_gemm_relu_f16_host")

    for _ in range(2):
        call()
    t0 = time.perf_counter()
    for _ in range(steps):
        call()
    dt = (time.perf_counter() - t0) / steps
    return {"value": wl.flops / dt / 1e12, "unit": "TFLOP/s",
            "h2d_bytes_per_step": (wl.M * wl.K + wl.K * wl.N) * 2,
            "d2h_bytes_per_step": wl.M * wl.N * 2, "ms_per_step": 1e3 * dt, "steps": steps}


def main():
    args = parse_args()
    wl = workloads.get(args.workload)
    if args.impl == "reference":
        run_reference(args, wl)
    else:
        run_ours(args, wl)


if __name__ == "__main__":
    main()
