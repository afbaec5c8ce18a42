"""Benchmark: C = A·B through the library's C ABI on the square bf16 8192^3 TN GEMM.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload W]

``--workload`` picks another row of the workload table: c1..c5 (16-bit operands),
c4-e4m3 (8-bit operands, per-tensor scales, gemm_run_ex), c4-mx (8-bit operands with
E8M0 scales per 32 K elements, gemm_run_mx) or c4-sp (a 2:4-sparse A, gemm_run_sp; TFLOP/s
counted dense-equivalent, 2MNK, against twice the dense peak).

One step = one full GEMM (the whole hot path: TMA ring, tcgen05 MMA, epilogue) on
inputs resident in HBM.  Prints one JSON line.  The library is a one-GPU library: with
--gpus > 1, or under a launcher that starts more than one rank (WORLD_SIZE > 1), the
benchmark refuses to run and exits with status 2.

The line also carries the CPU oracle timed on a sample of whole rows of C (``cpu_baseline``)
and the error of the GPU's result on those rows against the oracle's (``accuracy``: maximum
absolute and relative error, bit-identical fraction, the per-element tolerance check).

``--impl reference`` times the CPU oracle (fp64 triple loop) on bounded samples of the
same workload on the host cores: the slow reference arm, not a GPU implementation.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GEMM TFLOP/s at 1 GB300 and % of dense FP16/BF16 tensor roofline"
WORKLOAD = "c4"
# Roofline denominators when no measured peaks are present: one earlier measurement of a
# cuBLAS bf16 GEMM and of a device copy on a GB300.
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "hbm_gbs": 6800.0}
# NVIDIA's published dense FP16/BF16 tensor rate of one GB300 (2.25 PFLOP/s; its larger figures
# assume 2:4 sparsity).  Context only: the roofline uses the measured peaks.
NOMINAL_DENSE_TFLOPS = 2250.0
L2_BYTES = 129 * 10**6        # GB300 L2
FLUSH_BYTES = 512 * 2**20     # the buffer written between steps whose inputs fit in L2
KERNEL_DIR = os.path.join("dense_tiled_gemm_04_gb300", "csrc")


def _code_only(text: str) -> str:
    """C++ source without comments and blank space, so that a comment edit does not count as
    a kernel change (string literals in these sources hold no comment markers)."""
    import re

    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return re.sub(r"\s+", " ", text).strip()


# What a launch's DRAM traffic depends on besides the kernel's code: the launch shape.
PLAN_KEYS = ("config", "bm", "bn", "bk", "stages", "cluster", "grid", "dp_tiles", "sk_base", "sk_extra",
             "raster_group", "k_snake")
HOST_SOURCE = "gemm_api.cu"  # argument checks, tensor maps, plans and the host pipeline


def kernel_fingerprint() -> str:
    """Hash of the kernels' device sources (code only, see _code_only; the host side is left
    out, its launch shape is compared through PLAN_KEYS); a stored ncu traffic figure is only
    reported for the code and the launch shape it was measured on."""
    h = hashlib.sha256()
    d = os.path.join(ROOT, KERNEL_DIR)
    for name in sorted(os.listdir(d)):
        if name.endswith((".cu", ".cuh", ".h")) and name != HOST_SOURCE:
            with open(os.path.join(d, name), encoding="utf-8") as f:
                h.update(name.encode() + _code_only(f.read()).encode())
    return h.hexdigest()[:16]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def launch_shape(plan: dict) -> dict:
    return {k: int(plan[k]) for k in PLAN_KEYS}


def load_traffic(workload_key: str, plan: dict, path: str = os.path.join(ROOT, "profiles", "traffic.json")):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on this kernel
    code with this launch shape."""
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    entry = d.get(workload_key)
    if not entry or entry.get("kernel_sha") != kernel_fingerprint() or entry.get("plan") != launch_shape(plan):
        return None
    return entry.get("dram_bytes_per_launch")


# NVML clock-event reason bits (nvmlClocksEventReason*): the ones a bench line reports.
NVML_REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
                0x80: "hw_power_brake_slowdown"}
NVML_CLOCK_SM = 1
CLOCK_POLL_S = 0.002  # NVML is polled every 2 ms, so a 10 ms timed region still gets samples


class NvmlReader:
    """Reads the SM clock, its maximum, the power draw and the clock-event reasons of one GPU
    through the driver's NVML library (ctypes; nothing to install).  Read-only: it changes no
    setting of the GPU."""

    def __init__(self, uuid: str = "", index: int = 0, lib=None):
        import ctypes

        self.ct = ctypes
        self.lib = lib if lib is not None else ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.handle = ctypes.c_void_p()
        self.matched = "uuid"
        u = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        if not uuid or self.lib.nvmlDeviceGetHandleByUUID(u.encode(), ctypes.byref(self.handle)) != 0:
            self.matched = "index"
            if self.lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(self.handle)) != 0:
                raise OSError("no NVML handle for the device")
        mx = ctypes.c_uint(0)
        self.lib.nvmlDeviceGetMaxClockInfo(self.handle, NVML_CLOCK_SM, ctypes.byref(mx))
        self.sm_max = float(mx.value)

    def read(self):
        """(SM MHz, power W or None, reason bitmask or None)."""
        ct = self.ct
        clk, pw, rs = ct.c_uint(0), ct.c_uint(0), ct.c_ulonglong(0)
        if self.lib.nvmlDeviceGetClockInfo(self.handle, NVML_CLOCK_SM, ct.byref(clk)) != 0:
            return None
        power = pw.value / 1000.0 if self.lib.nvmlDeviceGetPowerUsage(self.handle, ct.byref(pw)) == 0 else None
        fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(self.lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
        reasons = rs.value if fn(self.handle, ct.byref(rs)) == 0 else None
        return float(clk.value), power, reasons


def summarize_clocks(samples, sm_max, t0: float, t1: float, source: str):
    """Clock record of the samples (t, SM MHz, power W, reason bits) taken inside [t0, t1]."""
    inside = [s for s in samples if t0 <= s[0] <= t1]
    if not inside:
        return {"sm_mhz": None, "sm_max_mhz": sm_max, "reasons": [], "samples": 0, "source": source,
                "note": f"no sample fell inside the {1e3 * (t1 - t0):.1f} ms region"}
    sm = [s[1] for s in inside]
    pw = [s[2] for s in inside if s[2] is not None]
    reasons = set()
    for s in inside:
        if s[3] is not None:
            reasons.update(name for bit, name in NVML_REASONS.items() if s[3] & bit)
    out = {"sm_mhz": statistics.median(sm), "sm_min_mhz": min(sm), "sm_max_mhz": sm_max,
           "reasons": sorted(reasons), "samples": len(sm), "source": source}
    if pw:
        out["power_w_max"] = max(pw)
    return out


class ClockSampler:
    """Samples the GPU's clocks in a background thread while timed regions run: NVML every
    CLOCK_POLL_S, or, without NVML, nvidia-smi every 50 ms."""

    SMI_FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active")

    def __init__(self, uuid: str = "", index: int = 0, reader=None):
        self.samples = []
        self.sm_max = None
        self.stop_flag = threading.Event()
        self.thread = None
        self.proc = None
        self.reader = reader
        self.source = "nvml"
        if self.reader is None:
            try:
                self.reader = NvmlReader(uuid, index)
            except OSError:
                self.reader = None
                self.source = "nvidia-smi"
        if self.reader is not None:
            self.sm_max = self.reader.sm_max
            self.source = f"nvml ({getattr(self.reader, 'matched', 'uuid')}), every {CLOCK_POLL_S * 1e3:.0f} ms"
        self.index = index

    def start(self):
        if self.reader is not None:
            self.thread = threading.Thread(target=self._poll, daemon=True)
        else:
            try:
                self.proc = subprocess.Popen(
                    ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.SMI_FIELDS}",
                     "--format=csv,noheader,nounits", "-lms", "50"], stdout=subprocess.PIPE,
                    stderr=subprocess.DEVNULL, text=True)
            except (FileNotFoundError, OSError):
                return
            self.thread = threading.Thread(target=self._read_smi, daemon=True)
        self.thread.start()

    def _poll(self):
        while not self.stop_flag.is_set():
            r = self.reader.read()
            if r is not None:
                self.samples.append((time.perf_counter(), *r))
            time.sleep(CLOCK_POLL_S)

    def _read_smi(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            try:
                sm, mx, pw, act = float(parts[0]), float(parts[1]), float(parts[2]), int(parts[3], 16)
            except (ValueError, IndexError):
                continue
            self.sm_max = mx
            self.samples.append((time.perf_counter(), sm, pw, act))

    def stop(self):
        self.stop_flag.set()
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)

    def region(self, t0: float, t1: float):
        return summarize_clocks(list(self.samples), self.sm_max, t0, t1, self.source)


def one_gpu_refusal(gpus: int, env=None):
    """None when the run asks for one GPU and one process; otherwise the reason it is refused.
    The library computes on one GPU: it has no multi-GPU path to measure."""
    env = os.environ if env is None else env
    world = int(env.get("WORLD_SIZE", "1"))
    if gpus != 1 or world != 1:
        return (f"bench.py measures a one-GPU library: --gpus {gpus} with WORLD_SIZE {world} is refused "
                "(run it with --gpus 1, without a multi-process launcher)")
    return None


# ------------------------------------------------------------------ CPU oracle timing


def oracle_rows_fn(A, B, w):
    """rows -> (those rows of C as output-type codes, threads used), from the oracle routine of
    the workload."""
    import oracle
    from dense_tiled_gemm_04_gb300.workloads import block_scales, tensor_scales

    threads = oracle.max_threads()
    if w.sparse:
        Ac, E, _ = oracle.sparse24_compress(A)
        return lambda rows: (oracle.gemm_sparse24(Ac, E, B, w.layout, w.dtype, rows=rows), threads)
    if w.elem_bytes == 2:
        def dense(rows):
            codes, _, used = oracle.gemm_rows(A, B, w.layout, w.dtype, rows)
            return codes, used
        return dense
    if w.scales == "block":
        sa, sb = block_scales(w)
        return lambda rows: (oracle.gemm_blockscaled(A, B, sa, sb, w.layout, w.dtype, w.out_dtype, rows=rows),
                             threads)
    s_a, s_b = tensor_scales(w)
    return lambda rows: (oracle.gemm_typed(A, B, w.layout, w.dtype, w.out_dtype, alpha=s_a * s_b, rows=rows),
                         threads)


def oracle_rows_sample(A, B, w, target_s: float):
    """Time the oracle on whole rows of C: calibrate on one batch, then run ~target_s.  Returns
    (the cpu_baseline object, the rows, the oracle's codes for them)."""
    import numpy as np

    import oracle

    threads = oracle.max_threads()
    fn = oracle_rows_fn(A, B, w)
    rng = np.random.default_rng(0)
    calib = rng.integers(0, w.M, threads)
    t0 = time.perf_counter()
    fn(calib)
    t_cal = time.perf_counter() - t0
    batches = max(1, int(target_s / max(t_cal, 1e-3)))
    rows = rng.integers(0, w.M, threads * batches)
    t0 = time.perf_counter()
    ref, used = fn(rows)
    dt = time.perf_counter() - t0
    flops = 2.0 * rows.size * w.N * w.K
    cpu = {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": int(used), "kind": "oracle",
           "sample": f"{rows.size} random rows of C ({rows.size}x{w.N} outputs, K={w.K}), fp64 sums, "
                     f"{dt:.1f} s on {used} threads"}
    return cpu, rows, ref


# Per-element tolerance on random inputs (fp16 / bf16 output): |gpu - ref| <= atol + rtol * |ref|.
TOLERANCE = {"f16": (1e-2, 1e-2), "bf16": (3e-2, 3e-2)}


def accuracy_line(got_codes, ref_codes, out_dtype: str):
    """Error of the GPU's rows of C against the oracle's (both rounded to the output type)."""
    import numpy as np

    import oracle

    g = oracle.decode(np.asarray(got_codes), out_dtype)
    r = oracle.decode(np.asarray(ref_codes), out_dtype)
    d = np.abs(g - r)
    atol, rtol = TOLERANCE[out_dtype]
    big = np.abs(r) >= atol / rtol  # where the relative term of the tolerance dominates
    ratio = d / (atol + rtol * np.abs(r))
    finite = bool(np.isfinite(g).all())
    return {"elements": int(g.size), "max_abs_err": float(d.max()) if finite else None,
            "max_rel_err": float((d[big] / np.abs(r[big])).max()) if finite and big.any() else None,
            "max_rel_err_where": f"|ref| >= {atol / rtol:g}",
            "bit_identical_frac": float(np.mean(np.asarray(got_codes) == np.asarray(ref_codes))),
            "worst_tolerance_ratio": float(ratio.max()) if finite else None,
            "within_tolerance": bool(finite and (ratio <= 1.0).all()),
            "tolerance": f"|gpu - ref| <= {atol:g} + {rtol:g} |ref| ({out_dtype} output)",
            "reference": "the CPU oracle: fp64 sums rounded once to the output type"}


def run_reference(args, w):
    """The reference arm: the CPU oracle on bounded samples of the workload, per step."""
    import numpy as np

    import oracle
    from dense_tiled_gemm_04_gb300.workloads import workload_inputs

    oracle.build()
    A, B = workload_inputs(w)
    threads = oracle.max_threads()
    if w.elem_bytes == 1 or w.sparse:
        return run_reference_rows(args, w, A, B, threads)
    rng = np.random.default_rng(1)
    # Elements per step sized so warm-up + timed steps take about a minute in total.
    probe = 64 * threads
    t0 = time.perf_counter()
    oracle.gemm_elems(A, B, w.layout, w.dtype, rng.integers(0, w.M, probe), rng.integers(0, w.N, probe))
    per_elem = (time.perf_counter() - t0) / probe
    total_steps = args.steps + args.warmup
    elems = int(max(threads, min(1 << 20, 60.0 / max(total_steps, 1) / max(per_elem, 1e-9))))
    samples = [(rng.integers(0, w.M, elems), rng.integers(0, w.N, elems)) for _ in range(total_steps)]
    for i in range(args.warmup):
        oracle.gemm_elems(A, B, w.layout, w.dtype, *samples[i])
    t0 = time.perf_counter()
    for i in range(args.warmup, total_steps):
        oracle.gemm_elems(A, B, w.layout, w.dtype, *samples[i])
    dt = time.perf_counter() - t0
    step_s = dt / max(args.steps, 1)
    value = 2.0 * elems * w.K / step_s / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_s * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": f"synthetic: seeded {w.dist} inputs x {w.scale:.3g} rounded to {w.dtype} "
                f"(torch CPU generator, seed {w.seed})",
        "config": {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "layout": w.layout, "in_dtype": w.dtype,
                   "sample_per_step": f"{elems} random elements of C"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": f"{elems} random elements of C per step (each a {w.K}-term fp64 dot product)"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_reference_rows(args, w, A, B, threads):
    """Reference arm for the 8-bit workloads: whole rows of C per step with the oracle."""
    import numpy as np

    fn = oracle_rows_fn(A, B, w)
    rng = np.random.default_rng(1)
    t0 = time.perf_counter()
    fn(rng.integers(0, w.M, threads))
    per_row = (time.perf_counter() - t0) / threads
    total_steps = args.steps + args.warmup
    nrows = int(max(threads, min(w.M, 60.0 / max(total_steps, 1) / max(per_row, 1e-9))))
    samples = [rng.integers(0, w.M, nrows) for _ in range(total_steps)]
    for i in range(args.warmup):
        fn(samples[i])
    t0 = time.perf_counter()
    for i in range(args.warmup, total_steps):
        fn(samples[i])
    step_s = (time.perf_counter() - t0) / max(args.steps, 1)
    value = 2.0 * nrows * w.N * w.K / step_s / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_s * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": f"synthetic: seeded {w.dist} {w.dtype} inputs (torch CPU generator, seed {w.seed})",
        "config": {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "layout": w.layout, "in_dtype": w.dtype,
                   "out": w.out_dtype, "scales": w.scales, "sample_per_step": f"{nrows} random rows of C"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": f"{nrows} random rows of C per step ({nrows}x{w.N} fp64 dot products of "
                                   f"{w.K} terms)"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ GPU arm


def roofline_line(w, ms_step: float, peaks: dict, peak_src: str, traffic):
    """The roofline object of the JSON line for workload w at ms_step per launch.

    8-bit operands take the bf16 peak times the nominal fp8 / bf16 dense ratio (4.5 / 2.25); a
    2:4-sparse A takes twice the dense peak (the sparse tensor rate), flops counted
    dense-equivalent.  The bound is whichever roofline time is longer: 2MNK at the tensor
    peak, or the algorithmic bytes at the measured copy bandwidth."""
    flops = float(w.flops)
    ratio = 2.0 if (w.elem_bytes == 1 or w.sparse) else 1.0
    peak = ratio * float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    achieved = flops / (ms_step * 1e-3) / 1e12
    achieved_gbs = w.algorithmic_bytes / (ms_step * 1e-3) / 1e9
    src = f"{peak_src}: cuBLAS bf16 8192^3 burst" if peak_src == "measured" else "fallback bf16"
    tensor = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
              "traffic": traffic,
              "peak_source": src + (" x 2 (2:4 sparse tensor rate, dense-equivalent flops)" if w.sparse else
                                    " x 2 (nominal fp8/bf16 dense ratio)" if ratio != 1.0 else "")}
    if w.algorithmic_bytes / (hbm * 1e9) > flops / (peak * 1e12):
        line = {"bound": "hbm", "achieved": achieved_gbs, "peak": hbm, "unit": "GB/s", "frac": achieved_gbs / hbm,
                "traffic": traffic,
                "peak_source": f"{peak_src}: copy bandwidth (read + write)" if peak_src == "measured"
                else "fallback copy bandwidth",
                "tensor": {k: tensor[k] for k in ("achieved", "peak", "unit", "frac")}}
    else:
        line = dict(tensor, achieved_gbs=achieved_gbs)
    line.update({"nominal_dense_peak_tflops": NOMINAL_DENSE_TFLOPS * ratio,
                 "frac_of_nominal": achieved / (NOMINAL_DENSE_TFLOPS * ratio),
                 "algorithmic_flops_per_launch": flops, "algorithmic_bytes_per_launch": w.algorithmic_bytes})
    if "bf16_tflops_sustained" in peaks:
        line["frac_of_sustained"] = achieved / (ratio * float(peaks["bf16_tflops_sustained"]))
    return line




def make_step(g, native, torch, w, A, B, C, stream):
    """The library call one step makes, for the workload's operand kind.  Returns
    (step(), plan dict, the device tensors a step reads, description of the kernel kind)."""
    from dense_tiled_gemm_04_gb300.workloads import block_scales, tensor_scales

    sp = stream.cuda_stream
    lay, dt = native.LAYOUTS[w.layout], native.DTYPES[w.dtype]
    base = (A.data_ptr(), B.data_ptr(), C.data_ptr())
    dims = (w.M, w.N, w.K, A.stride(0), B.stride(0), C.stride(0))

    if w.sparse:
        # The compression is a one-time preparation of A (like packing weights): outside the step.
        Ac, meta, bad = g.sp_compress(A, stream)
        torch.cuda.synchronize(A.device)
        if int(bad.item()) != 0:
            raise RuntimeError("A is not 2:4 sparse")

        def step():
            st = g.run_sp_raw(Ac.data_ptr(), B.data_ptr(), C.data_ptr(), meta.data_ptr(), w.M, w.N, w.K, Ac.stride(0),
                              B.stride(0), C.stride(0), lay, dt, 1.0, 0.0, 0, sp)
            if st != native.OK:
                raise native.GemmError(st, "gemm_run_sp")
        return step, g.plan(w.M, w.N, w.K, w.layout, w.dtype, "sparse24"), [Ac, meta, B], \
            "kind::f16 .sp (2:4-sparse A)"
    if w.elem_bytes == 2:
        def step():
            st = g.run_raw(*base, *dims, lay, dt, sp)
            if st != native.OK:
                raise native.GemmError(st, "gemm_run")
        return step, g.plan(w.M, w.N, w.K, w.layout, w.dtype), [A, B], "kind::f16"
    out = native.DTYPES[w.out_dtype]
    if w.scales == "tensor":
        s_a, s_b = tensor_scales(w)

        def step():
            st = g.run_ex_raw(*base, *dims, lay, dt, 1.0, 0.0, 0, sp, out, s_a, s_b)
            if st != native.OK:
                raise native.GemmError(st, "gemm_run_ex")
        return step, g.plan(w.M, w.N, w.K, w.layout, w.dtype), [A, B], "kind::f8f6f4, per-tensor scales"
    sa, sb = block_scales(w)
    psa = g.pack_scales(torch.from_numpy(sa).to(A.device), w.K, stream)
    psb = g.pack_scales(torch.from_numpy(sb).to(A.device), w.K, stream)

    def step():
        st = g.run_mx_raw(*base, psa.data_ptr(), psb.data_ptr(), *dims, lay, dt, out, stream=sp)
        if st != native.OK:
            raise native.GemmError(st, "gemm_run_mx")
    return step, g.plan(w.M, w.N, w.K, w.layout, w.dtype, "block_scaled"), [A, B, psa, psb], \
        "kind::mxf8f6f4.block_scale, E8M0 scales per 32 K"


# Tensor-pipe rate per SM and clock for 16-bit operands: one 128 x 256 x 16 MMA (524,288
# multiply-adds) every 128 clocks, measured with a one-thread issue loop on this GPU; 8-bit
# operands and a 2:4-sparse A (dense-equivalent) count twice as many.  The minimum cycles of a
# work unit's share of the tiles follow from it.
MACS_PER_CLK_SM_16BIT = 4096
SUSTAINED_S = 2.0  # length of the back-to-back sustained leg


def cycle_figures(w, plan: dict, ms_step: float, sm_mhz):
    """Clock-normalised view of a launch: SM cycles per launch and per output tile of one work
    unit (a CTA, or a CTA pair), and the tensor pipe's minimum for that tile."""
    if not sm_mhz:
        return None
    units = plan["grid"] // plan["cluster"]
    tiles = plan["tiles_m"] * plan["tiles_n"]
    cycles = ms_step * 1e-3 * sm_mhz * 1e6
    rate = MACS_PER_CLK_SM_16BIT * (2 if (w.elem_bytes == 1 or w.sparse) else 1)
    min_tile = plan["bm"] * plan["bn"] * w.K / (plan["cluster"] * rate)  # per SM of the unit
    per_tile = cycles * units / tiles
    return {"sm_mhz": sm_mhz, "cycles_per_launch": cycles, "cycles_per_tile": per_tile,
            "min_cycles_per_tile": min_tile, "tensor_busy_est": min_tile / per_tile}


def run_ours(args, w):
    import torch

    from dense_tiled_gemm_04_gb300 import build as lib_build
    from dense_tiled_gemm_04_gb300 import native
    from dense_tiled_gemm_04_gb300.workloads import TORCH_DTYPES, workload_inputs

    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA device")
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    lib_build.build()
    g = native.Gemm(0)
    g.set_option(native.OPT_CONFIG, {"auto": native.CONFIG_AUTO, "128x256": native.CONFIG_128x256,
                                     "128x128": native.CONFIG_128x128, "256x256": native.CONFIG_256x256,
                                     "128x64": native.CONFIG_128x64}[args.config])
    if args.sk_min_blocks:
        g.set_option(native.OPT_SK_MIN_BLOCKS, args.sk_min_blocks)
    if args.raster_group:
        g.set_option(native.OPT_RASTER_GROUP, args.raster_group)
    if args.k_snake >= 0:
        g.set_option(native.OPT_K_SNAKE, args.k_snake)

    A_cpu, B_cpu = workload_inputs(w)
    A, B = A_cpu.to(dev), B_cpu.to(dev)
    C = native.empty_output(w.M, w.N, TORCH_DTYPES[w.out_dtype], dev)
    stream = torch.cuda.current_stream(dev)
    step, plan, step_inputs, kind = make_step(g, native, torch, w, A, B, C, stream)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize(dev)

    props = torch.cuda.get_device_properties(dev)
    sampler = ClockSampler(str(getattr(props, "uuid", "")), 0)
    sampler.start()
    time.sleep(0.1)  # let the sampler start before the timed region
    # Inputs that fit in L2 would be served from it by the previous step: for those, every
    # timed step is preceded by a write of a buffer several times larger than L2 (outside
    # the step's own events), and the step time is the sum of the per-step event times.
    flush = w.algorithmic_bytes < L2_BYTES
    flush_buf = torch.empty(FLUSH_BYTES // 4, dtype=torch.int32, device=dev) if flush else None

    def timed(n):
        """Run n steps; (ms per step by CUDA events on the launching stream, wall t0, t1)."""
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        if flush:
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
            for i, (e0, e1) in enumerate(evs):
                flush_buf.fill_(i)
                e0.record(stream)
                step()
                e1.record(stream)
        else:
            ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            ev0.record(stream)
            for _ in range(n):
                step()
            ev1.record(stream)
        torch.cuda.synchronize(dev)
        t1 = time.perf_counter()
        ms = sum(e0.elapsed_time(e1) for e0, e1 in evs) if flush else ev0.elapsed_time(ev1)
        return ms / n, t0, t1

    # The timed region: exactly --steps steps.
    ms_step, t_wall0, t_wall1 = timed(args.steps)
    clocks = sampler.region(t_wall0, t_wall1)
    # The sustained leg: the same step back to back for about SUSTAINED_S seconds (the power
    # limit of the part settles within them), with its own clock record.
    sustained = None
    if not args.no_sustained:
        wall_per_step = (t_wall1 - t_wall0) / args.steps
        n_sus = int(min(20000, max(args.steps, math.ceil(SUSTAINED_S / max(wall_per_step, 1e-6)))))
        ms_sus, s0, s1 = timed(n_sus)
        sus_clocks = sampler.region(s0, s1)
        sustained = {"value": float(w.flops) / (ms_sus * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": ms_sus,
                     "steps": n_sus, "seconds": s1 - s0, "clocks": sus_clocks}
    sampler.stop()
    st = g.sync_status(stream)
    if st != native.OK:
        raise native.GemmError(st, "watchdog")
    del flush_buf
    flops = float(w.flops)
    value = flops / (ms_step * 1e-3) / 1e12
    if not clocks.get("samples") and sustained and sustained["clocks"].get("samples"):
        clocks["note"] += "; the sustained leg's clock record is the nearest one"

    # End to end through the public C ABI on pinned host buffers: H2D of A and B, the
    # kernel, D2H of C, synchronised every step.
    e2e = None
    if not args.no_e2e and (w.elem_bytes == 1 or w.sparse):
        # 8-bit or sparse operands: the same library call, with the step's inputs (A or its
        # compressed form, B, any block scales or metadata) copied in from pinned host memory
        # and C copied back, every step.
        hosts = [t.cpu().pin_memory() for t in step_inputs]
        devs = step_inputs
        Ch = torch.empty(C.shape, dtype=C.dtype).pin_memory()
        e2e_steps = max(3, min(args.steps, 20))
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        for _ in range(e2e_steps):
            for d_, h_ in zip(devs, hosts):
                d_.copy_(h_, non_blocking=True)
            step()
            Ch.copy_(C, non_blocking=True)
            stream.synchronize()
        e2e_s = (time.perf_counter() - t0) / e2e_steps
        e2e = {"value": flops / e2e_s / 1e12, "unit": "TFLOP/s", "ms_per_step": e2e_s * 1e3,
               "h2d_bytes_per_step": int(sum(h_.numel() * h_.element_size() for h_ in hosts)),
               "d2h_bytes_per_step": int(Ch.numel() * 2)}
    elif not args.no_e2e:
        Ah, Bh = A_cpu.pin_memory(), B_cpu.pin_memory()
        Ch = torch.empty((w.M, w.N), dtype=A_cpu.dtype).pin_memory()
        e2e_steps = max(3, min(args.steps, 20))
        if g.run_host(Ah, Bh, Ch, w.layout, stream) != native.OK:  # sizes the device staging buffers
            raise RuntimeError("gemm_run_host failed")
        t0 = time.perf_counter()
        for _ in range(e2e_steps):
            st = g.run_host(Ah, Bh, Ch, w.layout, stream)
            if st != native.OK:
                raise native.GemmError(st, "gemm_run_host")
        e2e_s = (time.perf_counter() - t0) / e2e_steps
        e2e = {"value": flops / e2e_s / 1e12, "unit": "TFLOP/s", "ms_per_step": e2e_s * 1e3,
               "h2d_bytes_per_step": int(Ah.numel() * 2 + Bh.numel() * 2), "d2h_bytes_per_step": int(Ch.numel() * 2)}

    peaks, peak_src = load_peaks()
    roofline = roofline_line(w, ms_step, peaks, peak_src, load_traffic(args.workload, plan))
    roofline["cycles"] = cycle_figures(w, plan, ms_step, clocks.get("sm_mhz"))
    if sustained:
        sustained["frac_of_sustained_peak"] = roofline_line(w, sustained["ms_per_step"], peaks, peak_src,
                                                            None).get("frac_of_sustained")
        sustained["cycles"] = cycle_figures(w, plan, sustained["ms_per_step"], sustained["clocks"].get("sm_mhz"))

    # The CPU baseline: the oracle timed on a sample of whole rows of C; the same rows of the
    # GPU's C (the last timed step's) are then compared with them.
    cpu = accuracy = None
    if not args.no_cpu_baseline:
        cpu, rows, ref = oracle_rows_sample(A_cpu, B_cpu, w, target_s=args.cpu_seconds)
        got = C[torch.from_numpy(rows).to(dev)].cpu().contiguous().view(torch.int16).numpy().view("uint16")
        accuracy = dict(accuracy_line(got, ref, w.out_dtype), rows=int(rows.size))

    g.close()
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype,
        "data": f"synthetic: seeded {w.dist} inputs x {w.scale:.3g} rounded to {w.dtype} "
                f"(torch CPU generator, seed {w.seed})"
                + (", E8M0 block scales uniform in 124..130 (numpy generator)" if w.scales == "block" else "")
                + (", A pruned to a seeded 2:4 pattern along K" if w.sparse else ""),
        "config": {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "layout": w.layout,
                   "accumulate": "fp32", "out": w.out_dtype,
                   "kernel": f"tcgen05 {kind}, {plan['bm']}x{plan['bn']}x{plan['bk']} tile, {plan['stages']}-stage "
                             f"ring, {plan['grid']} persistent CTAs"
                             + (f" in {plan['grid'] // plan['cluster']} CTA pairs (cta_group::2)"
                                if plan["cluster"] == 2 else ""),
                   "l2": (f"inputs larger than L2 (A, B, C = {w.algorithmic_bytes / 2**20:.0f} MiB > 129 MB), "
                          "no flush") if w.algorithmic_bytes >= L2_BYTES else
                         (f"inputs fit in L2 ({w.algorithmic_bytes / 2**20:.1f} MiB): a {FLUSH_BYTES >> 20} MiB "
                          "buffer is written before every step, outside its events (cold L2)"),
                   "parallelism": "1 GPU",
                   "plan": launch_shape(plan), "kernel_sha": kernel_fingerprint()},
        "roofline": roofline,
        "sustained": sustained,
        "cpu_baseline": cpu,
        "accuracy": accuracy,
        "e2e": e2e,
        "gpu_launches": args.steps,
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="target length of the CPU-oracle sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg (profiling runs)")
    ap.add_argument("--workload", default=WORKLOAD,
                    help="c1..c5, c4-e4m3, c4-mx, c4-sp (default c4, the headline workload)")
    ap.add_argument("--config", choices=["auto", "128x256", "128x128", "256x256", "128x64"], default="auto",
                    help="kernel configuration (default: the library's own choice)")
    ap.add_argument("--no-sustained", action="store_true", help="skip the back-to-back sustained leg")
    ap.add_argument("--sk-min-blocks", type=int, default=0,
                    help="shortest stream-K share in K blocks (default: the library's, 8)")
    ap.add_argument("--raster-group", type=int, default=0,
                    help="tile rows per group of the grouped raster (default: the library's, about 48 MiB of A, at most 16 rows)")
    ap.add_argument("--k-snake", type=int, choices=[0, 1], default=-1,
                    help="1: every second work item walks its K blocks backwards (default: the library's)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    refusal = one_gpu_refusal(args.gpus)
    if refusal:
        print(refusal, file=sys.stderr, flush=True)
        return 2
    from dense_tiled_gemm_04_gb300.workloads import WORKLOADS

    w = WORKLOADS[args.workload]
    if args.impl == "reference":
        return run_reference(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
