"""Benchmark: C = A·B through the library's C ABI on the square bf16 8192^3 TN GEMM.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload W]

``--workload`` picks another row of the workload table: c1..c5 (16-bit operands),
c4-e4m3 (8-bit operands, per-tensor scales, gemm_run_ex), c4-mx (8-bit operands with
E8M0 scales per 32 K elements, gemm_run_mx) or c4-sp (a 2:4-sparse A, gemm_run_sp; TFLOP/s
counted dense-equivalent, 2MNK, against twice the dense peak).

One step = one full GEMM (the whole hot path: TMA ring, tcgen05 MMA, epilogue) on
inputs resident in HBM.  Prints one JSON line (rank 0).  Under torchrun each rank runs
its own independent GEMM of the same size (weak scaling; no collective on the data
path); the timed region is bracketed by a barrier and the maximum over ranks is kept.

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
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "hbm_gbs": 6800.0}
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
PLAN_KEYS = ("config", "bm", "bn", "bk", "stages", "cluster", "grid", "dp_tiles", "sk_base", "sk_extra")
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


class ClockSampler:
    """nvidia-smi clock/throttle sampling while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line.strip()))

    def stop(self, t0: float, t1: float):
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, mx, pw, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ts, line in self.lines:
            if not (t0 <= ts <= t1):
                continue
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
                pw.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "power_w_max": max(pw),
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def reduce_max(values, world, device=None):
    """Max of per-rank floats over all ranks (identity when world == 1)."""
    if world == 1:
        return list(values)
    import torch
    import torch.distributed as dist

    t = torch.tensor(values, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


# ------------------------------------------------------------------ CPU oracle timing


def oracle_rows_fn(A, B, w):
    """rows -> threads used, computing those rows of C with the oracle routine of the workload."""
    import oracle
    from dense_tiled_gemm_04_gb300.workloads import block_scales, tensor_scales

    threads = oracle.max_threads()
    if w.sparse:
        Ac, E, _ = oracle.sparse24_compress(A)
        return lambda rows: (oracle.gemm_sparse24(Ac, E, B, w.layout, w.dtype, rows=rows), threads)[1]
    if w.elem_bytes == 2:
        return lambda rows: oracle.gemm_rows(A, B, w.layout, w.dtype, rows)[2]
    if w.scales == "block":
        sa, sb = block_scales(w)
        return lambda rows: (oracle.gemm_blockscaled(A, B, sa, sb, w.layout, w.dtype, w.out_dtype, rows=rows),
                             threads)[1]
    s_a, s_b = tensor_scales(w)
    return lambda rows: (oracle.gemm_typed(A, B, w.layout, w.dtype, w.out_dtype, alpha=s_a * s_b, rows=rows),
                         threads)[1]


def oracle_rows_sample(A, B, w, target_s: float):
    """Time the oracle on whole rows of C: calibrate on one batch, then run ~target_s."""
    import numpy as np

    import oracle

    threads = oracle.max_threads()
    fn = oracle_rows_fn(A, B, w)
    rng = np.random.default_rng(0)
    calib = rng.integers(0, w.M, threads)
    t0 = time.perf_counter()
    used = fn(calib)
    t_cal = time.perf_counter() - t0
    batches = max(1, int(target_s / max(t_cal, 1e-3)))
    rows = rng.integers(0, w.M, threads * batches)
    t0 = time.perf_counter()
    used = fn(rows)
    dt = time.perf_counter() - t0
    flops = 2.0 * rows.size * w.N * w.K
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": int(used), "kind": "oracle",
            "sample": f"{rows.size} random rows of C ({rows.size}x{w.N} outputs, K={w.K}), fp64 sums, "
                      f"{dt:.1f} s on {used} threads"}


def run_reference(args, w):
    """The reference arm: the CPU oracle on bounded samples of the workload, per step."""
    import numpy as np

    import oracle
    from dense_tiled_gemm_04_gb300.workloads import workload_inputs

    rank, world, _ = dist_env()
    if rank != 0:
        return 0
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
    line.update({"nominal_dense_peak_tflops": 2250.0 * ratio, "frac_of_nominal": achieved / (2250.0 * ratio),
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


def run_ours(args, w):
    import torch

    from dense_tiled_gemm_04_gb300 import build as lib_build
    from dense_tiled_gemm_04_gb300 import native
    from dense_tiled_gemm_04_gb300.workloads import workload_inputs

    rank, world, local = dist_env()
    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)
    lib_build.build()
    g = native.Gemm(local)
    g.set_option(native.OPT_CONFIG, {"auto": native.CONFIG_AUTO, "128x256": native.CONFIG_128x256,
                                     "128x128": native.CONFIG_128x128, "256x256": native.CONFIG_256x256,
                                     "512x256": native.CONFIG_512x256}[args.config])

    from dense_tiled_gemm_04_gb300.workloads import TORCH_DTYPES

    A_cpu, B_cpu = workload_inputs(w)
    A, B = A_cpu.to(dev), B_cpu.to(dev)
    C = native.empty_output(w.M, w.N, TORCH_DTYPES[w.out_dtype], dev)
    stream = torch.cuda.current_stream(dev)
    step, plan, step_inputs, kind = make_step(g, native, torch, w, A, B, C, stream)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize(dev)

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)  # let the sampler start before the timed region
    # Inputs that fit in L2 would be served from it by the previous step: for those, every
    # timed step is preceded by a write of a buffer several times larger than L2 (outside
    # the step's own events), and the step time is the sum of the per-step event times.
    flush = w.algorithmic_bytes < L2_BYTES
    flush_buf = torch.empty(FLUSH_BYTES // 4, dtype=torch.int32, device=dev) if flush else None
    barrier(world)
    torch.cuda.synchronize(dev)
    t_wall0 = time.perf_counter()
    if flush:
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        for i, (e0, e1) in enumerate(evs):
            flush_buf.fill_(i)
            e0.record(stream)
            step()
            e1.record(stream)
    else:
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        for _ in range(args.steps):
            step()
        ev1.record(stream)
    torch.cuda.synchronize(dev)
    t_wall1 = time.perf_counter()
    barrier(world)
    clocks = sampler.stop(t_wall0, t_wall1)
    st = g.sync_status(stream)
    if st != native.OK:
        raise native.GemmError(st, "watchdog")
    ms_total = sum(e0.elapsed_time(e1) for e0, e1 in evs) if flush else ev0.elapsed_time(ev1)
    del flush_buf
    ms_total = reduce_max([ms_total], world, dev)[0]
    ms_step = ms_total / args.steps
    flops = float(w.flops)
    value = flops * world / (ms_step * 1e-3) / 1e12

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
        barrier(world)
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        for _ in range(e2e_steps):
            for d_, h_ in zip(devs, hosts):
                d_.copy_(h_, non_blocking=True)
            step()
            Ch.copy_(C, non_blocking=True)
            stream.synchronize()
        e2e_s = (time.perf_counter() - t0) / e2e_steps
        e2e_s = reduce_max([e2e_s], world, dev)[0]
        e2e = {"value": flops * world / e2e_s / 1e12, "unit": "TFLOP/s", "ms_per_step": e2e_s * 1e3,
               "h2d_bytes_per_step": int(sum(h_.numel() * h_.element_size() for h_ in hosts)),
               "d2h_bytes_per_step": int(Ch.numel() * 2)}
    elif not args.no_e2e:
        Ah, Bh = A_cpu.pin_memory(), B_cpu.pin_memory()
        Ch = torch.empty((w.M, w.N), dtype=A_cpu.dtype).pin_memory()
        e2e_steps = max(3, min(args.steps, 20))
        if g.run_host(Ah, Bh, Ch, w.layout, stream) != native.OK:  # sizes the device staging buffers
            raise RuntimeError("gemm_run_host failed")
        barrier(world)
        t0 = time.perf_counter()
        for _ in range(e2e_steps):
            st = g.run_host(Ah, Bh, Ch, w.layout, stream)
            if st != native.OK:
                raise native.GemmError(st, "gemm_run_host")
        e2e_s = (time.perf_counter() - t0) / e2e_steps
        e2e_s = reduce_max([e2e_s], world, dev)[0]
        e2e = {"value": flops * world / e2e_s / 1e12, "unit": "TFLOP/s", "ms_per_step": e2e_s * 1e3,
               "h2d_bytes_per_step": int(Ah.numel() * 2 + Bh.numel() * 2), "d2h_bytes_per_step": int(Ch.numel() * 2)}

    peaks, peak_src = load_peaks()
    roofline = roofline_line(w, ms_step, peaks, peak_src, load_traffic(args.workload, plan))

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = oracle_rows_sample(A_cpu, B_cpu, w, target_s=args.cpu_seconds)

    g.close()
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
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
                                    if plan["cluster"] == 2 else
                                    f" in {plan['grid'] // 4} clusters of four (two CTA pairs sharing B by multicast)"
                                    if plan["cluster"] == 4 else ""),
                       "l2": (f"inputs larger than L2 (A, B, C = {w.algorithmic_bytes / 2**20:.0f} MiB > 129 MB), "
                              "no flush") if w.algorithmic_bytes >= L2_BYTES else
                             (f"inputs fit in L2 ({w.algorithmic_bytes / 2**20:.1f} MiB): a {FLUSH_BYTES >> 20} MiB "
                              "buffer is written before every step, outside its events (cold L2)"),
                       "parallelism": f"{world} independent GEMMs, one per GPU" if world > 1 else "1 GPU",
                       "plan": launch_shape(plan), "kernel_sha": kernel_fingerprint()},
            "roofline": roofline,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": args.steps,
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
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
    ap.add_argument("--config", choices=["auto", "128x256", "128x128", "256x256", "512x256"], default="auto",
                    help="kernel configuration (default: the library's own choice)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    from dense_tiled_gemm_04_gb300.workloads import WORKLOADS

    w = WORKLOADS[args.workload]
    if args.impl == "reference":
        return run_reference(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
