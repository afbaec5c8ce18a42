"""The benchmark's host-side logic on CPU: the one-GPU rule, the clock record and the
clock-normalised figures.  No GPU: a fake NVML library stands in for the driver's."""
import pytest

import bench
from dense_tiled_gemm_04_gb300.workloads import WORKLOADS


def test_more_than_one_gpu_is_refused():
    assert bench.one_gpu_refusal(1, {}) is None
    assert bench.one_gpu_refusal(1, {"WORLD_SIZE": "1"}) is None
    assert "refused" in bench.one_gpu_refusal(2, {})
    assert "refused" in bench.one_gpu_refusal(1, {"WORLD_SIZE": "2"})


def test_main_exits_2_before_any_gpu_work_when_asked_for_two(capsys):
    assert bench.main(["--gpus", "2", "--steps", "1", "--warmup", "3"]) == 2
    assert "one-GPU" in capsys.readouterr().err


class FakeNvml:
    """The few NVML calls the reader makes, answering from a script of (MHz, mW, reasons)."""

    def __init__(self, script):
        self.script = list(script)
        self.i = 0

    def nvmlInit_v2(self):
        return 0

    def nvmlDeviceGetHandleByUUID(self, uuid, handle):
        return 0 if uuid == b"GPU-1234" else 999

    def nvmlDeviceGetHandleByIndex_v2(self, index, handle):
        return 0

    def nvmlDeviceGetMaxClockInfo(self, handle, which, out):
        out._obj.value = 2070
        return 0

    def nvmlDeviceGetClockInfo(self, handle, which, out):
        out._obj.value = self.script[min(self.i, len(self.script) - 1)][0]
        return 0

    def nvmlDeviceGetPowerUsage(self, handle, out):
        out._obj.value = self.script[min(self.i, len(self.script) - 1)][1]
        return 0

    def nvmlDeviceGetCurrentClocksEventReasons(self, handle, out):
        out._obj.value = self.script[min(self.i, len(self.script) - 1)][2]
        self.i += 1
        return 0


def test_nvml_reader_decodes_clocks_power_and_reasons():
    r = bench.NvmlReader("1234", 0, lib=FakeNvml([(1980, 1_200_000, 0x4 | 0x1)]))
    assert r.matched == "uuid" and r.sm_max == 2070.0
    mhz, watts, reasons = r.read()
    assert (mhz, watts, reasons) == (1980.0, 1200.0, 0x5)
    assert bench.NvmlReader("ffff", 0, lib=FakeNvml([(1, 1, 0)])).matched == "index"


def test_clock_record_keeps_only_samples_inside_the_region():
    samples = [(0.5, 900.0, 100.0, 0), (1.0, 2070.0, 900.0, 0), (1.1, 1800.0, 1390.0, 0x4),
               (1.2, 1780.0, 1395.0, 0x4 | 0x40), (3.0, 500.0, 50.0, 0x8)]
    rec = bench.summarize_clocks(samples, 2070.0, 0.9, 1.25, "test")
    assert rec["samples"] == 3 and rec["sm_mhz"] == 1800.0 and rec["sm_min_mhz"] == 1780.0
    assert rec["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"] and rec["power_w_max"] == 1395.0
    empty = bench.summarize_clocks(samples, 2070.0, 1.3, 1.31, "test")
    assert empty["samples"] == 0 and "no sample" in empty["note"]


def test_sampler_polls_a_reader_in_the_background():
    import time

    s = bench.ClockSampler(reader=bench.NvmlReader("1234", 0, lib=FakeNvml([(2000, 1000_000, 0)] * 10000)))
    t0 = time.perf_counter()
    s.start()
    time.sleep(0.05)
    s.stop()
    rec = s.region(t0, time.perf_counter())
    assert rec["samples"] >= 3 and rec["sm_mhz"] == 2000.0 and rec["source"].startswith("nvml")


def test_cycle_figures_of_the_headline_plan():
    w = WORKLOADS["c4"]
    plan = {"grid": 152, "cluster": 2, "tiles_m": 32, "tiles_n": 32, "bm": 256, "bn": 256}
    c = bench.cycle_figures(w, plan, 0.6, 2000.0)
    assert c["cycles_per_launch"] == pytest.approx(1.2e6)
    assert c["cycles_per_tile"] == pytest.approx(1.2e6 * 76 / 1024)
    # One pair tile: 256 x 256 x 8192 multiply-adds over two SMs at 4096 per clock each.
    assert c["min_cycles_per_tile"] == pytest.approx(256 * 256 * 8192 / 2 / 4096)
    assert bench.cycle_figures(w, plan, 0.6, None) is None


def test_accuracy_line_against_the_oracles_codes():
    import numpy as np

    import oracle

    ref = oracle.encode(np.array([[1.0, -2.0, 0.5, 100.0]]), "bf16")
    same = bench.accuracy_line(ref, ref, "bf16")
    assert same["max_abs_err"] == 0.0 and same["within_tolerance"] and same["bit_identical_frac"] == 1.0
    off = ref.copy()
    off[0, 3] += 1  # one bf16 ulp at 100: 0.5, inside 3e-2 + 3e-2 * 100
    one = bench.accuracy_line(off, ref, "bf16")
    assert one["max_abs_err"] == 0.5 and one["within_tolerance"] and one["bit_identical_frac"] == 0.75
    assert one["max_rel_err"] == 0.5 / 100.0 and one["max_rel_err_where"] == "|ref| >= 1"
    far = oracle.encode(np.array([[1.0, -2.0, 0.5, 110.0]]), "bf16")
    assert not bench.accuracy_line(far, ref, "bf16")["within_tolerance"]
    nan = oracle.encode(np.array([[np.nan, -2.0, 0.5, 100.0]]), "bf16")
    assert not bench.accuracy_line(nan, ref, "bf16")["within_tolerance"]


def test_cpu_baseline_sample_returns_the_oracles_rows(oracle_lib):
    import numpy as np

    from dense_tiled_gemm_04_gb300.workloads import make_inputs
    from dense_tiled_gemm_04_gb300.workloads import WORKLOADS as W

    w = W["c1"]
    A, B = make_inputs(w.M, w.N, w.K, w.layout, w.dtype, "int", seed=3)
    cpu, rows, ref = bench.oracle_rows_sample(A, B, w, target_s=0.01)
    assert cpu["kind"] == "oracle" and cpu["cores"] >= 1 and ref.shape == (rows.size, w.N)
    assert np.array_equal(ref, oracle_lib.gemm(A, B, w.layout, w.dtype)[rows])
