"""The benchmark's roofline object and L2 policy, on CPU.

The bound is the longer of the two roofline times (2MNK at the tensor peak, algorithmic
bytes at the copy bandwidth); `achieved` and `peak` are then in that bound's unit.  Workloads
whose inputs fit in L2 are timed with a flush before every step.
"""
import pytest

import bench
from dense_tiled_gemm_04_gb300.workloads import WORKLOADS

PEAKS = {"bf16_tflops": 2000.0, "hbm_gbs": 8000.0, "bf16_tflops_sustained": 1600.0}


def test_square_8192_is_tensor_bound_against_the_dense_peak():
    w = WORKLOADS["c4"]
    ms = 1.0
    r = bench.roofline_line(w, ms, PEAKS, "measured", None)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert r["achieved"] == pytest.approx(2 * 8192**3 / 1e-3 / 1e12)
    assert r["frac"] == pytest.approx(r["achieved"] / 2000.0)
    assert r["frac_of_sustained"] == pytest.approx(r["achieved"] / 1600.0)
    assert r["achieved_gbs"] == pytest.approx(w.algorithmic_bytes / 1e-3 / 1e9)


def test_worked_example_shape_is_bandwidth_bound():
    # 128 x 256 x 192: 12.6 MFLOP against 213 KB -- the bytes take longer at any realistic peak.
    w = WORKLOADS["c1"]
    r = bench.roofline_line(w, 0.005, PEAKS, "measured", None)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] == 8000.0
    assert w.algorithmic_bytes == 2 * (128 * 192 + 192 * 256 + 128 * 256)
    assert r["achieved"] == pytest.approx(w.algorithmic_bytes / 5e-6 / 1e9)
    assert r["tensor"]["achieved"] == pytest.approx(2 * 128 * 256 * 192 / 5e-6 / 1e12)


def test_eight_bit_and_sparse_take_twice_the_dense_peak():
    for key in ("c4-e4m3", "c4-mx", "c4-sp"):
        r = bench.roofline_line(WORKLOADS[key], 1.0, PEAKS, "measured", None)
        assert r["bound"] == "tensor" and r["peak"] == 4000.0


def test_flush_policy_follows_the_inputs_size():
    small = [k for k, w in WORKLOADS.items() if w.algorithmic_bytes < bench.L2_BYTES]
    assert sorted(small) == ["c1", "c2", "c3"]
    assert bench.FLUSH_BYTES > 2 * bench.L2_BYTES


PLAN = {"config": 3, "bm": 256, "bn": 256, "bk": 64, "stages": 6, "cluster": 2, "tiles_m": 32, "tiles_n": 32,
        "k_blocks": 128, "grid": 152, "threads": 192, "smem_bytes": 200000, "dp_tiles": 988, "sk_base": 60,
        "sk_extra": 48, "raster_group": 8, "k_snake": 1}


def test_stored_traffic_needs_the_same_kernel_code_and_launch_shape(tmp_path):
    import json

    path = tmp_path / "traffic.json"
    entry = {"kernel_sha": bench.kernel_fingerprint(), "plan": bench.launch_shape(PLAN),
             "dram_bytes_per_launch": 123}
    path.write_text(json.dumps({"c4": entry}))
    assert bench.load_traffic("c4", PLAN, str(path)) == 123
    assert bench.load_traffic("c3", PLAN, str(path)) is None
    assert bench.load_traffic("c4", dict(PLAN, grid=148), str(path)) is None
    assert bench.load_traffic("c4", dict(PLAN, raster_group=12), str(path)) is None
    assert bench.load_traffic("c4", dict(PLAN, k_snake=0), str(path)) is None
    path.write_text(json.dumps({"c4": dict(entry, kernel_sha="0" * 16)}))
    assert bench.load_traffic("c4", PLAN, str(path)) is None


def test_fingerprint_ignores_comments_and_host_code():
    src = "int f(int x) { return x + 1; }"
    assert bench._code_only("// note\n" + src + " /* more */") == bench._code_only(src)
    assert bench.HOST_SOURCE == "gemm_api.cu"
