"""The benchmark line's host logic on CPU: both arms name the workload with
the same string, and the compact per-configuration block at the end of the
line stays short enough to survive in a reader that keeps only the line's
last 1500 characters."""
import json

import bench
import workloads as wl


def _entry(name):
    w = wl.make(name, n_rows=2) if name != "long_f32" else wl.make(name, n_rows=1)
    return {"shape": [wl.FULL_ROWS[name], wl.COLS[name]],
            "dtype": bench.DTYPE_NAMES[w.dtype],
            "GB/s": 5966.1234, "frac_of_measured_peak": 0.891934, "frac_of_8000": 0.745766,
            "rows_per_s": bench.sig(181234567.891), "median_ms_single": 0.024567,
            "p95_ms_single": 0.025678,
            "ncu_one_launch": {"frac_of_measured_peak": 0.79234, "traffic_over_algorithmic": 0.9702},
            "cpu_oracle": {"seconds": 0.32154, "GB/s": bench.sig(1.6694321)}}


def test_configs_block_is_last_and_short():
    per = {name: _entry(name) for name in wl.NAMES}
    per["attention_x"] = {"TFLOP/s": 1.0}
    block = bench.configs_block(per, 6689.1)
    assert [k for k in block if k.startswith("C")] == ["C1", "C2", "C3", "C4", "C5"]
    line = json.dumps({"value": 1.0, "per_config": per, "configs": block})
    tail = json.dumps({"configs": block})
    assert len(tail) < 1350, len(tail)
    assert line.endswith(tail[1:])
    assert block["C5"]["w"] == "long_f32 256x262144 f32"


def test_percentile_and_sig():
    xs = [5.0, 1.0, 3.0, 2.0, 4.0]
    assert bench.percentile(xs, 0.5) == 3.0
    assert bench.percentile(xs, 0.95) == 4.8
    assert bench.percentile([7.0], 0.95) == 7.0
    assert bench.sig(123456.789) == 123500.0


def test_both_arms_name_the_headline_alike():
    w = wl.make(bench.HEADLINE, n_rows=4)
    assert bench.workload_label(w) == "masked_f32: 4 x 4096 f32, row strides 4096/4096"
    assert bench.workload_label(w, True).endswith(", mask from indices, scale 0.125")
