"""bench.py keeps its JSON-line contract: one line with the metric, the
whole-job value, the roofline of the dominant kernel, the end-to-end number,
the clocks seen, the launch count and the CPU (oracle) baseline; the
reference arm (the oracle on the host cores) prints the same metric."""
import json
import os
import statistics
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*args, timeout=900):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                       capture_output=True, text=True, timeout=timeout)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    return json.loads(lines[0])


BASE_KEYS = {"metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
             "scaling", "vs_baseline", "dtype", "data", "config", "e2e"}


def test_reference_arm_line():
    d = _run("--impl", "reference", "--workload", "tiny", "--steps", "2", "--warmup", "1")
    assert BASE_KEYS <= set(d) and d["impl"] == "reference"
    assert d["value"] > 0 and d["unit"] == "elem/s" and d["higher_is_better"] is True
    assert d["steps"] == 2 and d["n_gpus"] == 1 and d["vs_baseline"] is None
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    assert "workload" in d["config"]


def test_list_workloads():
    """Every workload's configuration as JSON (no device needed), with the
    block counts of the configurations the workloads stand for."""
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--list-workloads"], cwd=ROOT,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    got = {d["name"]: d for d in map(json.loads, r.stdout.splitlines())}
    assert {k: v["n_blocks"] for k, v in got.items()} == {
        "tiny": 6, "dense": 15040, "moe": 86016, "ragged": 42706, "ragged_literal": 602268, "large": 244608,
        "large_literal": 204288}
    assert got["moe"]["n_real"] == 1409286144 and (got["moe"]["dp"], got["moe"]["rank"]) == (8, 3)
    assert got["ragged"]["n_params"] == 4000 and got["ragged"]["inf_step"] == 2


def _check_ours(d, steps):
    assert BASE_KEYS <= set(d) and "impl" not in d
    assert d["value"] > 0 and d["steps"] == steps and d["warmup"] >= 3
    assert d["scaling"] == "weak" and d["n_gpus"] == 1
    rf = d["roofline"]
    assert rf["bound"] == "hbm" and rf["unit"] == "GB/s" and rf["peak"] > 0
    assert rf["frac"] == pytest.approx(rf["achieved"] / rf["peak"])
    assert "traffic" in rf
    ck = d["clocks"]
    assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(ck)
    assert d["gpu_launches"] > 0
    assert "workload" in d["config"]


@pytest.mark.gpu
def test_bench_line_tiny():
    d = _run("--workload", "tiny", "--steps", "4", "--warmup", "3", "--compare", "1", "--e2e-steps", "2",
             "--cpu-sample-experts", "1", "--monitors", "2", "--other-workloads", "tiny,tiny@2:1,mx:moe",
             "--other-steps", "3")
    _check_ours(d, 4)
    ow, mx = d["other_workloads"][:2], d["other_workloads"][2]
    assert [o["blocks"] for o in ow] == [6, 3] and ow[1]["dp"].startswith("rank 1 of 2")
    # the MXFP8 variant's record: the norm and the step, 4 and 29 B per element (+ scales)
    n = 32 * (7168 * 4096 + 2048 * 7168)
    assert mx["scheme"] == "mx" and mx["elems_padded"] == mx["elems_real"] == n and mx["groups"] == n // 32
    assert mx["steps"] == 3 and mx["ms_per_step"] > 0 and mx["skipped_steps"] == 0
    assert mx["bytes_per_launch"] == {"norm": 4 * n, "step": 29 * n + n // 32}
    for k in ("norm", "step"):
        assert mx["kernels_gbs"][k] == pytest.approx(mx["bytes_per_launch"][k] / mx["kernels_ms"][k] / 1e6)
    for o in ow:
        assert o["steps"] == 3 and o["ms_per_step"] > 0 and o["skipped_steps"] == 0
        assert set(o["kernels_ms"]) == set(o["kernels_gbs"]) == set(o["frac_of_measured"]) == {"fold_norm", "step"}
        assert o["kernels_gbs"]["step"] == pytest.approx(o["bytes_per_launch"]["step"] / o["kernels_ms"]["step"] / 1e6)
        na = o["fold_norm_alone"]
        assert na["ms_median"] > 0 and na["gbs"] == pytest.approx(o["bytes_per_launch"]["fold_norm"] / na["ms_median"] / 1e6)
    e = d["e2e"]
    assert e["value"] > 0 and e["h2d_bytes_per_step"] == 4 * 60000 and e["d2h_bytes_per_step"] > 60000
    assert len(e["ms_per_step_reps"]) == len(e["ms_per_step_one_at_a_time_reps"]) == e["reps"] == 5
    assert e["ms_per_step"] == statistics.median(e["ms_per_step_reps"])
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] > 0
    assert d["other_path"]["path"] == "unfused"
    mon = d["monitors"]
    assert mon["step_ms"] > 0 and mon["step_gbs"] > 0 and mon["paramwise_split_ms"] >= 0
    lb = d["layout_build_ms"]
    assert 0 < lb["host"] and 0 < lb["host_and_upload"]
    # per step: the flat-run norm and the step (one launch for the tiny workload's
    # single padded run)
    assert d["gpu_launches"] == 2 * 4


@pytest.mark.gpu
def test_bench_line_shard_and_bf16_fold():
    d = _run("--workload", "dense", "--shard", "4:1", "--steps", "3", "--warmup", "3", "--compare", "0",
             "--e2e-steps", "0", "--cpu-sample-experts", "0", "--bf16-fold", "2", "--other-workloads", "")
    _check_ours(d, 3)
    assert d["config"]["dp"].startswith("rank 1 of 4")
    assert d["config"]["blocks"] == 3760 and d["e2e"] is None
    assert d["bf16_fold"]["fold_ms"] > 0 and d["bf16_fold"]["unfold_ms"] > 0


@pytest.mark.gpu
def test_bench_line_mx():
    d = _run("--scheme", "mx", "--workload", "moe", "--experts", "1", "--steps", "3", "--warmup", "3")
    _check_ours(d, 3)


def test_threaded_oracle_pass_equals_single_thread():
    """The all-cores CPU baseline runs the same oracle calls on block ranges in
    threads: its state and codes equal the single-thread pass's."""
    import numpy as np

    sys.path.insert(0, ROOT)
    import bench
    one, many = bench.OracleSample("tiny", 1), bench.OracleSample("tiny", 1)
    one.run()
    many.run_threads(3)
    for name in ("p", "m", "v"):
        assert np.array_equal(getattr(one, name).view(np.uint32), getattr(many, name).view(np.uint32))
    for a, b in zip(one.outs, many.outs):
        assert np.array_equal(a, b)
    d = bench.cpu_baseline_all_cores("tiny", 1)
    assert d["cores"] == (os.cpu_count() or 1) and d["value"] > 0 and d["host_cores"] >= 1
