"""The bench harness on a GPU: the default JSON line's contract keys, and the
output dump (--dump) compared offline against the f64 oracle on the same
seeded workload, the way a dumped step is checked after a run."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import oracle
from paged_gqa_decode_06_gb300 import workloads

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_bench(*extra):
    r = subprocess.run([sys.executable, "bench.py", *extra], cwd=ROOT, capture_output=True,
                       text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    return [json.loads(l) for l in lines]


@pytest.fixture(scope="module")
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@pytest.mark.parametrize("name", ["tiny", "llama"])
def test_bench_line_and_dump_match_the_oracle(gpu, tmp_path, name):
    path = str(tmp_path / f"{name}.npz")
    cpu = ["--cpu-budget", "1"] if name == "tiny" else ["--no-cpu-baseline"]
    (line,) = run_bench("--workload", name, "--steps", "5", "--warmup", "3", "--e2e-steps", "0",
                        "--config-steps", "0", *cpu, "--dump", path)
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "cpu_baseline", "e2e", "gpu_launches", "clocks"):
        assert key in line, key
    assert line["steps"] == 5 and line["gpu_launches"] == 5 and line["value"] > 0
    roof = line["roofline"]
    assert roof["bound"] == "hbm" and roof["unit"] == "GB/s" and roof["peak"] > 0
    assert abs(roof["frac"] - roof["achieved"] / roof["peak"]) < 1e-9
    if roof["traffic"] is None:
        assert roof["traffic_gbs"] is None
    else:
        assert abs(roof["traffic_gbs"] - roof["traffic"] / roof["launch_us"] / 1e3) < 1e-6
    for pc in (roof["launch_us_percentiles"], line["step_us_percentiles"]):
        assert 0 < pc["p10"] <= pc["p50"] <= pc["p90"]
    if name == "tiny":
        cb = line["cpu_baseline"]
        assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] > 0 and cb["cpu"]
        if cb["cores"] > 1:
            assert cb["one_thread"]["value"] > 0
    d = np.load(path)
    assert str(d["workload"]) == name and json.loads(str(d["plan"]))["variant"] == 2
    # the workloads draw from the device's own generator: regenerate on the
    # device the bench ran on, then compare on the host
    w = workloads.make(name, device="cuda:0").to("cpu")
    ref = oracle.decode_attn(w.q, w.k_pages, w.v_pages, w.page_table, w.seq_lens, w.scale,
                             w.window)
    got = d["out"].astype(np.float64).reshape(ref.shape)
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert rel <= 5e-4 and np.abs(got - ref).max() <= 2e-3, rel


def test_context_sweep_runs(gpu):
    lines = run_bench("--context-sweep", "--steps", "10")
    points = [l for l in lines if "context" in l]
    assert len(points) == 15 * 3 * 3
    for p in points:
        assert p["us_per_step_median"] > 0
        # the default threshold: single pass up to 256 positions, split above
        if p["mode"] == "threshold 256" and p["context"] > 1:
            assert p["split"] == (1 if p["context"] > 256 else 0), p
    assert "summary_mean_us" in lines[-1]


def test_per_config_block_and_reference_config(gpu):
    """The default line carries every other benchmark configuration, timed the
    same way, and the reference arm names the same configuration dict."""
    (line,) = run_bench("--workload", "tiny", "--steps", "5", "--warmup", "3", "--e2e-steps",
                        "0", "--no-cpu-baseline", "--config-steps", "10")
    pc = line["per_config"]
    assert set(pc) == {"llama", "sweep_d64", "sweep_d128", "sweep_d256", "batched", "long_w4096"}
    peak = line["roofline"]["peak"]
    for name, e in pc.items():
        assert e["us_per_step"] > 0 and e["steps"] == 10, name
        assert abs(e["frac"] - e["kv_tbs"] * 1e3 / peak) < 1e-9, name
        assert e["kv_tbs"] * 1e12 * e["us_per_step"] * 1e-6 == pytest.approx(e["kv_bytes_per_step"],
                                                                           rel=1e-9)
        assert e["kernel"].startswith("split_mma_kernel"), name
        assert 0 < e["us_percentiles"]["p10"] <= e["us_percentiles"]["p90"]
    (ref,) = run_bench("--impl", "reference", "--workload", "tiny", "--steps", "1", "--warmup",
                       "0")
    assert ref["impl"] == "reference" and ref["config"] == line["config"]
