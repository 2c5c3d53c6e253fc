"""The JSON line of bench.py's reference arm (the CPU oracle timed on the host, no GPU
needed): one line on stdout with the contract's keys, its value carried into
cpu_baseline and e2e, and no host-device transfers."""

import json
import subprocess
import sys
from pathlib import Path

REPO = Path(__file__).resolve().parent.parent

TOP_KEYS = {"impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
            "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
            "cpu_baseline", "e2e"}


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], cwd=REPO, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert TOP_KEYS <= set(line)
    assert line["impl"] == "reference" and line["n_gpus"] == 1
    assert (line["steps"], line["warmup"]) == (1, 0)
    assert line["higher_is_better"] is True and line["vs_baseline"] is None
    assert line["value"] > 0 and line["unit"] == "GB/s"
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"]
    assert cb["value"] == line["value"] and cb["unit"] == line["unit"]
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["unit"] == line["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
    assert "workload" in line["config"] and line["sample"]
    # the same config dict as the GPU arm's decode-step line, and a measured step time
    sys.path.insert(0, str(REPO))
    import bench

    assert line["config"] == bench.decode_config(1)
    assert line["ms_per_step"] > 0 and line["ms_per_full_step_extrapolated"] > line["ms_per_step"]


def test_reference_arm_other_workloads():
    for wl in ("gemv_94mb", "rmsnorm_big"):
        r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", wl,
                            "--steps", "1", "--warmup", "0"], cwd=REPO, capture_output=True,
                           text=True, timeout=300)
        assert r.returncode == 0, r.stderr
        line = json.loads(r.stdout.strip().splitlines()[-1])
        assert line["impl"] == "reference" and line["value"] > 0
        assert line["config"]["workload"] == wl


def test_reference_arm_persistent_step_is_unavailable():
    # the one-launch step computes exactly the decode step, whose oracle arm is decode_step
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload",
                        "persistent_step", "--steps", "1", "--warmup", "0"], cwd=REPO,
                       capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and "decode_step" in line["unavailable"]
