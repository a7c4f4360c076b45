"""bench.py's reference arm (the fp64 oracle on the host cores) runs without a GPU
and prints one JSON line with the keys the measurement contract fixes."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

KEYS = {"metric", "value", "unit", "impl", "n_gpus", "steps", "warmup", "ms_per_step",
        "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
        "cpu_baseline", "e2e"}


def test_reference_arm_prints_one_contract_line():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    out = json.loads(lines[0])
    assert KEYS <= set(out)
    assert out["impl"] == "reference" and out["unit"] == "tokens/s" and out["value"] > 0
    assert out["higher_is_better"] is True and out["vs_baseline"] is None
    assert out["config"]["workload"].startswith("packed training batch T=4096")
    cb, e2e = out["cpu_baseline"], out["e2e"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == out["value"]
    assert e2e["value"] == out["value"] and e2e["h2d_bytes_per_step"] == 0
    assert e2e["d2h_bytes_per_step"] == 0
