"""bench.py on the host: the reference arm (the CPU oracle timed on a bounded
sample) prints one JSON line with the contract's keys (CPU only, tiny workload)."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_json_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "tiny",
                          "--steps", "2", "--warmup", "0", "--cpu-seconds", "1"],
                         cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    assert len(lines) == 1, out.stdout
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["unit"] == "tokens/s" and d["higher_is_better"] is True
    assert d["value"] > 0 and d["steps"] == 2 and d["n_gpus"] == 1
    assert "workload" in d["config"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    # the same config dict the GPU arm prints for these arguments (batch 1: the context by prefill)
    sys.path.insert(0, ROOT)
    import bench
    import synth
    cfg = synth.CONFIGS["tiny"]
    assert d["config"] == bench.arm_config(cfg, cfg.ctx, 2, len(cfg.fence) - 1, 1, "prefill", True)


def test_fill_resolution():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.resolve_fill("auto", 1, 0) == "prefill"
    assert bench.resolve_fill("auto", 8, 0) == "synthetic"
    assert bench.resolve_fill("auto", 8, 8) == "synthetic"  # verify rows: batch = rows of one sequence
    assert bench.resolve_fill("decode", 1, 0) == "decode"
