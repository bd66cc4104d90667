"""bench.py's reference arm on the host cores: one JSON line with the fields of the bench
contract (the oracle timed on a bounded sample of the default workload), and the argument
checks of the timing rules.  No GPU."""

from __future__ import annotations

import json
import subprocess
import sys
from pathlib import Path

ROOT = Path(__file__).resolve().parents[1]


def run_bench(*args, timeout=600):
    return subprocess.run([sys.executable, str(ROOT / "bench.py"), *args], cwd=ROOT,
                          capture_output=True, text=True, timeout=timeout)


def test_reference_arm_prints_one_contract_line():
    r = run_bench("--impl", "reference", "--steps", "1", "--warmup", "3")
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config"):
        assert key in d, key
    assert d["impl"] == "reference"
    assert d["n_gpus"] == 1 and d["steps"] == 1 and d["warmup"] == 3
    assert d["unit"] == "GB/s" and d["higher_is_better"] is True and d["value"] > 0
    assert d["config"]["workload"] == "mix64"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0


def test_timing_rules_are_enforced_on_the_command_line():
    r = run_bench("--impl", "reference", "--steps", "1", "--warmup", "2")
    assert r.returncode != 0 and "--warmup must be >= 3" in r.stderr


def test_traffic_key_ignores_comments_and_tracks_code(tmp_path, monkeypatch):
    """roofline.traffic is keyed by a hash of the decode sources: editing a comment keeps the
    hash, editing code changes it (so a stale ncu capture is reported as null, never as current)."""
    import shutil
    sys.path.insert(0, str(ROOT))
    import bench
    base = bench.kernel_source_hash()
    fake = tmp_path / "paged_kv_cache_244_gb300" / "csrc"
    fake.mkdir(parents=True)
    for name in ("paged_decode.cu", "pa_device.cuh", "pa_launch.h"):
        shutil.copy(ROOT / "paged_kv_cache_244_gb300" / "csrc" / name, fake / name)
    monkeypatch.setattr(bench, "ROOT", tmp_path)
    assert bench.kernel_source_hash() == base
    src = fake / "paged_decode.cu"
    src.write_text(src.read_text() + "\n// a comment\n/* and a block comment */\n")
    assert bench.kernel_source_hash() == base
    src.write_text(src.read_text() + "\nconstexpr int kUnused = 1;\n")
    assert bench.kernel_source_hash() != base
