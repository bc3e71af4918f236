"""Host-side parts of bench.py that need no GPU: the reference arm (the
float64 oracle timed on the host cores) and its JSON line, the non-zero
ranks of a torchrun launch, and the helpers behind the roofline fields."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _run(args, env_extra=None):
    env = dict(os.environ)
    env.update(env_extra or {})
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                       capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0, r.stderr
    return r.stdout


def test_reference_arm_prints_the_contract_line():
    out = _run(["--impl", "reference", "--workload", "b1_t64", "--steps", "2", "--warmup", "3",
                "--reference-windows", "1"])
    lines = [l for l in out.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "windows/s" and d["value"] > 0
    assert d["metric"] == bench.METRIC and d["higher_is_better"] is True
    assert d["steps"] == 2 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["config"]["workload"] == "b1_t64"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "windows/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_reference_arm_other_ranks_do_no_work():
    out = _run(["--impl", "reference", "--workload", "b1_t64", "--steps", "2", "--warmup", "3"],
               {"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert out.strip() == ""


def test_warmup_below_three_is_refused():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--warmup", "2"],
                       cwd=ROOT, capture_output=True, text=True, timeout=120)
    assert r.returncode != 0 and "warmup" in r.stderr


def test_flop_counts():
    # 2 * rows * 1024 * K over the four layers' K = 60, 256, 256, 256
    assert bench.flops_projection(10) == 2.0 * 10 * 1024 * (60 + 3 * 256)
    # the 512 x 128 matrix-vector product per window, step and direction (one
    # launch runs both directions)
    assert bench.flops_recurrence_launch(3, 7) == 2.0 * 3 * 7 * 512 * 128 * 2
    assert bench.flops_recurrence_launch(3, 7, directions=1) == 2.0 * 3 * 7 * 512 * 128
    assert bench.flops_heads(5) == 2.0 * 5 * (256 * 128 + 128 * 128 + 128 * 7)


def test_ncu_traffic_scales_with_rows_and_tracks_the_source(tmp_path, monkeypatch):
    rec = json.load(open(os.path.join(ROOT, "profiles", "ncu_traffic.json")))["recurrence"]
    got = bench.ncu_traffic("recurrence", 2 * rec["rows"])
    import hashlib
    sha = hashlib.sha256(open(os.path.join(ROOT, rec["source"]), "rb").read()).hexdigest()[:16]
    if sha == rec["sha256_16"]:
        assert got == pytest.approx(2 * (rec["dram_read_bytes"] + rec["dram_write_bytes"]))
    else:
        assert got is None
    assert bench.ncu_traffic("no_such_kernel", 100) is None
