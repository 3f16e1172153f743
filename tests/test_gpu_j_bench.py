"""bench.py's own arm prints the one JSON line of the measurement contract
(run on the tiny workload so it takes seconds)."""
import json
import subprocess
import sys
from pathlib import Path

import pytest

pytestmark = pytest.mark.gpu
ROOT = Path(__file__).resolve().parents[1]


def test_bench_prints_one_contract_line():
    r = subprocess.run([sys.executable, "bench.py", "--workload", "tiny", "--steps", "3", "--warmup", "3",
                        "--no-cpu-baseline"], cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1
    j = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "clocks", "gpu_launches", "e2e"):
        assert key in j, key
    assert j["unit"] == "tokens/s" and j["higher_is_better"] is True and j["scaling"] == "weak"
    assert j["value"] > 0 and j["steps"] == 3 and j["warmup"] == 3 and j["n_gpus"] == 1
    assert j["gpu_launches"] > 0 and j["config"]["workload"].startswith("tiny")
    rl = j["roofline"]
    for key in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert key in rl, key
    assert rl["bound"] == "tensor" and rl["unit"] == "TFLOP/s" and abs(rl["frac"] - rl["achieved"] / rl["peak"]) < 1e-9
    for key in ("sm_mhz", "sm_max_mhz", "reasons"):
        assert key in j["clocks"], key
    e = j["e2e"]
    assert e["unit"] == "tokens/s" and e["value"] > 0
    assert e["h2d_bytes_per_step"] == e["d2h_bytes_per_step"] == 256 * 512 * 2


def test_graft_entry_smoke_runs_the_layer_on_cuda0():
    # the entry point's smoke(): one tiny forward through libmoe checked against the oracle
    r = subprocess.run([sys.executable, "-c", "import __graft_entry__ as g; g.smoke()"], cwd=ROOT,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    assert "smoke ok" in r.stdout
