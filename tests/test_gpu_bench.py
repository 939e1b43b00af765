"""bench.py's prefill arm on a small stack: one JSON line with the contract's keys.

The metric pass replays one captured step (a CUDA graph of every layer's gdn_layer launches), and
the line says so; with --no-graph the same stack is timed from direct launches.  Both lines carry
the contract's keys, the launch count of the timed region and a roofline record.
"""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
KEYS = ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
        "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e", "gpu_launches", "clocks")


def _line(*extra):
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--layers", "2", "--steps", "2", "--warmup", "3",
           "--no-e2e", "--no-cpu-baseline", *extra]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout[-3000:]
    return json.loads(lines[0])


@pytest.mark.parametrize("graph", [True, False], ids=["graph", "direct"])
def test_bench_prefill_line(graph):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    line = _line() if graph else _line("--no-graph")
    for key in KEYS:
        assert key in line, key
    assert line["config"]["launch"] == ("cuda graph of one step, replayed" if graph else "direct")
    assert line["steps"] == 2 and line["warmup"] == 3 and line["n_gpus"] == 1
    assert line["gpu_launches"] == 5 * 2 * 2  # pre, gram, prep, chain, post per layer and step
    assert line["value"] > 0 and line["ms_per_step"] > 0
    assert line["roofline"]["bound"] == "hbm" and 0 < line["roofline"]["frac"] < 2
    assert set(line["clocks"]) >= {"sm_mhz", "sm_max_mhz", "reasons"}
