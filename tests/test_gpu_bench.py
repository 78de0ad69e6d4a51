"""bench.py on the GPU: one JSON line with the contract's keys, for a
one-shape workload (with the oracle's CPU baseline) and for a slice of the
7B-class stack (several shapes, the group's host I/O over several chunks)."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
KEYS = {"metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
        "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e", "gpu_launches", "clocks"}


def _run(args):
    env = dict(os.environ)
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK", "MUON_TUNE_CACHE"):
        env.pop(k, None)
    out = subprocess.run([sys.executable, "bench.py"] + args, cwd=ROOT, env=env, capture_output=True, text=True,
                         timeout=900)
    assert out.returncode == 0, out.stderr[-3000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, out.stdout[-3000:]
    return json.loads(lines[0])


def _common(d, workload):
    assert KEYS <= set(d), KEYS - set(d)
    assert d["config"]["workload"] == workload
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["n_gpus"] == 1 and d["warmup"] >= 3
    assert d["gpu_launches"] > 0
    r = d["roofline"]
    assert {"bound", "achieved", "peak", "unit", "frac", "traffic"} <= set(r)
    assert r["achieved"] > 0 and r["peak"] > 0 and abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-9
    e = d["e2e"]
    assert e["unit"] == d["unit"] and e["value"] > 0 and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    c = d["clocks"]
    assert c is None or {"sm_mhz", "sm_max_mhz", "reasons"} <= set(c)


def test_bench_line_fp32_workload():
    d = _run(["--workload", "single_256x1024_f32", "--steps", "3", "--warmup", "3"])
    _common(d, "single_256x1024_f32")
    assert d["roofline"]["bound"] == "alu"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] > 0 and cb["cores"] >= 1 and cb["unit"] == d["unit"]
    assert d["e2e"]["h2d_bytes_per_step"] == 256 * 1024 * 4


def test_bench_line_stack_slice():
    d = _run(["--slice", "64", "--steps", "3", "--warmup", "3", "--no-cpu-baseline"])
    _common(d, "stack_32L_7b_bf16_f32mom/slice64")
    assert d["config"]["matrices"] == 4 and d["roofline"]["bound"] == "tensor"
    # every gradient in and every weight out: bf16, the four shapes once each
    elems = 4096 * 4096 + 1024 * 4096 + 2 * 14336 * 4096
    assert d["e2e"]["h2d_bytes_per_step"] == 2 * elems == d["e2e"]["d2h_bytes_per_step"]
    assert set(d["config"]["ns_paths"]) == {"4096x4096", "1024x4096", "4096x14336"}
