"""bench.py's reference arm (the oracle on the host cores) on CPU: one JSON
line with the contract's keys, for one-shape and several-shape Muon workloads
and the AdamW one."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
KEYS = {"impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
        "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"}


@pytest.mark.parametrize("workload", ["single_256x1024_f32", "bucket_512_small_bf16", "adamw_nonmatrix_7b"])
def test_reference_arm_json_line(workload):
    env = dict(os.environ)
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        env.pop(k, None)
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", workload,
                          "--steps", "1", "--warmup", "0"], cwd=ROOT, env=env, capture_output=True, text=True,
                         timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, out.stdout
    d = json.loads(lines[0])
    assert KEYS <= set(d), KEYS - set(d)
    # the timing rules ask for at least three warm-up steps: a smaller W is raised
    # a workload of several shapes runs every shape at least once
    nshapes = 2 if workload == "bucket_512_small_bf16" else 1
    assert d["impl"] == "reference" and d["steps"] == nshapes and d["warmup"] == 3
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["config"]["workload"] == workload
    if nshapes > 1:
        # extrapolated from one matrix per shape to the workload's 512 matrices
        assert d["cpu_baseline"]["extrapolated"] is True
        assert d["config"]["matrices"] == 512
        assert sorted(d["config"]["shapes"]) == [[128, 512, 256], [256, 256, 256]]
