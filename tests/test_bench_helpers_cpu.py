"""bench.py's host-side helpers, without a GPU: the workload slice used for
profiling runs, the distinct caller shapes the CPU baseline extrapolates
from, and the scaling of a traffic figure measured on a slice to one launch
of the full workload."""
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    sys.argv = ["bench.py"]
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    import bench as b
    return b


def test_slice_keeps_shape_proportions(bench):
    from workloads import WORKLOADS
    wl = WORKLOADS["stack_32L_7b_bf16_f32mom"]
    s = bench._sliced(wl, 32)
    assert [(r, c, k) for r, c, k in s.shapes] == [(4096, 4096, 2), (1024, 4096, 2), (14336, 4096, 2), (4096, 14336, 1)]
    assert s.count == 7 and s.name.endswith("/slice32")
    assert bench._sliced(wl, 1) is wl
    # a divisor larger than a count keeps one matrix of that shape
    assert all(k == 1 for _, _, k in bench._sliced(wl, 1000).shapes)


def test_distinct_shapes_cover_every_matrix(bench):
    from workloads import WORKLOADS
    for name in ("stack_32L_7b_bf16_f32mom", "stack_24L_h2048_bf16", "bucket_512_small_bf16", "single_2560x9728_bf16"):
        wl = WORKLOADS[name]
        shapes = bench._distinct_shapes(wl)
        assert sum(k for _, _, _, k in shapes) == wl.count
        assert len({(r, c) for _, r, c, _ in shapes}) == len(shapes)
        first = {}
        for idx, r, c in wl.matrices():
            first.setdefault((r, c), idx)
        for idx, r, c, _ in shapes:
            assert first[(r, c)] == idx


def test_oracle_path_follows_the_gpu_choice(bench):
    assert bench._oracle_path(4096, 14336) == "gram"
    assert bench._oracle_path(14336, 4096) == "gram"
    assert bench._oracle_path(4096, 4096) == "plain"
    assert bench._oracle_path(1024, 4096, {"1024x4096": "plain"}) == "plain"


def test_traffic_scales_from_the_slice(bench, tmp_path, monkeypatch):
    """An entry measured on a 1/D slice holds the instance's DRAM bytes per
    step of the slice; one launch of the full workload is D times that over
    the instance's launches per step.  A changed kernel source voids it."""
    prof = tmp_path / "profiles"
    prof.mkdir()
    h = bench._kernel_hash()
    (prof / "ncu_traffic.json").write_text(json.dumps({"entries": [
        {"workload": "w", "instance": "symmetric", "kernel_hash": h, "slice": 32,
         "dram_bytes_per_step_of_slice": 6.0e9},
        {"workload": "w", "instance": "apply", "kernel_hash": "0" * 16, "slice": 32,
         "dram_bytes_per_step_of_slice": 4.0e9},
        {"workload": "v", "instance": "symmetric", "kernel_hash": h, "dram_bytes_per_launch": 2.5e7}]}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "_kernel_hash", lambda: h)
    monkeypatch.setattr(bench, "WORKLOAD_SEL", ["w"])
    assert bench._measured_traffic("gemm_tc_kernel symmetric products (...)", 128) == pytest.approx(6.0e9 * 32 / 128)
    assert bench._measured_traffic("gemm_tc_kernel long apply QX", 36) is None        # other kernel sources
    assert bench._measured_traffic("small_ns_kernel (fused small matrices)", 1) is None
    monkeypatch.setattr(bench, "WORKLOAD_SEL", ["v"])
    assert bench._measured_traffic("gemm_tc_kernel symmetric products (...)", 10) == pytest.approx(2.5e7)
