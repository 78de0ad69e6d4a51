"""Benchmark of the Muon update hot path on GB300.

One step = one full Muon update (momentum, Frobenius normalisation,
Newton-Schulz with the path chosen by the measured-cost autotune, shape-scaled
decoupled-decay update) of every matrix of the workload, through the C ABI's
persistent group (muon_group_step, the optimizer object of a training loop),
with parameters, momentum and gradient resident in HBM.  L2 is flushed (256 MiB
write) between timed steps, outside the per-step CUDA events.

The default workload is the largest one that fits one GPU: the 32-layer
7B-class stack (hidden 4096, FFN 14336, 8 KV heads of dim 128; 224 bf16
matrices, fp32 momentum, about 7e9 parameters).  --workload selects another
(the single 2560x9728 matrix, the 512-matrix small bucket, the 24-layer stack,
the fp32 and fp16 cases, AdamW, packing); --slice D keeps 1/D of every shape
of a stack (for profiling runs that must stay small).

Usage:  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
                        [--workload NAME] [--slice D] [--no-cpu-baseline]
Under torchrun each rank runs its own replica of the workload (the matrices
are independent units; no collective on the data path) and rank 0 prints one
JSON line with the whole-job throughput.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "Muon-step matrices/s and NS TFLOP/s (fraction of GB300 dense BF16 peak)"
UNIT = "matrices/s"
WORKLOAD = "stack_32L_7b_bf16_f32mom"
L2_FLUSH_BYTES = 256 << 20


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def combine_over_ranks(local_ms, dist, device):
    """Slowest rank's step time (the job's step time); local value when not distributed."""
    if dist is None:
        return float(local_ms)
    import torch
    t = torch.tensor([float(local_ms)], device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(matrices_per_rank, world, step_ms):
    """Whole-job matrices/s: every rank runs its own replica of the workload."""
    return world * matrices_per_rank / (step_ms * 1e-3)


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the GPU works."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.path = os.path.join("/tmp", f"muon_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(self.dev)], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None

        def num(x):
            try:
                return float(x)
            except ValueError:
                return float("nan")

        sm = [num(r[1]) for r in rows]
        smax = max(num(r[2]) for r in rows)
        busy = [s for s in sm if s > 0.5 * smax] or sm
        reasons = set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for r in rows:
            for nm, v in zip(names, r[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(busy), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(rows), "power_w_max": max(num(r[3]) for r in rows)}


def _pinned_like(torch, tensors, copy):
    """Host copies of `tensors` as views of ONE pinned allocation per dtype.
    On the GB300 machines the copy engines read a single large pinned block at
    the full host link rate more reliably than hundreds of separately pinned
    buffers (measured: after earlier processes on a box, first passes over
    224 separate 128 MB buffers ran at 66-142 GB/s, one 28 GB block at
    152-210 GB/s)."""
    out = [None] * len(tensors)
    by_dtype = {}
    for i, t in enumerate(tensors):
        by_dtype.setdefault(t.dtype, []).append(i)
    for dt, idxs in by_dtype.items():
        total = sum(tensors[i].numel() for i in idxs)
        block = torch.empty(total, dtype=dt).pin_memory()
        off = 0
        for i in idxs:
            n = tensors[i].numel()
            v = block[off:off + n].view(tensors[i].shape)
            if copy:
                v.copy_(tensors[i])
            out[i] = v
            off += n
    return out


def _gen_inputs(torch, wl, device):
    """Seeded generator bytes for every matrix of the workload, moved to the device."""
    import numpy as np
    from workloads import gen_matrix, zeros_matrix
    params, grads, moms, host_grads = [], [], [], []
    for idx, r, c in wl.matrices():
        seed = wl.seed(idx)
        W = gen_matrix(seed, 1, r, c, wl.weight_std, wl.param_dtype)
        G = gen_matrix(seed, 0, r, c, wl.grad_std, wl.param_dtype)
        M = zeros_matrix(r, c, wl.mom_dtype)

        def dev(h):
            if h.dtype == "f32":
                return torch.from_numpy(np.ascontiguousarray(h.data)).to(device)
            t16 = torch.float16 if h.dtype == "f16" else torch.bfloat16
            return torch.from_numpy(np.ascontiguousarray(h.data).view(np.int16)).to(device).view(t16)

        params.append(dev(W))
        grads.append(dev(G))
        moms.append(dev(M))
        host_grads.append(G)
    return params, grads, moms, host_grads


def _blas_threads():
    """Threads of numpy's BLAS pool, where the oracle's matrix products run."""
    try:
        from threadpoolctl import threadpool_info
        n = [d["num_threads"] for d in threadpool_info() if d.get("user_api") == "blas"]
        if n:
            return max(n)
    except Exception:
        pass
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        try:
            return max(1, int(os.environ[var]))
        except (KeyError, ValueError):
            pass
    return os.cpu_count()


# numpy's elementwise operations and copies run on one thread
ELEMENTWISE_THREADS = 1


def _oracle_path(r, c, paths=None):
    """NS path the oracle runs for a caller shape: the one the GPU run chose
    (paths from muon_last_path), else Gram for rectangular and plain for
    square shapes (what the autotune picks for every workload shape)."""
    m, n = min(r, c), max(r, c)
    if paths and f"{m}x{n}" in paths:
        return paths[f"{m}x{n}"]
    return "gram" if n > m else "plain"


def _distinct_shapes(wl):
    """One entry per distinct caller shape of the workload, in parameter
    order: (index of its first matrix, rows, cols, matrices of that shape)."""
    out = {}
    for idx, r, c in wl.matrices():
        if (r, c) not in out:
            out[(r, c)] = [idx, 0]
        out[(r, c)][1] += 1
    return [(v[0], r, c, v[1]) for (r, c), v in out.items()]


class _OracleCase:
    """Generator bytes of one matrix of the workload and one full Muon step of
    the fp64 oracle on them (inputs made once, outside any timing)."""

    def __init__(self, wl, idx, r, c, path):
        from workloads import gen_matrix, zeros_matrix
        seed = wl.seed(idx)
        self.wl, self.r, self.c, self.path = wl, r, c, path
        self.W = gen_matrix(seed, 1, r, c, wl.weight_std, wl.param_dtype)
        self.G = gen_matrix(seed, 0, r, c, wl.grad_std, wl.param_dtype)
        self.M = zeros_matrix(r, c, wl.mom_dtype)

    def step(self):
        from oracle import muon_oracle as orc
        wl = self.wl
        t0 = time.perf_counter()
        orc.muon_step(self.W.data, self.M.data, self.G.data, lr=wl.lr, beta=wl.beta, wd=wl.wd,
                      nesterov=wl.nesterov, path=self.path, param_dtype=wl.param_dtype, mom_dtype=wl.mom_dtype,
                      segments=tuple(wl.extra.get("segments", (2, 2, 1))))
        return time.perf_counter() - t0


def run_cpu_baseline(wl, paths=None, max_seconds=30.0):
    """The fp64 oracle as it stands, timed on the host cores on a bounded sample.

    One-shape workloads: full Muon steps of the workload's first matrix, as
    many as fit in about max_seconds (at most three).  Workloads of several
    shapes (the transformer stacks): one full Muon step of one matrix of every
    distinct shape, extrapolated to the workload by its per-shape counts."""
    shapes = _distinct_shapes(wl)
    if len(shapes) == 1:
        idx, r, c, _ = shapes[0]
        case = _OracleCase(wl, idx, r, c, _oracle_path(r, c, paths))
        done, el = 0, 0.0
        while True:
            el += case.step()
            done += 1
            if el * (done + 1) / done > max_seconds or done >= 3:
                break
        return {"value": wl.count * done / el, "unit": UNIT, "cores": _blas_threads(), "kind": "oracle",
                "sample": f"{done} full Muon step(s) of one {r}x{c} {wl.param_dtype} matrix, {case.path} NS, "
                          f"numpy fp64 (BLAS threads = host cores)", "seconds": el}
    parts, total_s, el = [], 0.0, 0.0
    for idx, r, c, k in shapes:
        case = _OracleCase(wl, idx, r, c, _oracle_path(r, c, paths))
        t = case.step()
        el += t
        total_s += k * t
        parts.append(f"{k} x {r}x{c} {case.path} {t:.2f} s")
    return {"value": wl.count / total_s, "unit": UNIT, "cores": _blas_threads(), "kind": "oracle",
            "extrapolated": True,
            "sample": "extrapolated: one full Muon step of one matrix of every distinct shape "
                      f"(numpy fp64, BLAS threads = host cores), times the workload's counts: {'; '.join(parts)}; "
                      f"projected {total_s:.1f} s for all {wl.count} matrices",
            "seconds": el}


def bench_reference(args):
    """--impl reference: the oracle as it stands on the host cores, same metric.

    A step is one full Muon update of one matrix by the fp64 oracle.  The
    timed steps cycle through the workload's distinct shapes (every shape at
    least once, even when --steps is smaller), and the value extrapolates the
    mean time per shape to the whole workload by its per-shape counts.  The
    warm-up steps run the cheapest shape."""
    world, rank, _ = _dist()
    if rank != 0:
        return 0
    if args.workload == ADAMW_WORKLOAD:
        return bench_reference_adamw(args)
    if args.workload == PACK_WORKLOAD:
        return bench_reference_pack(args)
    from workloads import WORKLOADS
    wl = _sliced(WORKLOADS[args.workload], args.slice)
    shapes = _distinct_shapes(wl)
    cases = [_OracleCase(wl, idx, r, c, _oracle_path(r, c)) for idx, r, c, _ in shapes]
    cheapest = min(range(len(cases)), key=lambda i: cases[i].r * cases[i].c)
    for _ in range(args.warmup):
        cases[cheapest].step()
    nsteps = max(args.steps, len(cases))
    times = [[] for _ in cases]
    el = 0.0
    for i in range(nsteps):
        t = cases[i % len(cases)].step()
        times[i % len(cases)].append(t)
        el += t
    per_shape = [sum(ts) / len(ts) for ts in times]
    total_s = sum(k * t for (_, _, _, k), t in zip(shapes, per_shape))
    value = wl.count / total_s
    if len(cases) == 1:
        sample = (f"one full Muon step of one {cases[0].r}x{cases[0].c} matrix per step ({cases[0].path} NS, "
                  f"numpy fp64), scaled to the workload's {wl.count} matrices")
    else:
        sample = ("one full Muon step of one matrix per step, cycling through the distinct shapes "
                  + "; ".join(f"{k} x {r}x{c} {cs.path} {t:.2f} s" for (_, r, c, k), cs, t in
                              zip(shapes, cases, per_shape))
                  + f" (mean per step); extrapolated to all {wl.count} matrices by the per-shape counts")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": nsteps, "warmup": args.warmup, "ms_per_step": 1e3 * el / nsteps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic: seeded SplitMix64/Box-Muller generator bytes (workloads.py)",
            "config": {"workload": wl.name, "matrices": wl.count,
                       "shapes": [[r, c, k] for _, r, c, k in shapes],
                       "ns_paths": {f"{min(cs.r, cs.c)}x{max(cs.r, cs.c)}": cs.path for cs in cases}},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": _blas_threads(), "kind": "oracle",
                             "extrapolated": len(cases) > 1, "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def _sliced(wl, div):
    """The workload with every shape's count divided by div (at least one
    matrix each), for profiling runs that must hold only a few GB."""
    if not div or div <= 1:
        return wl
    import dataclasses
    shapes = [(r, c, max(1, k // div)) for r, c, k in wl.shapes]
    return dataclasses.replace(wl, shapes=shapes, name=f"{wl.name}/slice{div}")


def _kernel_hash():
    import hashlib
    h = hashlib.sha256()
    for f in ("gemm_tc.cu", "epilogue.cuh", "muon_internal.cuh"):
        with open(os.path.join(ROOT, "newton_schulz_frobenius_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def _instance_of(kernel_key):
    """Short name of a kernel instance group, as profiles/ncu_traffic.json keys it."""
    for prefix, name in (("gemm_tc_kernel symmetric", "symmetric"), ("gemm_tc_kernel long apply", "apply"),
                         ("small_ns_kernel", "small"), ("gemm_simt_kernel", "simt"), ("adamw", "adamw")):
        if kernel_key.startswith(prefix):
            return name
    return kernel_key


def _measured_traffic(kernel_key, launches_per_step=None):
    """Per-launch DRAM bytes (read + write) of the dominant kernel instance from
    the committed ncu summary, or None when absent or taken on different
    kernel sources.  An entry measured on a slice of the workload (1/D of
    every shape) holds the instance's DRAM bytes per step of the slice; the
    full workload's per-launch figure is that times D over the instance's
    launches per step here (traffic taken to grow with the matrices processed)."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
        inst = _instance_of(kernel_key)
        for e in d.get("entries", []):
            if e.get("instance") != inst or e.get("workload") != WORKLOAD_SEL[0]:
                continue
            if e.get("kernel_hash") != _kernel_hash():
                return None
            if "dram_bytes_per_launch" in e:
                return float(e["dram_bytes_per_launch"])
            if launches_per_step:
                return float(e["dram_bytes_per_step_of_slice"]) * float(e["slice"]) / float(launches_per_step)
    except Exception:
        pass
    return None


WORKLOAD_SEL = [WORKLOAD]


def _gen_device_inputs(torch, wl, device):
    """Large stacks: seeded device RNG (same distributions), no host round trip."""
    g = torch.Generator(device=device).manual_seed(1000 * wl.config_id)
    tdt = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}
    pdt, mdt = tdt[wl.param_dtype], tdt[wl.mom_dtype]
    params, grads, moms = [], [], []
    for _, r, c in wl.matrices():
        params.append((torch.randn((r, c), generator=g, device=device) * wl.weight_std).to(pdt))
        grads.append((torch.randn((r, c), generator=g, device=device) * wl.grad_std).to(pdt))
        moms.append(torch.zeros((r, c), device=device, dtype=mdt))
    return params, grads, moms


ADAMW_WORKLOAD = "adamw_nonmatrix_7b"


ADAMW_SIZES = [32000 * 4096, 32000 * 4096] + [4096] * 65
ADAMW_HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, wd=0.01)


def adamw_cpu_baseline(max_seconds=20.0):
    """The fp64 AdamW oracle as it stands on the host cores, on a bounded
    sample: consecutive 4M-element slices of the embedding table."""
    import numpy as np
    from oracle import adamw_oracle as ad
    from workloads import gen_matrix, zeros_matrix
    n = 1 << 22
    P = gen_matrix(4242, 1, 1, n, 0.02, "bf16").data.reshape(-1)
    G = gen_matrix(4242, 0, 1, n, 1e-3, "bf16").data.reshape(-1)
    M = zeros_matrix(1, n, "f32").data.reshape(-1)
    V = zeros_matrix(1, n, "f32").data.reshape(-1)
    done, t0 = 0, time.perf_counter()
    while True:
        r = ad.adamw_step(P, G, M, V, step=done + 1, param_dtype="bf16", state_dtype="f32", **ADAMW_HP)
        M, V = r["m_new"].astype(np.float32), r["v_new"].astype(np.float32)
        done += 1
        el = time.perf_counter() - t0
        if el * (done + 1) / done > max_seconds or done >= 8:
            break
    return {"value": 22.0 * n * done / el / 1e9, "unit": "GB/s", "cores": ELEMENTWISE_THREADS, "kind": "oracle",
            "sample": f"{done} AdamW step(s) over {n} bf16 parameters with fp32 moments (numpy fp64), "
                      f"22 algorithmic bytes per element", "seconds": el}


def bench_reference_adamw(args):
    """--impl reference for the AdamW workload: the fp64 oracle on 4M-element
    slices, one slice per step."""
    import numpy as np
    from oracle import adamw_oracle as ad
    from workloads import gen_matrix, zeros_matrix
    n = 1 << 22
    P = gen_matrix(4242, 1, 1, n, 0.02, "bf16").data.reshape(-1)
    G = gen_matrix(4242, 0, 1, n, 1e-3, "bf16").data.reshape(-1)
    M = zeros_matrix(1, n, "f32").data.reshape(-1)
    V = zeros_matrix(1, n, "f32").data.reshape(-1)
    t = 0

    def step():
        nonlocal t, M, V
        t += 1
        r = ad.adamw_step(P, G, M, V, step=t, param_dtype="bf16", state_dtype="f32", **ADAMW_HP)
        M, V = r["m_new"].astype(np.float32), r["v_new"].astype(np.float32)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = time.perf_counter() - t0
    value = 22.0 * n * args.steps / el / 1e9
    line = {"impl": "reference", "metric": "AdamW step over the non-matrix parameters (GB/s)", "value": value,
            "unit": "GB/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * el / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": ADAMW_WORKLOAD, "elements_per_step": n, "param_dtype": "bf16",
                       "state_dtype": "f32", "bytes_per_element": 22},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": ELEMENTWISE_THREADS, "kind": "oracle",
                             "sample": f"AdamW over {n} bf16 parameters per step (numpy fp64)"},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


PACK_WORKLOAD = "pack_7b_bf16"
PACK_RANKS = 8


def _pack_setup():
    """The 7B stack's 224 bf16 gradient matrices, owners for PACK_RANKS ranks
    by the owner planner, and the packed layout (16-byte starts)."""
    from workloads import WORKLOADS
    wl = WORKLOADS["stack_32L_7b_bf16_f32mom"]
    shapes = [(r, c) for _, r, c in wl.matrices()]
    return shapes


def pack_cpu_baseline(shapes, offsets, max_seconds=20.0):
    """The packing oracle (numpy) on the host cores, on a bounded sample: the
    first matrices of the layout, about 256 M elements per pass."""
    import numpy as np
    from oracle import pack_oracle as po
    take, n = [], 0
    for i, (m, c) in enumerate(shapes):
        if n + m * c > (1 << 28):
            break
        take.append(i)
        n += m * c
    mats = [np.zeros((shapes[i][0], shapes[i][1]), np.uint16) + np.uint16(i) for i in take]
    base = min(offsets[i] for i in take)
    end = max(offsets[i] + mats[k].size for k, i in enumerate(take))
    done, t0 = 0, time.perf_counter()
    while True:
        po.pack(mats, [offsets[i] - base for i in take], end - base)
        done += 1
        el = time.perf_counter() - t0
        if el * (done + 1) / done > max_seconds or done >= 5:
            break
    return {"value": 4.0 * n * done / el / 1e9, "unit": "GB/s", "cores": ELEMENTWISE_THREADS, "kind": "oracle",
            "sample": f"{done} pack(s) of the first {len(take)} matrices ({n} bf16 elements, read + write "
                      f"4 bytes per element) with the numpy packing oracle", "seconds": el}


def bench_reference_pack(args):
    """--impl reference for the pack workload: the numpy packing oracle on the
    bounded sample, one pack per step.  The layout is the oracle's, with
    owners round-robin (the owner choice moves the bytes, not their number)."""
    from oracle import pack_oracle as po
    shapes = _pack_setup()
    owners = [i % PACK_RANKS for i in range(len(shapes))]
    offsets, seg = po.layout(shapes, owners, PACK_RANKS, 8)
    cb = pack_cpu_baseline(shapes, offsets, max_seconds=5.0 * max(1, args.steps))
    value = cb["value"]
    line = {"impl": "reference", "metric": "packed exchange buffers: pack + unpack of the gradients (GB/s)",
            "value": value, "unit": "GB/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * cb["seconds"] / max(1, args.steps), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "u16", "data": "synthetic",
            "config": {"workload": PACK_WORKLOAD, "matrices": len(shapes), "ranks": PACK_RANKS},
            "cpu_baseline": {k: cb[k] for k in ("value", "unit", "cores", "kind", "sample")},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def bench_pack(args):
    """Packed exchange buffers for an 8-rank owner-centric step of the 7B
    stack: all 224 bf16 gradient matrices into the packed layout and back out,
    one launch each way.  HBM-bound: algorithmic bytes per element = 2 B read
    + 2 B written per direction = 8 B per step."""
    import torch
    torch.cuda.set_device(0)
    import __graft_entry__
    __graft_entry__.build()
    import newton_schulz_frobenius_gb300 as mg
    shapes = _pack_setup()
    owners, _, _, _ = mg.muon_owner_plan(shapes, PACK_RANKS)
    offsets, seg = mg.muon_pack_plan(shapes, owners, PACK_RANKS, 8)
    g = torch.Generator(device="cuda").manual_seed(777)
    mats = [torch.randn(s, generator=g, device="cuda").to(torch.bfloat16) for s in shapes]
    packed = torch.empty(PACK_RANKS * seg, dtype=torch.bfloat16, device="cuda")
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    elems = sum(m * n for m, n in shapes)
    nbytes = 8.0 * elems

    def step():
        mg.muon_pack(mats, offsets, packed, to_packed=True)
        mg.muon_pack(mats, offsets, packed, to_packed=False)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    clk = ClockSampler(0)
    clk.start()
    n0 = mg.muon_launch_count()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for i in range(args.steps):
        flush.zero_()
        evs[i][0].record()
        step()
        evs[i][1].record()
    torch.cuda.synchronize()
    launches = mg.muon_launch_count() - n0
    clocks = clk.stop()
    ms = sum(a.elapsed_time(b) for a, b in evs) / args.steps

    mg.muon_kernel_timing_read()
    mg.muon_set_kernel_timing(True)
    for _ in range(args.steps):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    mg.muon_set_kernel_timing(False)
    kl, kms, work = mg.muon_kernel_timing_read()["pack"]
    achieved = work / (kms * 1e-3) / 1e9

    # end to end: one rank's owned gradients H2D from pinned host, the two
    # launches, the same matrices D2H to pinned host
    mine = [i for i in range(len(shapes)) if owners[i] == 0]
    host = [mats[i].cpu().pin_memory() for i in mine]
    back = [torch.empty_like(h).pin_memory() for h in host]
    e2e_steps = max(3, min(args.steps, 10))
    eev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(e2e_steps)]
    for i in range(e2e_steps):
        flush.zero_()
        eev[i][0].record()
        for k, j in enumerate(mine):
            mats[j].copy_(host[k], non_blocking=True)
        step()
        for k, j in enumerate(mine):
            back[k].copy_(mats[j], non_blocking=True)
        eev[i][1].record()
    torch.cuda.synchronize()
    e2e_ms = sum(a.elapsed_time(b) for a, b in eev) / e2e_steps
    hbytes = sum(h.numel() * h.element_size() for h in host)

    peaks = _peaks()
    line = {"metric": "packed exchange buffers: pack + unpack of the gradients (GB/s)",
            "value": nbytes / (ms * 1e-3) / 1e9, "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "u16", "data": "synthetic: seeded torch device RNG",
            "config": {"workload": PACK_WORKLOAD, "matrices": len(shapes), "elements": elems, "ranks": PACK_RANKS,
                       "segment_elements": seg, "bytes_per_element": 8,
                       "l2": "flushed between timed steps (256 MiB device write outside the step events)"},
            "roofline": {"kernel": "pack_kernel", "bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                         "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"], "traffic": None, "launches": kl,
                         "peak_source": f"{peaks['source']} hbm_gbs"},
            "e2e": {"value": nbytes / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s", "h2d_bytes_per_step": hbytes,
                    "d2h_bytes_per_step": hbytes, "ms_per_step": e2e_ms,
                    "what": "rank 0's owned gradients H2D from pinned host, pack + unpack, the same D2H"},
            "gpu_launches": launches,
            "clocks": clocks}
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = {k: v for k, v in pack_cpu_baseline(shapes, offsets).items() if k != "seconds"}
    print(json.dumps(line), flush=True)
    return 0


def bench_adamw(args):
    """AdamW over the parameters a 7B-class model keeps off Muon: token
    embedding and output head (32000 x 4096 each, bf16), 65 RMSNorm vectors of
    4096 (bf16); fp32 moments.  HBM-bound: algorithmic bytes per element =
    read p, g (2+2) + read/write m, v (4+4+4+4) + write p (2) = 22."""
    import torch
    torch.cuda.set_device(0)
    import __graft_entry__
    __graft_entry__.build()
    import newton_schulz_frobenius_gb300 as mg
    g = torch.Generator(device="cuda").manual_seed(4242)
    sizes = ADAMW_SIZES
    P = [(torch.randn(n, generator=g, device="cuda") * 0.02).to(torch.bfloat16) for n in sizes]
    G = [(torch.randn(n, generator=g, device="cuda") * 1e-3).to(torch.bfloat16) for n in sizes]
    M = [torch.zeros(n, device="cuda") for n in sizes]
    V = [torch.zeros(n, device="cuda") for n in sizes]
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    t = 0

    def step():
        nonlocal t
        t += 1
        mg.muon_adamw_step(P, G, M, V, step=t, **ADAMW_HP)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    # timed pass (value): device events around each step, L2 flushed outside them
    clk = ClockSampler(0)
    clk.start()
    n0 = mg.muon_launch_count()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for i in range(args.steps):
        flush.zero_()
        evs[i][0].record()
        step()
        evs[i][1].record()
    torch.cuda.synchronize()
    launches = mg.muon_launch_count() - n0
    clocks = clk.stop()
    ms = sum(a.elapsed_time(b) for a, b in evs) / args.steps
    nbytes = 22.0 * sum(sizes)

    # instrumented pass: per-launch events on the library's stream
    mg.muon_kernel_timing_read()
    mg.muon_set_kernel_timing(True)
    for _ in range(args.steps):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    mg.muon_set_kernel_timing(False)
    kl, kms, work = mg.muon_kernel_timing_read()["adamw"]
    achieved = work / (kms * 1e-3) / 1e9

    # end to end: gradients H2D from pinned host, the step, parameters D2H to pinned host
    host_g = [x.cpu().pin_memory() for x in G]
    host_p = [torch.empty_like(x, device="cpu").pin_memory() for x in P]
    e2e_steps = max(3, min(args.steps, 10))
    eev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(e2e_steps)]
    for i in range(e2e_steps):
        flush.zero_()
        eev[i][0].record()
        for dg, hg in zip(G, host_g):
            dg.copy_(hg, non_blocking=True)
        step()
        for hp, dp in zip(host_p, P):
            hp.copy_(dp, non_blocking=True)
        eev[i][1].record()
    torch.cuda.synchronize()
    e2e_ms = sum(a.elapsed_time(b) for a, b in eev) / e2e_steps
    h2d = sum(x.numel() * x.element_size() for x in G)
    d2h = sum(x.numel() * x.element_size() for x in P)

    peaks = _peaks()
    line = {"metric": "AdamW step over the non-matrix parameters (GB/s)", "value": nbytes / (ms * 1e-3) / 1e9,
            "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic: seeded torch device RNG",
            "config": {"workload": ADAMW_WORKLOAD, "elements": sum(sizes), "param_dtype": "bf16",
                       "state_dtype": "f32", "bytes_per_element": 22, **ADAMW_HP,
                       "l2": "flushed between timed steps (256 MiB device write outside the step events)"},
            "roofline": {"kernel": "adamw_kernel", "bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                         "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"], "traffic": _measured_traffic("adamw"),
                         "launches": kl, "peak_source": f"{peaks['source']} hbm_gbs"},
            "e2e": {"value": nbytes / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                    "what": "gradients H2D from pinned host, muon_adamw_step, parameters D2H to pinned host"},
            "gpu_launches": launches,
            "clocks": clocks}
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = adamw_cpu_baseline()
    print(json.dumps(line), flush=True)
    return 0


def bench_gpu(args):
    import torch
    world, rank, local = _dist()
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if rank == 0:
        import __graft_entry__
        __graft_entry__.build()
    if dist is not None:
        dist.barrier()
    import newton_schulz_frobenius_gb300 as mg
    from workloads import WORKLOADS
    wl = _sliced(WORKLOADS[args.workload], args.slice)
    WORKLOAD_SEL[0] = wl.name
    segs = tuple(wl.extra.get("segments", (2, 2, 1)))
    mg.muon_set_ns_config(mg.QUINTIC, 5, segs, mg.MUON_PATH_AUTO)
    total_elems = sum(r * c for _, r, c in wl.matrices())
    if total_elems <= 64 << 20:
        params, grads, moms, _ = _gen_inputs(torch, wl, device)
        data = "synthetic: seeded SplitMix64/Box-Muller generator bytes (workloads.py)"
    else:
        params, grads, moms = _gen_device_inputs(torch, wl, device)
        data = "synthetic: seeded torch device RNG, same distributions (workloads.py shapes)"
    hp = dict(lr=wl.lr, beta=wl.beta, wd=wl.wd, nesterov=wl.nesterov)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    # the optimizer object of a training loop: registered once, stepped many times
    group = mg.MuonGroup(params, grads, moms)
    dtype_code = {"bf16": mg.MUON_BF16, "f16": mg.MUON_F16, "f32": mg.MUON_F32}[wl.param_dtype]

    # warm-up (the first step autotunes every distinct shape)
    for _ in range(args.warmup):
        group.step(**hp)
    torch.cuda.synchronize()
    st = mg.muon_sync_status()
    if st != mg.MUON_OK:
        raise RuntimeError(f"device status after warm-up: {mg.status_str(st)}")

    shapes = sorted({(min(r, c), max(r, c)) for _, r, c in wl.matrices()})
    paths = {f"{m}x{n}": ("gram" if mg.muon_last_path(m, n, dtype_code) == mg.MUON_PATH_GRAM else "plain")
             for m, n in shapes}
    alg_per_step = nom_per_step = 0.0
    for _, r, c in wl.matrices():
        m, n = min(r, c), max(r, c)
        code = mg.MUON_PATH_GRAM if paths[f"{m}x{n}"] == "gram" else mg.MUON_PATH_PLAIN
        nom, alg = mg.muon_ns_flops(m, n, code, segs)
        alg_per_step += alg
        nom_per_step += nom

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)

    def timed_pass(kernel_timing):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        mg.muon_kernel_timing_read()
        mg.muon_set_kernel_timing(kernel_timing)
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        l0 = mg.muon_launch_count()
        for i in range(args.steps):
            flush.zero_()                      # L2 flush, outside the step's events
            evs[i][0].record()
            group.step(**hp)
            evs[i][1].record()
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        mg.muon_set_kernel_timing(False)
        return [a.elapsed_time(b) for a, b in evs], mg.muon_launch_count() - l0, mg.muon_kernel_timing_read()

    # pass 1: the step as a user runs it (no per-launch instrumentation) -> value
    step_ms, launches, _ = timed_pass(False)
    # pass 2: same steps with per-launch CUDA events on the launching stream
    # -> per-kernel times and the roofline of the dominant kernel
    step_ms_instr, _, ktimes = timed_pass(True)
    clocks = sampler.stop()
    st = mg.muon_sync_status()
    if st != mg.MUON_OK:
        raise RuntimeError(f"device status after timed steps: {mg.status_str(st)}")
    ms = combine_over_ranks(sum(step_ms) / len(step_ms), dist, device)
    value = job_throughput(wl.count, world, ms)

    # end to end through the public API: the group copies every gradient in
    # from pinned host memory and every updated weight out to pinned host
    # memory inside each step (muon_group_set_host_io), chunk by chunk on its
    # copy streams, overlapping the update of the other chunks
    host_g = _pinned_like(torch, grads, copy=True)
    host_w = _pinned_like(torch, params, copy=False)
    group.set_host_io(host_g, host_w)
    for _ in range(max(3, args.warmup)):  # untimed: the first captures the step with its copies
        group.step(**hp)
    e2e_steps = max(3, min(args.steps, 20))
    eev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(e2e_steps)]
    torch.cuda.synchronize()
    # the host copies draw power too: the clocks of this pass are reported with it
    e2e_sampler = ClockSampler(local)
    e2e_sampler.start()
    time.sleep(0.3)
    for i in range(e2e_steps):
        flush.zero_()
        eev[i][0].record()
        group.step(**hp)
        eev[i][1].record()
        # a training loop reads its updated weights before the next step
        eev[i][1].synchronize()
    torch.cuda.synchronize()
    e2e_clocks = e2e_sampler.stop()
    group.set_host_io(None, None)
    e2e_ms = combine_over_ranks(sum(a.elapsed_time(b) for a, b in eev) / e2e_steps, dist, device)
    h2d = sum(g.numel() * g.element_size() for g in grads)
    d2h = sum(p.numel() * p.element_size() for p in params)

    peaks = _peaks()
    # the burst peak for a step of milliseconds; a step of tens of milliseconds
    # keeps the tensor cores busy long enough to run under the power cap, so it
    # is measured against the sustained figure
    if ms > 20.0:
        peak_key, peak_why = "bf16_tflops_sustained", "sustained: the step runs tens of ms of back-to-back products"
    else:
        peak_key, peak_why = "bf16_tflops", "burst: kernels timed inside a step of about a millisecond"
    # dominant kernel: the tensor-core product instance with the largest device time
    # grouped by kernel instance as ncu lists them: the symmetric products (XX^T
    # and the Gram-space products) share one instance, the long applies another
    groups = {"gemm_tc_kernel symmetric products (XX^T, G^2+poly, PG, (PG)P, PQ)": ("gemm_tc_syrk", "gemm_tc_square"),
              "gemm_tc_kernel long apply QX (incl. fused update)": ("gemm_tc_apply", "gemm_tc_apply_update"),
              "gemm_simt_kernel (fp32 path)": ("gemm_fp32",), "small_ns_kernel (fused small matrices)": ("small_ns_fused",)}
    best, best_ms, best_work, best_n = None, -1.0, 0.0, 0
    for gname, members in groups.items():
        tot = sum(ktimes.get(k, (0, 0.0, 0.0))[1] for k in members)
        if tot > best_ms:
            best, best_ms = gname, tot
            best_work = sum(ktimes.get(k, (0, 0.0, 0.0))[2] for k in members)
            best_n = sum(ktimes.get(k, (0, 0.0, 0.0))[0] for k in members)
    roofline = None
    if best_n:
        achieved = best_work / (best_ms * 1e-3) / 1e12
        if best.startswith("gemm_simt"):
            # fp32 FFMA: 152 SMs x 128 lanes x 2 FLOP x 2.07 GHz (unit counts and clock)
            peak, bound, src = 152 * 128 * 2 * 2.07e9 / 1e12, "alu", "derived FFMA peak (152 SMs x 128 lanes x 2 x 2.07 GHz)"
        else:
            peak, bound = peaks[peak_key], "tensor"
            src = f"{peaks['source']} {peak_key} ({peak_why})"
        roofline = {"kernel": best, "bound": bound, "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                    "frac": achieved / peak, "launches": best_n, "avg_launch_ms": best_ms / best_n,
                    "work_per_launch_flop": best_work / best_n,
                    "traffic": _measured_traffic(best, best_n / args.steps), "peak_source": src}
    step_total_kernel_ms = sum(v[1] for v in ktimes.values()) / args.steps
    ns_tflops = alg_per_step * world / (ms * 1e-3) / 1e12

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": wl.param_dtype, "data": data,
        "config": {"workload": wl.name, "matrices": wl.count,
                   "shapes": [[r, c, k] for r, c, k in wl.shapes], "param_dtype": wl.param_dtype,
                   "mom_dtype": wl.mom_dtype, "ns_paths": paths, "segments": "+".join(str(x) for x in segs), "steps_ns": 5,
                   "lr": wl.lr, "beta": wl.beta, "wd": wl.wd, "nesterov": wl.nesterov,
                   "l2": "flushed between timed steps (256 MiB device write outside the step events)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "api": "muon_group_step (CUDA graph replay after the first step); "
                          "kernel breakdown from a second pass with per-launch events (direct launches)"},
        "ns_tflops": {"algorithmic": ns_tflops, "nominal": nom_per_step * world / (ms * 1e-3) / 1e12,
                      "frac_of_bf16_peak": ns_tflops / world / peaks[peak_key],
                      "peak_tflops": peaks[peak_key], "peak_source": f"{peaks['source']} {peak_key} ({peak_why})"},
        "roofline": roofline,
        "kernels": {k: {"launches": v[0], "ms_per_step": v[1] / args.steps,
                        "work_per_launch": v[2] / max(v[0], 1),
                        "rate": (v[2] / (v[1] * 1e-3) / (1e12 if k.startswith(("gemm", "small")) else 1e9))
                        if v[1] else None,
                        "rate_unit": "TFLOP/s" if k.startswith(("gemm", "small")) else "GB/s"}
                    for k, v in ktimes.items()},
        "kernel_ms_per_step": step_total_kernel_ms,
        "ms_per_step_instrumented": sum(step_ms_instr) / len(step_ms_instr),
        "e2e": {"value": job_throughput(wl.count, world, e2e_ms), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "what": "muon_group_step with host I/O: every gradient copied in from pinned host memory and "
                        "every updated weight copied out to pinned host memory inside each step, overlapped "
                        "chunk by chunk with the update",
                "clocks": e2e_clocks},
        "gpu_launches": launches,
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = run_cpu_baseline(wl, paths)
    elif rank == 0 and world == 1:
        line["cpu_baseline"] = None
    group.close()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--slice", type=int, default=1,
                    help="keep 1/D of every shape of the workload (profiling runs)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return bench_reference(args)
    if args.workload == ADAMW_WORKLOAD:
        return bench_adamw(args)
    if args.workload == PACK_WORKLOAD:
        return bench_pack(args)
    return bench_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
