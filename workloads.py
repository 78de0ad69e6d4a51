"""Seeded synthetic inputs for the Muon update hot path.

This module is shared by the tests, ``bench.py`` and ``__graft_entry__.smoke``.
It holds no arithmetic of the method itself: it only turns a seed into the
bytes of a gradient, a weight or a momentum matrix, and it lists the workload
shapes.  Both the CUDA path and the CPU oracle consume exactly the bytes made
here, so neither side depends on the other.

Generator (written once, here):
    * SplitMix64 as a counter: draw ``k`` of a stream with key ``s`` is
      ``mix64(s + (k + 1) * GAMMA)`` with GAMMA = 0x9E3779B97F4A7C15 and the
      usual SplitMix64 finaliser ``mix64``.
    * key ``s = (seed << 8) | stream``; per-matrix seed = 1000 * config + index;
      stream 0 = gradient, 1 = weight, 2 = second-step gradient, 3 = momentum.
    * 53-bit uniforms ``u = ((draw >> 11) + 1) * 2**-53`` in (0, 1].
    * Box-Muller on draws (2j, 2j+1): r = sqrt(-2 ln u0), t = 2 pi u1;
      element 2j = r cos t, element 2j+1 = r sin t (fp64).
    * scale by the standard deviation, round to fp32 (round-to-nearest-even),
      and for bf16 round the fp32 value again to bf16 (round-to-nearest-even).

The workload shapes stand in for the private models the pages measured on
(LingBot-VLA 2.0, Wall-OSS, Qwen2.5-7B); only their matrix shapes and value
distributions are reproduced.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

STREAM_GRAD = 0
STREAM_WEIGHT = 1
STREAM_GRAD2 = 2
STREAM_MOM = 3


def _mix64(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def splitmix_draws(key: int, start: int, count: int) -> np.ndarray:
    """Draws ``start .. start+count-1`` of the SplitMix64 stream with this key."""
    k = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix64(np.uint64(key & 0xFFFFFFFFFFFFFFFF) + k * GAMMA)


def normal_f64(seed: int, stream: int, count: int) -> np.ndarray:
    """``count`` standard normal fp64 values of one (seed, stream)."""
    key = (int(seed) << 8) | int(stream)
    npairs = (count + 1) // 2
    out = np.empty(2 * npairs, dtype=np.float64)
    chunk = 1 << 22
    for p0 in range(0, npairs, chunk):
        p1 = min(npairs, p0 + chunk)
        d = splitmix_draws(key, 2 * p0, 2 * (p1 - p0))
        u = ((d >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)
        u0, u1 = u[0::2], u[1::2]
        r = np.sqrt(-2.0 * np.log(u0))
        t = 2.0 * math.pi * u1
        out[2 * p0:2 * p1:2] = r * np.cos(t)
        out[2 * p0 + 1:2 * p1:2] = r * np.sin(t)
    return out[:count]


def f32_to_bf16_bits(x32: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even); returns uint16 bits."""
    u = np.ascontiguousarray(x32, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    u = (u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    return u.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def f32_to_f16_bits(x32: np.ndarray) -> np.ndarray:
    """Round fp32 values to IEEE binary16 (nearest, ties to even, numpy's
    conversion); returns uint16 bits."""
    return np.ascontiguousarray(x32, dtype=np.float32).astype(np.float16).view(np.uint16)


@dataclass
class HostMatrix:
    """One generated matrix: raw storage bytes plus its shape and dtype name."""
    rows: int
    cols: int
    dtype: str                 # "f32", "bf16" or "f16"
    data: np.ndarray           # float32 (f32) or uint16 bits (bf16, f16), shape (rows, cols)

    def as_f32(self) -> np.ndarray:
        if self.dtype == "f16":
            return self.data.view(np.float16).astype(np.float32)
        return self.data if self.dtype == "f32" else bf16_bits_to_f32(self.data)


def gen_matrix(seed: int, stream: int, rows: int, cols: int, std: float, dtype: str) -> HostMatrix:
    x = (normal_f64(seed, stream, rows * cols) * float(std)).astype(np.float32)
    x = x.reshape(rows, cols)
    if dtype == "f32":
        return HostMatrix(rows, cols, dtype, x)
    if dtype == "bf16":
        return HostMatrix(rows, cols, dtype, f32_to_bf16_bits(x).reshape(rows, cols))
    if dtype == "f16":
        return HostMatrix(rows, cols, dtype, f32_to_f16_bits(x).reshape(rows, cols))
    raise ValueError(dtype)


def zeros_matrix(rows: int, cols: int, dtype: str) -> HostMatrix:
    if dtype == "f32":
        return HostMatrix(rows, cols, dtype, np.zeros((rows, cols), np.float32))
    return HostMatrix(rows, cols, dtype, np.zeros((rows, cols), np.uint16))


# ----------------------------------------------------------------------------
# Workloads.  Each is a list of (rows, cols, count) plus its dtypes and
# hyper-parameters.  "N(0, 1e-3)" in the workload descriptions is read as the
# variance 1e-3 (std ~ 0.0316); weights are N(0, 0.02^2).
# ----------------------------------------------------------------------------

QUINTIC = (3.4445, -4.7750, 2.0315)
STEPS = 5
GRAM_221 = (2, 2, 1)


@dataclass
class Workload:
    name: str
    config_id: int
    shapes: list               # [(rows, cols, count), ...] in parameter order
    param_dtype: str
    mom_dtype: str
    grad_std: float
    weight_std: float = 0.02
    lr: float = 0.02
    wd: float = 0.1
    beta: float = 0.95
    nesterov: bool = False
    note: str = ""
    extra: dict = field(default_factory=dict)

    def matrices(self):
        """Yields (index, rows, cols) for every matrix in parameter order."""
        idx = 0
        for r, c, k in self.shapes:
            for _ in range(k):
                yield idx, r, c
                idx += 1

    @property
    def count(self) -> int:
        return sum(k for _, _, k in self.shapes)

    def seed(self, index: int) -> int:
        return 1000 * self.config_id + index


def _transformer(layers, hidden, ffn, kv=None):
    kv = hidden if kv is None else kv
    return [(hidden, hidden, 2 * layers), (kv, hidden, 2 * layers),
            (ffn, hidden, 2 * layers), (hidden, ffn, layers)]


WORKLOADS = {
    "single_256x1024_f32": Workload(
        "single_256x1024_f32", 1, [(256, 1024, 1)], "f32", "f32", grad_std=1.0,
        note="one fp32 matrix, zero momentum, one gradient"),
    "single_2560x9728_bf16": Workload(
        "single_2560x9728_bf16", 2, [(2560, 9728, 1)], "bf16", "bf16", grad_std=0.02,
        nesterov=True, note="one bf16 momentum matrix, Nesterov, shape-scaled update"),
    "bucket_512_small_bf16": Workload(
        "bucket_512_small_bf16", 3, [(128, 512, 256), (256, 256, 256)], "bf16", "bf16",
        grad_std=math.sqrt(1e-3), note="256 x 128x512 (Gram) + 256 x 256x256 (plain), one call"),
    "stack_24L_h2048_bf16": Workload(
        "stack_24L_h2048_bf16", 4,
        [(2048, 2048, 96), (8192, 2048, 48), (2048, 8192, 24)], "bf16", "bf16",
        grad_std=math.sqrt(1e-3),
        note="24 layers: Wq,Wk,Wv,Wo 2048x2048; Wgate,Wup 8192x2048; Wdown 2048x8192"),
    "stack_32L_7b_bf16_f32mom": Workload(
        "stack_32L_7b_bf16_f32mom", 5, _transformer(32, 4096, 14336, kv=1024), "bf16", "f32",
        grad_std=math.sqrt(1e-3),
        note="32 layers: Wq,Wo 4096^2; Wk,Wv 1024x4096; Wgate,Wup 14336x4096; Wdown 4096x14336"),
    # the open-source Gram NS configuration the MuonX page (section 3.2) names:
    # fp16 working type, five steps as segments 2+3; same matrix as config 2
    "single_2560x9728_f16_2p3": Workload(
        "single_2560x9728_f16_2p3", 6, [(2560, 9728, 1)], "f16", "f16", grad_std=0.02,
        nesterov=True, note="fp16 parameters and momentum, NS in fp16, Gram segments 2+3",
        extra={"segments": (2, 3)}),
}
