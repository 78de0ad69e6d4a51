"""Plain, slow fp64 CPU oracle of the Muon update hot path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this module.  The library never
calls it; it shares no code with the CUDA path.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(closed forms, an SVD identity, special cases, the pages' FLOP counts).  No
function is "parity unpinned".

Sources (page title, section):
  [DMuon news]  "自变量发布 DMuon 优化器 ..." (agentren.cn), section 2
                "形状自适应执行栈": Gram-space recursion moves NS from the
                m x n space into the m x m Gram space.
  [MuonX]       "MuonX: DMuon 调整多卡分工, Gram NS 降低计算量" (CSDN), section 2
                (momentum smooths the gradient, NS orthogonalises it) and
                section 3.2 "Gram NS" (Gram matrix XX^T, accumulate the
                transform, apply it to the long matrix at segment boundaries,
                restart each segment; 2+2+1 rebuilds the Gram matrix after
                iterations 2 and 4; 10 -> 6 long products, 5 -> 11 square,
                1.443 -> 1.134 TFLOPs for a 2560 x 9728 matrix).
  [DMuon paper] "DMuon: Efficient Distributed Muon Training with Near-Adam
                Overhead" (gist.science summary), sections 1 and 2.2 (NS
                needs XX^T; Gram recursion in G = XX^T for m < n).
The pages print neither the momentum rule, the NS polynomial, eps nor the
weight update; they are taken in their plainest reading:
  * momentum M' = beta*M + G; Nesterov uses U = G + beta*M' (sum form);
  * Frobenius normalisation X0 = U / (||U||_F + eps), eps = 1e-7;
  * one NS iteration X <- aX + (bA + cA^2)X with A = XX^T, quintic
    coefficients (a, b, c) = (3.4445, -4.7750, 2.0315), 5 iterations;
  * Gram form: per segment of length L, G = XX^T, then L times
    P = aI + bG + cG^2, Q <- P (first) or P Q, G <- P G P (not after the
    last), then X <- Q X;  the Gram matrix is rebuilt from the new X;
  * orientation: a matrix with more rows than columns is processed as its
    transpose so that the Gram space is the smaller side;
  * update W' = W (1 - lr*wd) - lr * 0.2 * sqrt(max(rows, cols)) * O, both
    terms on the old W (decoupled weight decay);
  * M' and W' are stored by rounding to nearest, ties to even.
"""
from __future__ import annotations

import math

import numpy as np

EPS = 1e-7
QUINTIC = (3.4445, -4.7750, 2.0315)
CUBIC = (1.5, -0.5, 0.0)

PATH_PLAIN = "plain"
PATH_GRAM = "gram"


# ---------------------------------------------------------------------------
# storage formats
# ---------------------------------------------------------------------------

def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 storage bits -> exact fp64 values (bf16 is the top half of fp32)."""
    u32 = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u32.view(np.float32).astype(np.float64)


def f16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """IEEE binary16 storage bits -> exact fp64 values, decoded from the
    format's definition: sign bit, 5-bit exponent (bias 15), 10-bit fraction;
    exponent 0 holds the subnormals fraction * 2^-24, exponent 31 inf/nan."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.int64)
    sign = np.where(u >> 15, -1.0, 1.0)
    e = (u >> 10) & 0x1F
    f = (u & 0x3FF).astype(np.float64)
    normal = np.ldexp(1024.0 + f, np.maximum(e, 1) - 25)       # (1 + f/1024) * 2^(e-15)
    sub = np.ldexp(f, -24)
    val = np.where(e == 0, sub, normal)
    val = np.where(e == 31, np.where(f == 0, np.inf, np.nan), val)
    return sign * val


def to_f64(data: np.ndarray, dtype: str) -> np.ndarray:
    """Exact fp64 view of stored bytes (fp32 array, bf16 or fp16 uint16 bits)."""
    if dtype == "f32":
        return np.asarray(data, dtype=np.float32).astype(np.float64)
    if dtype == "bf16":
        return bf16_bits_to_f64(data)
    if dtype == "f16":
        return f16_bits_to_f64(data)
    raise ValueError(dtype)


def round_bf16(x: np.ndarray) -> np.ndarray:
    """fp64 -> nearest bf16 value (ties to even), returned as fp64.

    bf16 keeps 8 significant bits; the normal range suffices for every value
    this path stores, so the rounding is done on the frexp mantissa.
    """
    x = np.asarray(x, dtype=np.float64)
    mant, expo = np.frexp(x)                 # x = mant * 2**expo, |mant| in [0.5, 1)
    return np.ldexp(np.rint(np.ldexp(mant, 8)), expo - 8)   # rint: ties to even


def round_f16(x: np.ndarray) -> np.ndarray:
    """fp64 -> nearest binary16 value (ties to even), returned as fp64.

    Eleven significant bits for |x| >= 2^-14; below that the subnormal
    quantum 2^-24 applies; magnitudes that round beyond 65504 become inf.
    """
    x = np.asarray(x, dtype=np.float64)
    mant, expo = np.frexp(x)                          # |mant| in [0.5, 1)
    q = np.maximum(expo - 11, -24)                    # exponent of the last kept bit
    r = np.ldexp(np.rint(np.ldexp(x, -q)), q)         # rint: ties to even
    return np.where(np.abs(r) > 65504.0, np.copysign(np.inf, x), r)


def round_f32(x: np.ndarray) -> np.ndarray:
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


def round_to(x: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "f32":
        return round_f32(x)
    if dtype == "f16":
        return round_f16(x)
    return round_bf16(x)


def bf16_bits_from_f64(x: np.ndarray) -> np.ndarray:
    """Storage bits of values that are already exact bf16 numbers."""
    return (np.asarray(x, dtype=np.float64).astype(np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def f16_bits_from_f64(x: np.ndarray) -> np.ndarray:
    """Storage bits of values that are already exact binary16 numbers."""
    return np.asarray(x, dtype=np.float64).astype(np.float16).view(np.uint16)


def bits_from_f64(x: np.ndarray, dtype: str) -> np.ndarray:
    """Storage array (fp32 values or 16-bit bits) of values exact in `dtype`."""
    if dtype == "f32":
        return np.asarray(x, dtype=np.float64).astype(np.float32)
    return f16_bits_from_f64(x) if dtype == "f16" else bf16_bits_from_f64(x)


# ---------------------------------------------------------------------------
# product bookkeeping (the FLOP/GEMM counter the pages' section 3.2 quotes)
# ---------------------------------------------------------------------------

class ProductLog:
    """Records every matrix product the NS algorithms perform.

    With ``symbolic=True`` no arithmetic is done: the algorithms run on shape
    placeholders, so the log is the exact sequence of products the
    algorithm's control flow performs for a shape.  A product is "long" when
    its operand or result has the long side n, "square" when all three
    extents are m.
    """

    def __init__(self, symbolic: bool = False):
        self.symbolic = symbolic
        self.products = []          # (M, N, K, symmetric_result)

    def mm(self, A, B, symmetric_result=False):
        M, K = A.shape
        K2, N = B.shape
        assert K == K2
        self.products.append((M, N, K, symmetric_result))
        if self.symbolic:
            return _Shape((M, N))
        return A @ B

    def counts(self, m: int):
        long_ = sum(1 for (M, N, K, _) in self.products if not (M == N == K == m))
        square = sum(1 for (M, N, K, _) in self.products if M == N == K == m)
        return long_, square

    def nominal_flops(self) -> float:
        return float(sum(2 * M * N * K for (M, N, K, _) in self.products))

    def algorithmic_flops(self) -> float:
        """Symmetric results need only one triangle: count them as half."""
        return float(sum((M * N * K if s else 2 * M * N * K)
                         for (M, N, K, s) in self.products))


class _Shape:
    """Shape-only stand-in used by the symbolic product log."""

    def __init__(self, shape):
        self.shape = tuple(shape)

    @property
    def T(self):
        return _Shape(self.shape[::-1])

    def __mul__(self, other):
        return self

    __rmul__ = __mul__

    def __add__(self, other):
        return self

    __radd__ = __add__


def _eye_like(X, m):
    return _Shape((m, m)) if isinstance(X, _Shape) else np.eye(m)


def _mm(log, A, B, symmetric_result=False):
    if log is None:
        return A @ B
    return log.mm(A, B, symmetric_result)


# ---------------------------------------------------------------------------
# the steps of the method
# ---------------------------------------------------------------------------

def momentum(M: np.ndarray, G: np.ndarray, beta: float, nesterov: bool):
    """M' = beta M + G;  U = G + beta M' (Nesterov) or U = M'.

    [MuonX] section 2: the gradient is first smoothed with momentum.
    Returns (M', U) in fp64.
    """
    M_new = beta * M + G
    U = G + beta * M_new if nesterov else M_new
    return M_new, U


def orient(U: np.ndarray):
    """Work on U^T when U has more rows than columns, so m <= n.

    [DMuon paper] section 2.2: the Gram space is m x m with m < n.
    Returns (X, transposed).
    """
    if U.shape[0] > U.shape[1]:
        return U.T.copy(), True
    return U, False


def frobenius_normalise(X: np.ndarray, eps: float = EPS) -> np.ndarray:
    """X / (||X||_F + eps), which places every singular value at or below 1."""
    nrm = math.sqrt(float(np.sum(X * X)))
    return X / (nrm + eps)


def ns_plain(X, coeffs=QUINTIC, steps: int = 5, log: ProductLog | None = None):
    """Plain Newton-Schulz: ``steps`` times  A = XX^T, B = bA + cA^2, X = aX + BX.

    [MuonX] section 3.2 counts its products: per iteration one XX^T and one
    product with X (long), one A^2 (square).
    """
    a, b, c = coeffs
    for _ in range(steps):
        A = _mm(log, X, X.T, symmetric_result=True)
        B = b * A + c * _mm(log, A, A, symmetric_result=True)
        X = a * X + _mm(log, B, X)
    return X


def ns_gram(X, coeffs=QUINTIC, segments=(2, 2, 1), log: ProductLog | None = None):
    """Gram-space Newton-Schulz with segment restarts.

    [MuonX] section 3.2 / [DMuon paper] section 2.2: form G = XX^T, iterate on
    the m x m Gram matrix while accumulating the transform Q, apply Q to the
    long matrix only at the end of each segment, and restart (rebuild G from
    the new X) at the next segment.  For each segment of length L:
        G = X X^T
        for j = 1..L:
            P = aI + bG + cG^2
            Q = P if j == 1 else P Q
            if j < L:  G = P G P
        X = Q X
    """
    a, b, c = coeffs
    m = X.shape[0]
    for L in segments:
        G = _mm(log, X, X.T, symmetric_result=True)
        Q = None
        for j in range(1, L + 1):
            P = a * _eye_like(X, m) + b * G + c * _mm(log, G, G, symmetric_result=True)
            Q = P if j == 1 else _mm(log, P, Q, symmetric_result=True)
            if j < L:
                G = _mm(log, _mm(log, P, G, symmetric_result=True), P, symmetric_result=True)
        X = _mm(log, Q, X)
    return X


def newton_schulz(X, path: str, coeffs=QUINTIC, steps: int = 5, segments=(2, 2, 1),
                  log: ProductLog | None = None):
    if path == PATH_PLAIN:
        return ns_plain(X, coeffs, steps, log)
    if path == PATH_GRAM:
        if sum(segments) != steps:
            raise ValueError("segments must sum to steps")
        return ns_gram(X, coeffs, segments, log)
    raise ValueError(path)


def orthogonalize(U: np.ndarray, path: str, coeffs=QUINTIC, steps: int = 5,
                  segments=(2, 2, 1), eps: float = EPS) -> np.ndarray:
    """Orient, Frobenius-normalise, run NS, transpose back: the ortho output O."""
    X, transposed = orient(np.asarray(U, dtype=np.float64))
    X = frobenius_normalise(X, eps)
    X = newton_schulz(X, path, coeffs, steps, segments)
    return X.T.copy() if transposed else X


def update_scale(rows: int, cols: int) -> float:
    """Shape scale 0.2 * sqrt(max(rows, cols)) of the update."""
    return 0.2 * math.sqrt(max(rows, cols))


def weight_update(W: np.ndarray, O: np.ndarray, lr: float, wd: float) -> np.ndarray:
    """W' = W (1 - lr wd) - lr * 0.2 sqrt(max(rows, cols)) * O (decoupled decay)."""
    s = update_scale(*W.shape)
    return W * (1.0 - lr * wd) - lr * s * O


def muon_step(W, M, G, *, lr, beta, wd, nesterov, path, param_dtype, mom_dtype,
              coeffs=QUINTIC, steps=5, segments=(2, 2, 1), eps=EPS):
    """One Muon update of one matrix, from stored bytes to stored bytes.

    Inputs are the stored arrays (fp32, or bf16 as uint16 bits).  Returns a
    dict with the fp64 values before storage (``M_exact``, ``W_exact``), the
    stored values after rounding (``M_new``, ``W_new``, fp64 holding the exact
    stored numbers) and the ortho output ``O``.
    """
    W64 = to_f64(W, param_dtype)
    M64 = to_f64(M, mom_dtype)
    G64 = to_f64(G, param_dtype)
    M_exact, U = momentum(M64, G64, beta, nesterov)
    O = orthogonalize(U, path, coeffs, steps, segments, eps)
    W_exact = weight_update(W64, O, lr, wd)
    return {
        "M_exact": M_exact, "M_new": round_to(M_exact, mom_dtype),
        "W_exact": W_exact, "W_new": round_to(W_exact, param_dtype),
        "O": O, "W_old": W64,
    }


def ns_product_log(m: int, n: int, path: str, coeffs=QUINTIC, steps=5, segments=(2, 2, 1)):
    """Symbolic run of one NS update on an oriented m x n matrix (m <= n)."""
    log = ProductLog(symbolic=True)
    newton_schulz(_Shape((m, n)), path, coeffs, steps, segments, log)
    return log
