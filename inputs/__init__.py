"""Seeded synthetic inputs for the int8 decomposition linear.

This module is shared by the CUDA path's tests/bench and by the oracle's tests.
It holds only random draws and casts to fp16: none of the method's arithmetic
(no outlier test, no scale, no code, no product) lives here.

Workloads follow the shapes and value distributions of the five named
configurations of the int8 decomposition benchmark:

* ``tiny``    X[16,256] ~ N(0,1), columns 7 and 133 multiplied by 20,
              W[256,256] ~ N(0,0.02), tau = 6.
* ``decode``  X[T,4096] (T in 1..16) ~ N(0,1), 4 seeded columns x U(8,60),
              W[4096,4096] ~ N(0,0.02), tau = 6.
* ``prefill`` X[2048,4096], 6 seeded columns x U(8,60), W[11008,4096] ~ N(0,0.02).
* ``large``   X[4096,8192], round(0.1% * 8192) = 8 seeded columns x U(8,60),
              W[28672,8192] ~ N(0,0.015).
* ``sweep``   X[512,8192], W[8192,8192] ~ N(0,0.02), outlier-column fraction in
              {0, 0.1%, 0.5%, 2%} x U(8,60), tau in {inf, 6, 3, 0}.

Draw order for every workload (fixed so that both sides see identical data):
1. X standard normals (float32), T x K;
2. outlier columns, chosen without replacement from range(K), then sorted;
3. one U(8, 60) factor per chosen column, multiplying the whole column
   (signs kept);
4. W normals with the config's standard deviation, N x K.
Both are then rounded to fp16 (round to nearest even, numpy ``astype``).
``N(0, s)`` means standard deviation s.  The tiny workload fixes its outlier
columns and factor (7 and 133, x20) instead of drawing them.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

TAU_DEFAULT = 6.0  # llm_int8_threshold default ("Hugging Face Quantization with bitsandbytes", section 3)

SWEEP_FRACTIONS = (0.0, 0.001, 0.005, 0.02)
SWEEP_TAUS = (math.inf, 6.0, 3.0, 0.0)
DECODE_TS = (1, 2, 4, 8, 16)


@dataclass
class Workload:
    name: str
    T: int
    K: int
    N: int
    tau: float
    seed: int
    x_outlier_cols: tuple = ()
    w_std: float = 0.02
    X: np.ndarray = field(default=None, repr=False)   # float16 [T, K]
    W: np.ndarray = field(default=None, repr=False)   # float16 [N, K]

    @property
    def ops(self) -> int:
        """Effective operation count 2*T*N*K of one linear call."""
        return 2 * self.T * self.N * self.K


def _draw(T, K, N, n_cols, w_std, seed, fixed_cols=None, fixed_factor=None,
          with_w=True):
    rng = np.random.default_rng(seed)
    X = rng.standard_normal((T, K), dtype=np.float32)
    if fixed_cols is not None:
        cols = np.array(sorted(fixed_cols), dtype=np.int64)
        factors = np.full(len(cols), fixed_factor, dtype=np.float32)
    else:
        cols = np.sort(rng.choice(K, size=n_cols, replace=False)) if n_cols else \
            np.zeros(0, dtype=np.int64)
        factors = rng.uniform(8.0, 60.0, size=len(cols)).astype(np.float32)
    if len(cols):
        X[:, cols] *= factors[None, :]
    X16 = X.astype(np.float16)
    del X
    W16 = None
    if with_w:
        W = rng.standard_normal((N, K), dtype=np.float32)
        W *= np.float32(w_std)
        W16 = W.astype(np.float16)
        del W
    return X16, W16, tuple(int(c) for c in cols)


def tiny(seed: int = 0, tau: float = TAU_DEFAULT) -> Workload:
    X, W, cols = _draw(16, 256, 256, 0, 0.02, seed, fixed_cols=(7, 133), fixed_factor=20.0)
    return Workload("tiny", 16, 256, 256, tau, seed, cols, 0.02, X, W)


def decode(T: int = 16, seed: int = 0, tau: float = TAU_DEFAULT, K: int = 4096,
           N: int = 4096) -> Workload:
    X, W, cols = _draw(T, K, N, 4, 0.02, seed)
    return Workload(f"decode_T{T}", T, K, N, tau, seed, cols, 0.02, X, W)


def prefill(seed: int = 0, tau: float = TAU_DEFAULT) -> Workload:
    X, W, cols = _draw(2048, 4096, 11008, 6, 0.02, seed)
    return Workload("prefill", 2048, 4096, 11008, tau, seed, cols, 0.02, X, W)


def large(seed: int = 0, tau: float = TAU_DEFAULT) -> Workload:
    K = 8192
    X, W, cols = _draw(4096, K, 28672, round(0.001 * K), 0.015, seed)
    return Workload("large", 4096, K, 28672, tau, seed, cols, 0.015, X, W)


def sweep(frac: float, tau: float, seed: int = 0, T: int = 512, K: int = 8192,
          N: int = 8192) -> Workload:
    X, W, cols = _draw(T, K, N, round(frac * K), 0.02, seed)
    return Workload(f"sweep_f{frac}_t{tau}", T, K, N, tau, seed, cols, 0.02, X, W)


def random_small(T: int, K: int, N: int, n_cols: int, seed: int, tau: float = TAU_DEFAULT,
                 w_std: float = 0.02) -> Workload:
    """Small random shapes for parity sweeps (same recipe, any sizes)."""
    X, W, cols = _draw(T, K, N, n_cols, w_std, seed)
    return Workload(f"rand_T{T}_K{K}_N{N}", T, K, N, tau, seed, cols, w_std, X, W)


def int_valued(T: int, K: int, N: int, seed: int, adversarial: bool = False):
    """fp16 matrices holding integers in [-127, 127] with +-127 in every row.

    With ``adversarial`` every entry is +-127 with a shared sign pattern so the
    int32 dot products reach their largest magnitude 127*127*K.
    Returns (X16, W16).
    """
    rng = np.random.default_rng(seed)
    if adversarial:
        X = np.full((T, K), 127, dtype=np.int32)
        W = np.full((N, K), 127, dtype=np.int32)
        flip = rng.integers(0, 2, size=K).astype(bool)
        X[:, flip] *= -1
        W[:, flip] *= -1
        # a few rows of the opposite sign so both extremes appear
        X[1::3] *= -1
    else:
        X = rng.integers(-127, 128, size=(T, K), dtype=np.int32)
        W = rng.integers(-127, 128, size=(N, K), dtype=np.int32)
        X[np.arange(T), rng.integers(0, K, size=T)] = 127
        W[np.arange(N), rng.integers(0, K, size=N)] = -127
    return X.astype(np.float16), W.astype(np.float16)


def bias(N: int, K: int, seed: int = 0) -> np.ndarray:
    """fp16 bias [N] drawn like PyTorch Linear's default initialisation,
    uniform on [-1/sqrt(K), 1/sqrt(K)]."""
    rng = np.random.default_rng(seed + 7919)
    bound = 1.0 / math.sqrt(K)
    return rng.uniform(-bound, bound, size=N).astype(np.float16)
