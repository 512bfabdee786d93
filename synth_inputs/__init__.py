"""Seeded synthetic inputs for the CA-SGD outer iteration.

This module is shared by the CPU oracle and by the GPU path and holds none of the
method's arithmetic: it only draws FP32 data matrices, labels and planted weights.
Storage rounding (BF16), sampling of minibatch rows, the Gram matrix, margins,
loss derivatives and updates all live on each side separately.

The workloads follow the shapes the paper (Mixed-Precision Communication-Avoiding
SGD for Generalized Linear Models on GPUs, abstract) evaluates on: logistic, linear
least-squares and Poisson problems on dense data sets it names epsilon, SUSY, HIGGS,
synth and Poisson-synth.  Those data sets are not available here; the five seeded
recipes below stand in for them (same row/feature counts class, same loss family).

Each recipe draws from NumPy PCG64 streams seeded with (seed, config id, stream):
  1  logistic, X 4096x64 ~ N(0,1); w* ~ N(0,1/64); y = sign(Xw* + 0.1 N(0,1)) with
     sign(0) -> +1; b=16, s=4, eta=0.1, 20 outer iterations.
  2  logistic (epsilon-like), X 400000x2000 ~ N(0,1)/sqrt(2000); w* ~ N(0,1);
     y = sign(Xw*) with each label flipped independently with probability 0.05;
     b=256, s=32, eta=0.5, 50 outer iterations.
  3  logistic (SUSY-like), X 5000000x18, columns 0-8 ~ N(0,1), columns 9-17 ~ |N(0,1)|;
     w* ~ N(0,1/18); y = +1 iff x.w* + L > 0 with L ~ Logistic(0,1);
     b=1024, s=16, eta=0.05, ceil(m/(s*b)) = 306 outer iterations.
  4  least squares (HIGGS-like), X 11000000x28 ~ N(0,1); w* ~ N(0,1/28);
     y = Xw* + 0.1 N(0,1); b=2048, s=8 (also 4, 16, 32), eta=0.01,
     ceil(m/(s*b)) outer iterations (1343/672/336/168 for s=4/8/16/32).
  5  Poisson (Poisson-synth), X 1000000x512 ~ 0.05 N(0,1); w* ~ N(0,1/512);
     y ~ Poisson(exp(Xw*)); b=512, s=16, eta=0.01, 30 outer iterations.

Labels are computed in FP64 from the FP32 matrix (before any storage rounding).
`m` can be shrunk for tests; every other parameter stays that of the recipe.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

LOGISTIC, LSQ, POISSON = 0, 1, 2
LOSS_NAMES = {LOGISTIC: "logistic", LSQ: "least_squares", POISSON: "poisson"}


@dataclass(frozen=True)
class Recipe:
    cid: int
    name: str
    loss: int
    m: int
    n: int
    b: int
    s: int
    eta: float
    iters: int | None  # None: ceil(m / (s*b)), one epoch-equivalent

    def outer_iters(self, m: int | None = None, s: int | None = None) -> int:
        if self.iters is not None:
            return self.iters
        mm = self.m if m is None else m
        ss = self.s if s is None else s
        return int(math.ceil(mm / (ss * self.b)))


RECIPES = {
    1: Recipe(1, "logistic_4096x64", LOGISTIC, 4096, 64, 16, 4, 0.1, 20),
    2: Recipe(2, "logistic_400000x2000", LOGISTIC, 400_000, 2000, 256, 32, 0.5, 50),
    3: Recipe(3, "logistic_5000000x18", LOGISTIC, 5_000_000, 18, 1024, 16, 0.05, None),
    4: Recipe(4, "lsq_11000000x28", LSQ, 11_000_000, 28, 2048, 8, 0.01, None),
    5: Recipe(5, "poisson_1000000x512", POISSON, 1_000_000, 512, 512, 16, 0.01, 30),
}
S_SWEEP_CONFIG4 = (4, 8, 16, 32)


@dataclass
class Problem:
    """One synthetic problem: FP32 X (m x n, C-contiguous), FP32 y, FP64 w*."""
    recipe: Recipe
    X: np.ndarray
    y: np.ndarray
    w_star: np.ndarray
    extra: dict = field(default_factory=dict)

    @property
    def m(self) -> int:
        return self.X.shape[0]

    @property
    def n(self) -> int:
        return self.X.shape[1]


def _rng(seed: int, cid: int, stream: int) -> np.random.Generator:
    return np.random.default_rng([int(seed), int(cid), int(stream)])


_ROW_CHUNK = 16384


def _normal32(seed: int, cid: int, shape) -> np.ndarray:
    """FP32 N(0,1) matrix; row chunk i of 16384 rows comes from its own PCG64 stream
    (seed, cid, 0, i), so the result does not depend on how many threads fill it."""
    m, n = shape
    X = np.empty((m, n), dtype=np.float32)

    def fill(i: int) -> None:
        a = i * _ROW_CHUNK
        e = min(m, a + _ROW_CHUNK)
        np.random.default_rng([int(seed), int(cid), 0, i]).standard_normal(
            (e - a, n), dtype=np.float32, out=X[a:e])

    chunks = (m + _ROW_CHUNK - 1) // _ROW_CHUNK
    if chunks <= 1:
        for i in range(chunks):
            fill(i)
    else:
        with ThreadPoolExecutor(min(chunks, os.cpu_count() or 1)) as ex:
            list(ex.map(fill, range(chunks)))
    return X


def _margins64(X: np.ndarray, w: np.ndarray) -> np.ndarray:
    """x_i . w* in FP64, in chunks of about 4M elements so that big matrices are
    never copied whole."""
    out = np.empty(X.shape[0], dtype=np.float64)
    chunk = max(1, (1 << 22) // max(1, X.shape[1]))
    for a in range(0, X.shape[0], chunk):
        out[a:a + chunk] = X[a:a + chunk].astype(np.float64) @ w
    return out


def _sign_pm1(v: np.ndarray) -> np.ndarray:
    return np.where(v >= 0.0, 1.0, -1.0).astype(np.float32)


def make_problem(cid: int, seed: int = 0, m: int | None = None) -> Problem:
    """Draw recipe `cid` (1..5) with `seed`; `m` overrides the row count."""
    r = RECIPES[cid]
    mm = r.m if m is None else int(m)
    n = r.n
    rw, rl = _rng(seed, cid, 1), _rng(seed, cid, 2)
    if cid == 1:
        X = _normal32(seed, cid, (mm, n))
        w_star = rw.normal(0.0, 1.0 / math.sqrt(n), n)
        y = _sign_pm1(_margins64(X, w_star) + 0.1 * rl.standard_normal(mm))
    elif cid == 2:
        X = _normal32(seed, cid, (mm, n))
        X *= np.float32(1.0 / math.sqrt(n))
        w_star = rw.normal(0.0, 1.0, n)
        y = _sign_pm1(_margins64(X, w_star))
        flip = rl.random(mm) < 0.05
        y[flip] = -y[flip]
    elif cid == 3:
        X = _normal32(seed, cid, (mm, n))
        half = n // 2
        np.abs(X[:, half:], out=X[:, half:])
        w_star = rw.normal(0.0, 1.0 / math.sqrt(n), n)
        v = _margins64(X, w_star) + rl.logistic(0.0, 1.0, mm)  # y=+1 iff v > 0
        y = np.where(v > 0.0, 1.0, -1.0).astype(np.float32)
    elif cid == 4:
        X = _normal32(seed, cid, (mm, n))
        w_star = rw.normal(0.0, 1.0 / math.sqrt(n), n)
        y = (_margins64(X, w_star) + 0.1 * rl.standard_normal(mm)).astype(np.float32)
    elif cid == 5:
        X = _normal32(seed, cid, (mm, n))
        X *= np.float32(0.05)
        w_star = rw.normal(0.0, 1.0 / math.sqrt(n), n)
        y = rl.poisson(np.exp(_margins64(X, w_star))).astype(np.float32)
    else:
        raise ValueError(f"unknown recipe {cid}")
    return Problem(r, np.ascontiguousarray(X), np.ascontiguousarray(y, dtype=np.float32),
                   w_star)


def make_random(m: int, n: int, loss: int, seed: int = 0, scale: float | None = None) -> Problem:
    """A small free-shape problem for ragged-size tests: X ~ N(0,1)*scale
    (scale defaults to 1/sqrt(n)), w* ~ N(0,1), labels as in recipes 1/4/5."""
    rw, rl = _rng(seed, 100 + loss, 1), _rng(seed, 100 + loss, 2)
    sc = (1.0 / math.sqrt(max(n, 1))) if scale is None else scale
    X = _normal32(seed, 100 + loss, (m, n))
    X *= np.float32(sc)
    w_star = rw.normal(0.0, 1.0, n)
    z = _margins64(X, w_star) if m > 0 else np.zeros(0)
    if loss == LOGISTIC:
        y = _sign_pm1(z + 0.1 * rl.standard_normal(m))
    elif loss == LSQ:
        y = (z + 0.1 * rl.standard_normal(m)).astype(np.float32)
    else:
        y = rl.poisson(np.exp(np.clip(z, -20, 5))).astype(np.float32)
    rec = Recipe(0, f"random_{m}x{n}", loss, m, n, 0, 0, 0.0, 0)
    return Problem(rec, X, y, w_star)


def random_weights(n: int, seed: int, scale: float = 0.1) -> np.ndarray:
    """A seeded non-zero FP32 starting point (margins are trivially zero at w=0)."""
    return (_rng(seed, 999, 0).standard_normal(n) * scale).astype(np.float32)
