"""8-level Lloyd-Max codebook for a unit Gaussian, as used by TQ3.

The Minima-KV pages name the packed "TQ3" format for Stale pages (abstract,
mlsanity.com paper page; "Technical Deep Dive" on the setupai.cc summary
calls it 3-bit) but do not define it.  The library's format spec
(``include/mkv.h``) fixes the quantiser as the 8-level Lloyd-Max quantiser
for N(0, 1) (Lloyd 1957/1982; Max 1960), stored as follows:

* levels: the fp64 Lloyd-Max fixed point rounded to IEEE fp16,
  ``L_0 < ... < L_7`` (symmetric: ``L_{7-k} = -L_k``);
* thresholds: exact midpoints of adjacent stored levels,
  ``tau_k = (L_{k-1} + L_k) / 2`` for k = 1..7 (exact in fp32);
* a value u gets code ``#{k : tau_k <= u}``, i.e. the nearest stored level,
  ties going to the upper code.

Rounding the levels to fp16 keeps the quantiser a nearest-level quantiser
and moves the mean-squared error only at second order (the Lloyd-Max point
is stationary); it makes a dequantised level exact in fp16 arithmetic.
"""
from __future__ import annotations

import math

import numpy as np

from .fp8 import round_to_fp16


def _phi(x: float) -> float:
    return math.exp(-0.5 * x * x) / math.sqrt(2.0 * math.pi) if math.isfinite(x) else 0.0


def _Phi(x: float) -> float:
    if x == math.inf:
        return 1.0
    if x == -math.inf:
        return 0.0
    return 0.5 * math.erfc(-x / math.sqrt(2.0))


def lloyd_max_gaussian(n_levels: int = 8, iters: int = 10000, tol: float = 1e-15):
    """Lloyd's alternation for N(0,1), in fp64.

    Step 1: thresholds are midpoints of adjacent levels.
    Step 2: each level becomes the conditional mean of its cell,
            E[X | a < X < b] = (phi(a) - phi(b)) / (Phi(b) - Phi(a)).
    Iterated from a uniform start until the levels stop moving.
    Returns (levels[n], thresholds[n-1]) as fp64 arrays.
    """
    levels = np.linspace(-2.0, 2.0, n_levels)
    for _ in range(iters):
        thr = 0.5 * (levels[1:] + levels[:-1])
        edges = np.concatenate(([-math.inf], thr, [math.inf]))
        new = np.array([
            (_phi(edges[k]) - _phi(edges[k + 1])) / (_Phi(edges[k + 1]) - _Phi(edges[k]))
            for k in range(n_levels)
        ])
        if np.max(np.abs(new - levels)) < tol:
            levels = new
            break
        levels = new
    thr = 0.5 * (levels[1:] + levels[:-1])
    return levels, thr


def gaussian_mse(levels: np.ndarray, thresholds: np.ndarray) -> float:
    """Mean-squared error of a scalar quantiser on N(0,1), in closed form:
    sum over cells of E[(X - c)^2; cell] using the Gaussian moments."""
    edges = np.concatenate(([-math.inf], thresholds, [math.inf]))
    total = 0.0
    for k, c in enumerate(levels):
        a, b = edges[k], edges[k + 1]
        p = _Phi(b) - _Phi(a)
        m1 = _phi(a) - _phi(b)                                   # E[X; cell]
        m2 = p + (a * _phi(a) if math.isfinite(a) else 0.0) \
               - (b * _phi(b) if math.isfinite(b) else 0.0)      # E[X^2; cell]
        total += m2 - 2.0 * c * m1 + c * c * p
    return total


def tq3_codebook():
    """The stored TQ3 codebook: (levels fp16-valued float64[8], thresholds float64[7])."""
    lv, _ = lloyd_max_gaussian(8)
    levels = np.array([round_to_fp16(x) for x in lv], dtype=np.float64)
    thresholds = 0.5 * (levels[1:] + levels[:-1])   # exact: fp16 inputs, fp64 sum
    return levels, thresholds


def quantize_scalar(u: float, thresholds: np.ndarray) -> int:
    """code = #{k : tau_k <= u} (ascending code order, ties to the upper code)."""
    return int(np.sum(thresholds <= u))


def quantize_array(u, thresholds: np.ndarray) -> np.ndarray:
    u = np.asarray(u, dtype=np.float64)
    return np.searchsorted(thresholds, u, side="right").astype(np.uint8)
