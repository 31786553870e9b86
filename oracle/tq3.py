"""TQ3 codec (Stale pages): rotate, scale, 3-bit Lloyd-Max codes.

Pages: "older non-anchor pages move to packed TQ3" (Minima-KV abstract,
mlsanity.com paper page); "packed into TQ3 (3-bit) format" ("Technical Deep
Dive", setupai.cc summary).  TQ3 is not defined on the pages; the library's
format spec (``include/mkv.h``) fixes it, and this module follows that spec
step by step, in fp64:

1. input is the FP8-dequantised row x_hat (demotion re-quantises what the
   FP8 page holds);
2. y = R x_hat (``oracle.rotation``);
3. sigma = fp16_rn( ||x_hat||_2 / sqrt(d) )  -- the RMS of the row, which
   equals the RMS of y because R is orthogonal;
4. u_i = y_i / sigma (u_i = 0 when sigma = 0);
5. code_i = #{k : tau_k <= u_i} with the stored codebook
   (``oracle.codebook``);
6. dequantisation x_tilde = R^T (sigma * L[code]).

The byte layout of codes inside a page is in ``oracle.layout``.
"""
from __future__ import annotations

import numpy as np

from .codebook import quantize_array, tq3_codebook
from .fp8 import round_to_fp16_array
from .rotation import rotate, unrotate


def tq3_sigma_raw(xhat: np.ndarray) -> np.ndarray:
    """RMS of each row before fp16 rounding (fp64)."""
    xhat = np.asarray(xhat, dtype=np.float64)
    d = xhat.shape[-1]
    return np.sqrt(np.sum(xhat * xhat, axis=-1) / d)


def tq3_encode_rows(xhat: np.ndarray, seed: int, sigma: np.ndarray | None = None):
    """Encode rows (last axis = head_dim).

    Returns (codes uint8[..., d], sigma float64[...] holding fp16 values,
    u float64[..., d] = the pre-decision values y/sigma).
    If ``sigma`` is given it is used instead of being computed (used to
    re-encode with another implementation's stored scale)."""
    xhat = np.asarray(xhat, dtype=np.float64)
    levels, thresholds = tq3_codebook()
    y = rotate(xhat, seed)
    if sigma is None:
        sigma = round_to_fp16_array(tq3_sigma_raw(xhat))
    sigma = np.asarray(sigma, dtype=np.float64)
    safe = np.where(sigma == 0.0, 1.0, sigma)
    u = np.where(sigma[..., None] == 0.0, 0.0, y / safe[..., None])
    codes = quantize_array(u, thresholds)
    return codes, sigma, u


def tq3_dequant_rows_rotated(codes: np.ndarray, sigma: np.ndarray) -> np.ndarray:
    """sigma * L[code]: the dequantised row in the rotated domain."""
    levels, _ = tq3_codebook()
    return np.asarray(sigma, dtype=np.float64)[..., None] * levels[np.asarray(codes, dtype=np.int64)]


def tq3_dequant_rows(codes: np.ndarray, sigma: np.ndarray, seed: int) -> np.ndarray:
    """x_tilde = R^T (sigma * L[code])."""
    return unrotate(tq3_dequant_rows_rotated(codes, sigma), seed)


def boundary_distance(u: np.ndarray) -> np.ndarray:
    """Relative distance of each pre-decision value to its nearest threshold:
    |u - b| / max(1, |b|).  Used for the boundary exemption in parity tests."""
    _, thresholds = tq3_codebook()
    u = np.asarray(u, dtype=np.float64)
    dist = np.abs(u[..., None] - thresholds) / np.maximum(1.0, np.abs(thresholds))
    return dist.min(axis=-1)


def fp16_tie_distance(v: np.ndarray) -> np.ndarray:
    """Relative distance |v - m| / |v| of a real value to the nearest fp16
    rounding boundary m (a midpoint between adjacent fp16 values).  Used for
    the scale exemption.

    The two candidate boundaries are the midpoints on either side of the
    largest fp16 value at or below |v|: the one above it and the one below
    it (the latter lies in the binade below when that value is a power of
    two, where the spacing halves)."""
    v = np.abs(np.asarray(v, dtype=np.float64))
    lo = v.astype(np.float16)
    lo = np.where(lo.astype(np.float64) > v, np.nextafter(lo, np.float16(0)), lo)   # largest fp16 <= v
    up = np.nextafter(lo, np.float16(np.inf)).astype(np.float64)
    down = np.nextafter(lo, np.float16(0)).astype(np.float64)
    lo64 = lo.astype(np.float64)
    mid_up = (lo64 + up) / 2.0
    mid_down = np.where(lo64 > 0.0, (lo64 + down) / 2.0, np.inf)
    dist = np.minimum(np.abs(v - mid_up), np.abs(v - mid_down))
    return dist / np.maximum(v, 1e-300)
