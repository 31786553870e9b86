"""Seeded random-sign Walsh-Hadamard rotation used by TQ3.

The pages name TQ3 without defining it; the library's format spec
(``include/mkv.h``) fixes the rotation as

    R = (1/sqrt(d)) * H_d * D,   D = diag(sign_0 .. sign_{d-1}),

with ``H_d`` the Sylvester Hadamard matrix in natural order
(H_1 = [1], H_2n = [[H_n, H_n], [H_n, -H_n]]): signs are applied first,
then H.  R is orthogonal and R^T = (1/sqrt(d)) D H_d.  The same R serves K
and V, every layer and head, for the pool's lifetime.

Signs come from SplitMix64 (Steele, Lea and Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014) seeded with the pool's
``rotation_seed``: output word w (w = 0 is the first output) supplies
sign_i for i in [64w, 64w + 64); sign_i = -1 when bit (i mod 64) of that
word is 1, else +1.
"""
from __future__ import annotations

import numpy as np

_MASK64 = (1 << 64) - 1


def splitmix64(seed: int, n: int) -> list[int]:
    """First n outputs of SplitMix64 started from ``seed`` (published definition:
    state += golden gamma; mix with two xor-shift-multiply rounds and a final
    xor-shift)."""
    state = seed & _MASK64
    out = []
    for _ in range(n):
        state = (state + 0x9E3779B97F4A7C15) & _MASK64
        z = state
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK64
        z = z ^ (z >> 31)
        out.append(z)
    return out


def rotation_signs(seed: int, d: int) -> np.ndarray:
    """sign_i in {+1, -1} as float64[d]."""
    words = splitmix64(seed, (d + 63) // 64)
    return np.array([-1.0 if (words[i // 64] >> (i % 64)) & 1 else 1.0 for i in range(d)])


def hadamard(d: int) -> np.ndarray:
    """Sylvester Hadamard matrix H_d (entries +-1), built by the doubling rule."""
    if d < 1 or d & (d - 1):
        raise ValueError("d must be a power of two")
    H = np.ones((1, 1))
    while H.shape[0] < d:
        H = np.block([[H, H], [H, -H]])
    return H


def rotation_matrix(seed: int, d: int) -> np.ndarray:
    """R = H D / sqrt(d), explicit d x d matrix (fp64)."""
    return hadamard(d) * rotation_signs(seed, d)[None, :] / np.sqrt(d)


def rotate(x: np.ndarray, seed: int) -> np.ndarray:
    """y = R x along the last axis (explicit matrix product, fp64)."""
    x = np.asarray(x, dtype=np.float64)
    R = rotation_matrix(seed, x.shape[-1])
    return x @ R.T


def unrotate(y: np.ndarray, seed: int) -> np.ndarray:
    """x = R^T y along the last axis (explicit matrix product, fp64)."""
    y = np.asarray(y, dtype=np.float64)
    R = rotation_matrix(seed, y.shape[-1])
    return y @ R
