"""Pins for the TQ3 codebook and rotation in the oracle.

Codebook: Max (1960) table values, the Lloyd-Max fixed-point conditions
checked with an independent numerical integrator, brute-force
nearest-level decisions.  Rotation: the published SplitMix64 test vector,
Hadamard closed forms, orthogonality, and an independently written fast
Walsh-Hadamard transform."""
import math
import os

import numpy as np
from scipy import integrate

from oracle.codebook import (gaussian_mse, lloyd_max_gaussian, quantize_array, quantize_scalar,
                             tq3_codebook)
from oracle.rotation import hadamard, rotate, rotation_matrix, rotation_signs, splitmix64, unrotate

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


def test_codebook_matches_max_1960():
    lv, th = lloyd_max_gaussian(8)
    rows = _golden_rows("max1960_gaussian_8level.txt")
    levels = [float(v) for k, v in rows if k == "level"]
    thr = [float(v) for k, v in rows if k == "threshold"]
    mse = [float(v) for k, v in rows if k == "mse"][0]
    assert np.allclose(lv[4:], levels, atol=6e-4)
    assert np.allclose(th[3:], thr, atol=6e-4)
    assert abs(gaussian_mse(lv, th) - mse) < 5e-5


def test_lloyd_max_fixed_point_independent_integrator():
    lv, th = lloyd_max_gaussian(8)
    pdf = lambda x: math.exp(-0.5 * x * x) / math.sqrt(2 * math.pi)
    edges = [-np.inf] + list(th) + [np.inf]
    for k in range(8):
        num = integrate.quad(lambda x: x * pdf(x), edges[k], edges[k + 1], epsabs=1e-14)[0]
        den = integrate.quad(pdf, edges[k], edges[k + 1], epsabs=1e-14)[0]
        assert abs(num / den - lv[k]) < 1e-9          # centroid condition
    assert np.allclose(th, 0.5 * (lv[1:] + lv[:-1]))  # midpoint condition
    # closed-form MSE agrees with direct numerical integration
    direct = sum(integrate.quad(lambda x, c=lv[k]: (x - c) ** 2 * pdf(x), edges[k], edges[k + 1])[0]
                 for k in range(8))
    assert abs(direct - gaussian_mse(lv, th)) < 1e-10


def test_stored_codebook_properties():
    L, T = tq3_codebook()
    assert np.array_equal(L, L.astype(np.float16).astype(np.float64))   # fp16 values
    assert np.array_equal(L[::-1], -L)                                   # symmetric
    assert T[3] == 0.0
    assert np.array_equal(T, T.astype(np.float32).astype(np.float64))   # exact in fp32
    assert np.array_equal(T, 0.5 * (L[1:] + L[:-1]))
    assert abs(gaussian_mse(L, T) - 0.0345478) < 1e-6                   # second-order change only


def test_quantizer_is_nearest_level_ties_up():
    L, T = tq3_codebook()
    rng = np.random.default_rng(5)
    u = np.concatenate([rng.standard_normal(20000) * 1.5, T, -T, [0.0, -0.0, 9.0, -9.0]])
    got = quantize_array(u, T)
    for x, c in zip(u, got):
        d = np.abs(L - x)
        best = np.flatnonzero(np.isclose(d, d.min(), rtol=0, atol=0))
        assert c == best.max()                 # nearest level, upper on a tie
        assert quantize_scalar(x, T) == c


def test_splitmix64_published_vector():
    exp = [int(r[0]) for r in _golden_rows("splitmix64_seed1234567.txt")]
    assert splitmix64(1234567, 5) == exp


def test_signs_bit_order():
    w = splitmix64(1234567, 4)
    s = rotation_signs(1234567, 256)
    for i in range(256):
        assert s[i] == (-1.0 if (w[i // 64] >> (i % 64)) & 1 else 1.0)


def test_hadamard_closed_forms():
    assert np.array_equal(hadamard(2), np.array([[1, 1], [1, -1]]))
    assert np.array_equal(hadamard(4)[:, 0], np.ones(4))
    H = hadamard(256)
    assert np.array_equal(H @ H.T, 256 * np.eye(256))
    assert np.array_equal(H, H.T)


def _fwht(x):
    """Independent in-place fast Walsh-Hadamard transform (natural order)."""
    x = np.array(x, dtype=np.float64)
    h = 1
    while h < x.shape[-1]:
        for i in range(0, x.shape[-1], 2 * h):
            a = x[..., i:i + h].copy()
            b = x[..., i + h:i + 2 * h].copy()
            x[..., i:i + h] = a + b
            x[..., i + h:i + 2 * h] = a - b
        h *= 2
    return x


def test_rotation_properties():
    seed = 0xC0FFEE
    R = rotation_matrix(seed, 256)
    assert np.max(np.abs(R @ R.T - np.eye(256))) < 1e-15
    assert np.all(np.abs(np.abs(R) - 1.0 / 16.0) == 0.0)          # R e_j entries are +-1/16
    rng = np.random.default_rng(6)
    x = rng.standard_normal((10, 256))
    y = rotate(x, seed)
    assert np.allclose(np.linalg.norm(y, axis=1), np.linalg.norm(x, axis=1), rtol=1e-14)
    # signs first, then H: compare with the independent FWHT
    assert np.allclose(y, _fwht(x * rotation_signs(seed, 256)) / 16.0, atol=1e-13)
    assert np.allclose(unrotate(y, seed), x, atol=1e-13)
    # R^T = D H / sqrt(d)
    assert np.allclose(unrotate(x, seed), rotation_signs(seed, 256) * _fwht(x) / 16.0, atol=1e-13)


def test_signs_literal_prefix():
    # sign_i = -1 iff bit (i mod 64) of SplitMix64 output floor(i/64) is set.
    # The published first output for seed 1234567 is 6457827717110365317 =
    # 0x599ED017FB08FC85; its low 16 bits 0xFC85 = 1111 1100 1000 0101 (bit 15
    # .. bit 0) give the first 16 signs.  The second output 3203168211198807973
    # = 0x2C73F08458540FA5 has low byte 0xA5 = 1010 0101: signs 64..71.
    s = rotation_signs(1234567, 256)
    assert list(s[:16]) == [-1, 1, -1, 1, 1, 1, 1, -1, 1, 1, -1, -1, -1, -1, -1, -1]
    assert list(s[64:72]) == [-1, 1, -1, 1, 1, -1, 1, -1]
