"""Pins for the oracle's FP8 (E4M3fn) codec and fp16 rounding.

Each check ties the oracle to something other than itself: the OCP E4M3
grid facts, a brute-force nearest-value search, and library conversions
(``torch.float8_e4m3fn``, ``numpy.float16``)."""
import numpy as np
import pytest
import torch

from oracle.fp8 import (E4M3_TABLE, e4m3_round, e4m3_round_array, fp8_dequant_row,
                        fp8_quantize_row, fp8_quantize_rows, fp8_scale, round_to_fp16_array)

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def test_grid_facts():
    assert E4M3_TABLE[0x7E] == 448.0
    assert np.isnan(E4M3_TABLE[0x7F]) and np.isnan(E4M3_TABLE[0xFF])
    assert E4M3_TABLE[0x08] == 2.0 ** -6          # smallest normal
    assert E4M3_TABLE[0x01] == 2.0 ** -9          # smallest subnormal
    pos = E4M3_TABLE[:0x7F]
    assert np.all(np.diff(pos) > 0)               # codes 0x00..0x7E increase
    assert np.array_equal(E4M3_TABLE[0x80:0xFF], -pos)
    assert 1.0 / np.min(np.diff(pos)) == 512.0    # uniform subnormal spacing 2^-9


def _brute(v):
    """Nearest finite non-negative grid value, ties to the even code, then sign."""
    a = min(abs(v), 448.0)
    grid = E4M3_TABLE[:0x7F]
    dist = np.abs(grid - a)
    cands = np.flatnonzero(dist == dist.min())
    c = int(cands[0]) if len(cands) == 1 else int([x for x in cands if x % 2 == 0][0])
    return c | (0x80 if np.signbit(v) else 0)


def test_round_matches_brute_force_random():
    rng = np.random.default_rng(1)
    v = rng.standard_normal(4000) * np.exp(rng.uniform(-9, 7, 4000))
    got = e4m3_round_array(v)
    exp = np.array([_brute(x) for x in v], dtype=np.uint8)
    assert np.array_equal(got, exp)


def test_round_ties_and_edges():
    grid = E4M3_TABLE[:0x7F]
    mids = 0.5 * (grid[1:] + grid[:-1])          # every exact tie between neighbours
    vals = np.concatenate([mids, -mids, grid, [0.0, -0.0, 448.0, 460.0, 464.0, 1e9, -1e9,
                                                 2.0 ** -10, 2.0 ** -11, 3 * 2.0 ** -11]])
    got = e4m3_round_array(vals)
    exp = np.array([_brute(x) for x in vals], dtype=np.uint8)
    assert np.array_equal(got, exp)
    assert all(e4m3_round(x) == _brute(x) for x in vals[:300])
    assert e4m3_round(-0.0) == 0x80 and e4m3_round(0.0) == 0x00


def test_round_matches_torch_conversion():
    rng = np.random.default_rng(2)
    v = rng.standard_normal(20000) * np.exp(rng.uniform(-10, 6, 20000))
    v = np.clip(v, -448.0, 448.0)
    grid = E4M3_TABLE[:0x7F]
    v = np.concatenate([v, 0.5 * (grid[1:] + grid[:-1])])
    ref = torch.tensor(v, dtype=torch.float64).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(e4m3_round_array(v), ref)


def test_fp16_rounding_matches_numpy():
    rng = np.random.default_rng(3)
    v = rng.standard_normal(50000) * np.exp(rng.uniform(-22, 12, 50000))
    spacing = np.ldexp(1.0, np.maximum(np.frexp(np.abs(v))[1] - 1, -14) - 10)
    ties = (np.floor(v / spacing) + 0.5) * spacing            # exact fp16 ties
    v = np.concatenate([v, ties, [65504.0, 65519.9, 65520.0, 2.0 ** -25, 3 * 2.0 ** -26]])
    assert np.array_equal(round_to_fp16_array(v), v.astype(np.float16).astype(np.float64))


def test_scale_closed_forms():
    assert fp8_scale(np.array([448.0, -3.0])) == 1.0
    assert fp8_scale(np.array([-448.0 * 2, 1.0])) == 2.0
    s = fp8_scale(np.array([1.0, 0.5]))
    assert s == float(np.float16(np.float32(1.0) / np.float32(448.0)))
    codes, s0 = fp8_quantize_row(np.zeros(16))
    assert s0 == 0.0 and not codes.any()


def test_quantize_error_bound_and_exact_dequant():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((64, 256)).astype(np.float32)
    x[:, 3] += 8.0
    codes, s = fp8_quantize_rows(x)
    for r in range(64):
        xh = fp8_dequant_row(codes[r], s[r])
        # x_hat is exactly representable in fp32 (4-bit x 11-bit significands)
        assert np.array_equal(xh.astype(np.float32).astype(np.float64), xh)
        # relative half-ulp of E4M3 (2^-4) in the normal range, 2^-10*s absolute below
        err = np.abs(xh - x[r])
        bound = np.maximum(np.abs(x[r]) * 2.0 ** -4, 2.0 ** -10 * s[r]) * (1 + 1e-6)
        assert np.all(err <= bound + 1e-3 * s[r])  # + fp32-division slack
        # the row maximum maps near 448 and never overflows the grid
        assert np.max(np.abs(E4M3_TABLE[codes[r]])) <= 448.0
    # row-wise and single-row forms agree
    c1, s1 = fp8_quantize_row(x[5])
    assert np.array_equal(c1, codes[5]) and s1 == s[5]
