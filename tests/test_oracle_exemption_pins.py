"""Pins for the two helpers that decide which GPU/oracle differences the
parity tests excuse (the boundary exemption of the TQ3 codes and of the fp16
scales): a value within 1e-6 (relative, max(1, |b|)) of a decision boundary
b may decide either way.  Each case is computed by hand below, so that a slip
in a helper (an absolute instead of a relative distance, the wrong nearest
boundary, a binade off by one) fails here rather than silently widening the
exemption."""
import numpy as np

from oracle.codebook import tq3_codebook
from oracle.tq3 import boundary_distance, fp16_tie_distance


def test_boundary_distance_on_and_near_thresholds():
    _, T = tq3_codebook()
    T = np.asarray(T, dtype=np.float64)
    # the codebook is symmetric, so the middle threshold is exactly 0
    assert T[3] == 0.0
    assert np.all(boundary_distance(T) == 0.0)
    # |b| < 1: the distance is absolute (max(1, |b|) = 1)
    assert np.isclose(boundary_distance(np.array([1e-6]))[0], 1e-6, rtol=1e-9, atol=0)
    assert np.isclose(boundary_distance(np.array([-3e-7]))[0], 3e-7, rtol=1e-9, atol=0)
    # |b| > 1 (the outer thresholds, about +-1.7479): relative to |b|
    b = T[-1]
    assert b > 1.5
    for u in (b * (1 + 1e-6), b * (1 - 1e-6), -b * (1 + 1e-6)):
        assert np.isclose(boundary_distance(np.array([u]))[0], 1e-6, rtol=1e-6, atol=0)
    # an absolute distance at the outer threshold would be 1e-6 * |b| > 1e-6
    # for u = b + 1e-6 * |b|; a relative one is exactly 1e-6
    # far from every threshold: the nearest one decides
    assert np.isclose(boundary_distance(np.array([5.0]))[0], (5.0 - b) / b, rtol=1e-12)
    # halfway between T[4] (about 0.5005) and T[5] (about 1.0498): the same
    # absolute gap to both, but relative to max(1, |b|) the outer one (|b| > 1)
    # is nearer, so the distance is gap / |T[5]|
    mid = (T[4] + T[5]) / 2.0
    gap = (T[5] - T[4]) / 2.0
    assert T[4] < 1.0 < T[5]
    assert np.isclose(boundary_distance(np.array([mid]))[0], gap / T[5], rtol=1e-12)


def test_fp16_tie_distance_hand_cases():
    # exact midpoints between adjacent fp16 values are at distance 0
    ties = np.array([1 + 2.0 ** -11,                # normal binade [1, 2): spacing 2^-10
                     1000.25,                        # [512, 1024): spacing 0.5
                     2.0 ** -14 + 2.0 ** -25,        # first normal binade: spacing 2^-24
                     3 * 2.0 ** -25,                 # subnormals: spacing 2^-24, tie between 2^-24 and 2^-23
                     2.0 ** -25])                    # tie between 0 and the smallest subnormal
    assert np.all(fp16_tie_distance(ties) == 0.0)
    # one fp64 ulp away from a tie: a tiny positive relative distance
    v = 1 + 2.0 ** -11 + 2.0 ** -52
    assert np.isclose(fp16_tie_distance(np.array([v]))[0], 2.0 ** -52 / v, rtol=1e-9)
    # relative, not absolute: 0.01 away from the tie 1000.25
    assert np.isclose(fp16_tie_distance(np.array([1000.26]))[0], 0.01 / 1000.26, rtol=1e-6)
    # a power of two: the nearest tie is in the binade below, 1 - 2^-12
    assert fp16_tie_distance(np.array([1.0]))[0] == 2.0 ** -12
    assert fp16_tie_distance(np.array([2.0 ** -3]))[0] == 2.0 ** -12
    # an fp16 value inside a binade: half a spacing to either side
    assert fp16_tie_distance(np.array([1.5]))[0] == 2.0 ** -11 / 1.5
    # sign does not matter
    assert fp16_tie_distance(np.array([-(1 + 2.0 ** -11)]))[0] == 0.0
