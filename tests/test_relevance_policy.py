"""Relevance-based Anchor policy (harness.RelevanceAnchors): decisions from
given page masses, applied to a host-only pool through the C ABI.  The
policy is the library's own design (the pages name "age and relevance" for
protected Anchor pages without defining either)."""
import pytest

from mixed_format_paged_gb300 import MkvPool
from mixed_format_paged_gb300.harness import RelevanceAnchors

A, R, S = 2, 1, 3


def _pool():
    return MkvPool(1, 24, 4, 256, 64, 32, 32, max_seqs=2, max_pages_per_seq=16, host_only=True)


def test_anchor_budget_swap_and_hysteresis():
    pool = _pool()
    pool.extend([0], [64 * 12])
    pol = RelevanceAnchors(frac=0.1, kappa=2.0, beta=1.0, hysteresis=0.25)
    mass = [[0.01] * 12]
    for j, m in ((2, 0.5), (3, 0.05), (5, 0.3), (6, 0.7), (7, 0.8)):
        mass[0][j] = m
    pol.observe([0], mass, [12])
    older = 10                      # even share 0.1: kappa = 2 asks for a mass >= 0.2; budget 1
    steps = {}
    for j in (2, 3, 5, 6, 7):
        steps[j] = pol.decide(0, j, older)
        pol.apply(pool, 0, steps[j])
    assert steps[2] == [("anchor", 2)]                     # strong, room in the budget
    assert steps[3] == [("demote", 3)]                     # weak
    assert steps[5] == [("demote", 5)]                     # strong but not 1.25 x the Anchor held (0.5)
    assert steps[6] == [("release", 2), ("anchor", 6)]     # 0.7 > 1.25 x 0.5: swap
    assert steps[7] == [("demote", 7)]                     # 0.8 < 1.25 x 0.7: no flap
    tiers = {j: pool.page_info(0, j)[0] for j in (2, 3, 5, 6, 7)}
    assert tiers == {2: S, 3: S, 5: S, 6: A, 7: S}
    assert pol.anchors[0] == {6}


def test_moving_average_and_no_observation():
    pol = RelevanceAnchors(frac=0.5, kappa=1.0, beta=0.5)
    assert pol.decide(0, 0, 4) == [("demote", 0)]          # nothing observed: no page is relevant
    pol.observe([0], [[0.4, 0.0]], [2])
    pol.observe([0], [[0.0, 0.0]], [2])
    assert pol.rho[(0, 0)] == pytest.approx(0.1)          # 0.5 * (0.5 * 0.4) + 0.5 * 0
    assert pol.decide(0, 0, 10) == [("anchor", 0)]        # 0.1 * 10 >= kappa 1


def test_released_anchor_goes_back_to_fp8_then_tq3():
    pool = _pool()
    pool.extend([0], [64 * 4])
    pool.set_tier(0, 1, A)
    pol = RelevanceAnchors()
    pol.anchors[0] = {1}
    pol.apply(pool, 0, [("release", 1), ("anchor", 2)])
    assert pool.page_info(0, 1)[0] == S and pool.page_info(0, 2)[0] == A
