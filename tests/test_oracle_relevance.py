"""Pins for the oracle's page relevance (attention mass per page), the
signal of the relevance-based Anchor policy.  Each check is independent of
the function's own formula: a normalisation invariant, closed forms, a
hand-computed two-token case, and the identity with decode attention when
each value row is the indicator vector of its token's page."""
import numpy as np

from oracle.attention import attention_dense
from oracle.paged import (TIER_ANCHOR, TIER_RECENT, TIER_STALE, demote_page, encode_fp8_page,
                          page_attention_mass, dequant_pages)

SEED = 4321


def _pages(rng, P, Hkv, D, tiers, last_n, same_key=None):
    pages = []
    for i, t in enumerate(tiers):
        n = last_n if i == len(tiers) - 1 else P
        K = rng.standard_normal((n, Hkv, D)).astype(np.float32)
        if same_key is not None:
            K[:] = same_key
        V = rng.standard_normal((n, Hkv, D)).astype(np.float32)
        pg = encode_fp8_page(K, V, P)
        if t == TIER_STALE:
            pg, _ = demote_page(pg, P, Hkv, D, SEED)
        pages.append((t, pg, n))
    return pages


def test_masses_sum_to_one_and_single_page():
    rng = np.random.default_rng(1)
    P, Hkv, D = 64, 2, 64
    pages = _pages(rng, P, Hkv, D, [TIER_ANCHOR, TIER_STALE, TIER_STALE, TIER_RECENT], 17)
    q = rng.standard_normal((6, D)) * 2
    m = page_attention_mass(q, pages, P, Hkv, D, SEED)
    assert m.shape == (4,) and np.all(m >= 0)
    assert abs(m.sum() - 1.0) < 1e-12
    one = page_attention_mass(q, pages[:1], P, Hkv, D, SEED)
    assert np.allclose(one, [1.0], atol=1e-15)


def test_identical_keys_give_mass_in_proportion_to_tokens():
    rng = np.random.default_rng(2)
    P, Hkv, D = 64, 2, 64
    key = (np.arange(D) % 5 - 2).astype(np.float32) * 0.5          # exactly representable in FP8 x scale
    pages = _pages(rng, P, Hkv, D, [TIER_ANCHOR, TIER_RECENT, TIER_RECENT], 10, same_key=key)
    q = rng.standard_normal((4, D))
    m = page_attention_mass(q, pages, P, Hkv, D, SEED)
    assert np.allclose(m, np.array([64, 64, 10]) / 138.0, atol=1e-12)


def test_two_tokens_by_hand():
    # one FP8 page per token, d = 16, keys along two axes with amplitude 448
    # (the FP8 scale is then exactly 1 and the key is stored exactly):
    # q = [4/448, 0, ...], k1 = 448 e_0, k2 = 448 e_1: s1 = 4/sqrt(16) = 1, s2 = 0
    P, Hkv, D = 64, 1, 16
    k1 = np.zeros((1, 1, D), np.float32)
    k1[0, 0, 0] = 448.0
    k2 = np.zeros((1, 1, D), np.float32)
    k2[0, 0, 1] = 448.0
    v = np.zeros((1, 1, D), np.float32)
    pages = [(TIER_RECENT, encode_fp8_page(k1, v, P), 1), (TIER_RECENT, encode_fp8_page(k2, v, P), 1)]
    q = np.zeros((1, D))
    q[0, 0] = 4.0 / 448.0
    m = page_attention_mass(q, pages, P, Hkv, D, SEED)
    e = np.exp(1.0)
    assert np.allclose(m, [e / (e + 1.0), 1.0 / (e + 1.0)], atol=1e-14)


def test_mass_is_decode_attention_onto_page_indicators():
    rng = np.random.default_rng(3)
    P, Hkv, D = 64, 2, 64
    tiers = [TIER_ANCHOR, TIER_STALE, TIER_STALE, TIER_STALE, TIER_RECENT]
    pages = _pages(rng, P, Hkv, D, tiers, 33)
    q = rng.standard_normal((6, D)) * 3
    K, _ = dequant_pages(pages, P, Hkv, D, SEED)
    # V row of token t: the indicator of its page (same for every kv head)
    owner = np.concatenate([np.full(nv, j) for j, (_, _, nv) in enumerate(pages)])
    Vind = np.zeros((K.shape[0], Hkv, D))          # the first len(pages) columns hold the indicator
    Vind[np.arange(K.shape[0]), :, owner] = 1.0
    out, _ = attention_dense(q, K, Vind)          # out[h, j]: head h's weight on page j
    assert np.allclose(page_attention_mass(q, pages, P, Hkv, D, SEED), out[:, :len(pages)].mean(axis=0),
                       atol=1e-12)
