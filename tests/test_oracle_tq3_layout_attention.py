"""Pins for the oracle's TQ3 codec, page layouts, attention, merge and byte
accounting: closed forms, hand-derived bit patterns, brute force on tiny
shapes and the online-softmax invariants the pages state."""
import numpy as np
import pytest

from oracle import layout
from oracle.accounting import (bytes_per_token, bytes_per_token_layer, fp8_fraction_for_ratio_vs_bf16,
                               mixed_bytes_per_token)
from oracle.attention import attention_dense, merge_states, partial_state
from oracle.codebook import tq3_codebook
from oracle.paged import (TIER_ANCHOR, TIER_RECENT, TIER_STALE, decode_attention,
                          decode_attention_partials, demote_page, encode_fp8_page,
                          fp8_page_dequant, tq3_page_dequant)
from oracle.rotation import rotation_matrix, rotation_signs, unrotate
from oracle.tq3 import tq3_dequant_rows, tq3_encode_rows

SEED = 20260824


# ----------------------------------------------------------------- TQ3 codec
def test_tq3_round_trip_of_representable_row():
    L, _ = tq3_codebook()
    rng = np.random.default_rng(7)
    codes = rng.integers(0, 8, (20, 256)).astype(np.uint8)
    sigma = np.array([np.float16(s) for s in rng.uniform(0.1, 3.0, 20)], dtype=np.float64)
    x = unrotate(sigma[:, None] * L[codes], SEED)            # R x = sigma * L[code]
    got, sg, u = tq3_encode_rows(x, SEED, sigma=sigma)
    assert np.array_equal(got, codes)
    assert np.allclose(tq3_dequant_rows(got, sigma, SEED), x, atol=1e-12)


def test_tq3_one_hot_closed_form():
    # x = a e_0: y = R x has every entry a*sign_0/16, RMS = |a|/16, so u = +-1
    # (up to fp16 rounding of sigma) and every code is 5 (u=+1) or 2 (u=-1).
    for a in (3.0, -5.5):
        x = np.zeros((1, 256))
        x[0, 0] = a
        codes, sigma, u = tq3_encode_rows(x, SEED)
        s0 = rotation_signs(SEED, 256)[0]
        assert sigma[0] == float(np.float16(abs(a) / 16.0))
        assert np.all(codes == (5 if a * s0 > 0 else 2))


def test_tq3_zero_row():
    codes, sigma, _ = tq3_encode_rows(np.zeros((2, 256)), SEED)
    assert np.all(codes == 4) and np.all(sigma == 0.0)
    assert np.all(tq3_dequant_rows(codes, sigma, SEED) == 0.0)


def test_tq3_distortion_statistics():
    # For Gaussian rows the relative distortion is the codebook's Gaussian MSE
    # (0.03455) because the rotated, RMS-scaled coordinates are ~N(0,1).
    rng = np.random.default_rng(8)
    x = rng.standard_normal((400, 256))
    codes, sigma, _ = tq3_encode_rows(x, SEED)
    xt = tq3_dequant_rows(codes, sigma, SEED)
    rel = np.sum((xt - x) ** 2) / np.sum(x ** 2)
    assert abs(rel - 0.03455) < 0.05 * 0.03455


def test_tq3_decision_brute_force():
    L, _ = tq3_codebook()
    rng = np.random.default_rng(9)
    x = rng.standard_normal((8, 256)) * 2
    codes, sigma, u = tq3_encode_rows(x, SEED)
    y = x @ rotation_matrix(SEED, 256).T
    for r in range(8):
        for i in range(256):
            v = y[r, i] / sigma[r]
            d = np.abs(L - v)
            assert codes[r, i] == np.flatnonzero(d == d.min()).max()


# ----------------------------------------------------------------- layouts
def test_unit_bit_pattern_hand_derived():
    # codes 0..31 mod 8.  W0: nibbles 0..7 -> 0x76543210, plus bit 0 of codes
    # 24..31 (= 0..7) in bits 3,7,..,31 -> odd i set bits 7,15,23,31 -> 0x80808080.
    # W1 = W2 nibbles the same; W1 takes bit 1 of 0..7 (i = 2,3,6,7 -> bits
    # 11,15,27,31 = 0x88008800); W2 takes bit 2 (i = 4..7 -> 0x88880000).
    words = layout.pack_units((np.arange(32) % 8).astype(np.uint8))
    assert [int(w) for w in words] == [0x76543210 | 0x80808080,
                                       0x76543210 | 0x88008800,
                                       0x76543210 | 0x88880000]
    assert [int(w) for w in words] == [0xF6D4B290, 0xFE54BA10, 0xFEDC3210]
    assert layout.pack_units(np.full(32, 7, np.uint8)).tolist() == [0xFFFFFFFF] * 3
    assert layout.pack_units(np.zeros(32, np.uint8)).tolist() == [0, 0, 0]


def test_unit_round_trip():
    rng = np.random.default_rng(10)
    c = rng.integers(0, 8, (100, 32)).astype(np.uint8)
    assert np.array_equal(layout.unpack_units(layout.pack_units(c)), c)


def test_page_sizes_closed_form():
    assert layout.fp8_page_bytes(64, 4, 256) == 64 * 4 * 2 * 258 == 132096
    assert layout.tq3_page_bytes(64, 4, 256) == 64 * 4 * 2 * 98 == 50176
    assert layout.fp8_page_bytes(128, 4, 256) == 264192
    assert layout.tq3_page_bytes(128, 4, 256) == 100352


def test_fp8_page_positions():
    P, H, D = 16, 2, 32
    kc = np.zeros((P, H, D), np.uint8)
    vc = np.zeros((P, H, D), np.uint8)
    kc[5, 1, 7] = 11
    vc[5, 1, 7] = 22     # token 5 = pair 2, odd
    vc[4, 0, 3] = 33     # token 4 = pair 2, even
    ks = np.zeros((P, H))
    vs = np.zeros((P, H))
    ks[3, 1] = 1.5
    pg = layout.pack_fp8_page(kc, ks, vc, vs)
    plane = P * D + 2 * P
    assert pg[1 * 2 * plane + 5 * D + 7] == 11
    assert pg[1 * 2 * plane + plane + 2 * 2 * D + 2 * 7 + 1] == 22
    assert pg[0 * 2 * plane + plane + 2 * 2 * D + 2 * 3 + 0] == 33
    off = 1 * 2 * plane + P * D + 2 * 3
    assert np.frombuffer(pg[off:off + 2].tobytes(), np.float16)[0] == 1.5


def test_tq3_page_positions_and_round_trip():
    P, H, D = 16, 2, 64
    rng = np.random.default_rng(11)
    kc = rng.integers(0, 8, (P, H, D)).astype(np.uint8)
    vc = rng.integers(0, 8, (P, H, D)).astype(np.uint8)
    ks = rng.uniform(0, 2, (P, H)).astype(np.float16).astype(np.float64)
    vs = rng.uniform(0, 2, (P, H)).astype(np.float16).astype(np.float64)
    pg = layout.pack_tq3_page(kc, ks, vc, vs)
    out = layout.unpack_tq3_page(pg, P, H, D)
    for a, b in zip(out, (kc, ks, vc, vs)):
        assert np.array_equal(a, b)
    plane = P * 3 * D // 8 + 2 * P
    # K token 3, dim 40 -> unit 3*2+1, code 8 -> word 1 nibble 0
    w = np.frombuffer(pg[(3 * 2 + 1) * 12: (3 * 2 + 1) * 12 + 12].tobytes(), np.uint32)
    assert w[1] & 7 == kc[3, 0, 40]
    # V token 7 (pair 3, odd), dim 18 -> unit 3*4+1, code 2*2+1 = 5 -> word 0 nibble 5
    vb = plane
    w = np.frombuffer(pg[vb + (3 * 4 + 1) * 12: vb + (3 * 4 + 1) * 12 + 12].tobytes(), np.uint32)
    assert (w[0] >> 20) & 7 == vc[7, 0, 18]


# ----------------------------------------------------------------- attention
def test_attention_closed_forms():
    rng = np.random.default_rng(12)
    q = rng.standard_normal((6, 16))
    K = rng.standard_normal((1, 1, 16))
    V = rng.standard_normal((1, 1, 16))
    out, lse = attention_dense(q, K, V)
    assert np.allclose(out, V[0, 0][None, :], atol=1e-15)
    assert np.allclose(lse, q @ K[0, 0] / 4.0, atol=1e-14)
    n = 7
    Kn = np.repeat(K, n, axis=0)
    Vn = rng.standard_normal((n, 1, 16))
    out, lse = attention_dense(q, Kn, Vn)
    assert np.allclose(out, Vn[:, 0].mean(axis=0)[None, :], atol=1e-14)
    assert np.allclose(lse, q @ K[0, 0] / 4.0 + np.log(n), atol=1e-13)


def test_attention_brute_force_tiny():
    rng = np.random.default_rng(13)
    for d in (8, 16):
        Hq, Hkv, T = 4, 2, 11
        q = rng.standard_normal((Hq, d))
        K = rng.standard_normal((T, Hkv, d))
        V = rng.standard_normal((T, Hkv, d))
        out, lse = attention_dense(q, K, V)
        for h in range(Hq):
            kv = h // 2
            s = [sum(q[h, i] * K[t, kv, i] for i in range(d)) / d ** 0.5 for t in range(T)]
            z = sum(np.exp(x) for x in s)
            o = [sum(np.exp(s[t]) * V[t, kv, i] for t in range(T)) / z for i in range(d)]
            assert np.allclose(out[h], o, atol=1e-13)
            assert abs(lse[h] - np.log(z)) < 1e-13


def test_merge_invariance_random_splits():
    rng = np.random.default_rng(14)
    q = rng.standard_normal((6, 32)) * 3
    K = rng.standard_normal((50, 32))
    V = rng.standard_normal((50, 32))
    ref_out, ref_lse = attention_dense(q, K[:, None, :], V[:, None, :])
    for trial in range(20):
        cuts = np.sort(rng.choice(np.arange(51), size=rng.integers(0, 8), replace=True))
        bounds = [0] + list(cuts) + [50]
        states = [partial_state(q, K[a:b], V[a:b]) for a, b in zip(bounds[:-1], bounds[1:])]
        states.append(partial_state(q, K[:0], V[:0]))               # an empty split
        out, lse = merge_states(states)
        assert np.allclose(out, ref_out, atol=1e-12)
        assert np.allclose(lse, ref_lse, atol=1e-12)


def _pages(rng, P, Hkv, D, tiers, last_n):
    pages = []
    for i, t in enumerate(tiers):
        n = last_n if i == len(tiers) - 1 else P
        K = rng.standard_normal((n, Hkv, D)).astype(np.float32)
        K[..., 5] += 8.0
        V = rng.standard_normal((n, Hkv, D)).astype(np.float32)
        pg = encode_fp8_page(K, V, P)
        if t == TIER_STALE:
            pg, _ = demote_page(pg, P, Hkv, D, SEED)
        pages.append((t, pg, n))
    return pages


def test_all_fp8_partials_equal_dense():
    rng = np.random.default_rng(15)
    P, Hkv, D = 16, 2, 64
    pages = _pages(rng, P, Hkv, D, [TIER_ANCHOR, TIER_RECENT, TIER_RECENT], 9)
    q = rng.standard_normal((6, D))
    a = decode_attention(q, pages, P, Hkv, D, SEED)
    b = decode_attention_partials(q, pages, P, Hkv, D, SEED)
    assert np.allclose(a[0], b[0], atol=1e-12) and np.allclose(a[1], b[1], atol=1e-12)


def test_mixed_partials_rotated_domain_equal_dense():
    rng = np.random.default_rng(16)
    P, Hkv, D = 16, 2, 64
    tiers = [TIER_ANCHOR, TIER_STALE, TIER_STALE, TIER_STALE, TIER_RECENT, TIER_RECENT]
    pages = _pages(rng, P, Hkv, D, tiers, 3)
    q = rng.standard_normal((6, D))
    ref = decode_attention(q, pages, P, Hkv, D, SEED)
    for split in (None, [[0, 1, 2, 3, 4, 5]], [[1], [0, 3], [2, 4, 5]], [[5], [], [0, 1, 2, 3, 4]]):
        got = decode_attention_partials(q, pages, P, Hkv, D, SEED, split=split)
        assert np.allclose(got[0], ref[0], atol=1e-11)
        assert np.allclose(got[1], ref[1], atol=1e-11)


def test_demote_reencodes_fp8_dequant():
    rng = np.random.default_rng(17)
    P, Hkv, D = 16, 2, 64
    K = rng.standard_normal((P, Hkv, D)).astype(np.float32)
    V = rng.standard_normal((P, Hkv, D)).astype(np.float32)
    f8 = encode_fp8_page(K, V, P)
    t3, _ = demote_page(f8, P, Hkv, D, SEED)
    Kh, Vh = fp8_page_dequant(f8, P, Hkv, D)
    Kt, Vt = tq3_page_dequant(t3, P, Hkv, D, SEED)
    rel = np.sum((Kt - Kh) ** 2) / np.sum(Kh ** 2)
    assert 0.02 < rel < 0.05


# ----------------------------------------------------------------- accounting
def test_bytes_per_token_closed_form():
    assert bytes_per_token_layer("fp8") == 2 * 4 * 258 == 2064
    assert bytes_per_token_layer("tq3") == 2 * 4 * 98 == 784
    assert bytes_per_token_layer("bf16") == 4096
    assert bytes_per_token("bf16") == 64 * 1024          # 64 KiB: 16 layers x 2 x 4 x 256 x 2 B
    assert bytes_per_token("fp8") / 1024 == 32.25
    assert bytes_per_token("tq3") / 1024 == 12.25
    # the pages' figures are mutually consistent: 64/18.3 ~ 3.50, 32/18.3 ~ 1.75
    assert abs(64 / 18.3 - 3.50) < 0.01 and abs(32 / 18.3 - 1.75) < 0.01
    # the canary geometry under this spec (44 FP8 + 878 TQ3 pages per request)
    r = bytes_per_token("bf16") / mixed_bytes_per_token(44 * 64, 878 * 64)
    assert abs(r - 4.847) < 1e-3
    assert abs(fp8_fraction_for_ratio_vs_bf16(3.5) - 0.3018) < 1e-3


def test_streaming_equals_dense():
    rng = np.random.default_rng(18)
    P, Hkv, D = 16, 2, 64
    tiers = [TIER_ANCHOR, TIER_STALE, TIER_STALE, TIER_RECENT, TIER_RECENT]
    pages = _pages(rng, P, Hkv, D, tiers, 5)
    q = rng.standard_normal((6, D))
    from oracle.paged import decode_attention_streaming
    a = decode_attention(q, pages, P, Hkv, D, SEED)
    b = decode_attention_streaming(q, pages, P, Hkv, D, SEED)
    assert np.allclose(a[0], b[0], atol=1e-12) and np.allclose(a[1], b[1], atol=1e-12)
    c = decode_attention_streaming(q, pages, P, Hkv, D, SEED, kv_heads=[1])
    assert np.allclose(c[0][3:], a[0][3:], atol=1e-12) and np.all(np.isnan(c[0][:3]))


# ----------------------------------------------------------------- several query tokens
def _masked_matrix_attention(q, K, V):
    """Causal attention written as one masked score matrix: S = Q K^T / sqrt(d)
    with S[i, t] = -inf for t > T - nq + i, row-wise softmax, times V."""
    nq, T = q.shape[0], K.shape[0]
    S = (q @ K.T) / np.sqrt(q.shape[1])
    mask = np.arange(T)[None, :] > (T - nq + np.arange(nq))[:, None]
    S = np.where(mask, -np.inf, S)
    m = S.max(axis=1, keepdims=True)
    E = np.exp(S - m)
    return (E @ V) / E.sum(axis=1, keepdims=True), m[:, 0] + np.log(E.sum(axis=1))


def test_multi_query_equals_masked_matrix():
    from oracle.paged import decode_attention_multi, dequant_pages
    rng = np.random.default_rng(19)
    P, Hkv, D = 16, 2, 64
    tiers = [TIER_ANCHOR, TIER_STALE, TIER_STALE, TIER_RECENT, TIER_RECENT]
    pages = _pages(rng, P, Hkv, D, tiers, 5)          # tail page: 5 tokens
    K, V = dequant_pages(pages, P, Hkv, D, SEED)
    for nq in (1, 3, 5, 9):                            # 9 reaches into the page before the tail
        q = rng.standard_normal((nq, 6, D))
        out, lse = decode_attention_multi(q, pages, P, Hkv, D, SEED)
        for h in range(6):
            kv = h // 3
            ro, rl = _masked_matrix_attention(q[:, h], K[:, kv], V[:, kv])
            assert np.allclose(out[:, h], ro, atol=1e-12) and np.allclose(lse[:, h], rl, atol=1e-12)


def test_multi_query_token_is_decode_over_its_prefix():
    from oracle.paged import decode_attention_multi
    rng = np.random.default_rng(20)
    P, Hkv, D = 16, 2, 64
    tiers = [TIER_STALE, TIER_ANCHOR, TIER_RECENT, TIER_RECENT]
    pages = _pages(rng, P, Hkv, D, tiers, 3)
    T = 3 * P + 3
    nq = 7
    q = rng.standard_normal((nq, 6, D))
    out, lse = decode_attention_multi(q, pages, P, Hkv, D, SEED)
    # nq = 1 is the decode step itself
    o1, l1 = decode_attention_multi(q[-1:], pages, P, Hkv, D, SEED)
    d1 = decode_attention(q[-1], pages, P, Hkv, D, SEED)
    assert np.allclose(o1[0], d1[0], atol=1e-12) and np.allclose(l1[0], d1[1], atol=1e-12)
    # query i equals a single decode over the cache cut after its own token:
    # the page list truncated and its last page's valid count lowered
    for i in range(nq):
        visible = T - nq + i + 1
        cut = []
        for t, pg, n in pages:
            start = sum(x[2] for x in cut)
            if start >= visible:
                break
            cut.append((t, pg, min(n, visible - start)))
        ref = decode_attention(q[i], cut, P, Hkv, D, SEED)
        assert np.allclose(out[i], ref[0], atol=1e-12) and np.allclose(lse[i], ref[1], atol=1e-12)
    # more query tokens than cached tokens is an error
    with pytest.raises(ValueError):
        decode_attention_multi(rng.standard_normal((T + 1, 6, D)), pages, P, Hkv, D, SEED)
