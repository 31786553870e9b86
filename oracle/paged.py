"""Paged, mixed-format cache in the oracle: page encode/decode and attention
over a list of pages of either tier.

Pages (Minima-KV abstract, mlsanity.com paper page): Recent and protected
Anchor pages stay in FP8, older non-anchor pages move to packed TQ3, and every
live-request page stays addressable; the setupai.cc "Technical Deep Dive"
adds that the mixed formats live "within the same memory block structure"
as PagedAttention.  Each page here is (tier, bytes, n_valid tokens); the
byte layout is ``oracle.layout``.
"""
from __future__ import annotations

import numpy as np

from . import layout
from .attention import attention_dense, merge_states, merge_unnormalised, partial_state
from .fp8 import E4M3_TABLE, fp8_quantize_rows
from .rotation import rotate, unrotate
from .tq3 import tq3_dequant_rows_rotated, tq3_encode_rows

TIER_RECENT, TIER_ANCHOR, TIER_STALE = 1, 2, 3


def encode_fp8_page(K: np.ndarray, V: np.ndarray, P: int):
    """Quantise up to P tokens (K/V [n, Hkv, D], fp32-representable values)
    into FP8 page bytes; token slots past n hold code 0 and scale 0."""
    n, Hkv, D = K.shape
    kc = np.zeros((P, Hkv, D), np.uint8)
    vc = np.zeros((P, Hkv, D), np.uint8)
    ks = np.zeros((P, Hkv))
    vs = np.zeros((P, Hkv))
    kc[:n], ks[:n] = fp8_quantize_rows(K)
    vc[:n], vs[:n] = fp8_quantize_rows(V)
    return layout.pack_fp8_page(kc, ks, vc, vs)


def fp8_page_dequant(page: np.ndarray, P: int, Hkv: int, D: int):
    kc, ks, vc, vs = layout.unpack_fp8_page(page, P, Hkv, D)
    return E4M3_TABLE[kc] * ks[..., None], E4M3_TABLE[vc] * vs[..., None]


def demote_page(fp8_page: np.ndarray, P: int, Hkv: int, D: int, seed: int):
    """FP8 page bytes -> TQ3 page bytes (re-quantising the dequantised rows).
    Also returns the pre-decision values (uK, uV) and the raw (pre-fp16) RMS
    scales, for the boundary exemption."""
    Kh, Vh = fp8_page_dequant(fp8_page, P, Hkv, D)
    kc, ks, uK = tq3_encode_rows(Kh, seed)
    vc, vs, uV = tq3_encode_rows(Vh, seed)
    return layout.pack_tq3_page(kc, ks, vc, vs), (uK, uV)


def tq3_page_dequant(page: np.ndarray, P: int, Hkv: int, D: int, seed: int):
    kc, ks, vc, vs = layout.unpack_tq3_page(page, P, Hkv, D)
    return (unrotate(tq3_dequant_rows_rotated(kc, ks), seed),
            unrotate(tq3_dequant_rows_rotated(vc, vs), seed))


def tq3_page_dequant_rotated(page: np.ndarray, P: int, Hkv: int, D: int):
    kc, ks, vc, vs = layout.unpack_tq3_page(page, P, Hkv, D)
    return tq3_dequant_rows_rotated(kc, ks), tq3_dequant_rows_rotated(vc, vs)


def dequant_pages(pages, P: int, Hkv: int, D: int, seed: int):
    """Concatenate the dequantised valid tokens of a page list.
    pages: iterable of (tier, bytes, n_valid)."""
    Ks, Vs = [], []
    for tier, page, n in pages:
        if tier == TIER_STALE:
            K, V = tq3_page_dequant(page, P, Hkv, D, seed)
        else:
            K, V = fp8_page_dequant(page, P, Hkv, D)
        Ks.append(K[:n])
        Vs.append(V[:n])
    return np.concatenate(Ks), np.concatenate(Vs)


def decode_attention(q: np.ndarray, pages, P: int, Hkv: int, D: int, seed: int):
    """The method's result by definition: exact softmax attention of q
    [Hq, D] over every valid token of every page, dequantised per tier."""
    K, V = dequant_pages(pages, P, Hkv, D, seed)
    return attention_dense(q, K, V)


def decode_attention_partials(q: np.ndarray, pages, P: int, Hkv: int, D: int, seed: int,
                              split=None):
    """The method's structure: per-format partial states merged by online
    softmax.  FP8 pages are scored as stored; TQ3 pages are scored in the
    rotated domain with q' = R q, their partial outputs are merged there and
    rotated back once (R^T), then merged with the FP8 partial.
    ``split`` optionally groups page indices into sets (each one partial)."""
    q = np.asarray(q, dtype=np.float64)
    Hq = q.shape[0]
    G = Hq // Hkv
    pages = list(pages)
    groups = split if split is not None else [[i] for i in range(len(pages))]
    out = np.zeros((Hq, D))
    lse = np.zeros(Hq)
    qr = rotate(q, seed)
    for kv in range(Hkv):
        qh = q[kv * G:(kv + 1) * G]
        qrh = qr[kv * G:(kv + 1) * G]
        fp8_states, tq3_states = [], []
        for grp in groups:
            for tier in (TIER_STALE, None):
                Ks, Vs = [], []
                for i in grp:
                    t, page, n = pages[i]
                    if (t == TIER_STALE) != (tier == TIER_STALE):
                        continue
                    if t == TIER_STALE:
                        K, V = tq3_page_dequant_rotated(page, P, Hkv, D)
                    else:
                        K, V = fp8_page_dequant(page, P, Hkv, D)
                    Ks.append(K[:n, kv])
                    Vs.append(V[:n, kv])
                K = np.concatenate(Ks) if Ks else np.zeros((0, D))
                V = np.concatenate(Vs) if Vs else np.zeros((0, D))
                if tier == TIER_STALE:
                    tq3_states.append(partial_state(qrh, K, V))
                else:
                    fp8_states.append(partial_state(qh, K, V))
        # TQ3 partials merged in the rotated domain, rotated back once
        Ms, Ls, Os = merge_unnormalised(tq3_states)
        Os = unrotate(Os, seed)
        Mf, Lf, Of = merge_unnormalised(fp8_states)
        o, l = merge_states([(Ms, Ls, Os), (Mf, Lf, Of)])
        out[kv * G:(kv + 1) * G] = o
        lse[kv * G:(kv + 1) * G] = l
    return out, lse


def decode_attention_streaming(q: np.ndarray, pages, P: int, Hkv: int, D: int, seed: int,
                               kv_heads=None):
    """Same result as ``decode_attention`` computed page by page: one partial
    state per page (FP8 pages scored as stored, TQ3 pages dequantised to the
    original domain), merged at the end.  Memory stays O(page) so large
    contexts can be checked.  ``kv_heads`` restricts the work to some kv
    heads (other outputs are NaN)."""
    q = np.asarray(q, dtype=np.float64)
    Hq = q.shape[0]
    G = Hq // Hkv
    heads = range(Hkv) if kv_heads is None else kv_heads
    out = np.full((Hq, D), np.nan)
    lse = np.full(Hq, np.nan)
    states = {kv: [] for kv in heads}
    for tier, page, n in pages:
        if tier == TIER_STALE:
            K, V = tq3_page_dequant(page, P, Hkv, D, seed)
        else:
            K, V = fp8_page_dequant(page, P, Hkv, D)
        for kv in heads:
            states[kv].append(partial_state(q[kv * G:(kv + 1) * G], K[:n, kv], V[:n, kv]))
    for kv in heads:
        o, l = merge_states(states[kv])
        out[kv * G:(kv + 1) * G] = o
        lse[kv * G:(kv + 1) * G] = l
    return out, lse


def decode_attention_multi(q: np.ndarray, pages, P: int, Hkv: int, D: int, seed: int):
    """Several query tokens per request with a causal mask: q [nq, Hq, D]
    are the request's last nq tokens, and query token i (position
    T - nq + i, T the valid tokens of all pages) attends to tokens
    0 .. T - nq + i of the dequantised cache.  Returns out [nq, Hq, D] and
    lse [nq, Hq].

    The pages describe one query per decode step; a chunk of queries (prefill
    of a chunk, or verification of speculative tokens) is the same softmax
    attention under the decoder's causal mask: each token sees itself and
    every earlier token."""
    K, V = dequant_pages(pages, P, Hkv, D, seed)
    q = np.asarray(q, dtype=np.float64)
    nq, T = q.shape[0], K.shape[0]
    if nq > T:
        raise ValueError("more query tokens than cached tokens")
    outs, lses = [], []
    for i in range(nq):
        visible = T - nq + i + 1
        o, l = attention_dense(q[i], K[:visible], V[:visible])
        outs.append(o)
        lses.append(l)
    return np.stack(outs), np.stack(lses)


def page_attention_mass(q: np.ndarray, pages, P: int, Hkv: int, D: int, seed: int):
    """Relevance of each page to a query: the softmax weight its tokens get,
    averaged over the query heads, i.e. for page j

        mass_j = (1 / Hq) * sum_h sum_{t in page j} softmax_h(s_h)_t,
        s_h,t  = q_h . k_t / sqrt(D)  (kv head floor(h / G), K dequantised
                 per the page's tier).

    The pages speak of protecting Anchor pages by "age and relevance"
    (insight.aitobox.com post, "执行摘要") without defining relevance; this is
    the library's definition (attention mass, the weight decode attention
    itself puts on the page).  Returns float64 [npages]; the masses sum to 1."""
    q = np.asarray(q, dtype=np.float64)
    Hq = q.shape[0]
    G = Hq // Hkv
    K, _ = dequant_pages(pages, P, Hkv, D, seed)
    n = K.shape[0]
    owner = np.concatenate([np.full(nv, j) for j, (_, _, nv) in enumerate(pages)])
    mass = np.zeros(len(pages))
    for h in range(Hq):
        s = K[:, h // G, :] @ q[h] / np.sqrt(D)
        w = np.exp(s - s.max())
        w /= w.sum()
        mass += np.bincount(owner, weights=w, minlength=len(pages))
    assert owner.shape[0] == n
    return mass / Hq
