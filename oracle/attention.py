"""Decode attention over a mixed-format paged cache: definition, partial
states and the online-softmax merge (fp64).

Pages: "Format-specific kernels compute partial attention states and combine
them through a globally normalized online-softmax merge, enabling direct
heterogeneous decode without a cache-sized dense shadow" (Minima-KV abstract,
mlsanity.com paper page; restated as the "Online-Softmax Recurrence" in the
setupai.cc "Technical Deep Dive").  The merge is exact, so the method computes
plain softmax attention over the dequantised stored cache; that definition is
``attention_dense``.  The partial/merge pair is the recurrence itself, used to
check the definition (invariant: any split of the tokens merges to the
one-pass result) and to stream large contexts.

Readings (silent on the pages): softmax scale 1/sqrt(d); the log-sum-exp is
the natural log of sum_t exp(s_t) over the scaled scores; query head h reads
kv head floor(h / G) with G = H_q / H_kv.
"""
from __future__ import annotations

import numpy as np


def scores(q: np.ndarray, K: np.ndarray) -> np.ndarray:
    """s[h, t] = q_h . K_t / sqrt(d) for one kv head: q [G, d], K [T, d]."""
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    return (q @ K.T) / np.sqrt(q.shape[-1])


def attention_dense(q: np.ndarray, K: np.ndarray, V: np.ndarray):
    """Plain softmax attention for one request.

    q: [Hq, d]; K, V: [T, Hkv, d] (already dequantised).  Returns
    out [Hq, d] and lse [Hq] (natural log)."""
    q = np.asarray(q, dtype=np.float64)
    Hq, d = q.shape
    Hkv = K.shape[1]
    G = Hq // Hkv
    out = np.zeros((Hq, d))
    lse = np.zeros(Hq)
    for h in range(Hq):
        kv = h // G
        s = scores(q[h:h + 1], K[:, kv, :])[0]
        m = np.max(s)
        e = np.exp(s - m)
        out[h] = (e @ np.asarray(V[:, kv, :], dtype=np.float64)) / np.sum(e)
        lse[h] = m + np.log(np.sum(e))
    return out, lse


def partial_state(q: np.ndarray, K: np.ndarray, V: np.ndarray):
    """(m, l, o) of one token set for one kv head: q [G, d], K/V [T, d].

    m = max_t s_t, l = sum_t exp(s_t - m), o = sum_t exp(s_t - m) V_t
    (unnormalised).  An empty set gives (-inf, 0, 0)."""
    q = np.asarray(q, dtype=np.float64)
    G, d = q.shape
    if K.shape[0] == 0:
        return np.full(G, -np.inf), np.zeros(G), np.zeros((G, d))
    s = scores(q, K)
    m = np.max(s, axis=1)
    e = np.exp(s - m[:, None])
    return m, e.sum(axis=1), e @ np.asarray(V, dtype=np.float64)


def merge_states(states):
    """Combine partial states (m_j, l_j, o_j):
    M = max_j m_j, L = sum_j l_j e^{m_j - M}, O = sum_j o_j e^{m_j - M};
    out = O / L, lse = M + ln L.  Empty states (m = -inf) contribute nothing."""
    states = list(states)
    G, d = states[0][2].shape
    ms = np.stack([s[0] for s in states])          # [J, G]
    M = np.max(ms, axis=0)
    L = np.zeros(G)
    O = np.zeros((G, d))
    for m, l, o in states:
        with np.errstate(invalid="ignore"):
            w = np.where(np.isneginf(m), 0.0, np.exp(np.where(np.isneginf(m), 0.0, m - M)))
        L += l * w
        O += o * w[:, None]
    return O / L[:, None], M + np.log(L)


def merge_unnormalised(states):
    """Like ``merge_states`` but returns the merged (M, L, O) state itself."""
    states = list(states)
    G, d = states[0][2].shape
    ms = np.stack([s[0] for s in states])
    M = np.max(ms, axis=0)
    L = np.zeros(G)
    O = np.zeros((G, d))
    for m, l, o in states:
        with np.errstate(invalid="ignore"):
            w = np.where(np.isneginf(m), 0.0, np.exp(np.where(np.isneginf(m), 0.0, m - M)))
        L += l * w
        O += o * w[:, None]
    return M, L, O
