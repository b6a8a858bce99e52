"""Attention with the row softmax inside it, in double on the CPU.

TEST INFRASTRUCTURE ONLY, like the rest of this package: only tests/,
``__graft_entry__.smoke()`` and bench.py's CPU legs may use it.  It shares no
code with the CUDA path.

"Triton GPU programming deep dive" (ybb.press), section 3.1, writes attention
as ``softmax(Q K^T / sqrt(d)) V``; section 3.3 computes it a tile of keys at a
time with a running max m_i and running sum l_i: per key tile the scores
qk = Q K^T (masked to -inf where a key index exceeds the query index),
m_ij = max(m_i, rowmax(qk)), p = exp(qk - m_ij), l_ij = rowsum(p),
alpha = exp(m_i - m_ij), l_i = l_i * alpha + l_ij, acc = acc * alpha + p V,
m_i = m_ij; finally acc / l_i.

``attention`` is the definition (scores, row softmax, weighted sum of V);
``attention_online`` follows section 3.3's steps in their order.  Shapes:
q [BH, n_q, d], k and v [BH, n_k, d], float64; the causal mask keeps key j
for query i iff j <= i + offset (offset 0: the page's mask).  A query row with
no visible key (every key masked, or no key at all) is the softmax of only
-inf: NaN, and its logsumexp is -inf.
"""
from __future__ import annotations

import numpy as np


def _visible(n_q: int, n_k: int, causal: bool, offset: int) -> np.ndarray:
    if not causal:
        return np.ones((n_q, n_k), dtype=bool)
    return np.arange(n_k)[None, :] <= np.arange(n_q)[:, None] + offset


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float | None = None,
              causal: bool = False, offset: int = 0) -> np.ndarray:
    """softmax(scale * q k^T, masked) v for each of the BH (batch, head) pairs."""
    q, k, v = (np.asarray(a, dtype=np.float64) for a in (q, k, v))
    d = q.shape[-1]
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    out = np.empty(q.shape[:-1] + (v.shape[-1],), dtype=np.float64)
    keep = _visible(q.shape[1], k.shape[1], causal, offset)
    with np.errstate(invalid="ignore"):
        for b in range(q.shape[0]):
            s = scale * (q[b] @ k[b].T)
            s = np.where(keep, s, -np.inf)
            # The max of no score is -inf; the weights' sum then is 0 and the
            # weighted sum of V over no key, divided by it, is 0/0 = NaN.
            m = s.max(axis=1, keepdims=True, initial=-np.inf)
            e = np.exp(s - m)
            out[b] = (e @ v[b]) / e.sum(axis=1, keepdims=True)
    return out


def attention_online(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float | None = None,
                     causal: bool = False, offset: int = 0, block_n: int = 64) -> np.ndarray:
    """The same result, one tile of block_n keys at a time (section 3.3).  A
    tile whose running max is still -inf adds nothing (as in the row oracle)."""
    q, k, v = (np.asarray(a, dtype=np.float64) for a in (q, k, v))
    d = q.shape[-1]
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    n_q, n_k = q.shape[1], k.shape[1]
    keep = _visible(n_q, n_k, causal, offset)
    out = np.empty(q.shape[:-1] + (v.shape[-1],), dtype=np.float64)
    with np.errstate(invalid="ignore"):
        for b in range(q.shape[0]):
            m_i = np.full(n_q, -np.inf)
            l_i = np.zeros(n_q)
            acc = np.zeros((n_q, v.shape[-1]))
            for start_n in range(0, n_k, block_n):
                kt, vt = k[b, start_n:start_n + block_n], v[b, start_n:start_n + block_n]
                qk = scale * (q[b] @ kt.T)
                qk = np.where(keep[:, start_n:start_n + block_n], qk, -np.inf)
                m_ij = np.maximum(m_i, qk.max(axis=1))
                live = m_ij > -np.inf
                ref = np.where(live, m_ij, 0.0)
                p = np.exp(qk - ref[:, None])
                l_ij = p.sum(axis=1)
                alpha = np.where(live, np.exp(m_i - ref), 1.0)
                l_i = l_i * alpha + l_ij
                acc = acc * alpha[:, None] + p @ vt
                m_i = m_ij
            out[b] = acc / l_i[:, None]
    return out


def logsumexp(q: np.ndarray, k: np.ndarray, scale: float | None = None, causal: bool = False,
              offset: int = 0) -> np.ndarray:
    """Natural-log logsumexp of each query row's masked, scaled scores [BH, n_q]."""
    q, k = (np.asarray(a, dtype=np.float64) for a in (q, k))
    d = q.shape[-1]
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    keep = _visible(q.shape[1], k.shape[1], causal, offset)
    out = np.empty(q.shape[:2])
    with np.errstate(invalid="ignore", divide="ignore"):
        for b in range(q.shape[0]):
            s = np.where(keep, scale * (q[b] @ k[b].T), -np.inf)
            m = s.max(axis=1, initial=-np.inf)
            ref = np.where(m > -np.inf, m, 0.0)
            out[b] = ref + np.log(np.exp(s - ref[:, None]).sum(axis=1))
    return out
