"""The pages' online-softmax recurrences, step by step, in fp64.

Test infrastructure (see package docstring).  These are not what GPU outputs are compared
with (that is the plain definition in ``attention.py`` / ``softmax.py``); they restate the
method's own steps so that tests can pin them against the definition (block-size and
split-count invariance, the worked rescale example).
"""
from __future__ import annotations

import numpy as np


def _block_update(m: float, l: float, block: np.ndarray):
    """One step of the boxed recurrence of [SO] "Online Softmax".

    ``m' = max(m, max(block))``; ``l' = l * exp(m - m') + sum(exp(block - m'))``.
    With ``m = m' = -inf`` (nothing seen yet, block all ``-inf``) the state stays
    ``(-inf, 0)``; this guard is a reading (the pages start from ``m = -inf``, ``l = 0``
    and never feed an all ``-inf`` block first).
    """
    m_new = max(m, float(np.max(block))) if block.size else m
    if m_new == -np.inf:
        return m, l
    alpha = np.exp(m - m_new)
    return m_new, l * alpha + float(np.sum(np.exp(block - m_new)))


def online_softmax_state(x, block: int, trace: list | None = None):
    """Streaming ``(m, l)`` over a 1-D ``x`` in blocks of ``block`` elements.

    Invariant after every block ([SO] "Online Softmax"): ``l = sum_{seen} exp(x_j - m)`` with
    ``m`` the maximum seen so far.  ``trace`` (optional list) receives ``(m, l, alpha)``
    after each block, where ``alpha = exp(m_prev - m)`` is the rescale factor of [SA]
    "实现思路".
    """
    x = np.asarray(x, dtype=np.float64).ravel()
    m, l = -np.inf, 0.0
    for s in range(0, x.size, block):
        m_prev = m
        m, l = _block_update(m, l, x[s:s + block])
        if trace is not None:
            alpha = 0.0 if m_prev == -np.inf else float(np.exp(m_prev - m))
            trace.append((m, l, alpha))
    return m, l


def online_softmax(x, block: int) -> np.ndarray:
    """Two-pass online softmax of a 1-D ``x`` ([TP] "Optimized Approach (Two Loops with
    Online Softmax)"; [SO] "Online Softmax"): pass 1 builds ``(m, l)`` block by block,
    pass 2 writes ``exp(x - m) / l``."""
    x = np.asarray(x, dtype=np.float64).ravel()
    m, l = online_softmax_state(x, block)
    return np.exp(x - m) / l


def online_attention_row(q, K, V, block: int, scale: float | None = None,
                         n_keys: int | None = None):
    """One query row through the blocked recurrence of [SA] "实现思路" (its pseudocode).

    Per key block: scores ``s = q . k * scale`` (keys at or beyond ``n_keys`` score
    ``-inf``, the tail mask), ``m' = max(m, max s)``, ``alpha = exp(m - m')``,
    ``p = exp(s - m')``, ``l = l * alpha + sum p``, ``acc = acc * alpha + p @ v``.  The row
    is ``acc / l``.  Returns ``(o, m, l)``.
    """
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    d = q.shape[0]
    if scale is None:
        scale = d ** -0.5
    N = K.shape[0] if n_keys is None else n_keys
    m, l = -np.inf, 0.0
    acc = np.zeros(V.shape[1])
    for start in range(0, K.shape[0], block):
        k = K[start:start + block]
        v = V[start:start + block]
        s = (k @ q) * scale
        idx = np.arange(start, start + k.shape[0])
        s = np.where(idx < N, s, -np.inf)
        m_new = max(m, float(np.max(s)))
        if m_new == -np.inf:
            continue
        alpha = np.exp(m - m_new)
        p = np.exp(s - m_new)
        l = l * alpha + float(np.sum(p))
        acc = acc * alpha + p @ v
        m = m_new
    return acc / l, m, l


def combine_partials(ms, ls, accs):
    """Merge partial states ``(m_s, l_s, acc_s)`` of disjoint key chunks.

    The boxed rule of [SO] "Online Softmax" applied to whole partial states instead of one
    block: ``M = max_s m_s``, ``l = sum_s exp(m_s - M) l_s``,
    ``acc = sum_s exp(m_s - M) acc_s``; the row is ``acc / l`` and its log-sum-exp is
    ``M + log l``.  Chunks with ``m_s = -inf`` (no keys) contribute nothing.  This is the
    split-K decode combine; the pages give the rule, not the split (a reading).
    Returns ``(o, lse)``.
    """
    ms = np.asarray(ms, dtype=np.float64)
    ls = np.asarray(ls, dtype=np.float64)
    accs = np.asarray(accs, dtype=np.float64)
    M = np.max(ms)
    w = np.where(np.isneginf(ms), 0.0, np.exp(ms - M))
    l = float(np.sum(w * ls))
    acc = np.sum(w[:, None] * accs, axis=0)
    return acc / l, M + np.log(l)
