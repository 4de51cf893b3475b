"""Three-pass stable softmax in fp64 -- test infrastructure (see package docstring).

Follows the three-loop form of [TP] "Puzzle 8: Long Softmax", "Brute-Force Approach (Three
Loops)", and the three-stage stable softmax of [SO] "Triton 版本 · Baseline": subtracting
the row maximum is allowed because softmax is invariant under a common shift of its
inputs, and it keeps every exponent <= 0.
"""
from __future__ import annotations

import numpy as np


def softmax(x) -> np.ndarray:
    """Row softmax along the last axis, in fp64.

    1. ``m = max_j x_j``                       (pass 1)
    2. ``e_j = exp(x_j - m)``, ``L = sum_j e_j`` (pass 2)
    3. ``z_j = e_j / L``                       (pass 3)

    A row whose entries are all ``-inf`` has no defined softmax; it yields zeros (a reading:
    the pages never meet that case).  An empty last axis returns an empty array.
    """
    x = np.asarray(x, dtype=np.float64)
    if x.shape[-1] == 0:
        return x.copy()
    m = np.max(x, axis=-1, keepdims=True)
    m_safe = np.where(np.isneginf(m), 0.0, m)
    e = np.exp(x - m_safe)
    L = np.sum(e, axis=-1, keepdims=True)
    with np.errstate(invalid="ignore", divide="ignore"):
        z = e / L
    return np.where(L > 0, z, 0.0)


def softmax_masked(x, scale: float = 1.0, causal_period: int = 0) -> np.ndarray:
    """Row softmax of ``scale * x`` over ``x[rows, T]`` with an optional causal mask, in fp64.

    The softmax of [Q3] "自注意力原理" / "使用triton实现" (a softmax over attention-weight rows
    with a scale and, for causal attention, the load condition "column <= row", which fills
    the part above the diagonal with -inf so it becomes 0 after the exponential):

    1. ``s_j = scale * x_j``
    2. if ``causal_period > 0``: ``s_j = -inf`` for ``j > r % causal_period``, ``r`` the row
       number -- the row within its own ``[Sq, Sk]`` score matrix when rows of several heads are
       stacked (``causal_period = Sq``; a single matrix has ``causal_period = rows``)
    3. :func:`softmax` of ``s``
    """
    x = np.asarray(x, dtype=np.float64)
    s = x * float(scale)
    if causal_period > 0:
        rows, T = s.shape
        r = np.arange(rows) % causal_period
        s = np.where(np.arange(T)[None, :] > r[:, None], -np.inf, s)
    return softmax(s)
