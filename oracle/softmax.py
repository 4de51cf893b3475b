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
