"""Gradients of scaled dot-product attention, written out as their definition, in fp64.

Test infrastructure (see package docstring).  The pages describe only the forward pass
``O = softmax(mask(Q K^T * scale)) V`` ([SA] "实现思路", [Q3] "自注意力原理" / "GQA"); the
backward pass here is the plain chain rule through that definition for a scalar loss whose
gradient with respect to ``O`` is ``dO``:

* ``P = softmax(S)`` with ``S = mask(Q K^T * scale)`` (masked entries ``-inf`` so ``P = 0``)
* ``dV = P^T dO``
* ``dP = dO V^T``
* ``dS = P * (dP - rowsum(dP * P))``  -- the Jacobian of a row softmax applied to ``dP``
* ``dQ = scale * dS K``,  ``dK = scale * dS^T Q``

Grouped-query attention: a kv head's ``dK`` and ``dV`` are the sums over its ``G`` query heads
(each query head reads the same K, V).  Nothing is blocked or fused.
"""
from __future__ import annotations

import numpy as np

from .attention import _group, _q_index


def attention_bwd(Q, K, V, dO, scale: float | None = None, q_index=None):
    """Single head: ``Q[M, d]``, ``K/V[N, d]``, ``dO[M, d]`` -> ``(dQ, dK, dV)``.

    ``q_index[i]`` is the last key row ``i`` may see (``None``: every key), as in
    :func:`oracle.attention`.  Rows that see no key contribute nothing.
    """
    Q, K, V, dO = (np.asarray(a, dtype=np.float64) for a in (Q, K, V, dO))
    M, d = Q.shape
    N = K.shape[0]
    if scale is None:
        scale = d ** -0.5
    S = (Q @ K.T) * scale
    if q_index is not None:
        S = np.where(np.arange(N)[None, :] > np.asarray(q_index)[:, None], -np.inf, S)
    m = np.max(S, axis=1, keepdims=True) if N else np.zeros((M, 1))
    m_safe = np.where(np.isneginf(m), 0.0, m)
    E = np.exp(S - m_safe)
    L = np.sum(E, axis=1, keepdims=True)
    with np.errstate(invalid="ignore", divide="ignore"):
        P = np.where(L > 0, E / L, 0.0)
    dV = P.T @ dO
    dP = dO @ V.T
    dS = P * (dP - np.sum(dP * P, axis=1, keepdims=True))
    dQ = scale * (dS @ K)
    dK = scale * (dS.T @ Q)
    return dQ, dK, dV


def attention_gqa_bwd(Q, K, V, dO, mask: str = "none", scale: float | None = None):
    """Batched GQA on ``[B, H, S, D]``: ``(dQ[B,Hq,Sq,D], dK[B,Hkv,Sk,D], dV[B,Hkv,Sk,D])``.

    ``mask`` as in :func:`oracle.attention_gqa` (``none``, ``top_left``, ``bottom_right``).
    """
    Q, K, V, dO = (np.asarray(a, dtype=np.float64) for a in (Q, K, V, dO))
    B, Hq, Sq, D = Q.shape
    Hkv, Sk = K.shape[1], K.shape[2]
    G = _group(Hq, Hkv)
    qi = _q_index(mask, Sq, Sk)
    dQ = np.zeros_like(Q)
    dK = np.zeros_like(K)
    dV = np.zeros_like(V)
    for b in range(B):
        for hq in range(Hq):
            kvh = hq // G
            gq, gk, gv = attention_bwd(Q[b, hq], K[b, kvh], V[b, kvh], dO[b, hq], scale, qi)
            dQ[b, hq] = gq
            dK[b, kvh] += gk
            dV[b, kvh] += gv
    return dQ, dK, dV
