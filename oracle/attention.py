"""Scaled dot-product attention, written out as its definition, in fp64.

Test infrastructure (see package docstring).  The definition is
``O = softmax(mask(Q K^T * scale)) V`` with ``scale = d ** -0.5``, as in [SA] "实现思路"
(the naive PyTorch ``solve``) and [Q3] "自注意力原理" (the torch GQA + causal block).  The
scores are formed explicitly; nothing is blocked, fused or reordered.
"""
from __future__ import annotations

import numpy as np


def attention(Q, K, V, scale: float | None = None, causal: bool = False, q_index=None):
    """Single-head attention.  ``Q[M, d]``, ``K[N, d]``, ``V[N, d]`` -> ``(O[M, d], lse[M])``.

    Steps (each one line of the definition):

    1. ``S = (Q @ K^T) * scale`` -- explicit ``[M, N]`` scores ([SA] "实现思路"; the scale
       multiplies the scores before the maximum).
    2. Causal mask: key ``j`` is dropped (score ``-inf``) when ``j > q_index[i]``; this is
       the top-left aligned ``tril(ones(Sq, Sk))`` of [Q3] "自注意力原理".  ``q_index``
       defaults to ``0..M-1``.
    3. ``m_i = max_j S_ij``; ``E = exp(S - m)``; ``L_i = sum_j E_ij`` (three-pass stable
       softmax, [SO] "Triton 版本 · Baseline").
    4. ``O = (E @ V) / L``; ``lse = m + log L``.

    A row with no unmasked key (``N == 0``, or ``q_index[i] < 0``) gets ``O = 0`` and
    ``lse = -inf`` -- a reading, the pages never meet that case.
    """
    Q = np.asarray(Q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    M, d = Q.shape
    N = K.shape[0]
    if scale is None:
        scale = d ** -0.5
    S = (Q @ K.T) * scale
    if causal:
        qi = np.arange(M) if q_index is None else np.asarray(q_index)
        S = np.where(np.arange(N)[None, :] > qi[:, None], -np.inf, S)
    if N == 0:
        return np.zeros((M, V.shape[1])), np.full(M, -np.inf)
    m = np.max(S, axis=1, keepdims=True)
    m_safe = np.where(np.isneginf(m), 0.0, m)
    E = np.exp(S - m_safe)
    L = np.sum(E, axis=1, keepdims=True)
    with np.errstate(invalid="ignore", divide="ignore"):
        O = np.where(L > 0, (E @ V) / L, 0.0)
        lse = np.where(L[:, 0] > 0, m_safe[:, 0] + np.log(L[:, 0]), -np.inf)
    return O, lse


def _group(Hq: int, Hkv: int) -> int:
    if Hkv <= 0 or Hq % Hkv != 0:
        raise ValueError(f"Hq ({Hq}) must be a positive multiple of Hkv ({Hkv})")
    return Hq // Hkv


MASKS = ("none", "top_left", "bottom_right")


def _q_index(mask: str, Sq: int, Sk: int, i0: int = 0, n: int | None = None):
    """Last key each query row may see, or ``None`` for no mask.

    ``top_left``: row ``i`` sees keys ``0..i`` -- the ``tril(ones(Sq, Sk))`` of [Q3]
    "自注意力原理", which applies it only when ``Sq > 1`` (a single decode row sees every key).
    ``bottom_right``: row ``i`` sees keys ``0..i + Sk - Sq``, i.e. the last query row is the
    last key (a KV cache of ``Sk - Sq`` earlier tokens followed by the ``Sq`` new ones).  The
    pages do not describe this alignment; it is the plainest reading of "the new rows come
    after the cache", and it coincides with ``top_left`` when ``Sq == Sk`` and with no mask
    when ``Sq == 1``.
    """
    if mask not in MASKS:
        raise ValueError(f"mask must be one of {MASKS}")
    n = Sq if n is None else n
    if mask == "none" or (mask == "top_left" and Sq <= 1):
        return None
    off = Sk - Sq if mask == "bottom_right" else 0
    return np.arange(i0, i0 + n) + off


def attention_gqa(Q, K, V, causal: bool = False, scale: float | None = None, mask: str | None = None):
    """Batched grouped-query attention on ``[B, H, S, D]`` tensors.

    ``Q[B, Hq, Sq, D]``, ``K/V[B, Hkv, Sk, D]`` -> ``(O[B, Hq, Sq, D], lse[B, Hq, Sq])``.
    Query head ``hq`` reads kv head ``hq // (Hq // Hkv)``: consecutive query heads share a
    kv head ([Q3] "GQA"; the reshape to ``[B, Hkv, G, Sq, D]`` in "自注意力原理").  The
    causal mask applies only when ``Sq > 1``, as in [Q3] "自注意力原理", so a single query
    row (decode) sees every key.  ``mask`` (``"none"``, ``"top_left"``, ``"bottom_right"``;
    see :func:`_q_index`) overrides ``causal`` (``causal=True`` is ``"top_left"``).
    """
    Q = np.asarray(Q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    B, Hq, Sq, D = Q.shape
    Hkv, Sk = K.shape[1], K.shape[2]
    G = _group(Hq, Hkv)
    qi = _q_index(mask if mask is not None else ("top_left" if causal else "none"), Sq, Sk)
    O = np.empty((B, Hq, Sq, V.shape[3]))
    lse = np.empty((B, Hq, Sq))
    for b in range(B):
        for hq in range(Hq):
            kvh = hq // G
            O[b, hq], lse[b, hq] = attention(Q[b, hq], K[b, kvh], V[b, kvh], scale,
                                             qi is not None, q_index=qi)
    return O, lse


def attention_rows(Q, K, V, rows, causal: bool = False, scale: float | None = None,
                   mask: str | None = None):
    """Selected output rows of :func:`attention_gqa`, one by one.

    ``rows`` is a list of ``(b, hq, i)``; returns ``(O[len(rows), D], lse[len(rows)])``.
    Used to check full-size outputs at sampled positions without the full score matrix.
    """
    B, Hq, Sq, D = Q.shape
    Hkv, Sk = K.shape[1], K.shape[2]
    G = _group(Hq, Hkv)
    mask = mask if mask is not None else ("top_left" if causal else "none")
    outs, lses = [], []
    for b, hq, i in rows:
        kvh = hq // G
        qi = _q_index(mask, Sq, Sk, i0=i, n=1)
        o, l = attention(np.asarray(Q[b, hq, i:i + 1], dtype=np.float64),
                         np.asarray(K[b, kvh], dtype=np.float64),
                         np.asarray(V[b, kvh], dtype=np.float64), scale,
                         qi is not None, q_index=qi)
        outs.append(o[0])
        lses.append(l[0])
    return np.stack(outs), np.array(lses)
