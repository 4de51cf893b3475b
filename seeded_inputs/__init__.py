"""Seeded synthetic inputs, shared by the oracle-side tests and the CUDA-side harness.

This module holds none of the attention or softmax arithmetic. It holds only:

* SplitMix64, the counter-based 64-bit hash of Steele, Lea and Flood ("Fast splittable
  pseudorandom number generators", OOPSLA 2014), with the constants of its published
  reference implementation.  Element ``i`` of stream ``(seed, stream)`` is
  ``mix(key + (i + 1) * GAMMA)`` so any element can be drawn independently, in any order,
  on any machine, with bit-identical results (x86 here, aarch64 on the GPU host).
* The Box-Muller transform (Box and Muller, 1958) turning two uniforms into one N(0, 1)
  draw, evaluated in float64.
* IEEE round-to-nearest-even narrowing float64 -> float32 -> bfloat16.

Workload recipes (shapes and value distributions) follow the synthetic workloads the
attention/softmax pages describe: i.i.d. N(0, 1) Q/K/V, and softmax rows of 8*N(0, 1) with a
single +30 spike at a seeded column.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_MASK = (1 << 64) - 1
_GAMMA = 0x9E3779B97F4A7C15
_M1 = 0xBF58476D1CE4E5B9
_M2 = 0x94D049BB133111EB

# Stream ids: one independent stream per tensor role.
STREAM_Q, STREAM_K, STREAM_V, STREAM_X, STREAM_SPIKE = 0, 1, 2, 3, 4

_CHUNK = 1 << 18


def _mix_scalar(z: int) -> int:
    z &= _MASK
    z = ((z ^ (z >> 30)) * _M1) & _MASK
    z = ((z ^ (z >> 27)) * _M2) & _MASK
    return z ^ (z >> 31)


def _mix(z: np.ndarray) -> np.ndarray:
    """SplitMix64 finaliser on a uint64 array (numpy uint64 arithmetic wraps mod 2**64)."""
    z ^= z >> np.uint64(30)
    z *= np.uint64(_M1)
    z ^= z >> np.uint64(27)
    z *= np.uint64(_M2)
    z ^= z >> np.uint64(31)
    return z


def stream_key(seed: int, stream: int) -> int:
    """64-bit key of stream ``stream`` under ``seed``."""
    return _mix_scalar(((seed * 1024 + stream + 1) * _GAMMA) & _MASK)


def u64(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """Elements ``start .. start+count-1`` of the counter-based stream, as uint64."""
    key = np.uint64(stream_key(seed, stream))
    idx = np.arange(start + 1, start + 1 + count, dtype=np.uint64)
    idx *= np.uint64(_GAMMA)
    idx += key
    return _mix(idx)


def _normal_chunk(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """Draw ``n`` uses stream elements ``2n`` (u1) and ``2n + 1`` (u2)."""
    key = np.uint64(stream_key(seed, stream))
    ctr = np.arange(2 * start + 1, 2 * (start + count) + 1, 2, dtype=np.uint64)
    a = ctr * np.uint64(_GAMMA)
    a += key
    ctr += np.uint64(1)
    b = ctr * np.uint64(_GAMMA)
    b += key
    a = _mix(a)
    b = _mix(b)
    a >>= np.uint64(11)
    b >>= np.uint64(11)
    u1 = a.astype(np.float64)
    u1 += 1.0
    u1 *= 2.0 ** -53                                      # (0, 1]
    u2 = b.astype(np.float64)
    u2 *= 2.0 * np.pi * 2.0 ** -53                        # 2*pi*[0, 1)
    np.log(u1, out=u1)
    u1 *= -2.0
    np.sqrt(u1, out=u1)
    np.cos(u2, out=u2)
    u1 *= u2
    return u1


def _threads() -> int:
    return max(1, min(32, os.cpu_count() or 1))


def normal_f64(n: int, seed: int, stream: int, scale: float = 1.0,
               out_dtype=np.float64) -> np.ndarray:
    """``n`` draws of ``scale * N(0, 1)`` (Box-Muller on SplitMix64 uniforms, in float64).

    With ``out_dtype=np.float32`` each float64 draw is rounded once, nearest-even.
    """
    out = np.empty(n, dtype=out_dtype)

    def fill(s: int) -> None:
        e = min(n, s + _CHUNK)
        v = _normal_chunk(seed, stream, s, e - s)
        if scale != 1.0:
            v *= scale
        out[s:e] = v

    starts = range(0, n, _CHUNK)
    if n > _CHUNK:
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(fill, starts))
    else:
        for s in starts:
            fill(s)
    return out


def normal_f32(shape, seed: int, stream: int, scale: float = 1.0) -> np.ndarray:
    """``scale * N(0, 1)`` rounded once (nearest-even) to float32, C-contiguous."""
    n = int(np.prod(shape, dtype=np.int64))
    return normal_f64(n, seed, stream, scale, np.float32).reshape(shape)


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest-even); returns the 16-bit patterns as uint16.

    Inputs here are finite, so no NaN handling is needed.
    """
    bits = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    rounding = ((bits >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((bits + rounding) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns to float32."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def qkv(shape_q, shape_kv, seed: int, dtype: str = "f32"):
    """i.i.d. N(0, 1) Q, K, V.

    Returns ``(Q, K, V)`` as float32 arrays when ``dtype == "f32"``; for ``"bf16"`` returns
    uint16 bit patterns (round-to-nearest-even of the float32 draws).
    """
    q = normal_f32(shape_q, seed, STREAM_Q)
    k = normal_f32(shape_kv, seed, STREAM_K)
    v = normal_f32(shape_kv, seed, STREAM_V)
    if dtype == "f32":
        return q, k, v
    if dtype == "bf16":
        return f32_to_bf16_bits(q), f32_to_bf16_bits(k), f32_to_bf16_bits(v)
    raise ValueError(f"unknown dtype {dtype!r}")


def spike_columns(rows: int, T: int, seed: int) -> np.ndarray:
    """Seeded spike column per row: ``u64(seed, SPIKE, r) mod T``."""
    return (u64(seed, STREAM_SPIKE, 0, rows) % np.uint64(T)).astype(np.int64)


def softmax_rows_input(rows: int, T: int, seed: int, sigma: float = 8.0,
                       spike: float = 30.0) -> np.ndarray:
    """``x[rows, T]`` float32: ``sigma * N(0, 1)`` plus ``+spike`` at one seeded column per row.

    Each element is formed in float64 and rounded once to float32.
    """
    base = normal_f64(rows * T, seed, STREAM_X, sigma).reshape(rows, T)
    cols = spike_columns(rows, T, seed)
    base[np.arange(rows), cols] += spike
    return base.astype(np.float32)
