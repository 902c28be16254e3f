"""Seeded synthetic inputs shared by the CUDA path's tests, the oracle's tests and the bench.

This module draws numbers and rounds them to bf16; it holds none of the attention
arithmetic. Both sides of every parity check receive the very same bf16 bit patterns
from here, so neither side ever generates its own inputs.

Recipe (counter-based, so any element can be regenerated independently):

* ``key = mix(seed * 256 + tensor_id)`` where ``mix`` is the SplitMix64 finaliser
  (Steele, Lea and Flood, "Fast splittable pseudorandom number generators", OOPSLA 2014,
  with Vigna's published constants).
* The raw 64-bit word for counter ``c`` is ``mix(key + (c + 1) * 0x9E3779B97F4A7C15)``.
* Normal pair ``n`` uses the words for counters ``2n`` and ``2n + 1``: their top 53 bits give
  ``u1, u2`` in [0, 1); Box-Muller gives ``r = sqrt(-2 ln(1 - u1))``, element ``2n`` is
  ``r cos(2 pi u2)`` and element ``2n + 1`` is ``r sin(2 pi u2)`` (computed in float64).
* The float64 normal is multiplied by ``sigma``, rounded to float32 (round to nearest even),
  then rounded to bf16 (round to nearest even on the float32 bits).

Tensor ids: 0 = Q, 1 = K, 2 = V, 3 = dO.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

TENSOR_Q, TENSOR_K, TENSOR_V, TENSOR_DO = 0, 1, 2, 3


def _mix(z: np.ndarray) -> np.ndarray:
    """SplitMix64 finaliser on a uint64 array (wrapping arithmetic)."""
    z = z.copy()
    z ^= z >> np.uint64(30)
    z *= _M1
    z ^= z >> np.uint64(27)
    z *= _M2
    z ^= z >> np.uint64(31)
    return z


def stream_key(seed: int, tensor_id: int) -> np.uint64:
    base = np.array([(int(seed) * 256 + int(tensor_id)) & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64)
    return _mix(base)[0]


def _normals_chunk(key: np.uint64, start_pair: int, npairs: int) -> np.ndarray:
    pair = np.arange(start_pair, start_pair + npairs, dtype=np.uint64)
    c1 = pair * np.uint64(2)
    w1 = _mix(key + (c1 + np.uint64(1)) * GAMMA)
    w2 = _mix(key + (c1 + np.uint64(2)) * GAMMA)
    scale53 = float(2.0 ** -53)
    u1 = (w1 >> np.uint64(11)).astype(np.float64) * scale53
    u2 = (w2 >> np.uint64(11)).astype(np.float64) * scale53
    r = np.sqrt(-2.0 * np.log1p(-u1))
    t = 2.0 * np.pi * u2
    out = np.empty(2 * npairs, dtype=np.float64)
    out[0::2] = r * np.cos(t)
    out[1::2] = r * np.sin(t)
    return out


def float32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest even); returns uint16 bit patterns."""
    bits = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((bits >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((bits + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_float64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float64."""
    b = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def normal_bf16_bits(shape, seed: int, tensor_id: int, sigma: float = 1.0,
                     threads: int | None = None) -> np.ndarray:
    """uint16 bf16 bit patterns of i.i.d. N(0, sigma^2) draws, row-major ``shape``."""
    n = int(np.prod(shape)) if len(shape) else 1
    out = np.empty(n, dtype=np.uint16)
    if n == 0:
        return out.reshape(shape)
    key = stream_key(seed, tensor_id)
    npairs = (n + 1) // 2
    chunk = 1 << 21  # pairs per chunk
    starts = list(range(0, npairs, chunk))

    def work(p0: int) -> None:
        cnt = min(chunk, npairs - p0)
        z = _normals_chunk(key, p0, cnt) * float(sigma)
        e0 = 2 * p0
        e1 = min(n, e0 + 2 * cnt)
        out[e0:e1] = float32_to_bf16_bits(z[: e1 - e0].astype(np.float32))

    if threads is None:
        threads = min(len(starts), max(1, len(os.sched_getaffinity(0))))
    if threads <= 1 or len(starts) == 1:
        for p0 in starts:
            work(p0)
    else:
        with ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(work, starts))
    return out.reshape(shape)


def attention_inputs(B: int, H: int, N: int, d: int, seed: int, qk_sigma: float = 1.0,
                     v_sigma: float = 1.0, with_dout: bool = False) -> dict:
    """Q, K, V (and dO) as bf16 bit arrays of shape [B, H, N, d]."""
    shape = (B, H, N, d)
    res = {
        "q": normal_bf16_bits(shape, seed, TENSOR_Q, qk_sigma),
        "k": normal_bf16_bits(shape, seed, TENSOR_K, qk_sigma),
        "v": normal_bf16_bits(shape, seed, TENSOR_V, v_sigma),
    }
    if with_dout:
        res["do"] = normal_bf16_bits(shape, seed, TENSOR_DO, 1.0)
    return res


def attention_inputs_ex(B: int, Hq: int, Hkv: int, Tq: int, Tk: int, d: int, seed: int,
                        qk_sigma: float = 1.0, v_sigma: float = 1.0,
                        with_dout: bool = False) -> dict:
    """Q [B, Hq, Tq, d], K and V [B, Hkv, Tk, d] (and dO like Q) as bf16 bit arrays, for
    grouped KV heads and query blocks shorter than the key sequence."""
    res = {
        "q": normal_bf16_bits((B, Hq, Tq, d), seed, TENSOR_Q, qk_sigma),
        "k": normal_bf16_bits((B, Hkv, Tk, d), seed, TENSOR_K, qk_sigma),
        "v": normal_bf16_bits((B, Hkv, Tk, d), seed, TENSOR_V, v_sigma),
    }
    if with_dout:
        res["do"] = normal_bf16_bits((B, Hq, Tq, d), seed, TENSOR_DO, 1.0)
    return res


def sample_rows(N: int, count: int, seed: int, tile: int = 128) -> np.ndarray:
    """Sorted unique row indices: ``count`` seeded rows plus the tile-boundary rows
    {0, tile-1, tile, 2*tile-1, N-tile-1, N-1} that fall inside [0, N)."""
    key = stream_key(seed, 0xA5)
    words = _mix(key + (np.arange(count, dtype=np.uint64) + np.uint64(1)) * GAMMA)
    picks = (words % np.uint64(max(N, 1))).astype(np.int64) if N > 0 else np.zeros(0, np.int64)
    fixed = np.array([0, tile - 1, tile, 2 * tile - 1, N - tile - 1, N - 1], dtype=np.int64)
    fixed = fixed[(fixed >= 0) & (fixed < N)]
    return np.unique(np.concatenate([picks, fixed]))
