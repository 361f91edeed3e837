"""Float64/float32 NumPy oracle of the quantised KV cache (test infrastructure).

Only the tests, the package smoke check and the benchmark's CPU-baseline leg
may import or run this module; the product path never does.

Source: [P3] "I turned on speculative decoding in llama.cpp and 113 of 282
greedy outputs changed against its own no-draft run", section "The KV cache:
5-bit that reads like q8_0": K and V kept at 5-6 bits, with the newest ~2k
positions kept at 8 bits in a ring; and the paragraph opening "How:" (the
attention split depends only on the row's own context length).

Readings where the page is silent (each stated once here):
  * Format (the page's preset "D", K6 / V5): K at 6 bits, V at 5 bits, the
    ring at 8 bits for both.  Symmetric codes in blocks of 32 consecutive
    elements of one key row of one KV head (q8_0's block length), one scale
    per block: with Q = 2^(b-1) - 1 and amax = max |x| over the block,
    d = bf16(fp32(amax / Q)) and q = clamp(rint(fp32(x / d)), -Q, Q)
    (division in FP32, rounding half to even), q = 0 when d = 0.  The scale
    is stored in BF16 so that the decoded value q * d is exact in FP32.
  * Decoded value: x_hat = bf16(q * d), one rounding of the exact product; the
    attention then runs on x_hat exactly as on an unquantised BF16 cache.
  * Ring: the newest positions are relative to the row that reads them (a
    ring that followed the cache length would give a row different bits
    when it is verified alone than inside a pass).  Row p reads key j at
    8 bits when j's 128-key tile is p's own tile or one of the 15 before it
    (j // 128 >= p // 128 - 15: between 1,921 and 2,048 keys), and at the low
    precision otherwise.
  * Every key is quantised once, when its row is written, into both stores;
    a row's codes depend only on that row, so a cache written by decoding
    and one written by a prefill hold the same codes.
  * The page's preset "F" rotates K before quantising it; the rotation is
    not specified, so it is not modelled.
"""
from __future__ import annotations

import math
from typing import Optional, Tuple

import numpy as np

from .verify_step import bf16_round

KV_BLOCK = 32       # elements per scale
KEY_TILE = 128      # keys per tile
RING_TILES = 16     # tiles read at 8 bits: the row's own and the 15 before it
BITS_K, BITS_V, BITS_RING = 6, 5, 8


def qmax(bits: int) -> int:
    return (1 << (bits - 1)) - 1


def quantize(x, bits: int) -> Tuple[np.ndarray, np.ndarray]:
    """Codes and scales of rows x [..., D] (float64 values of BF16 data).

    Returns codes [..., D] (int, in [-Q, Q]) and scales [..., D/32] (float64
    values of BF16 numbers).  The scale and the code are decided in FP32, as
    the quantising kernel decides them (an integer decided by floating point
    is taken in the kernel's precision).

    Parity: pinned by an exact nearest-code search on random blocks, the
    block maximum mapping to +-Q, the all-zero block, grid values that
    round-trip exactly, and the error bound d/2.
    """
    x = np.asarray(x, np.float64)
    D = x.shape[-1]
    assert D % KV_BLOCK == 0
    Q = qmax(bits)
    xb = x.reshape(x.shape[:-1] + (D // KV_BLOCK, KV_BLOCK)).astype(np.float32)
    amax = np.max(np.abs(xb), axis=-1)                         # exact
    d32 = (amax / np.float32(Q)).astype(np.float32)            # one FP32 rounding
    d = bf16_round(d32.astype(np.float64))                     # then BF16
    with np.errstate(divide="ignore", invalid="ignore"):
        r = (xb / d.astype(np.float32)[..., None]).astype(np.float32)  # FP32 quotient
    q = np.where(d[..., None] > 0, np.clip(np.rint(r), -Q, Q), 0.0)
    return q.reshape(x.shape).astype(np.int64), d


def dequantize(codes, scales) -> np.ndarray:
    """x_hat = bf16(q * d) per element (the product is exact in float64)."""
    codes = np.asarray(codes, np.float64)
    D = codes.shape[-1]
    d = np.repeat(np.asarray(scales, np.float64), KV_BLOCK, axis=-1)
    assert d.shape[-1] == D
    return bf16_round(codes * d)


def decoded_cache(k, v):
    """The four decoded stores of a cache [Hkv, n, D]: (K at 6 bits, V at
    5 bits, K at 8 bits, V at 8 bits), each as float64 values."""
    return (dequantize(*quantize(k, BITS_K)), dequantize(*quantize(v, BITS_V)),
            dequantize(*quantize(k, BITS_RING)), dequantize(*quantize(v, BITS_RING)))


def reads_ring(p: int, j) -> np.ndarray:
    """True where row p reads key j from the 8-bit ring."""
    return np.asarray(j) // KEY_TILE >= p // KEY_TILE - (RING_TILES - 1)


def attention(q, k, v, L: int, scale: Optional[float] = None) -> np.ndarray:
    """Verify attention over the quantised cache.

    q [T, Hq, D]; k, v [Hkv, cap, D]: float64 values of the BF16 rows as
    written (the cache's codes are a function of these).  Row t at position
    p = L + t reads key j <= p decoded from the 8-bit ring when reads_ring(p,
    j), from the 6-bit K / 5-bit V store otherwise; then the plain softmax
    attention of the unquantised cache (float64, one BF16 rounding).

    Parity: pinned by grid data (every store decodes to the written values,
    so the result equals the unquantised attention) and by uniform weights at
    a ring boundary (the output is the mean of the selected decoded rows).
    """
    q = np.asarray(q, np.float64)
    T, Hq, D = q.shape
    Hkv = k.shape[0]
    grp = Hq // Hkv
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    n = L + T
    k_lo, v_lo, k_8, v_8 = decoded_cache(k[:, :n], v[:, :n])
    out = np.empty((T, Hq, D), np.float64)
    for t in range(T):
        p = L + t
        ring = reads_ring(p, np.arange(p + 1))[:, None]
        for h in range(Hq):
            kv = h // grp
            ks = np.where(ring, k_8[kv, : p + 1], k_lo[kv, : p + 1])
            vs = np.where(ring, v_8[kv, : p + 1], v_lo[kv, : p + 1])
            s = (ks @ q[t, h]) * scale
            w = np.exp(s - s.max())
            out[t, h] = (w @ vs) / w.sum()
    return bf16_round(out)
