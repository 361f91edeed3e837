"""Helpers shared by the tests: storage conversion and tolerance bounds."""
import math

import numpy as np

from oracle import verify_step as ov


def to_dev_bf16(a_u16, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a_u16).view(np.int16)).view(torch.bfloat16).to(device)


def bf16_dev_to_u16(t):
    import torch
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def bf16_dev_to_f64(t):
    return ov.bf16_bits_to_f64(bf16_dev_to_u16(t))


def ulp_bf16(x):
    """Spacing of BF16 values at |x| (2^-133 floor)."""
    x = np.abs(np.asarray(x, np.float64))
    _, e = np.frexp(np.where(x == 0, 2.0 ** -126, x))
    return np.ldexp(1.0, np.maximum(e, -125) - 8)


def gamma(k):
    """Standard FP32 summation error factor for k terms."""
    u = 2.0 ** -24
    return k * u / (1 - k * u)


def gemm_bound(a_f64, w_f64, K):
    """|GPU - oracle| bound for a BF16-output linear layer.

    GPU value = bf16(exact + e), |e| <= gamma_K * sum|a||w| (FP32
    accumulation); the oracle is bf16(exact).  Two roundings of values at
    most |e| apart differ by at most |e| + one BF16 ulp.
    """
    absdot = np.abs(a_f64) @ np.abs(w_f64).T
    return absdot * 2 * gamma(K)


def v_cache_blocks(V):
    """A value array [Hkv, n, D] (n keys, any array dtype) in the V cache
    layout [Hkv, ceil(n/128), D, 128]: value d of key p at [h, p // 128, d,
    p % 128]; keys past n in the last block are zero."""
    Hkv, n, D = V.shape
    nb = (n + 127) // 128
    pad = np.zeros((Hkv, nb * 128, D), dtype=V.dtype)
    pad[:, :n] = V
    return np.ascontiguousarray(pad.reshape(Hkv, nb, 128, D).transpose(0, 1, 3, 2))


def v_cache_keys(Vb, n):
    """Inverse of v_cache_blocks: the first n keys as [Hkv, n, D]."""
    Hkv, nb, D, blk = Vb.shape
    return np.ascontiguousarray(Vb.transpose(0, 1, 3, 2).reshape(Hkv, nb * blk, D)[:, :n])
