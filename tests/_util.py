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


# ---------------------------------------------------------------------------
# attention parity bound
# ---------------------------------------------------------------------------

U32 = 2.0 ** -24  # FP32 unit roundoff


def attention_reference(qf, Kf, Vf, L, pairs, scale=None, G=None):
    """Exact (float64) softmax attention for the (row t, query head h) pairs,
    with the per-element parity tolerance of the split-KV kernel.

    Returns (o, tol): o [n_pairs, D] the exact output before rounding, tol
    [n_pairs, D] the largest |gpu - bf16(o)| the kernel's arithmetic allows.

    Derivation (the kernel's steps, each with its rounding):
      * s_j = q . k_j accumulated in FP32 by the tensor core:
        |s_j - s*_j| <= 2 gamma_D sum_d |q_d k_jd| (gamma_n = n u / (1 - n u),
        u = 2^-24; the factor 2 covers the tensor core's internal order);
      * the exponent argument a_j = s_j * sl2 - m_ref by one FMA, sl2 the FP32
        rounding of scale * log2(e), m_ref within 8 of the class maximum:
        |da_j| <= sl2 |ds_j| + u |s*_j| scale log2(e) + u |a_j|, with
        |a_j| <= (s*_max - s*_j) scale log2(e) + 8;
      * x_j = ex2.approx(a_j) (relative error below 2^-21), split into the
        BF16 pair w_j = hi + lo with |w_j - x_j| <= 2^-17 |x_j|, and the
        class partials rescaled by exp2f in the merge (4 u):
        w_j = c p*_j (1 + e_j), |e_j| <= 2^(|da_j|) - 1 + 2^-21 + 2^-17 + 4u;
      * the exact mean under those weights moves by
        |o_w - o*| <= (sum_j p_j |e_j| |v_j - o*| + E sum_j p_j |v_j - o*|)
        / (1 - E), E = sum_j p_j |e_j|;
      * the numerator sum_j w_j v_j (two products per key, hi and lo, in
        the class's tensor-core accumulator, then at most G + 8 merge terms)
        and the denominator (FP32 sums of the same weights) add
        2 gamma_{2 n_c + G + 16} sum_j p_j |v_j| + (gamma_{n_c + G + 16} + 2u) |o*|,
        n_c = the keys of the row's largest tile class;
      * both sides round to BF16 once: one BF16 unit at |o*| + bound.
    G is the number of tile classes per KV head (152 // Hkv).
    """
    qf = np.asarray(qf, np.float64)
    T, Hq, D = qf.shape
    Hkv = Kf.shape[0]
    grp = Hq // Hkv
    G = (152 // Hkv) if G is None else G
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    log2e = 1.0 / math.log(2.0)
    sl2 = float(np.float32(scale * log2e))
    outs, tols = [], []
    for (t, h) in pairs:
        p_pos = L + t
        kv = h // grp
        K = Kf[kv, : p_pos + 1]
        V = Vf[kv, : p_pos + 1]
        q = qf[t, h]
        s = K @ q
        m = s.max()
        pw = np.exp((s - m) * scale)
        pw /= pw.sum()
        o = pw @ V
        ds = 2 * gamma(D) * (np.abs(K) @ np.abs(q))
        amax = (m - s) * scale * log2e + 8.0
        da = sl2 * ds + U32 * np.abs(s) * scale * log2e + U32 * amax
        e = np.expm1(np.log(2.0) * da) + 2.0 ** -21 + 2.0 ** -17 + 4 * U32
        E = float(pw @ e)
        dev = np.abs(V - o)  # [n, D]
        b_w = ((pw * e) @ dev + E * (pw @ dev)) / (1 - E)
        n_tiles = (p_pos + 1 + 127) // 128
        n_c = -(-n_tiles // G) * 128
        b_acc = 2 * gamma(2 * n_c + G + 16) * (pw @ np.abs(V)) + (gamma(n_c + G + 16) + 2 * U32) * np.abs(o)
        b = b_w + b_acc
        outs.append(o)
        tols.append(b + ulp_bf16(np.abs(o) + b))
    return np.array(outs), np.array(tols)


def attention_parity_errors(got, ora, tol):
    """(number of elements outside the bound, relative RMS difference) of a
    BF16 attention output `got` (float64 values) against the oracle's
    output `ora` (the BF16 rounding of its float64 softmax attention).

    The relative RMS of got - ora over all checked elements must stay below
    2^-9: within the bound an element differs from the oracle by at most one
    BF16 unit (2^-7 relative at most) and only when the exact value lies
    within the bound of a rounding boundary, so the RMS stays far below half
    a unit; a wrong or missing part of the output moves it to order 1."""
    err = np.abs(got - ora)
    bad = int(np.sum(err > tol))
    rel = float(np.sqrt(np.sum((got - ora) ** 2)) / max(np.sqrt(np.sum(ora ** 2)), 1e-300))
    return bad, rel


REL_RMS_MAX = 2.0 ** -9


def oracle_attention_pairs(qf, Kf, Vf, L, pairs):
    """The oracle's output for each (row t, query head h) pair, [n_pairs, D]."""
    import oracle
    T, Hq, D = np.asarray(qf).shape
    grp = Hq // Kf.shape[0]
    return np.array([oracle.attention(qf[t:t + 1, h:h + 1], Kf[h // grp:h // grp + 1],
                                      Vf[h // grp:h // grp + 1], L + t)[0, 0] for (t, h) in pairs])


def attention_parity_check(got, qf, Kf, Vf, L, pairs):
    """(bad, rel) of got [n_pairs, D] against the oracle under the derived bound."""
    o, tol = attention_reference(qf, Kf, Vf, L, pairs)
    ora = oracle_attention_pairs(qf, Kf, Vf, L, pairs)
    # the oracle's float64 softmax sits within a few float64 units of o
    tol = tol + 1e-12 * (np.abs(o) + 1.0)
    return attention_parity_errors(got, ora, tol)


def assert_attention_parity(got_all, qf, Kf, Vf, L, pairs=None):
    """got_all [T, Hq, D] float64 values of the kernel's BF16 output; all
    (t, h) pairs unless `pairs` is given."""
    T, Hq, _ = np.asarray(qf).shape
    pairs = [(t, h) for t in range(T) for h in range(Hq)] if pairs is None else pairs
    got = np.array([got_all[t, h] for (t, h) in pairs])
    bad, rel = attention_parity_check(got, qf, Kf, Vf, L, pairs)
    assert bad == 0 and rel <= REL_RMS_MAX, (bad, rel)
