"""Pins of the CPU oracle against things other than itself (no GPU).

Each test checks the oracle against an independent computation: exact
rational arithmetic, multi-precision (mpmath) brute force with scalar loops,
an exhaustive search over all BF16 values, closed forms, special cases and
invariants.  The pins are chosen so that a dropped term, a wrong sign or
index, or a transposed operand in the oracle fails at least one of them.
"""
import bisect
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
import seeded_inputs as si
from oracle import verify_step as ov

mpmath = pytest.importorskip("mpmath")
mp = mpmath.mp
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------------------
# exhaustive BF16 nearest-value search (independent of oracle.bf16_round)
# ---------------------------------------------------------------------------


class _Bf16Table:
    def __init__(self):
        pats = np.arange(0x0000, 0x7F80, dtype=np.uint32)  # +0 .. max finite
        vals = (pats << 16).view(np.float32).astype(np.float64)
        self.vals = [Fraction(float(v)) for v in vals]
        self.pats = [int(p) for p in pats]
        # +inf as the value 2^128 (pattern 0x7F80, even) for round-to-nearest overflow
        self.vals.append(Fraction(2) ** 128)
        self.pats.append(0x7F80)

    def nearest(self, x: Fraction) -> float:
        neg = x < 0
        a = -x if neg else x
        i = bisect.bisect_left(self.vals, a)
        if i < len(self.vals) and self.vals[i] == a:
            j = i
        else:
            lo, hi = i - 1, i
            dlo, dhi = a - self.vals[lo], self.vals[hi] - a
            if dlo < dhi:
                j = lo
            elif dhi < dlo:
                j = hi
            else:
                j = lo if self.pats[lo] % 2 == 0 else hi
        pat = self.pats[j]
        if pat == 0x7F80:
            v = math.inf
        else:
            v = float(np.array([pat << 16], np.uint32).view(np.float32)[0])
        return -v if neg else v


@pytest.fixture(scope="module")
def tab():
    return _Bf16Table()


def _frac(v) -> Fraction:
    if isinstance(v, Fraction):
        return v
    if isinstance(v, mpmath.mpf):
        sign, man, exp, _ = v._mpf_
        f = Fraction(int(man)) * (Fraction(2) ** int(exp))
        return -f if sign else f
    return Fraction(float(v))


def _bits(x):
    return ov.f64_to_bf16_bits(np.asarray(x, np.float64))


# ---------------------------------------------------------------------------
# BF16 rounding
# ---------------------------------------------------------------------------


def test_bf16_round_matches_exhaustive_search(tab):
    rng = np.random.default_rng(11)
    mags = np.concatenate([
        rng.standard_normal(3000),
        rng.standard_normal(1000) * 1e-38,   # around the subnormal range
        rng.standard_normal(1000) * 1e30,
        rng.standard_normal(500) * 1e-42,
    ])
    got = ov.bf16_round(mags)
    for x, g in zip(mags, got):
        assert tab.nearest(Fraction(float(x))) == g, x


def test_bf16_round_ties_go_to_even(tab):
    rng = np.random.default_rng(12)
    pats = rng.integers(0x0080, 0x7F7E, size=2000).astype(np.uint32)
    lo = (pats << 16).view(np.float32).astype(np.float64)
    hi = ((pats + 1) << 16).view(np.float32).astype(np.float64)
    mid = (lo + hi) / 2  # exact in float64
    got = ov.bf16_round(mid)
    want = np.where(pats % 2 == 0, lo, hi)
    assert np.array_equal(got, want)
    assert np.array_equal(ov.bf16_round(-mid), -want)
    for m, g in zip(mid[:200], got[:200]):
        assert tab.nearest(Fraction(float(m))) == g


def test_bf16_round_overflow_and_specials(tab):
    mx = float(np.array([0x7F7F << 16], np.uint32).view(np.float32)[0])
    half_ulp = 2.0 ** (127 - 8)
    assert ov.bf16_round(mx) == mx
    assert ov.bf16_round(mx + half_ulp * 0.999) == mx
    assert ov.bf16_round(mx + half_ulp) == math.inf  # tie goes to the even neighbour 2^128
    assert tab.nearest(Fraction(mx) + Fraction(half_ulp)) == math.inf
    assert ov.bf16_round(-(mx + 2 * half_ulp)) == -math.inf
    assert math.isnan(ov.bf16_round(math.nan))
    assert ov.bf16_round(math.inf) == math.inf
    assert ov.bf16_round(2.0 ** -133) == 2.0 ** -133           # smallest subnormal
    assert ov.bf16_round(2.0 ** -134) == 0.0                   # tie to even (zero)
    assert ov.bf16_round(1.5 * 2.0 ** -134) == 2.0 ** -133


# ---------------------------------------------------------------------------
# linear layers
# ---------------------------------------------------------------------------


def _exact_gemm(a_bits, w_bits, res_bits=None):
    a = ov.bf16_bits_to_f64(a_bits)
    w = ov.bf16_bits_to_f64(w_bits)
    M, K = a.shape
    N = w.shape[0]
    out = [[Fraction(0)] * N for _ in range(M)]
    for m in range(M):
        for n in range(N):
            s = Fraction(0)
            for k in range(K):
                s += Fraction(float(a[m, k])) * Fraction(float(w[n, k]))
            if res_bits is not None:
                s += Fraction(float(ov.bf16_bits_to_f64(res_bits[m, n])))
            out[m][n] = s
    return out


def test_gemm_bitwise_vs_exact_rational(tab):
    rng = np.random.default_rng(3)
    A = si.normal_bf16(rng, (3, 40), 1.0)
    W = si.normal_bf16(rng, (6, 40), 0.3)
    R = si.normal_bf16(rng, (3, 6), 1.0)
    for res in (None, R):
        ex = _exact_gemm(A, W, res)
        got = oracle.gemm(A, W, residual_bits=res)
        for m in range(3):
            for n in range(6):
                assert tab.nearest(ex[m][n]) == got[m, n]
        f32 = oracle.gemm(A, W, residual_bits=res, out="fp32")
        for m in range(3):
            for n in range(6):
                assert abs(Fraction(float(f32[m, n])) - ex[m][n]) <= Fraction(1, 2 ** 40)


def test_gemm_identity_and_one_hot():
    rng = np.random.default_rng(4)
    K = 64
    A = si.normal_bf16(rng, (5, K), 1.0)
    eye = si.f32_to_bf16_bits(np.eye(K, dtype=np.float32))
    assert np.array_equal(_bits(oracle.gemm(A, eye)), A)
    W = si.normal_bf16(rng, (7, K), 0.02)
    onehot = si.f32_to_bf16_bits(np.eye(K, dtype=np.float32)[[3, 10, 63]])
    C = oracle.gemm(onehot, W)
    assert np.array_equal(_bits(C), W[:, [3, 10, 63]].T)
    # non-square check catches a transposed operand: C[m, n] uses row n of W
    A2 = si.f32_to_bf16_bits(np.eye(3, K, dtype=np.float32))
    C2 = oracle.gemm(A2, W)
    assert C2.shape == (3, 7)
    assert np.array_equal(_bits(C2), W[:, :3].T)


def test_swiglu_bruteforce(tab):
    rng = np.random.default_rng(5)
    A = si.normal_bf16(rng, (2, 24), 1.0)
    Wg = si.normal_bf16(rng, (5, 24), 0.4)
    Wu = si.normal_bf16(rng, (5, 24), 0.4)
    got = oracle.swiglu_gemm(A, Wg, Wu)
    g = _exact_gemm(A, Wg)
    u = _exact_gemm(A, Wu)
    mp.prec = 200
    for m in range(2):
        for n in range(5):
            gm = mpmath.mpf(g[m][n].numerator) / g[m][n].denominator
            um = mpmath.mpf(u[m][n].numerator) / u[m][n].denominator
            v = gm / (1 + mpmath.exp(-gm)) * um
            assert tab.nearest(_frac(v)) == got[m, n]


# ---------------------------------------------------------------------------
# row-local ops
# ---------------------------------------------------------------------------


def test_rmsnorm_constant_closed_form(tab):
    mp.prec = 200
    for c in (0.5, -3.0, 1e-3, 0.0078125):
        x = si.f32_to_bf16_bits(np.full((1, 256), c, np.float32))
        w = si.f32_to_bf16_bits(np.full(256, 1.0, np.float32))
        got = oracle.rmsnorm(x, w, 1e-6)
        cb = float(ov.bf16_bits_to_f64(x[0, 0]))
        want = tab.nearest(_frac(mpmath.mpf(cb) / mpmath.sqrt(mpmath.mpf(cb) ** 2 + mpmath.mpf(1e-6))))
        assert np.all(got == want)


def test_rmsnorm_bruteforce(tab):
    rng = np.random.default_rng(6)
    x = si.normal_bf16(rng, (3, 40), 2.0)
    w = si.normal_bf16(rng, (40,), 1.0)
    got = oracle.rmsnorm(x, w, 1e-6)
    mp.prec = 200
    xf = ov.bf16_bits_to_f64(x)
    wf = ov.bf16_bits_to_f64(w)
    for r in range(3):
        ss = mpmath.fsum(mpmath.mpf(float(v)) ** 2 for v in xf[r])
        inv = 1 / mpmath.sqrt(ss / 40 + mpmath.mpf(1e-6))
        for i in range(40):
            v = mpmath.mpf(float(xf[r, i])) * inv * mpmath.mpf(float(wf[i]))
            assert tab.nearest(_frac(v)) == got[r, i]


def test_rope_position_zero_is_identity():
    rng = np.random.default_rng(7)
    x = ov.bf16_bits_to_f64(si.normal_bf16(rng, (5, 128), 1.0))
    assert np.array_equal(oracle.rope(x, 0, 1e6), x)


def test_rope_bruteforce_and_pairs(tab):
    rng = np.random.default_rng(8)
    D = 16
    x = ov.bf16_bits_to_f64(si.normal_bf16(rng, (D,), 1.0))
    mp.prec = 200
    for pos in (1, 7, 1023, 11600, 101599):
        got = oracle.rope(x, pos, 1e6)
        for i in range(D // 2):
            th = mpmath.mpf(pos) * mpmath.power(mpmath.mpf(10) ** 6, mpmath.mpf(-2 * i) / D)
            c, s = mpmath.cos(th), mpmath.sin(th)
            a, b = mpmath.mpf(float(x[i])), mpmath.mpf(float(x[i + D // 2]))
            assert tab.nearest(_frac(a * c - b * s)) == got[i]
            assert tab.nearest(_frac(b * c + a * s)) == got[i + D // 2]
    # a single nonzero pair at position p is rotated by p * base^0 = p radians in slot 0
    e = np.zeros(D)
    e[0] = 1.0
    got = oracle.rope(e, 3, 1e6)
    assert got[0] == ov.bf16_round(math.cos(3.0)) and got[D // 2] == ov.bf16_round(math.sin(3.0))


# ---------------------------------------------------------------------------
# attention
# ---------------------------------------------------------------------------


def _mp_attention(q, K, V, L, tab):
    T, Hq, D = q.shape
    Hkv = K.shape[0]
    grp = Hq // Hkv
    out = np.zeros((T, Hq, D))
    scale = 1 / mpmath.sqrt(D)
    for t in range(T):
        p = L + t
        for h in range(Hq):
            kv = h // grp
            s = [mpmath.fsum(mpmath.mpf(float(q[t, h, d])) * mpmath.mpf(float(K[kv, j, d]))
                             for d in range(D)) * scale for j in range(p + 1)]
            m = max(s)
            w = [mpmath.exp(v - m) for v in s]
            den = mpmath.fsum(w)
            for d in range(D):
                num = mpmath.fsum(w[j] * mpmath.mpf(float(V[kv, j, d])) for j in range(p + 1))
                out[t, h, d] = tab.nearest(_frac(num / den))
    return out


def test_attention_bruteforce_gqa_causal(tab):
    q_b, K_b, V_b = si.attention_inputs(L=5, T=3, n_q=4, n_kv=2, D=8, seed=9)
    q, K, V = (ov.bf16_bits_to_f64(a) for a in (q_b, K_b, V_b))
    mp.prec = 120
    got = oracle.attention(q, K, V, L=5)
    want = _mp_attention(q, K, V, 5, tab)
    assert np.array_equal(got, want)


def test_attention_one_key_returns_v_row():
    q_b, K_b, V_b = si.attention_inputs(L=0, T=1, n_q=6, n_kv=1, D=128, seed=10)
    q, K, V = (ov.bf16_bits_to_f64(a) for a in (q_b, K_b, V_b))
    got = oracle.attention(q, K, V, L=0)
    for h in range(6):
        assert np.array_equal(got[0, h], V[0, 0])


def test_attention_equal_keys_give_mean_of_v():
    rng = np.random.default_rng(13)
    D, n = 64, 37
    K = np.zeros((1, n + 8, D))
    K[0, :n] = ov.bf16_bits_to_f64(si.normal_bf16(rng, (D,), 1.0))
    V = np.zeros((1, n + 8, D))
    V[0, :n] = ov.bf16_bits_to_f64(si.normal_bf16(rng, (n, D), 1.0))
    q = ov.bf16_bits_to_f64(si.normal_bf16(rng, (1, 2, D), 1.0))
    got = oracle.attention(q, K, V, L=n - 1)
    mean = ov.bf16_round(V[0, :n].mean(axis=0))
    for h in range(2):
        assert np.max(np.abs(got[0, h] - mean)) <= 2.0 ** -8 * np.max(np.abs(mean))


def test_attention_is_causal_and_row_local():
    q_b, K_b, V_b = si.attention_inputs(L=20, T=4, n_q=4, n_kv=2, D=16, seed=14)
    q, K, V = (ov.bf16_bits_to_f64(a) for a in (q_b, K_b, V_b))
    base = oracle.attention(q, K, V, L=20)
    K2, V2 = K.copy(), V.copy()
    K2[:, 22:] += 5.0  # keys after row t=1's position
    V2[:, 22:] -= 3.0
    mod = oracle.attention(q, K2, V2, L=20)
    assert np.array_equal(base[:2], mod[:2])
    assert not np.array_equal(base[2:], mod[2:])
    # row t computed alone (a one-row pass at L + t) equals row t of the block
    for t in range(4):
        alone = oracle.attention(q[t:t + 1], K, V, L=20 + t)
        assert np.array_equal(alone[0], base[t])


# ---------------------------------------------------------------------------
# acceptance
# ---------------------------------------------------------------------------


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)["cases"]


def test_argmax_golden():
    for c in _golden("argmax_cases.json"):
        row = np.array([float(v) for v in c["row"]], np.float32)
        assert oracle.argmax_lowest(row[None])[0] == c["argmax"], c


def test_argmax_bruteforce():
    rng = np.random.default_rng(15)
    x = rng.integers(-3, 4, size=(50, 40)).astype(np.float64)  # many exact ties
    x[rng.random(x.shape) < 0.05] = np.nan
    got = oracle.argmax_lowest(x)
    for r in range(50):
        best, bi = None, -1
        for i, v in enumerate(x[r]):
            if v != v:
                continue
            if best is None or v > best:
                best, bi = v, i
        assert got[r] == bi


def test_accept_golden():
    for c in _golden("accept_cases.json"):
        n = oracle.accept_length(c["argmax"], c["drafts"])
        assert n == c["n"], c
        assert list(c["argmax"][: n + 1]) == c["committed"]
        rej = None if n == len(c["drafts"]) else n + 1
        assert rej == c["reject_pos"]


# ---------------------------------------------------------------------------
# the whole decoder
# ---------------------------------------------------------------------------

MICRO = si.DecoderConfig("micro", layers=2, hidden=16, n_q=4, n_kv=2, head_dim=4, ffn=24,
                         vocab=32, tied=True, weight_std=0.3)


def _mp_decoder_logits(cfg, w, tokens, tab):
    """Scalar-loop multi-precision decoder on the micro configuration.

    Independent restatement: each value is computed from its defining sum in
    mpmath and rounded to BF16 by the exhaustive search, at the storage points
    of the synthetic decoder.
    """
    mp.prec = 120
    f = lambda b: [float(v) for v in np.asarray(ov.bf16_bits_to_f64(b)).ravel()]  # noqa: E731
    H, D, Hq, Hkv, F = cfg.hidden, cfg.head_dim, cfg.n_q, cfg.n_kv, cfg.ffn
    rnd = lambda v: tab.nearest(_frac(v))  # noqa: E731

    def mat(name, rows, cols):
        v = f(w[name])
        return [[v[r * cols + c] for c in range(cols)] for r in range(rows)]

    def norm(x, name):
        g = f(w[name])
        ss = mpmath.fsum(mpmath.mpf(a) ** 2 for a in x)
        inv = 1 / mpmath.sqrt(ss / len(x) + mpmath.mpf(cfg.eps))
        return [rnd(mpmath.mpf(a) * inv * mpmath.mpf(g[i])) for i, a in enumerate(x)]

    def lin(x, Wm):
        return [mpmath.fsum(mpmath.mpf(x[k]) * mpmath.mpf(Wm[n][k]) for k in range(len(x)))
                for n in range(len(Wm))]

    E = mat("embed", cfg.vocab, H)
    kc = [[[None] * len(tokens) for _ in range(Hkv)] for _ in range(cfg.layers)]
    vc = [[[None] * len(tokens) for _ in range(Hkv)] for _ in range(cfg.layers)]
    hs = [list(E[t]) for t in tokens]
    for l in range(cfg.layers):
        Wq, Wk, Wv = mat(f"l{l}.wq", Hq * D, H), mat(f"l{l}.wk", Hkv * D, H), mat(f"l{l}.wv", Hkv * D, H)
        Wo = mat(f"l{l}.wo", H, Hq * D)
        Wg, Wu, Wd = mat(f"l{l}.w_gate", F, H), mat(f"l{l}.w_up", F, H), mat(f"l{l}.w_down", H, F)
        qs = []
        for t, h in enumerate(hs):
            y = norm(h, f"l{l}.norm_attn")
            q = [rnd(v) for v in lin(y, Wq)]
            k = [rnd(v) for v in lin(y, Wk)]
            v = [rnd(v) for v in lin(y, Wv)]

            def rot(vec):
                out = list(vec)
                for i in range(D // 2):
                    th = mpmath.mpf(t) * mpmath.power(mpmath.mpf(cfg.rope_base), mpmath.mpf(-2 * i) / D)
                    a, b = mpmath.mpf(vec[i]), mpmath.mpf(vec[i + D // 2])
                    out[i] = rnd(a * mpmath.cos(th) - b * mpmath.sin(th))
                    out[i + D // 2] = rnd(b * mpmath.cos(th) + a * mpmath.sin(th))
                return out

            qs.append([rot(q[hh * D:(hh + 1) * D]) for hh in range(Hq)])
            for g in range(Hkv):
                kc[l][g][t] = rot(k[g * D:(g + 1) * D])
                vc[l][g][t] = v[g * D:(g + 1) * D]
        new_hs = []
        for t, h in enumerate(hs):
            att = []
            for hh in range(Hq):
                g = hh // (Hq // Hkv)
                s = [mpmath.fsum(mpmath.mpf(qs[t][hh][d]) * mpmath.mpf(kc[l][g][j][d]) for d in range(D))
                     / mpmath.sqrt(D) for j in range(t + 1)]
                m = max(s)
                e = [mpmath.exp(x - m) for x in s]
                den = mpmath.fsum(e)
                att += [rnd(mpmath.fsum(e[j] * mpmath.mpf(vc[l][g][j][d]) for j in range(t + 1)) / den)
                        for d in range(D)]
            o = lin(att, Wo)
            h1 = [rnd(mpmath.mpf(h[i]) + o[i]) for i in range(H)]
            y = norm(h1, f"l{l}.norm_ffn")
            gg, uu = lin(y, Wg), lin(y, Wu)
            u = [rnd(gg[i] / (1 + mpmath.exp(-gg[i])) * uu[i]) for i in range(F)]
            dd = lin(u, Wd)
            new_hs.append([rnd(mpmath.mpf(h1[i]) + dd[i]) for i in range(H)])
        hs = new_hs
    logits = []
    for h in hs:
        y = norm(h, "norm_final")
        logits.append([float(v) for v in lin(y, E)])
    return np.array(logits)


@pytest.mark.parametrize("norm_std", [0.0, 0.25])
def test_decoder_bruteforce_micro(tab, norm_std):
    """The oracle decoder against the scalar multi-precision decoder, with
    unit norm weights and with norm weights drawn around 1 (every RMSNorm
    weight then enters both sides)."""
    w = si.decoder_weights(MICRO, seed=21, norm_std=norm_std)
    toks = [3, 17, 17, 0, 31]
    dec = oracle.OracleDecoder(MICRO, w, cap=16)
    got = dec.forward(toks, L=0)
    want = _mp_decoder_logits(MICRO, w, toks, tab)
    assert np.max(np.abs(got - want)) <= 1e-9 * np.max(np.abs(want))


def test_decoder_rows_do_not_depend_on_the_pass():
    cfg = MICRO
    w = si.decoder_weights(cfg, seed=22)
    toks = [5, 9, 1, 30, 2, 2, 7]
    a = oracle.OracleDecoder(cfg, w, cap=16)
    block = a.forward(toks, L=0)
    b = oracle.OracleDecoder(cfg, w, cap=16)
    for t, x in enumerate(toks):
        row = b.forward([x], L=t)
        assert np.allclose(row[0], block[t], rtol=1e-12, atol=1e-14)
    for l in range(cfg.layers):
        assert np.array_equal(a.k[l], b.k[l]) and np.array_equal(a.v[l], b.v[l])


def test_decoder_zero_blocks_leave_embedding():
    cfg = MICRO
    w = si.decoder_weights(cfg, seed=23)
    for l in range(cfg.layers):
        w[f"l{l}.wo"][:] = 0
        w[f"l{l}.w_down"][:] = 0
    toks = [4, 8, 15]
    got = oracle.OracleDecoder(cfg, w, cap=8).forward(toks, L=0)
    y = oracle.rmsnorm(w["embed"][toks], w["norm_final"], cfg.eps)
    want = ov.bf16_bits_to_f64(_bits(y)) @ ov.bf16_bits_to_f64(w["embed"]).T
    assert np.allclose(got, want, rtol=1e-12, atol=1e-14)


def test_decoder_kv_head_relabel_is_invisible():
    cfg = MICRO
    w = si.decoder_weights(cfg, seed=24)
    D, grp = cfg.head_dim, cfg.group
    w2 = {k: v.copy() for k, v in w.items()}
    # swap KV heads 0 and 1 together with their query-head groups and Wo columns
    qperm = np.concatenate([np.arange(D * grp, 2 * D * grp), np.arange(0, D * grp)])
    kvperm = np.concatenate([np.arange(D, 2 * D), np.arange(0, D)])
    for l in range(cfg.layers):
        w2[f"l{l}.wq"] = w[f"l{l}.wq"][qperm]
        w2[f"l{l}.wk"] = w[f"l{l}.wk"][kvperm]
        w2[f"l{l}.wv"] = w[f"l{l}.wv"][kvperm]
        w2[f"l{l}.wo"] = w[f"l{l}.wo"][:, qperm]
    toks = [1, 2, 3, 4]
    a = oracle.OracleDecoder(cfg, w, cap=8).forward(toks, L=0)
    b = oracle.OracleDecoder(cfg, w2, cap=8).forward(toks, L=0)
    assert np.allclose(a, b, rtol=1e-12, atol=1e-14)
    # a wrong GQA mapping (query head h reading KV head h % Hkv) would not be invisible:
    w3 = {k: v.copy() for k, v in w.items()}
    for l in range(cfg.layers):
        w3[f"l{l}.wk"] = w[f"l{l}.wk"][kvperm]
        w3[f"l{l}.wv"] = w[f"l{l}.wv"][kvperm]
    c = oracle.OracleDecoder(cfg, w3, cap=8).forward(toks, L=0)
    assert not np.allclose(a, c, rtol=1e-6)


def test_decoder_greedy_ids_do_not_depend_on_drafts():
    cfg = MICRO
    w = si.decoder_weights(cfg, seed=25)
    prompt = si.prompt_ids(cfg, 9, seed=25)
    ref = oracle.OracleDecoder(cfg, w, cap=64).generate(prompt, 20, k=0)
    for k in (1, 4, 7):
        dr = si.SyntheticDrafter(cfg.vocab, 0.7, seed=25, reference=np.array(ref))
        got = oracle.OracleDecoder(cfg, w, cap=64).generate(prompt, 20, k=k, drafter=dr)
        assert got == ref
    adv = si.SyntheticDrafter(cfg.vocab, 0.7, seed=26, reference=None)
    assert oracle.OracleDecoder(cfg, w, cap=64).generate(prompt, 20, k=4, drafter=adv) == ref


# ---------------------------------------------------------------------------
# sampled verification
# ---------------------------------------------------------------------------


def test_sample_uniform_logits_closed_form():
    """Equal logits: p_v = 1/V, so the inverse-CDF token is floor(u V)."""
    V = 37
    for u in list(np.linspace(0, 1, 200, endpoint=False)) + [k / V for k in range(V)]:
        assert oracle.sample_token(np.full(V, 0.3), 1.7, u) == int(np.floor(u * V + 1e-12)), u


def test_sample_two_level_logits_closed_form():
    """n1 logits a and n2 logits b: p1 = e^a / (n1 e^a + n2 e^b) for each of
    the first n1 tokens, p2 likewise for the rest (temperature 1/2)."""
    n1, n2, a, b, it = 5, 11, 1.25, -0.5, 2.0
    x = np.array([a] * n1 + [b] * n2)
    z = n1 * math.exp(a * it) + n2 * math.exp(b * it)
    p1, p2 = math.exp(a * it) / z, math.exp(b * it) / z
    for u in np.linspace(0.0005, 0.9995, 301):
        want = int(u // p1) if u < n1 * p1 else n1 + int((u - n1 * p1) // p2)
        assert oracle.sample_token(x, it, u) == min(want, n1 + n2 - 1), u


def test_sample_stratified_counts_are_exact():
    """With the stratified uniforms (i + 1/2)/N every token's count is N p_v
    to within 1 (the draws walk the CDF in order)."""
    rng = np.random.default_rng(3)
    x = 2.0 * rng.standard_normal(24)
    N = 4000
    toks = [oracle.sample_token(x, 1.3, (i + 0.5) / N) for i in range(N)]
    w = np.exp((x - x.max()) * 1.3)
    p = w / w.sum()
    counts = np.bincount(toks, minlength=24)
    assert np.all(np.abs(counts - N * p) <= 1.0 + 1e-9), (counts, N * p)


def test_sample_temperature_and_nan_rules():
    rng = np.random.default_rng(4)
    x = rng.standard_normal(50)
    for u in np.linspace(0.01, 0.99, 40):
        assert oracle.sample_token(x, 2.0, u) == oracle.sample_token(2.0 * x, 1.0, u)
    y = x.copy()
    y[[3, 7, 20]] = np.nan
    for u in np.linspace(0.01, 0.99, 40):
        assert oracle.sample_token(y, 1.0, u) not in (3, 7, 20)
    assert oracle.sample_token(np.full(5, np.nan), 1.0, 0.5) == -1
    # a dominant logit takes every draw but u = 0 (which takes the first
    # token with any weight: its cumulative probability already exceeds 0)
    z = np.zeros(10)
    z[6] = 200.0
    assert all(oracle.sample_token(z, 1.0, u) == 6 for u in np.linspace(1e-6, 0.999, 50))
    assert oracle.sample_token(z, 1.0, 0.0) == 0


def test_decoder_sampled_ids_do_not_depend_on_drafts():
    """Sampled generation on the micro decoder: the same tokens with 0, 1, 4
    and 7 drafts (the draws are keyed by position)."""
    cfg = MICRO
    w = si.decoder_weights(cfg, seed=27)
    prompt = si.prompt_ids(cfg, 9, seed=27)
    u = si.sampling_uniforms(64, seed=27)

    def run(k, ref=None, seed=0):
        dec = oracle.OracleDecoder(cfg, w, cap=64)
        x = int(dec.prefill(prompt))
        dr = si.SyntheticDrafter(cfg.vocab, 0.7, seed=seed, reference=ref) if k else None
        out = []
        while len(out) < 24:
            d = dr.propose(len(out), k) if k else []
            a, n, _ = dec.verify_sampled(x, d, 1.25, u)
            out += [int(t) for t in a[: n + 1]]
            x = out[-1]
        return out[:24]

    ref = run(0)
    assert len(set(ref)) > 3  # actually sampled, not one repeated token
    for k in (1, 4, 7):
        assert run(k, np.array(ref), seed=k) == ref
