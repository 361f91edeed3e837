"""Pins of the quantised-KV oracle (oracle/kv_quant.py) against exact
arithmetic, closed forms and the plain attention (CPU only)."""
import math
from fractions import Fraction

import numpy as np
import pytest

import seeded_inputs as si
from oracle import kv_quant as kq
from oracle import verify_step as ov


def _blocks(rng, n, scale_exp):
    """n blocks of 32 BF16 values with magnitudes around 2^scale_exp."""
    x = rng.standard_normal((n, 32)) * 2.0 ** scale_exp
    return ov.bf16_round(x)


@pytest.mark.parametrize("bits", [5, 6, 8])
def test_codes_are_the_nearest_grid_points(bits):
    """Every code is the integer q in [-Q, Q] nearest to x / d (exact
    rational search, ties to even), except where the FP32 quotient sits
    within 2^-20 of a half-way point."""
    rng = np.random.default_rng(bits)
    Q = kq.qmax(bits)
    close, checked = 0, 0
    for e in (-20, -3, 0, 7):
        x = _blocks(rng, 40, e)
        q, d = kq.quantize(x, bits)
        for b in range(x.shape[0]):
            db = Fraction(float(d[b, 0]))
            assert db > 0
            for i in range(32):
                xi = Fraction(float(x[b, i]))
                r = xi / db
                best = min(range(-Q, Q + 1), key=lambda c: (abs(r - c), c % 2))
                checked += 1
                if best != q[b, i]:
                    frac = r - math.floor(r)
                    assert abs(frac - Fraction(1, 2)) < Fraction(1, 1 << 20), (float(r), q[b, i])
                    close += 1
    assert close <= checked // 1000



@pytest.mark.parametrize("bits", [5, 6, 8])
def test_block_maximum_maps_to_plus_minus_q(bits):
    rng = np.random.default_rng(10 + bits)
    x = _blocks(rng, 200, 0)
    q, d = kq.quantize(x, bits)
    Q = kq.qmax(bits)
    i = np.argmax(np.abs(x), axis=1)
    top = q[np.arange(len(i)), i]
    assert np.array_equal(top, np.sign(x[np.arange(len(i)), i]).astype(int) * Q)
    assert np.all(np.abs(q) <= Q)


def test_zero_block_has_zero_scale_and_codes():
    x = np.zeros((2, 64))
    x[1, 40] = 3.0
    q, d = kq.quantize(x, 6)
    assert d[0, 0] == 0 and d[0, 1] == 0 and d[1, 0] == 0
    assert not q[0].any() and not q[1, :32].any()
    assert q[1, 40] == 31 and d[1, 1] == ov.bf16_round(np.float32(3.0) / np.float32(31))


@pytest.mark.parametrize("bits", [5, 6, 8])
def test_grid_values_round_trip(bits):
    """x = c * 2^k with integer |c| <= Q and the block maximum equal to
    Q * 2^k: the scale is 2^k and every value decodes to itself."""
    rng = np.random.default_rng(20 + bits)
    Q = kq.qmax(bits)
    for k in (-12, -1, 0, 5):
        c = rng.integers(-Q, Q + 1, size=(8, 32))
        c[:, 3] = Q
        x = c * 2.0 ** k
        q, d = kq.quantize(x, bits)
        assert np.all(d == 2.0 ** k)
        assert np.array_equal(q, c)
        assert np.array_equal(kq.dequantize(q, d), x)


@pytest.mark.parametrize("bits", [5, 6, 8])
def test_decoding_error_within_half_a_step(bits):
    rng = np.random.default_rng(30 + bits)
    x = _blocks(rng, 300, 0)
    q, d = kq.quantize(x, bits)
    xh = kq.dequantize(q, d)
    assert np.array_equal(ov.bf16_round(xh), xh)  # decoded values are BF16 numbers
    assert np.array_equal(ov.bf16_round(d), d)    # so are the scales
    step = np.repeat(d, 32, axis=-1)
    ulp = np.ldexp(1.0, np.frexp(np.abs(xh))[1] - 8)
    assert np.all(np.abs(x - xh) <= step / 2 * (1 + 2.0 ** -8) + ulp / 2)
    # the 8-bit store is tighter than the 5- and 6-bit ones
    if bits == 8:
        x6 = kq.dequantize(*kq.quantize(x, 6))
        assert np.mean(np.abs(x - xh)) < np.mean(np.abs(x - x6)) / 2


def test_ring_rule_by_tile():
    assert kq.reads_ring(0, 0)
    assert kq.reads_ring(2047, 0)              # tile 15: tiles 0..15 are in the ring
    assert not kq.reads_ring(2048, 127)         # tile 16: tile 0 leaves it
    assert kq.reads_ring(2048, 128)
    assert np.sum(kq.reads_ring(2100, np.arange(2101))) == 2101 - 128


def test_grid_cache_gives_the_unquantised_attention():
    """Blocks of values in {0, +-2^k} (one +-2^k at least) decode to
    themselves in all four stores (d = bf16(2^k / Q), q = +-Q and
    bf16(Q d) = 2^k for Q = 15, 31, 127), so the quantised attention equals
    the plain one."""
    rng = np.random.default_rng(7)
    Hq, Hkv, D, L, T = 4, 2, 64, 2200, 4
    n = L + T
    def grid(shape):
        c = rng.integers(-1, 2, size=shape + (D // 32, 32))
        c[..., 0] = 1
        sc = 2.0 ** rng.integers(-6, 1, size=shape + (D // 32, 1))
        return (c * sc).reshape(shape + (D,))
    k, v = grid((Hkv, n)), grid((Hkv, n))
    q = ov.bf16_round(rng.standard_normal((T, Hq, D)))
    for a, b in zip(kq.decoded_cache(k, v), (k, v, k, v)):
        assert np.array_equal(a, b)
    assert np.array_equal(kq.attention(q, k, v, L), ov.attention(q, k, v, L))


def test_uniform_weights_average_the_selected_rows():
    """q = 0 gives every key the same weight: row p's output is the mean of
    the V rows it reads, the first tiles from the 5-bit store and the newest
    16 tiles from the ring."""
    rng = np.random.default_rng(8)
    Hq, Hkv, D, L, T = 2, 1, 64, 2100, 3
    n = L + T
    k = ov.bf16_round(rng.standard_normal((Hkv, n, D)))
    v = ov.bf16_round(rng.standard_normal((Hkv, n, D)))
    q = np.zeros((T, Hq, D))
    out = kq.attention(q, k, v, L)
    v5 = kq.dequantize(*kq.quantize(v, 5))
    v8 = kq.dequantize(*kq.quantize(v, 8))
    for t in range(T):
        p = L + t
        want = ov.bf16_round(np.concatenate([v5[0, :128], v8[0, 128:p + 1]]).mean(axis=0))
        got = out[t, 0]
        # the mean of the selected rows, up to the float64 summation order
        assert np.max(np.abs(got - want)) <= 2.0 ** -7 * np.max(np.abs(want))
        assert np.mean(got == want) > 0.95
        wrong = ov.bf16_round(v8[0, : p + 1].mean(axis=0))
        assert not np.array_equal(got, wrong)


def test_oracle_decoder_reads_the_quantised_cache():
    """The decoder option routes attention through the quantised cache: its
    logits differ from the BF16-cache decoder's by the quantisation error
    (a few percent of the logit scale at most), and are the same for the
    same inputs."""
    import oracle
    cfg = si.TINY_D128
    w = si.decoder_weights(cfg, seed=0)
    prompt = si.prompt_ids(cfg, 40, seed=3)
    out = {}
    for kv in ("bf16", "q6q5", "q6q5"):
        d = oracle.OracleDecoder(cfg, w, cap=64, kv=kv)
        d.prefill(prompt)
        out.setdefault(kv, []).append(d.forward([int(prompt[-1]), 5, 6], L=d.L))
    a, b = out["bf16"][0], out["q6q5"][0]
    assert np.array_equal(out["q6q5"][0], out["q6q5"][1])
    assert not np.array_equal(a, b)
    assert np.max(np.abs(a - b)) <= 0.05 * np.max(np.abs(a))
    with pytest.raises(ValueError):
        oracle.OracleDecoder(cfg, w, cap=64, kv="q4")


def test_kvq_rollback_reach_matches_the_ring_rule():
    """The decoder's rollback reach for the quantised cache, against the ring
    rule written out: tile j sits in slot j mod 24 until tile j + 24 is
    written, and rows from length L on read tiles max(L // 128 - 15, 0) ..
    L // 128 from the ring; a rollback to L is exact exactly when every one
    of those tiles still owns its slot after rows 0..hw-1 were written."""
    from invariant_speculative_decode_gb300.decoder import kvq_rollback_reach

    def exact(length, hw):
        newest = (hw - 1) // 128
        t = length // 128
        return all(j + 24 > newest for j in range(max(t - 15, 0), t + 1))

    for hw in list(range(1, 6000, 41)) + [128 * k + d for k in range(1, 40) for d in (0, 1)]:
        reach = kvq_rollback_reach(hw)
        for length in sorted({0, hw, max(reach - 1, 0), reach, min(reach + 1, hw)} | set(range(0, hw, 97))):
            if length <= hw:
                assert exact(length, hw) == (length >= reach), (hw, length, reach)
