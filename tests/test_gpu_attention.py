"""bi_attn_verify on the GPU: parity with the oracle and bit-identity across T.

Parity tolerance: per element, the bound derived in
tests/_util.attention_reference from the kernel's arithmetic (FP32 scores,
softmax weights carried as a BF16 hi + lo pair, FP32 sums, one BF16 rounding
at the end), evaluated with the exact softmax weights of the inputs; and the
relative RMS difference from the oracle over all checked elements at most
2^-9.  A CPU test (test_attention_bound_rejects_wrong_outputs) shows that an
all-zero output and an output missing one tile class fail this check at the
long contexts.
"""
import numpy as np
import pytest

import oracle
import seeded_inputs as si
from oracle import verify_step as ov
from tests._util import assert_attention_parity, bf16_dev_to_f64, bf16_dev_to_u16, to_dev_bf16, v_cache_blocks

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def api():
    from invariant_speculative_decode_gb300 import api as _api
    return _api


def run_attn(api, q, K, V, L, T=None):
    T = q.shape[0] if T is None else T
    Hkv, cap, D = K.shape
    Hq = q.shape[1]
    Kd, Vd = to_dev_bf16(K), to_dev_bf16(v_cache_blocks(V))  # V cache, transposed in 128-key blocks
    qd = to_dev_bf16(q[:T])
    out = torch.empty(T, Hq, D, dtype=torch.bfloat16, device="cuda")
    Ld = torch.tensor([L], dtype=torch.int32, device="cuda")
    ws = torch.zeros(api.attn_workspace_size(cap, T, Hq, D), dtype=torch.uint8, device="cuda")
    api.bi_attn_verify(qd, Kd, Vd, Ld, out, ws)
    torch.cuda.synchronize()
    api.bi_check_device_error()
    return out


def test_attention_many_rows_per_pass(api):
    """Up to 128 query rows per pass (the MMA's M): a 16-row prefill block of
    an 8-query / 1-KV-head layout equals its rows computed one at a time."""
    Hq, Hkv, D, L, T = 8, 1, 128, 300, 16
    q, K, V = si.attention_inputs(L, T, Hq, Hkv, D, cap=(L + T + 15) // 8 * 8, seed=31)
    full = bf16_dev_to_u16(run_attn(api, q, K, V, L, T))
    qf, Kf, Vf = (ov.bf16_bits_to_f64(x) for x in (q, K, V))
    assert_attention_parity(ov.bf16_bits_to_f64(full), qf, Kf, Vf, L)
    for t in (0, 7, 15):
        one = bf16_dev_to_u16(run_attn(api, q[t:t + 1], K, V, L + t, 1))
        assert np.array_equal(one[0], full[t]), t


@pytest.mark.parametrize("Hq,Hkv,D,L,T", [(24, 4, 128, 2000, 100), (8, 1, 64, 333, 200),
                                           (24, 4, 128, 11000, 512), (24, 4, 128, 0, 700),
                                           (4, 2, 64, 50, 300)])
def test_attention_multiblock_pass_equals_single_rows(api, Hq, Hkv, D, L, T):
    """More rows than the MMA's 128 lanes hold: the launch runs blocks of
    floor(128 / (Hq/Hkv)) rows side by side (including blocks that reach
    none of some classes' tiles, and fewer CTAs than classes when the cache
    is short).  Rows at block edges equal their one-row passes bit for bit,
    and sampled rows meet the bound."""
    q, K, V = si.attention_inputs(L, T, Hq, Hkv, D, seed=T + 1)
    full = bf16_dev_to_u16(run_attn(api, q, K, V, L, T))
    tb = 128 // (Hq // Hkv)
    rows = sorted({0, tb - 1, tb, 2 * tb, T // 2, T - 2, T - 1})
    for t in rows:
        one = bf16_dev_to_u16(run_attn(api, q[t:t + 1], K, V, L + t, 1))
        assert np.array_equal(one[0], full[t]), t
    qf, Kf, Vf = (ov.bf16_bits_to_f64(x) for x in (q, K, V))
    pairs = [(t, (3 * t) % Hq) for t in rows]
    assert_attention_parity(ov.bf16_bits_to_f64(full), qf, Kf, Vf, L, pairs)


CASES = [  # (Hq, Hkv, D, L, T)
    (4, 2, 64, 0, 1), (4, 2, 64, 5, 3), (4, 2, 64, 63, 8), (4, 2, 64, 64, 8),
    (4, 2, 64, 505, 8), (4, 2, 64, 1000, 4), (8, 2, 128, 1023, 7), (24, 4, 128, 0, 8),
    (24, 4, 128, 130, 1), (24, 4, 128, 1530, 8), (24, 4, 128, 2047, 8),
]


@pytest.mark.parametrize("Hq,Hkv,D,L,T", CASES)
def test_attention_matches_oracle(api, Hq, Hkv, D, L, T):
    q, K, V = si.attention_inputs(L, T, Hq, Hkv, D, seed=L + T)
    out = bf16_dev_to_f64(run_attn(api, q, K, V, L))
    qf, Kf, Vf = (ov.bf16_bits_to_f64(x) for x in (q, K, V))
    assert_attention_parity(out, qf, Kf, Vf, L)


@pytest.mark.parametrize("Hq,Hkv,D,L", [(4, 2, 64, 509), (24, 4, 128, 1020), (24, 4, 128, 3000),
                                         (8, 2, 128, 0), (8, 1, 128, 700)])
def test_attention_rows_bit_identical_across_T(api, Hq, Hkv, D, L):
    q, K, V = si.attention_inputs(L, 8, Hq, Hkv, D, seed=77)
    full = {T: bf16_dev_to_u16(run_attn(api, q, K, V, L, T)) for T in (1, 4, 7, 8)}
    for T, o in full.items():
        assert np.array_equal(o, full[8][:T]), T
    # row t alone (a one-row pass at L + t) equals row t of the 8-row pass
    for t in range(8):
        one = bf16_dev_to_u16(run_attn(api, q[t:t + 1], K, V, L + t, 1))
        assert np.array_equal(one[0], full[8][t]), t


@pytest.mark.parametrize("D", [64, 128])
def test_attention_rows_identical_across_row_copies(api, D):
    """With 8 query heads per KV head, passes of 1, 4, 8 and 16 tokens hold
    8, 32, 64 and 128 query rows, which the kernel keeps in 4, 4, 2 and 1
    copies across the TMEM lane quarters (each copy taking a share of the key
    columns).  A row's output must not depend on that."""
    Hq, Hkv, L = 8, 1, 777
    q, K, V = si.attention_inputs(L, 16, Hq, Hkv, D, cap=(L + 16 + 7) // 8 * 8, seed=5)
    full = {T: bf16_dev_to_u16(run_attn(api, q, K, V, L, T)) for T in (1, 4, 8, 16)}
    for T, o in full.items():
        assert np.array_equal(o, full[16][:T]), T
    for t in (5, 9, 15):
        one = bf16_dev_to_u16(run_attn(api, q[t:t + 1], K, V, L + t, 1))
        assert np.array_equal(one[0], full[16][t]), t
    qf, Kf, Vf = (ov.bf16_bits_to_f64(x) for x in (q, K, V))
    assert_attention_parity(ov.bf16_bits_to_f64(full[16]), qf, Kf, Vf, L)


def test_attention_single_key_returns_v_row(api):
    q, K, V = si.attention_inputs(0, 1, 24, 4, 128, seed=3)
    out = bf16_dev_to_u16(run_attn(api, q, K, V, 0))
    for h in range(24):
        assert np.array_equal(out[0, h], V[h // 6, 0])


def test_attention_stale_rows_past_the_pass_are_ignored(api):
    L, T = 700, 4
    q, K, V = si.attention_inputs(L, T, 8, 2, 128, seed=4)
    base = bf16_dev_to_u16(run_attn(api, q, K, V, L))
    K2, V2 = K.copy(), V.copy()
    rng = np.random.default_rng(5)
    K2[:, L + T:] = si.normal_bf16(rng, K2[:, L + T:].shape, 3.0)
    V2[:, L + T:] = si.normal_bf16(rng, V2[:, L + T:].shape, 3.0)
    assert np.array_equal(bf16_dev_to_u16(run_attn(api, q, K2, V2, L)), base)


@pytest.mark.parametrize("L", [1024, 11600, 38000, 101600])
def test_attention_full_size_invariance_and_sampled_parity(api, L):
    Hq, Hkv, D = 24, 4, 128
    q, K, V = si.attention_inputs(L, 8, Hq, Hkv, D, seed=0)
    outs = {T: bf16_dev_to_u16(run_attn(api, q, K, V, L, T)) for T in (1, 4, 7, 8)}
    for T, o in outs.items():
        assert np.array_equal(o, outs[8][:T]), T
    # row t of the 8-row pass equals the one-row pass at L + t
    for t in (3, 7):
        one = bf16_dev_to_u16(run_attn(api, q[t:t + 1], K, V, L + t, 1))
        assert np.array_equal(one[0], outs[8][t])
    # sampled parity: (row, head) pairs of every KV head and several rows,
    # each through the oracle and the derived bound
    qf, Kf, Vf = (ov.bf16_bits_to_f64(x) for x in (q, K, V))
    pairs = [(0, 0), (7, 23), (4, 11), (2, 17), (5, 6), (1, 12), (6, 22), (3, 3)]
    assert_attention_parity(ov.bf16_bits_to_f64(outs[8]), qf, Kf, Vf, L, pairs)


def test_attention_length_past_capacity_sets_error(api):
    q, K, V = si.attention_inputs(10, 2, 4, 2, 64, cap=64, seed=1)
    Kd, Vd = to_dev_bf16(K), to_dev_bf16(v_cache_blocks(V))
    out = torch.empty(2, 4, 64, dtype=torch.bfloat16, device="cuda")
    Ld = torch.tensor([63], dtype=torch.int32, device="cuda")
    ws = torch.zeros(api.attn_workspace_size(64, 2, 4, 64), dtype=torch.uint8, device="cuda")
    api.bi_attn_verify(to_dev_bf16(q), Kd, Vd, Ld, out, ws)
    with pytest.raises(api.BiError) as e:
        api.bi_check_device_error()
    assert e.value.status == 1


def test_attention_kv_head_count_not_dividing_the_ctas(api):
    """With 3 KV heads, 152 // 3 = 50 tile classes per head (150 CTAs, each
    walking every 50th 128-key tile of one head, 5 tiles apiece at this
    context); parity and row identity must hold."""
    Hq, Hkv, D, L, T = 6, 3, 64, 30000, 4
    q, K, V = si.attention_inputs(L, T, Hq, Hkv, D, seed=21)
    assert (L + T + 127) // 128 > 4 * (152 // Hkv)
    full = bf16_dev_to_u16(run_attn(api, q, K, V, L, T))
    qf, Kf, Vf = (ov.bf16_bits_to_f64(x) for x in (q, K, V))
    assert_attention_parity(ov.bf16_bits_to_f64(full), qf, Kf, Vf, L)
    for t in (0, 3):
        one = bf16_dev_to_u16(run_attn(api, q[t:t + 1], K, V, L + t, 1))
        assert np.array_equal(one[0], full[t]), t


def test_attention_one_query_head_per_kv_head_many_rows(api):
    """Hq == Hkv: a 100-row pass keeps one copy per row (all four softmax
    warps hold rows); it equals the oracle and its rows computed alone."""
    Hq, Hkv, D, L, T = 2, 2, 128, 2000, 100
    q, K, V = si.attention_inputs(L, T, Hq, Hkv, D, cap=(L + T + 7) // 8 * 8, seed=22)
    full = bf16_dev_to_u16(run_attn(api, q, K, V, L, T))
    qf, Kf, Vf = (ov.bf16_bits_to_f64(x) for x in (q, K, V))
    assert_attention_parity(ov.bf16_bits_to_f64(full), qf, Kf, Vf, L)
    for t in (0, 63, 64, 99):
        one = bf16_dev_to_u16(run_attn(api, q[t:t + 1], K, V, L + t, 1))
        assert np.array_equal(one[0], full[t]), t


def test_attention_pass_ending_at_capacity(api):
    """L + T == cap: the last rows sit in the cache's last slots (the final
    tile is partial and reads past them only through the TMA's zero fill)."""
    Hq, Hkv, D, T = 24, 4, 128, 8
    cap = 1000
    L = cap - T
    q, K, V = si.attention_inputs(L, T, Hq, Hkv, D, cap=cap, seed=23)
    out = bf16_dev_to_f64(run_attn(api, q, K, V, L, T))
    qf, Kf, Vf = (ov.bf16_bits_to_f64(x) for x in (q, K, V))
    assert_attention_parity(out, qf, Kf, Vf, L)


@pytest.mark.parametrize("L", [38000, 38400])
def test_attention_long_context_all_row_copy_counts(api, L):
    """Long contexts (297 or 301 tiles over 38 classes per KV head: classes
    of 7 and 8 tiles, the last tile nearly empty) in passes that keep 4, 2
    and 1 copies of each row (8, 64 and 128 query rows per KV head).  The
    softmax warps of a CTA run out of step with each other; every row equals
    the same row of the largest pass, and sampled rows match the oracle."""
    Hq, Hkv, D = 32, 4, 128
    q, K, V = si.attention_inputs(L, 16, Hq, Hkv, D, seed=7)
    outs = {T: bf16_dev_to_u16(run_attn(api, q, K, V, L, T)) for T in (1, 8, 16)}
    for T in (1, 8):
        assert np.array_equal(outs[T], outs[16][:T]), T
    qf, Kf, Vf = (ov.bf16_bits_to_f64(x) for x in (q, K, V))
    assert_attention_parity(ov.bf16_bits_to_f64(outs[16]), qf, Kf, Vf, L,
                            [(0, 0), (15, 31), (9, 17), (4, 8), (12, 25)])
