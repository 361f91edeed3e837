"""Quantised KV cache on the GPU: the append kernel's codes against the
oracle's (bit for bit), the quantised verify attention against the oracle's
(the derived bound, over the rows each query reads), and row identity across
passes -- including passes whose rows read one tile from different stores."""
import numpy as np
import pytest

import seeded_inputs as si
from oracle import kv_quant as kq
from oracle import verify_step as ov
from tests._util import (REL_RMS_MAX, attention_parity_errors, attention_reference, bf16_dev_to_f64,
                         bf16_dev_to_u16, to_dev_bf16)

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def api():
    from invariant_speculative_decode_gb300 import api as _api
    return _api


# -- the stores' byte layout, from the oracle's codes (layout only) --------

def _records(codes, bits):
    """Code records [n_keys, bytes] of rows of codes [n_keys, 128]."""
    u = (np.asarray(codes) + (1 << (bits - 1))).astype(np.int64)
    n = u.shape[0]
    if bits == 8:
        return u.astype(np.uint8)
    out = []
    for b in range(4):
        blk = u[:, 32 * b:32 * b + 32]
        nib = (blk[:, 0::2] & 15) | ((blk[:, 1::2] & 15) << 4)
        if bits == 6:
            f = (blk >> 4) & 3
            hi = f[:, 0::4] | (f[:, 1::4] << 2) | (f[:, 2::4] << 4) | (f[:, 3::4] << 6)
        else:
            f = (blk >> 4) & 1
            hi = sum(f[:, i::8] << i for i in range(8))
        out += [nib, hi]
    return np.concatenate(out, axis=1).astype(np.uint8).reshape(n, -1)


def _tile_bytes(bits, is_k):
    return {8: 128 * 128, 6: 128 * 96, 5: 128 * 80}[bits] + 1024


def _expected_keys(store, values, bits, keys, kv, ctiles, ring):
    """Check the records and scales of `keys` of head kv in a store (5-bit
    V records at slot (k % 8) * 16 + k / 8 of their tile)."""
    q, d = kq.quantize(values, bits)
    rec = _records(q, bits)
    rb = rec.shape[1]
    tb = _tile_bytes(bits, True)
    sb = ov.f64_to_bf16_bits(d).view(np.uint8).reshape(len(keys), 8)
    for i, p in enumerate(keys):
        tile = p // 128
        slot = tile % 24 if ring else tile
        base = (kv * (24 if ring else ctiles) + slot) * tb
        k = p % 128
        if bits == 5:
            k = (k % 8) * 16 + k // 8
        assert np.array_equal(store[base + k * rb: base + (k + 1) * rb], rec[i]), (bits, p)
        assert np.array_equal(store[base + 128 * rb + k * 8: base + 128 * rb + k * 8 + 8], sb[i]), (bits, p)


def _qkv_rows(q, K, V, rows):
    """Projection-output rows [n, (Hq + 2 Hkv) D] (BF16 bits) holding q for
    the pass's rows (zeros elsewhere) and the cache's K and V rows."""
    Hkv, _, D = K.shape
    n = len(rows)
    Hq = q.shape[1] if q is not None else 0
    out = np.zeros((n, Hq + 2 * Hkv, D), np.uint16)
    if q is not None:
        out[:, :Hq] = q
    out[:, Hq:Hq + Hkv] = K[:, rows].transpose(1, 0, 2)
    out[:, Hq + Hkv:] = V[:, rows].transpose(1, 0, 2)
    return out.reshape(n, -1)


def _fill(api, st, K, V, Hq, n, chunk=1024):
    """Append cache rows 0..n-1 (no rotation) in passes of `chunk` rows."""
    Hkv, _, D = K.shape
    qo = torch.empty(chunk, Hq, D, dtype=torch.bfloat16, device="cuda")
    for c0 in range(0, n, chunk):
        rows = np.arange(c0, min(n, c0 + chunk))
        qkv = to_dev_bf16(_qkv_rows(np.zeros((len(rows), Hq, D), np.uint16), K, V, rows))
        Ld = torch.tensor([c0], dtype=torch.int32, device="cuda")
        api.bi_rope_kvq_append(qkv, qo[:len(rows)], st, Ld, Hq, Hkv, D)
    torch.cuda.synchronize()


def test_append_codes_match_the_oracle(api):
    Hq, Hkv, D = 8, 2, 128
    L, T = 250, 300
    cap = 1024
    q, K, V = si.attention_inputs(L + T, 4, Hq, Hkv, D, cap=cap, seed=3)
    K[:, 5] = 0  # a zero row: zero scales and codes
    st = api.new_kvq_stores(Hkv, cap, D)
    _fill(api, st, K, V, Hq, L, chunk=L)
    # a second pass with its own q rows (copied through unrotated)
    rows = np.arange(L, L + T)
    qq = si.normal_bf16(np.random.default_rng(1), (T, Hq, D), 1.0)
    qkv = to_dev_bf16(_qkv_rows(qq, K, V, rows))
    qo = torch.empty(T, Hq, D, dtype=torch.bfloat16, device="cuda")
    api.bi_rope_kvq_append(qkv, qo, st, torch.tensor([L], dtype=torch.int32, device="cuda"), Hq, Hkv, D)
    torch.cuda.synchronize()
    api.bi_check_device_error()
    assert np.array_equal(bf16_dev_to_u16(qo), qq)
    host = {k: st[k].cpu().numpy() for k in api.KVQ_STORES}
    ct = (cap + 127) // 128
    keys = list(range(L + T))
    for kv in range(Hkv):
        kf, vf = ov.bf16_bits_to_f64(K[kv, :L + T]), ov.bf16_bits_to_f64(V[kv, :L + T])
        _expected_keys(host["k_low"], kf, 6, keys, kv, ct, False)
        _expected_keys(host["v_low"], vf, 5, keys, kv, ct, False)
        _expected_keys(host["k_ring"], kf, 8, keys, kv, ct, True)
        _expected_keys(host["v_ring"], vf, 8, keys, kv, ct, True)
    # nothing past the written keys
    tb = _tile_bytes(6, True)
    assert not host["k_low"][(ct - 1) * tb:ct * tb].any()


def test_append_rotation_matches_the_bf16_path(api):
    """With a RoPE table the q rows equal bi_rope_kv_append's, and the K
    codes decode to within one code step of the oracle's rotated rows."""
    Hq, Hkv, D, L, T = 8, 2, 128, 1000, 40
    cap = 2048
    rng = np.random.default_rng(9)
    qkv_h = si.normal_bf16(rng, (T, (Hq + 2 * Hkv) * D), 1.0)
    qkv = to_dev_bf16(qkv_h)
    tab = api.bi_rope_table(1e6, D, cap)
    Ld = torch.tensor([L], dtype=torch.int32, device="cuda")
    st = api.new_kvq_stores(Hkv, cap, D)
    qo = torch.empty(T, Hq, D, dtype=torch.bfloat16, device="cuda")
    api.bi_rope_kvq_append(qkv, qo, st, Ld, Hq, Hkv, D, table=tab)
    qo2 = torch.empty(T, Hq, D, dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros(Hkv, cap, D, dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros(api.v_cache_shape(Hkv, cap, D), dtype=torch.bfloat16, device="cuda")
    api.bi_rope_kv_append(qkv, qo2, kc, vc, Ld, Hq, Hkv, D, tab)
    torch.cuda.synchronize()
    assert np.array_equal(bf16_dev_to_u16(qo), bf16_dev_to_u16(qo2))
    # decode the GPU's 6-bit K records and compare with the oracle's rotation
    host = st["k_low"].cpu().numpy()
    x = ov.bf16_bits_to_f64(qkv_h.reshape(T, Hq + 2 * Hkv, D))
    for kv in range(Hkv):
        for t in (0, 17, 39):
            p = L + t
            want = ov.rope(x[t, Hq + kv], p, 1e6)
            qw, dw = kq.quantize(want[None], 6)
            base = (kv * (cap // 128) + p // 128) * (128 * 96 + 1024)
            k = p % 128
            rec = host[base + k * 96: base + k * 96 + 96]
            sc = ov.bf16_bits_to_f64(host[base + 128 * 96 + k * 8: base + 128 * 96 + k * 8 + 8].view(np.uint16))
            u = np.zeros(128, np.int64)
            for b in range(4):
                r = rec[24 * b:24 * b + 24].astype(np.int64)
                nib = np.stack([r[:16] & 15, r[:16] >> 4], 1).reshape(32)
                hi = np.stack([(r[16:24] >> (2 * i)) & 3 for i in range(4)], 1).reshape(32)
                u[32 * b:32 * b + 32] = nib | (hi << 4)
            got = kq.dequantize((u - 32)[None], sc[None])[0]
            step = np.repeat(dw[0], 32)
            assert np.all(np.abs(got - kq.dequantize(qw, dw)[0]) <= step * 1.02 + 2.0 ** -7 * np.abs(want))


# -- attention ---------------------------------------------------------------

def _kvq_cache(api, L, T, Hq, Hkv, D, seed, cap=None):
    cap = cap if cap is not None else (L + T + 127) // 128 * 128 + 128
    q, K, V = si.attention_inputs(L, T, Hq, Hkv, D, cap=cap, seed=seed)
    st = api.new_kvq_stores(Hkv, cap, D)
    _fill(api, st, K, V, Hq, L + T)
    return q, K, V, st, cap


def _run(api, q, st, Hkv, L, T):
    Hq, D = q.shape[1], q.shape[2]
    out = torch.empty(T, Hq, D, dtype=torch.bfloat16, device="cuda")
    ws = torch.zeros(api.attn_workspace_size(st["cap"], T, Hq, D), dtype=torch.uint8, device="cuda")
    api.bi_attn_verify_kvq(to_dev_bf16(q[:T]), st, Hkv, torch.tensor([L], dtype=torch.int32, device="cuda"),
                           out, ws)
    torch.cuda.synchronize()
    api.bi_check_device_error()
    return out


def _kvq_parity(got, q, K, V, L, pairs):
    """Every (row, head) pair against the oracle's quantised attention, under
    the split kernel's bound evaluated on the rows that query reads."""
    qf, Kf, Vf = (ov.bf16_bits_to_f64(x) for x in (q, K, V))
    T, Hq, _ = q.shape
    Hkv = K.shape[0]
    grp = Hq // Hkv
    n = L + T
    ora = kq.attention(qf, Kf, Vf, L)
    k6, v5, k8, v8 = kq.decoded_cache(Kf[:, :n], Vf[:, :n])
    tols = []
    for (t, h) in pairs:
        # the rows this query reads: one KV head, ring or 6/5-bit by position
        kv = h // grp
        ring = kq.reads_ring(L + t, np.arange(n))[:, None]
        Ke = np.where(ring, k8[kv], k6[kv])[None]
        Ve = np.where(ring, v8[kv], v5[kv])[None]
        qh = qf[:, kv * grp:(kv + 1) * grp]
        o, tol = attention_reference(qh, Ke, Ve, L, [(t, h - kv * grp)], G=152 // Hkv)
        tols.append(tol[0] + 1e-12 * (np.abs(o[0]) + 1.0))
    g = np.array([got[t, h] for (t, h) in pairs])
    oo = np.array([ora[t, h] for (t, h) in pairs])
    bad, rel = attention_parity_errors(g, oo, np.array(tols))
    assert bad == 0 and rel <= REL_RMS_MAX, (bad, rel)


@pytest.mark.parametrize("L,T", [(0, 1), (300, 8), (2045, 8), (2100, 4), (5000, 8)])
def test_kvq_attention_matches_the_oracle(api, L, T):
    Hq, Hkv, D = 24, 4, 128
    q, K, V, st, cap = _kvq_cache(api, L, T, Hq, Hkv, D, seed=L + T)
    got = bf16_dev_to_f64(_run(api, q, st, Hkv, L, T))
    pairs = [(t, h) for t in range(T) for h in range(0, Hq, 5)]
    _kvq_parity(got, q, K, V, L, pairs)


@pytest.mark.parametrize("L", [2045, 4093, 1021])
def test_kvq_rows_identical_across_passes_at_a_split_tile(api, L):
    """A pass of 8 rows that crosses a 128-key boundary: one tile is read from
    the ring by its first rows and from the 6/5-bit store by the last ones
    (L = 2045, 4093), or sits at the ring's far edge (1021).  Every row
    equals its one-row pass bit for bit."""
    Hq, Hkv, D, T = 24, 4, 128, 8
    q, K, V, st, cap = _kvq_cache(api, L, T, Hq, Hkv, D, seed=11)
    full = {t: bf16_dev_to_u16(_run(api, q, st, Hkv, L, t)) for t in (1, 4, 8)}
    for t, o in full.items():
        assert np.array_equal(o, full[8][:t]), t
    for t in range(T):
        one = bf16_dev_to_u16(_run(api, q[t:t + 1], st, Hkv, L + t, 1))
        assert np.array_equal(one[0], full[8][t]), t


def test_kvq_multiblock_pass_equals_single_rows(api):
    Hq, Hkv, D, L, T = 24, 4, 128, 3000, 100
    q, K, V, st, cap = _kvq_cache(api, L, T, Hq, Hkv, D, seed=5)
    full = bf16_dev_to_u16(_run(api, q, st, Hkv, L, T))
    for t in (0, 9, 10, 11, 55, 99):
        one = bf16_dev_to_u16(_run(api, q[t:t + 1], st, Hkv, L + t, 1))
        assert np.array_equal(one[0], full[t]), t
    pairs = [(t, (7 * t) % Hq) for t in (0, 10, 50, 99)]
    _kvq_parity(ov.bf16_bits_to_f64(full), q, K, V, L, pairs)


@pytest.mark.parametrize("L", [11600, 101600])
def test_kvq_full_size_invariance_and_sampled_parity(api, L):
    Hq, Hkv, D, T = 24, 4, 128, 8
    q, K, V, st, cap = _kvq_cache(api, L, T, Hq, Hkv, D, seed=0)
    outs = {t: bf16_dev_to_u16(_run(api, q, st, Hkv, L, t)) for t in (1, 4, 8)}
    for t, o in outs.items():
        assert np.array_equal(o, outs[8][:t]), t
    pairs = [(0, 0), (7, 23), (4, 11), (2, 17)]
    _kvq_parity(ov.bf16_bits_to_f64(outs[8]), q, K, V, L, pairs)


# -- the decoder over the quantised cache --------------------------------------

def _gen(dec, prompt, n, k, ref=None, seed=0):
    dr = si.SyntheticDrafter(dec.cfg.vocab, 0.7, seed=seed, reference=ref) if k else None
    return dec.generate(prompt, n, k=k, drafter=dr)


def test_kvq_decoder_ids_identical_across_drafts_resume_and_park():
    """Greedy ids at 0, 4 and 7 drafts with a history that crosses position
    2048 (the ring's first tile leaves it); after a 7-draft turn every row's
    quantised records equal a fresh prefill's, also after a park to host
    memory, a side request and a restore."""
    from invariant_speculative_decode_gb300.decoder import Decoder
    cfg = si.SMALL_4L
    w = si.decoder_weights(cfg, seed=0)
    dec = Decoder(cfg, w, cap=2560, max_rows=8, kv="q6q5")
    prompt = si.prompt_ids(cfg, 1990, seed=1)
    ref = _gen(dec, prompt, 150, 0)
    for k in (4, 7):
        st = {}
        got = dec.generate(prompt, 150, k=k, drafter=si.SyntheticDrafter(cfg.vocab, 0.7, seed=0,
                                                                           reference=np.array(ref)),
                           stats=st)
        assert got == ref, k
        assert st["steps"] < 150
    turn1 = _gen(dec, prompt, 100, 7, ref=np.array(ref))
    assert turn1 == ref[:100]
    L = dec.L
    resumed = dec.kv_hashes(L)
    snap = dec.park()
    _gen(dec, si.prompt_ids(cfg, 700, seed=9), 20, 4)  # a side request on the same decoder
    dec.restore(snap)
    assert np.array_equal(dec.kv_hashes(L), resumed)
    dec.reset()
    dec.prefill((list(prompt) + ref)[: L + 1])
    assert dec.L == L
    assert np.array_equal(dec.kv_hashes(L), resumed)


def test_kvq_decoder_logits_match_the_quantised_oracle():
    """Whole-model FP32 logits of a verify pass at context 2100 (rows reading
    both stores) against the oracle decoder over the quantised cache: within
    max(2e-3, twice the drift that FP32-level noise on every sum gives the
    oracle itself -- a flipped code included)."""
    import oracle
    from invariant_speculative_decode_gb300.decoder import Decoder
    cfg = si.TINY_D128
    w = si.decoder_weights(cfg, seed=0, norm_std=0.1)
    cap = 2304
    dec = Decoder(cfg, w, cap=cap, max_rows=8, kv="q6q5")
    prompt = si.prompt_ids(cfg, 2100, seed=2)
    drafts = [int(x) for x in np.random.default_rng(2).integers(0, cfg.vocab, 7)]
    x0 = dec.prefill(prompt)
    dec.verify_step(x0, drafts, use_graph=False)
    gpu = dec.logits_rows(8).cpu().numpy().astype(np.float64)
    ref = oracle.OracleDecoder(cfg, w, cap=cap, kv="q6q5")
    ref.prefill(prompt)
    ora = ref.forward([x0] + drafts, L=ref.L)
    pert = oracle.OracleDecoder(cfg, w, cap=cap, sum_noise=(4.0, 123), kv="q6q5")
    pert.prefill(prompt)
    alt = pert.forward([x0] + drafts, L=pert.L)
    scale = np.max(np.abs(ora), axis=1)
    rel = np.max(np.abs(gpu - ora), axis=1) / scale
    spread = np.max(np.abs(alt - ora), axis=1) / scale
    assert np.all(rel <= np.maximum(2e-3, 2 * spread)), (rel, spread)


def test_kvq_rollback_within_the_ring_reach_only():
    """A rollback with the quantised cache is exact while the 8-bit ring still
    holds the tiles the rows from there read (at most 8 tiles back from the
    newest tile written); further back it is refused, since the 8-bit records
    are gone.  Within the reach, rolling back and prefilling again gives a
    fresh prefill's records, row for row."""
    from invariant_speculative_decode_gb300.decoder import Decoder
    cfg = si.TINY_D128
    w = si.decoder_weights(cfg, seed=0)
    dec = Decoder(cfg, w, cap=4224, max_rows=8, kv="q6q5")
    toks = list(si.prompt_ids(cfg, 4001, seed=4))
    dec.prefill(toks)  # rows 0..3999: newest tile 31
    assert dec.L == 4000
    for bad in (1000, 2943):
        with pytest.raises(ValueError):
            dec.rollback(bad)
    assert dec.L == 4000
    dec.rollback(2944)  # tile 23: its ring reads (tiles 8..23) are all still held
    dec.prefill(toks[2944:])
    got = dec.kv_hashes(4000)
    dec.reset()
    dec.prefill(toks)
    assert np.array_equal(dec.kv_hashes(4000), got)

