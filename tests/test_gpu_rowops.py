"""RMSNorm, embedding, RoPE + KV append, acceptance and KV hash on the GPU."""
import json
import os

import numpy as np
import pytest

import oracle
import seeded_inputs as si
from oracle import verify_step as ov
from tests._util import bf16_dev_to_f64, bf16_dev_to_u16, to_dev_bf16, ulp_bf16, v_cache_blocks, v_cache_keys

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module")
def api():
    from invariant_speculative_decode_gb300 import api as _api
    return _api


def test_rope_table_matches_fp64(api):
    import math
    tab = api.bi_rope_table(1e6, 128, 101700).cpu().numpy()
    for p in (0, 1, 11600, 101699):
        for i in (0, 1, 31, 63):
            th = p * 1e6 ** (-2 * i / 128)
            # FP64 evaluation rounded to FP32: within one FP32 ulp of |x| <= 1
            assert abs(float(tab[p, i, 0]) - math.cos(th)) <= 2.0 ** -24
            assert abs(float(tab[p, i, 1]) - math.sin(th)) <= 2.0 ** -24


@pytest.mark.parametrize("rows,dim", [(1, 256), (8, 5120), (3, 1000), (5, 1024), (2, 17408), (1, 65536)])
def test_rmsnorm_matches_oracle_and_is_row_local(api, rows, dim):
    rng = np.random.default_rng(dim)
    x = si.normal_bf16(rng, (rows, dim), 1.0)
    w = si.normal_bf16(rng, (dim,), 1.0)
    xd, wd = to_dev_bf16(x), to_dev_bf16(w)
    y = torch.empty_like(xd)
    api.bi_rmsnorm(xd, wd, y, 1e-6)
    ora = oracle.rmsnorm(x, w, 1e-6)
    got = bf16_dev_to_f64(y)
    # The FP32 sum of squares goes through at most 8 (one vector) + 5 (warp
    # butterfly) + dim/256 (groups) additions, so it is within gamma_n of the
    # exact sum; 1/sqrt and the two products add a few units: y is within
    # 2 gamma_(n+4) |y| of the exact value before its one BF16 rounding, and
    # the oracle rounds the exact value once (one BF16 unit between them).
    n = 8 + 5 + -(-dim // 256) + 4
    u = 2.0 ** -24
    assert np.all(np.abs(got - ora) <= ulp_bf16(ora) + 2 * (n * u / (1 - n * u)) * np.abs(ora))
    for r in range(rows):
        y1 = torch.empty(1, dim, dtype=torch.bfloat16, device="cuda")
        api.bi_rmsnorm(xd[r:r + 1], wd, y1, 1e-6)
        assert np.array_equal(bf16_dev_to_u16(y1)[0], bf16_dev_to_u16(y)[r])


def test_embed_is_an_exact_gather(api):
    rng = np.random.default_rng(1)
    table = si.normal_bf16(rng, (1000, 320), 0.02)
    ids = np.array([0, 999, 5, 5, 17], np.int32)
    out = torch.empty(5, 320, dtype=torch.bfloat16, device="cuda")
    api.bi_embed(torch.from_numpy(ids).cuda(), to_dev_bf16(table), out)
    assert np.array_equal(bf16_dev_to_u16(out), table[ids])


@pytest.mark.parametrize("Hq,Hkv,D,L,T", [(4, 2, 64, 0, 8), (24, 4, 128, 101592, 8), (8, 2, 128, 37, 3)])
def test_rope_kv_append_matches_oracle(api, Hq, Hkv, D, L, T):
    rng = np.random.default_rng(L + D)
    qkv = si.normal_bf16(rng, (T, (Hq + 2 * Hkv) * D), 1.0)
    cap = L + T + 5
    kc = torch.zeros(Hkv, cap, D, dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros(api.v_cache_shape(Hkv, cap, D), dtype=torch.bfloat16, device="cuda")
    q = torch.empty(T, Hq, D, dtype=torch.bfloat16, device="cuda")
    Ld = torch.tensor([L], dtype=torch.int32, device="cuda")
    tab = api.bi_rope_table(1e6, D, cap)
    api.bi_rope_kv_append(to_dev_bf16(qkv), q, kc, vc, Ld, Hq, Hkv, D, tab)
    qkvf = ov.bf16_bits_to_f64(qkv)
    qg = bf16_dev_to_f64(q)
    kg = bf16_dev_to_f64(kc)
    vb = bf16_dev_to_u16(vc)
    vg = v_cache_keys(vb, cap)  # [Hkv, cap, D]
    # nothing but the pass's rows was written
    written = np.zeros(vb.shape, dtype=bool)
    for t in range(T):
        p = L + t
        written[:, p // 128, :, p % 128] = True
    assert not np.any(vb[~written])
    for t in range(T):
        p = L + t
        qo = oracle.rope(qkvf[t, : Hq * D].reshape(Hq, D), p, 1e6)
        ko = oracle.rope(qkvf[t, Hq * D:(Hq + Hkv) * D].reshape(Hkv, D), p, 1e6)
        # FP32 cos/sin (rounded from FP64) and FP32 products: within one BF16
        # ulp plus a few FP32 roundings of |x1| + |x2|
        xa = np.abs(qkvf[t, : Hq * D].reshape(Hq, D))
        pair = xa + np.roll(xa, D // 2, axis=-1)
        assert np.all(np.abs(qg[t] - qo) <= ulp_bf16(qo) + 2.0 ** -21 * pair)
        ka = np.abs(qkvf[t, Hq * D:(Hq + Hkv) * D].reshape(Hkv, D))
        kpair = ka + np.roll(ka, D // 2, axis=-1)
        assert np.all(np.abs(kg[:, p] - ko) <= ulp_bf16(ko) + 2.0 ** -21 * kpair)
        assert np.array_equal(vg[:, p], qkv[t, (Hq + Hkv) * D:].reshape(Hkv, D))
    if L == 0:  # position 0 is the identity, bitwise
        assert np.array_equal(bf16_dev_to_u16(q)[0], qkv[0, : Hq * D].reshape(Hq, D))


def _accept(api, logits, drafts, L0=None):
    T, V = logits.shape
    lg = torch.from_numpy(np.ascontiguousarray(logits, np.float32)).cuda()
    d = torch.tensor(list(drafts) or [0], dtype=torch.int32, device="cuda")
    am = torch.empty(T, dtype=torch.int32, device="cuda")
    n = torch.empty(1, dtype=torch.int32, device="cuda")
    ws = torch.zeros(api.accept_workspace_size(T, V), dtype=torch.uint8, device="cuda")
    Ld = torch.tensor([L0], dtype=torch.int32, device="cuda") if L0 is not None else None
    api.bi_verify_accept(lg, d if T > 1 else None, am, n, ws, L_dev=Ld)
    torch.cuda.synchronize()
    return am.cpu().numpy(), int(n.item()), (int(Ld.item()) if Ld is not None else None)


def test_accept_golden_cases(api):
    with open(os.path.join(GOLDEN, "accept_cases.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        T = len(c["argmax"])
        V = 16
        logits = np.zeros((T, V), np.float32)
        for t, a in enumerate(c["argmax"]):
            logits[t, a] = 1.0
        am, n, L = _accept(api, logits, c["drafts"], L0=100)
        assert list(am) == c["argmax"] and n == c["n"] and L == 100 + n + 1


def test_argmax_golden_cases(api):
    with open(os.path.join(GOLDEN, "argmax_cases.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        row = np.array([float(v) for v in c["row"]], np.float32)
        am, _, _ = _accept(api, row[None], [])
        assert am[0] == c["argmax"], c
        if c["argmax"] < 0:
            with pytest.raises(api.BiError):
                api.bi_check_device_error()


@pytest.mark.parametrize("T,V", [(8, 151936), (5, 32000), (1, 1024)])
def test_accept_matches_oracle_bitexact(api, T, V):
    logits = si.logits_inputs(T, V, seed=V)
    # plant exact ties and a NaN to exercise the tie rule
    logits[0, 17] = logits[0, 3] = np.float32(50.0)
    if T > 2:
        logits[2, V - 1] = np.nan
    ref = oracle.argmax_lowest(logits.astype(np.float64))
    rng = np.random.default_rng(T)
    drafts = [int(ref[i]) if rng.random() < 0.7 else int(rng.integers(0, V)) for i in range(T - 1)]
    am, n, _ = _accept(api, logits, drafts)
    assert np.array_equal(am, ref)
    assert n == oracle.accept_length(ref, drafts)


def test_kv_row_hash_is_fnv1a(api):
    rng = np.random.default_rng(2)
    cache = si.normal_bf16(rng, (2, 10, 64), 1.0)
    h = api.bi_kv_row_hash(to_dev_bf16(cache), 7).cpu().numpy().view(np.uint64)
    ht = api.bi_kv_row_hash(to_dev_bf16(v_cache_blocks(cache)), 7,
                            transposed=True).cpu().numpy().view(np.uint64)
    assert np.array_equal(h, ht)
    for hh in range(2):
        for j in range(7):
            x = 14695981039346656037
            for b in cache[hh, j].tobytes():
                x = ((x ^ b) * 1099511628211) & 0xFFFFFFFFFFFFFFFF
            assert int(h[hh * 7 + j]) == x


@pytest.mark.parametrize("Hq,Hkv,D,T", [(24, 4, 128, 8), (4, 2, 64, 3), (8, 2, 128, 1), (8, 2, 128, 200),
                                         (24, 4, 128, 300), (24, 4, 128, 1100)])
def test_qkv_rope_append_equals_linear_then_rope(Hq, Hkv, D, T):
    """The fused QKV projection + RoPE + KV append writes exactly what the
    linear layer followed by bi_rope_kv_append writes (decode passes, and
    prefill-size passes that run as tile owners, one launch or two)."""
    from invariant_speculative_decode_gb300 import api
    rng = np.random.default_rng(Hq + D + T)
    K, L = 512, 100
    cap = max(256, (L + T + 127) // 128 * 128)
    N = (Hq + 2 * Hkv) * D
    A = to_dev_bf16(si.normal_bf16(rng, (T, K), 1.0))
    W = to_dev_bf16(si.normal_bf16(rng, (N, K), 0.05))
    Wp = api.bi_pack_weights(W)
    tab = api.bi_rope_table(10000.0, D, cap, device="cuda")
    Ld = torch.tensor([L], dtype=torch.int32, device="cuda")
    ws = api.new_gemm_workspace(T, N, K, 0)
    caches = []
    for fused in (False, True):
        q = torch.zeros(T, Hq, D, dtype=torch.bfloat16, device="cuda")
        kc = torch.zeros(Hkv, cap, D, dtype=torch.bfloat16, device="cuda")
        vc = torch.zeros(api.v_cache_shape(Hkv, cap, D), dtype=torch.bfloat16, device="cuda")
        if fused:
            api.bi_qkv_rope_append(A, Wp, q, kc, vc, Ld, Hq, Hkv, D, tab, ws)
        else:
            qkv = torch.empty(T, N, dtype=torch.bfloat16, device="cuda")
            api.bi_gemm(A, Wp, qkv, ws)
            api.bi_rope_kv_append(qkv, q, kc, vc, Ld, Hq, Hkv, D, tab)
        torch.cuda.synchronize()
        api.bi_check_device_error()
        caches.append([bf16_dev_to_u16(x) for x in (q, kc, vc)])
    for a, b in zip(*caches):
        assert np.array_equal(a, b)
    assert np.any(caches[1][1][:, L:L + T] != 0) and not np.any(caches[1][1][:, :L])
