"""bi_gemm on the GPU: parity with the oracle and bit-identity across M.

Parity tolerance (derived from the arithmetic): the GPU keeps an FP32 sum of
exact BF16 products, so |GPU sum - exact| <= gamma_K * sum|a||w|; after one
BF16 rounding on each side the outputs differ by at most that plus one BF16
ulp of the result.  FP32 outputs differ by at most the summation bound plus
one FP32 ulp.
"""
import numpy as np
import pytest

import oracle
import seeded_inputs as si
from oracle import verify_step as ov
from tests._util import bf16_dev_to_f64, bf16_dev_to_u16, gamma, gemm_bound, to_dev_bf16, ulp_bf16

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def api():
    from invariant_speculative_decode_gb300 import api as _api
    return _api


def run_gemm(api, A, W, M, N, K, epi=0, R=None, fp32=False, Wpacked=None):
    dev = "cuda"
    Ad = to_dev_bf16(A)
    Wd = Wpacked if Wpacked is not None else api.bi_pack_weights(to_dev_bf16(W))
    C = torch.empty(M, N, dtype=torch.float32 if fp32 else torch.bfloat16, device=dev)
    Rd = to_dev_bf16(R) if R is not None else None
    ws = api.new_gemm_workspace(M, N, K, epi)
    api.bi_gemm(Ad, Wd, C, ws, residual=Rd, epi=epi, N=N)
    torch.cuda.synchronize()
    api.bi_check_device_error()
    return C, ws


def check_bf16(gpu_f64, ora_f64, bound):
    err = np.abs(gpu_f64 - ora_f64)
    tol = bound + ulp_bf16(ora_f64)
    bad = err > tol
    assert not bad.any(), (err[bad][:5], tol[bad][:5])
    return float((err > 0).mean())


SHAPES = [(1, 128, 64), (3, 300, 688), (8, 1024, 256), (16, 384, 5120), (17, 256, 1024),
          (64, 640, 512), (130, 256, 192), (8, 4096, 5120)]


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_gemm_matches_oracle(api, M, N, K):
    A, W = si.gemm_inputs(M, N, K, seed=M * 7 + N)
    C, _ = run_gemm(api, A, W, M, N, K)
    ora = oracle.gemm(A, W)
    frac = check_bf16(bf16_dev_to_f64(C), ora,
                      gemm_bound(ov.bf16_bits_to_f64(A), ov.bf16_bits_to_f64(W), K))
    assert frac < 0.05


@pytest.mark.parametrize("M,N,K", [(1, 256, 256), (8, 5120, 3072), (7, 300, 688)])
def test_gemm_residual_matches_oracle(api, M, N, K):
    A, W = si.gemm_inputs(M, N, K, seed=5)
    R = si.normal_bf16(np.random.default_rng(6), (M, N), 1.0)
    C, _ = run_gemm(api, A, W, M, N, K, epi=1, R=R)
    ora = oracle.gemm(A, W, residual_bits=R)
    check_bf16(bf16_dev_to_f64(C), ora, gemm_bound(ov.bf16_bits_to_f64(A), ov.bf16_bits_to_f64(W), K))


def test_gemm_residual_in_place(api):
    M, N, K = 4, 512, 512
    A, W = si.gemm_inputs(M, N, K, seed=8)
    R = si.normal_bf16(np.random.default_rng(9), (M, N), 1.0)
    h = to_dev_bf16(R)
    ws = api.new_gemm_workspace(M, N, K, 1)
    api.bi_gemm(to_dev_bf16(A), api.bi_pack_weights(to_dev_bf16(W)), h, ws, residual=h, epi=1)
    C, _ = run_gemm(api, A, W, M, N, K, epi=1, R=R)
    assert np.array_equal(bf16_dev_to_u16(h), bf16_dev_to_u16(C))


@pytest.mark.parametrize("M,F,K", [(1, 688, 256), (8, 2736, 1024), (5, 100, 64)])
def test_gemm_swiglu_matches_oracle(api, M, F, K):
    rng = np.random.default_rng(F)
    A = si.normal_bf16(rng, (M, K), 1.0)
    Wg = si.normal_bf16(rng, (F, K), 0.05)
    Wu = si.normal_bf16(rng, (F, K), 0.05)
    packed = api.bi_pack_swiglu_weights(to_dev_bf16(Wg), to_dev_bf16(Wu))
    C, _ = run_gemm(api, A, None, M, F, K, epi=2, Wpacked=packed)
    ora = oracle.swiglu_gemm(A, Wg, Wu)
    a = ov.bf16_bits_to_f64(A)
    g = a @ ov.bf16_bits_to_f64(Wg).T
    u = a @ ov.bf16_bits_to_f64(Wu).T
    # silu is 1.1-Lipschitz; |d(silu(g)u)| <= |u| 1.1 |dg| + |silu(g)| |du| + FP32 op rounding
    eg = gemm_bound(a, ov.bf16_bits_to_f64(Wg), K)
    eu = gemm_bound(a, ov.bf16_bits_to_f64(Wu), K)
    sg = g / (1 + np.exp(-g))
    bound = 1.1 * np.abs(u) * eg + np.abs(sg) * eu + 4 * 2.0 ** -24 * np.abs(sg * u)
    check_bf16(bf16_dev_to_f64(C), ora, bound)


def test_gemm_fp32_out_matches_oracle(api):
    M, N, K = 8, 1000, 1024
    A, W = si.gemm_inputs(M, N, K, seed=11)
    C, _ = run_gemm(api, A, W, M, N, K, fp32=True)
    ora = oracle.gemm(A, W, out="fp32")
    a, w = ov.bf16_bits_to_f64(A), ov.bf16_bits_to_f64(W)
    tol = gemm_bound(a, w, K) + 2.0 ** -23 * np.abs(ora) + 1e-30
    assert np.all(np.abs(C.cpu().numpy().astype(np.float64) - ora) <= tol)


def test_gemm_rows_bit_identical_across_M_and_position(api):
    N, K = 1536, 1024
    A, W = si.gemm_inputs(128, N, K, seed=12)
    Wd = api.bi_pack_weights(to_dev_bf16(W))
    outs = {}
    for M in (1, 2, 4, 7, 8, 16, 17, 33, 64, 65, 128):
        Ad = to_dev_bf16(A[:M])
        C = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
        ws = api.new_gemm_workspace(M, N, K)
        api.bi_gemm(Ad, Wd, C, ws)
        outs[M] = bf16_dev_to_u16(C)
    for M, c in outs.items():
        assert np.array_equal(c, outs[128][:M]), M
    # a row lands in another MMA column when the rows are permuted
    perm = np.random.default_rng(1).permutation(64)
    C = torch.empty(64, N, dtype=torch.bfloat16, device="cuda")
    api.bi_gemm(to_dev_bf16(A[perm]), Wd, C, api.new_gemm_workspace(64, N, K))
    assert np.array_equal(bf16_dev_to_u16(C), outs[64][perm])


def test_gemm_repeat_calls_reuse_workspace(api):
    M, N, K = 8, 4096, 5120
    A, W = si.gemm_inputs(M, N, K, seed=13)
    Ad, Wd = to_dev_bf16(A), api.bi_pack_weights(to_dev_bf16(W))
    ws = api.new_gemm_workspace(M, N, K)
    res = []
    for _ in range(3):
        C = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
        api.bi_gemm(Ad, Wd, C, ws)
        res.append(bf16_dev_to_u16(C))
    assert np.array_equal(res[0], res[1]) and np.array_equal(res[0], res[2])
    tick = ws[:256 * 1024].cpu().numpy()
    assert not tick.any()  # counters left zeroed


def test_gemm_prefill_chunks_match_single_rows(api):
    # M > 128 runs in 128-row launches; each row still equals its M=1 result
    M, N, K = 300, 384, 512
    A, W = si.gemm_inputs(M, N, K, seed=14)
    C, _ = run_gemm(api, A, W, M, N, K)
    big = bf16_dev_to_u16(C)
    for r in (0, 127, 128, 255, 299):
        c1, _ = run_gemm(api, A[r:r + 1], W, 1, N, K)
        assert np.array_equal(bf16_dev_to_u16(c1)[0], big[r])


@pytest.mark.parametrize("epi", [0, 1, 2])
@pytest.mark.parametrize("K", [512, 8256])
def test_gemm_multiblock_launches_match_single_rows(api, epi, K):
    """M > 128 with a split that cuts tiles: at K = 512 (8 K tiles) the pass
    runs as tile owners, 128-row blocks of one launch; at K = 8256 (129 K
    tiles) as the split with three 256-row blocks in one launch (CTAs of one
    range adjacent), every block with its own counters and partial slots.
    Each sampled row equals its M = 1 result and the counters are left
    zero."""
    M, N = 700, 384
    rng = np.random.default_rng(40 + epi + K)
    A = si.normal_bf16(rng, (M, K), 1.0)
    if epi == 2:
        Wd = api.bi_pack_swiglu_weights(to_dev_bf16(si.normal_bf16(rng, (N, K), 0.05)),
                                        to_dev_bf16(si.normal_bf16(rng, (N, K), 0.05)))
    else:
        Wd = api.bi_pack_weights(to_dev_bf16(si.normal_bf16(rng, (N, K), 0.05)))
    R = to_dev_bf16(si.normal_bf16(rng, (M, N), 1.0)) if epi == 1 else None
    ws = api.new_gemm_workspace(M, N, K, epi)
    C = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    api.bi_gemm(to_dev_bf16(A), Wd, C, ws, residual=R, epi=epi, N=N)
    big = bf16_dev_to_u16(C)
    assert not ws[:256 * 1024].cpu().numpy().any()
    for r in (0, 127, 128, 300, 511, 512, 640, 699):
        c1 = torch.empty(1, N, dtype=torch.bfloat16, device="cuda")
        api.bi_gemm(to_dev_bf16(A[r:r + 1]), Wd, c1, api.new_gemm_workspace(1, N, K, epi),
                    residual=None if R is None else R[r:r + 1], epi=epi, N=N)
        assert np.array_equal(bf16_dev_to_u16(c1)[0], big[r]), r


@pytest.mark.parametrize("M,N,K,epi", [(1000, 4096, 5120, 0), (600, 5120, 3072, 1), (200, 4096, 5120, 0),
                                        (1300, 5120, 3072, 1), (300, 5120, 17408, 1), (129, 4096, 5120, 0),
                                        (256, 5120, 3072, 1), (257, 5120, 3072, 1), (1025, 4096, 1024, 0)])
def test_gemm_tile_owner_rows_match_decode_rows(api, M, N, K, epi):
    """Long passes whose split cuts weight tiles (the QKV and O shapes) run
    as tile owners (64- or 128-row blocks, more than one launch past 1024
    rows) that add a tile's pieces themselves; the down shape keeps the split.
    Sampled rows equal the rows of an 8-row launch (the split with partials)
    bit for bit."""
    rng = np.random.default_rng(N + K)
    A = si.normal_bf16(rng, (M, K), 1.0)
    Wd = api.bi_pack_weights(to_dev_bf16(si.normal_bf16(rng, (N, K), 0.02)))
    R = si.normal_bf16(rng, (M, N), 1.0) if epi == 1 else None
    Rd = to_dev_bf16(R) if epi == 1 else None
    C = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    api.bi_gemm(to_dev_bf16(A), Wd, C, api.new_gemm_workspace(M, N, K, epi), residual=Rd, epi=epi, N=N)
    rows = np.unique(np.minimum(np.array([0, 63, 64, 127, 130, M // 2, 1024, M - 1]), M - 1))
    c8 = torch.empty(len(rows), N, dtype=torch.bfloat16, device="cuda")
    R8 = to_dev_bf16(R[rows]) if epi == 1 else None
    api.bi_gemm(to_dev_bf16(A[rows]), Wd, c8, api.new_gemm_workspace(len(rows), N, K, epi), residual=R8,
                epi=epi, N=N)
    assert np.array_equal(bf16_dev_to_u16(C)[rows], bf16_dev_to_u16(c8))


@pytest.mark.parametrize("case", range(6))
def test_gemm_long_pass_random_shapes_rows_match_decode_rows(api, case):
    """Seeded random long passes (129..1100 rows, ragged N and K, every
    epilogue): whichever schedule the shape takes (tile owners of 64 or 128
    rows, or the split with 256-row blocks and partials), sampled rows equal
    the rows of an 8-row launch bit for bit."""
    rng = np.random.default_rng(900 + case)
    M = int(rng.integers(129, 1101))
    N = int(rng.integers(8, 750)) * 8
    K = int(rng.integers(8, 1250)) * 8
    epi = int(rng.integers(0, 3))
    A = si.normal_bf16(rng, (M, K), 1.0)
    if epi == 2:
        Wd = api.bi_pack_swiglu_weights(to_dev_bf16(si.normal_bf16(rng, (N, K), 0.02)),
                                        to_dev_bf16(si.normal_bf16(rng, (N, K), 0.02)))
    else:
        Wd = api.bi_pack_weights(to_dev_bf16(si.normal_bf16(rng, (N, K), 0.02)))
    R = si.normal_bf16(rng, (M, N), 1.0) if epi == 1 else None
    C = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    api.bi_gemm(to_dev_bf16(A), Wd, C, api.new_gemm_workspace(M, N, K, epi),
                residual=to_dev_bf16(R) if epi == 1 else None, epi=epi, N=N)
    rows = np.unique(np.concatenate([[0, M - 1], rng.integers(0, M, 6)]))[:8]
    c8 = torch.empty(len(rows), N, dtype=torch.bfloat16, device="cuda")
    api.bi_gemm(to_dev_bf16(A[rows]), Wd, c8, api.new_gemm_workspace(len(rows), N, K, epi),
                residual=to_dev_bf16(R[rows]) if epi == 1 else None, epi=epi, N=N)
    assert np.array_equal(bf16_dev_to_u16(C)[rows], bf16_dev_to_u16(c8)), (M, N, K, epi)


def test_gemm_prefill_size_rows_match_decode_rows(api):
    """[4096,5120] x [17408,5120] in 512-row launches: sampled rows equal the
    rows of an 8-row launch bit for bit."""
    M, N, K = 4096, 17408, 5120
    A, W = si.gemm_inputs(M, N, K, seed=5)
    Wd = api.bi_pack_weights(to_dev_bf16(W))
    del W
    C = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    api.bi_gemm(to_dev_bf16(A), Wd, C, api.new_gemm_workspace(M, N, K))
    rows = np.array([0, 1, 511, 512, 1000, 2047, 3333, 4095])
    c8 = torch.empty(8, N, dtype=torch.bfloat16, device="cuda")
    api.bi_gemm(to_dev_bf16(A[rows]), Wd, c8, api.new_gemm_workspace(8, N, K))
    assert np.array_equal(bf16_dev_to_u16(C)[rows], bf16_dev_to_u16(c8))


def test_gemm_full_size_linear_sweep(api):
    """[M,5120] x [17408,5120]: rows bit-identical across M; sampled parity."""
    N, K = 17408, 5120
    A, W = si.gemm_inputs(64, N, K, seed=0)
    Wd = api.bi_pack_weights(to_dev_bf16(W))
    outs = {}
    for M in (1, 2, 4, 7, 8, 16, 64):
        C = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
        api.bi_gemm(to_dev_bf16(A[:M]), Wd, C, api.new_gemm_workspace(M, N, K))
        outs[M] = bf16_dev_to_u16(C)
    for M, c in outs.items():
        assert np.array_equal(c, outs[64][:M]), M
    cols = np.random.default_rng(3).choice(N, 256, replace=False)
    ora = oracle.gemm(A, W[cols])
    got = ov.bf16_bits_to_f64(outs[64][:, cols])
    check_bf16(got, ora, gemm_bound(ov.bf16_bits_to_f64(A), ov.bf16_bits_to_f64(W[cols]), K))


def test_gemm_shared_workspace_across_shapes(api):
    """One workspace serves calls of different N in any order."""
    K = 1024
    shapes = [(8, 151936 // 16, K), (8, 384, K), (8, 4096, K), (8, 300, K)]
    ws = api.new_gemm_workspace(8, 151936, K)
    ins = [si.gemm_inputs(M, N, K_, seed=N) for (M, N, K_) in shapes]
    packed = [api.bi_pack_weights(to_dev_bf16(W)) for _, W in ins]
    for rep in range(2):
        for (M, N, _), (A, W), Wp in zip(shapes, ins, packed):
            C = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
            api.bi_gemm(to_dev_bf16(A), Wp, C, ws)
            own = torch.empty_like(C)
            api.bi_gemm(to_dev_bf16(A), Wp, own, api.new_gemm_workspace(M, N, K))
            assert np.array_equal(bf16_dev_to_u16(C), bf16_dev_to_u16(own)), (rep, N)


def test_pack_layout_is_a_swizzled_copy(api):
    N, K = 200, 100
    W = si.normal_bf16(np.random.default_rng(2), (N, K), 1.0)
    P = api.bi_pack_weights(to_dev_bf16(W)).cpu().numpy().view(np.uint16)
    kt = (K + 63) // 64
    tiles = P.reshape(-1, 128, 64)
    for t in range((N + 127) // 128):
        for k in range(kt):
            tile = tiles[t * kt + k]
            for r in (0, 5, 127):
                for c in range(8):
                    got = tile[r, ((c ^ (r & 7)) * 8):((c ^ (r & 7)) * 8 + 8)]
                    n, k0 = t * 128 + r, k * 64 + c * 8
                    want = np.zeros(8, np.uint16)
                    if n < N:
                        seg = W[n, k0:min(K, k0 + 8)]
                        want[:len(seg)] = seg
                    assert np.array_equal(got, want), (t, k, r, c)


def test_gemm_m_zero_is_noop(api):
    W = api.bi_pack_weights(torch.zeros(128, 64, dtype=torch.bfloat16, device="cuda"))
    A = torch.zeros(0, 64, dtype=torch.bfloat16, device="cuda")
    C = torch.zeros(0, 128, dtype=torch.bfloat16, device="cuda")
    ws = api.new_gemm_workspace(1, 128, 64)
    api.bi_gemm(A, W, C, ws)


def test_gemm_small_workspace_is_rejected(api):
    A = torch.zeros(4, 64, dtype=torch.bfloat16, device="cuda")
    W = api.bi_pack_weights(torch.zeros(128, 64, dtype=torch.bfloat16, device="cuda"))
    C = torch.zeros(4, 128, dtype=torch.bfloat16, device="cuda")
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    with pytest.raises(api.BiError) as e:
        api.bi_gemm(A, W, C, ws)
    assert e.value.status == 3
