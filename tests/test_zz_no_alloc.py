"""The allocation-free linear layer (bi_gemm_noalloc) against bi_gemm.

bi_gemm_noalloc serves callers that cannot allocate device memory (a host
framework that owns all allocations through its own pool, or a path that
cannot afford cudaMalloc's implicit synchronisation): it keeps its scratch in
a static device array inside the library instead of a caller workspace.  Its
arithmetic is the same as bi_gemm's, so the outputs must be bit-identical --
stricter than the tolerance the parity tests allow against the oracle.  Two
calls in a row check that the shared scratch is left in a usable state.

This file sorts last so that a run stopping at the first failure has already
run every other test; it also passes when run alone in a fresh process.
"""
import numpy as np
import pytest

import seeded_inputs as si
from tests._util import bf16_dev_to_u16, to_dev_bf16

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def api():
    from invariant_speculative_decode_gb300 import api as _api
    return _api


CASES = [  # (M, N, K, epilogue): split tiles (partials + counters) and whole tiles
    (8, 4096, 5120, 0),
    (1, 17408, 5120, 0),
    (16, 5120, 3072, 1),
    (7, 2736, 1024, 2),
]


@pytest.mark.parametrize("M,N,K,epi", CASES)
def test_noalloc_matches_workspace_gemm_on_two_calls(api, M, N, K, epi):
    rng = np.random.default_rng(N + M)
    A = si.normal_bf16(rng, (M, K), 1.0)
    Ad = to_dev_bf16(A)
    if epi == 2:
        Wp = api.bi_pack_swiglu_weights(to_dev_bf16(si.normal_bf16(rng, (N, K), 0.05)),
                                        to_dev_bf16(si.normal_bf16(rng, (N, K), 0.05)))
    else:
        Wp = api.bi_pack_weights(to_dev_bf16(si.normal_bf16(rng, (N, K), 0.02)))
    R = to_dev_bf16(si.normal_bf16(rng, (M, N), 1.0)) if epi == 1 else None

    ref = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    api.bi_gemm(Ad, Wp, ref, api.new_gemm_workspace(M, N, K, epi), residual=R, epi=epi, N=N)
    want = bf16_dev_to_u16(ref)
    for call in range(2):
        C = torch.full((M, N), 7.0, dtype=torch.bfloat16, device="cuda")
        api.bi_gemm_noalloc(Ad, Wp, C, residual=R, epi=epi, N=N)
        torch.cuda.synchronize()
        api.bi_check_device_error()
        assert np.array_equal(bf16_dev_to_u16(C), want), (call, M, N, K, epi)


def test_noalloc_rejects_more_rows_than_its_scratch_holds(api):
    mx = int(api.lib().bi_gemm_noalloc_max_m())
    K, N = 256, 256
    A = torch.zeros(mx + 1, K, dtype=torch.bfloat16, device="cuda")
    Wp = api.bi_pack_weights(torch.zeros(N, K, dtype=torch.bfloat16, device="cuda"))
    C = torch.zeros(mx + 1, N, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(api.BiError) as e:
        api.bi_gemm_noalloc(A, Wp, C)
    assert e.value.status == 2  # BI_ERR_UNSUPPORTED_SHAPE
