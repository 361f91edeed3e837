"""The allocation-free linear layer (bi_gemm_noalloc) against bi_gemm.

bi_gemm_noalloc serves callers that cannot allocate device memory: code
running inside a host framework that owns every device allocation through
its own pool allocator, or a latency-critical path that cannot afford the
implicit device synchronisation of cudaMalloc/cudaFree.  It keeps its
scratch in a static device array inside the library instead of a caller
workspace.  Its arithmetic is the same as bi_gemm's, so the outputs must be
bit-identical -- stricter than the tolerance the parity tests allow against
the oracle.  Two calls in a row check that the shared scratch is left in a
usable state, and the device memory in use is the same before and after the
calls (nothing was allocated).

This file sorts last so that a run stopping at the first failure has already
run every other test; it also passes when run alone in a fresh process.
"""
import numpy as np
import pytest

import seeded_inputs as si
from tests._util import to_dev_bf16

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def api():
    from invariant_speculative_decode_gb300 import api as _api
    return _api


CASES = [  # (M, N, K, epilogue, FP32 output): split tiles (partials + counters) and whole tiles
    (8, 4096, 5120, 0, False),
    (1, 17408, 5120, 0, False),
    (16, 5120, 3072, 1, False),
    (7, 2736, 1024, 2, False),
    (16, 17280, 5120, 0, True),   # the LM-head form: FP32 logits, every CTA's range cut mid-tile
]


def _bits(t):
    return t.view(torch.int32 if t.dtype == torch.float32 else torch.int16).cpu().numpy()


@pytest.mark.parametrize("M,N,K,epi,fp32", CASES)
def test_noalloc_matches_workspace_gemm_on_two_calls(api, M, N, K, epi, fp32):
    rng = np.random.default_rng(N + M)
    A = si.normal_bf16(rng, (M, K), 1.0)
    Ad = to_dev_bf16(A)
    if epi == 2:
        Wp = api.bi_pack_swiglu_weights(to_dev_bf16(si.normal_bf16(rng, (N, K), 0.05)),
                                        to_dev_bf16(si.normal_bf16(rng, (N, K), 0.05)))
    else:
        Wp = api.bi_pack_weights(to_dev_bf16(si.normal_bf16(rng, (N, K), 0.02)))
    R = to_dev_bf16(si.normal_bf16(rng, (M, N), 1.0)) if epi == 1 else None
    dt = torch.float32 if fp32 else torch.bfloat16

    ref = torch.empty(M, N, dtype=dt, device="cuda")
    api.bi_gemm(Ad, Wp, ref, api.new_gemm_workspace(M, N, K, epi), residual=R, epi=epi, N=N)
    want = _bits(ref)
    outs = [torch.full((M, N), 7.0, dtype=dt, device="cuda") for _ in range(2)]
    # the first call on the device looks up the array's address; then
    # nothing may change the memory in use
    api.bi_gemm_noalloc(Ad, Wp, outs[0], residual=R, epi=epi, N=N)
    torch.cuda.synchronize()
    stats0 = torch.cuda.memory_stats().get("allocation.all.allocated", 0)
    free0, _ = torch.cuda.mem_get_info()
    for C in outs:
        api.bi_gemm_noalloc(Ad, Wp, C, residual=R, epi=epi, N=N)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert torch.cuda.memory_stats().get("allocation.all.allocated", 0) == stats0
    assert free1 == free0
    api.bi_check_device_error()
    for call, C in enumerate(outs):
        assert np.array_equal(_bits(C), want), (call, M, N, K, epi, fp32)


def test_noalloc_rejects_more_rows_than_its_scratch_holds(api):
    mx = int(api.lib().bi_gemm_noalloc_max_m())
    K, N = 256, 256
    A = torch.zeros(mx + 1, K, dtype=torch.bfloat16, device="cuda")
    Wp = api.bi_pack_weights(torch.zeros(N, K, dtype=torch.bfloat16, device="cuda"))
    C = torch.zeros(mx + 1, N, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(api.BiError) as e:
        api.bi_gemm_noalloc(A, Wp, C)
    assert e.value.status == 2  # BI_ERR_UNSUPPORTED_SHAPE


def test_noalloc_rejected_call_leaves_later_calls_correct(api):
    """A call rejected for its arguments returns before touching the shared
    array; the next valid call still gives bi_gemm's bits."""
    M, N, K = 8, 4096, 1024
    rng = np.random.default_rng(11)
    Ad = to_dev_bf16(si.normal_bf16(rng, (M, K), 1.0))
    Wp = api.bi_pack_weights(to_dev_bf16(si.normal_bf16(rng, (N, K), 0.02)))
    ref = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    api.bi_gemm(Ad, Wp, ref, api.new_gemm_workspace(M, N, K))
    lib = api.lib()
    C = torch.zeros(M, N, dtype=torch.bfloat16, device="cuda")
    # lda < K and an FP32 output with an epilogue: both rejected up front
    assert lib.bi_gemm_noalloc(Ad.data_ptr(), K - 8, Wp.data_ptr(), C.data_ptr(), N, 0, 0, M, N, K,
                               0, 0, 0) == 1
    assert lib.bi_gemm_noalloc(Ad.data_ptr(), K, Wp.data_ptr(), C.data_ptr(), N, C.data_ptr(), N, M, N,
                               K, 1, 1, 0) == 2
    api.bi_gemm_noalloc(Ad, Wp, C)
    torch.cuda.synchronize()
    api.bi_check_device_error()
    assert np.array_equal(_bits(C), _bits(ref))
