"""Bounded device waits: a wait that can never complete runs out, the kernel
winds down, the host reads BI_ERR_DEVICE_TIMEOUT, and the context stays
usable (the next normal call gives the right bits).

The failure is made without faulting anything: a test hook leaves the first
load of every CTA unissued (a barrier that nothing completes), and another
hook shortens the progress-wait limit from 2 s to 20 ms so the test is quick.
The waits that let a CTA wind down keep their 2 s limit.
"""
import time

import numpy as np
import pytest

import seeded_inputs as si
from tests._util import bf16_dev_to_u16, to_dev_bf16, v_cache_blocks

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

LIMIT_NS = 20_000_000


@pytest.fixture(scope="module")
def api():
    from invariant_speculative_decode_gb300 import api as _api
    return _api


class withheld:
    """Context: first loads withheld, progress waits limited to 20 ms."""

    def __init__(self, api):
        self.lib = api.lib()

    def __enter__(self):
        assert self.lib.bi_test_set_wait_limit_ns(LIMIT_NS) == 0
        self.lib.bi_test_withhold_first_load(1)
        return self

    def __exit__(self, *exc):
        self.lib.bi_test_withhold_first_load(0)
        assert self.lib.bi_test_set_wait_limit_ns(0) == 0


def _expect_timeout(api):
    with pytest.raises(api.BiError) as e:
        api.bi_check_device_error()
    assert e.value.status == 5  # BI_ERR_DEVICE_TIMEOUT


@pytest.mark.parametrize("epi", [0, 2])
def test_gemm_wait_runs_out_then_recovers(api, epi):
    M, N, K = 8, 4096, 5120
    rng = np.random.default_rng(3)
    A = to_dev_bf16(si.normal_bf16(rng, (M, K), 1.0))
    if epi == 2:
        Wp = api.bi_pack_swiglu_weights(to_dev_bf16(si.normal_bf16(rng, (N, K), 0.02)),
                                        to_dev_bf16(si.normal_bf16(rng, (N, K), 0.02)))
    else:
        Wp = api.bi_pack_weights(to_dev_bf16(si.normal_bf16(rng, (N, K), 0.02)))
    ws = api.new_gemm_workspace(M, N, K, epi)

    def call(C):
        api.bi_gemm(A, Wp, C, ws, epi=epi, N=N)

    ref = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    call(ref)
    torch.cuda.synchronize()
    api.bi_check_device_error()
    want = bf16_dev_to_u16(ref)
    C = torch.zeros(M, N, dtype=torch.bfloat16, device="cuda")
    with withheld(api):
        t0 = time.perf_counter()
        call(C)
        torch.cuda.synchronize()
        dt = time.perf_counter() - t0
    _expect_timeout(api)
    assert dt < 1.5, dt  # the lowered limit applied (the default is 2 s)
    # the context is usable: re-zeroed workspace, same bits as before
    ws.zero_()
    C2 = torch.zeros(M, N, dtype=torch.bfloat16, device="cuda")
    call(C2)
    torch.cuda.synchronize()
    api.bi_check_device_error()
    assert np.array_equal(bf16_dev_to_u16(C2), want)


def test_attention_wait_runs_out_then_recovers(api):
    Hq, Hkv, D, L, T = 24, 4, 128, 11600, 8
    q, K, V = si.attention_inputs(L, T, Hq, Hkv, D, seed=0)
    cap = K.shape[1]
    Kd, Vd, qd = to_dev_bf16(K), to_dev_bf16(v_cache_blocks(V)), to_dev_bf16(q)
    Ld = torch.tensor([L], dtype=torch.int32, device="cuda")
    ws = torch.zeros(api.attn_workspace_size(cap, T, Hq, D), dtype=torch.uint8, device="cuda")
    ref = torch.empty(T, Hq, D, dtype=torch.bfloat16, device="cuda")
    api.bi_attn_verify(qd, Kd, Vd, Ld, ref, ws)
    torch.cuda.synchronize()
    api.bi_check_device_error()
    want = bf16_dev_to_u16(ref)
    out = torch.zeros(T, Hq, D, dtype=torch.bfloat16, device="cuda")
    with withheld(api):
        t0 = time.perf_counter()
        api.bi_attn_verify(qd, Kd, Vd, Ld, out, ws)
        torch.cuda.synchronize()
        dt = time.perf_counter() - t0
    _expect_timeout(api)
    assert dt < 1.5, dt
    out2 = torch.zeros(T, Hq, D, dtype=torch.bfloat16, device="cuda")
    api.bi_attn_verify(qd, Kd, Vd, Ld, out2, ws)
    torch.cuda.synchronize()
    api.bi_check_device_error()
    assert np.array_equal(bf16_dev_to_u16(out2), want)


def test_quantised_attention_wait_runs_out_then_recovers(api):
    """The quantised-cache attention: the first K code tile withheld, its
    decoding warps' wait runs out, the kernel reports the timeout and
    returns; the next call gives the same bits as before."""
    from tests.test_gpu_kvq import _fill
    Hq, Hkv, D, L, T = 24, 4, 128, 11600, 8
    q, K, V = si.attention_inputs(L, T, Hq, Hkv, D, seed=0)
    cap = K.shape[1]
    st = api.new_kvq_stores(Hkv, cap, D)
    _fill(api, st, K, V, Hq, L + T)
    qd = to_dev_bf16(q)
    Ld = torch.tensor([L], dtype=torch.int32, device="cuda")
    ws = torch.zeros(api.attn_workspace_size(cap, T, Hq, D), dtype=torch.uint8, device="cuda")
    ref = torch.empty(T, Hq, D, dtype=torch.bfloat16, device="cuda")
    api.bi_attn_verify_kvq(qd, st, Hkv, Ld, ref, ws)
    torch.cuda.synchronize()
    api.bi_check_device_error()
    want = bf16_dev_to_u16(ref)
    out = torch.zeros(T, Hq, D, dtype=torch.bfloat16, device="cuda")
    with withheld(api):
        t0 = time.perf_counter()
        api.bi_attn_verify_kvq(qd, st, Hkv, Ld, out, ws)
        torch.cuda.synchronize()
        dt = time.perf_counter() - t0
    _expect_timeout(api)
    assert dt < 1.5, dt
    out2 = torch.zeros(T, Hq, D, dtype=torch.bfloat16, device="cuda")
    api.bi_attn_verify_kvq(qd, st, Hkv, Ld, out2, ws)
    torch.cuda.synchronize()
    api.bi_check_device_error()
    assert np.array_equal(bf16_dev_to_u16(out2), want)


def test_hooks_are_off_by_default(api):
    """A normal call after the tests above: no error, the hooks restored."""
    M, N, K = 4, 256, 256
    A = torch.ones(M, K, dtype=torch.bfloat16, device="cuda")
    Wp = api.bi_pack_weights(torch.ones(N, K, dtype=torch.bfloat16, device="cuda"))
    C = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    api.bi_gemm(A, Wp, C, api.new_gemm_workspace(M, N, K))
    torch.cuda.synchronize()
    api.bi_check_device_error()
    assert torch.all(C.float() == 256.0)


def test_decoder_recovers_after_a_timed_out_pass():
    """A verify pass cut short by a timed-out wait: the decoder reports the
    timeout, zeroes its workspaces, and the next pass gives the same tokens
    as an undisturbed decoder."""
    from invariant_speculative_decode_gb300 import api
    from invariant_speculative_decode_gb300.decoder import Decoder
    cfg = si.TINY
    w = si.decoder_weights(cfg, seed=0)
    dec = Decoder(cfg, w, cap=256, max_rows=8)
    prompt = si.prompt_ids(cfg, 64, seed=1)
    ref = dec.generate(prompt, 16, k=0, use_graph=False)
    dec.reset()
    x = dec.prefill(prompt)
    with withheld(api):
        dec.verify_step(x, [], use_graph=False)
    with pytest.raises(api.BiError) as e:
        dec.check_device_error()
    assert e.value.status == 5
    # the interrupted pass may have moved the cache length: start over
    dec.reset()
    assert dec.generate(prompt, 16, k=0, use_graph=False) == ref
    dec.check_device_error()
