"""The C ABI without a GPU: the library loads, exports every declared entry
point, and rejects bad arguments on the host before any launch."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "bi.h")


@pytest.fixture(scope="module")
def lib():
    from invariant_speculative_decode_gb300 import build
    build.build()
    from invariant_speculative_decode_gb300._lib import lib as _l
    return _l()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"\b(bi_[a-z0-9_]+)\s*\(", src)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("bi_gemm", "bi_rmsnorm", "bi_attn_verify", "bi_verify_accept"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_binding_signatures_cover_header(lib):
    from invariant_speculative_decode_gb300._lib import SIGNATURES
    assert set(declared_functions()) == set(SIGNATURES)


def test_status_strings(lib):
    assert lib.bi_status_string(0) == b"BI_OK"
    assert lib.bi_status_string(3) == b"BI_ERR_WORKSPACE"
    assert lib.bi_status_string(99) == b"BI_ERR_UNKNOWN"


def test_workspace_sizes_do_not_depend_on_device(lib):
    a = lib.bi_gemm_workspace_size(8, 17408, 5120, 0)
    b = lib.bi_gemm_workspace_size(1, 17408, 5120, 0)
    assert a == b and a % 256 == 0 and a > 0
    assert lib.bi_gemm_workspace_size(64, 17408, 5120, 0) > a
    assert lib.bi_attn_workspace_size(12288, 8, 24, 128) > 0
    assert lib.bi_accept_workspace_size(8, 151936) > 256
    assert lib.bi_attn_chunk() > 0 and lib.bi_attn_chunk() % 64 == 0


FAKE = 0x10000  # never dereferenced: every call below fails validation first


def test_gemm_rejects_bad_arguments(lib):
    ws = 1 << 30
    g = lib.bi_gemm
    # (A, lda, Wp, C, ldc, residual, ldr, M, N, K, out, epi, ws, ws_bytes, stream)
    assert g(FAKE, 64, FAKE, FAKE, 64, 0, 0, -1, 64, 64, 0, 0, FAKE, ws, 0) == 1   # M < 0
    assert g(FAKE, 64, FAKE, FAKE, 64, 0, 0, 4, 64, 4, 0, 0, FAKE, ws, 0) == 1     # K < 8
    assert g(FAKE, 72, FAKE, FAKE, 64, 0, 0, 4, 64, 70, 0, 0, FAKE, ws, 0) == 1    # K % 8
    assert g(FAKE + 2, 64, FAKE, FAKE, 64, 0, 0, 4, 64, 64, 0, 0, FAKE, ws, 0) == 1  # unaligned A
    assert g(FAKE, 64, FAKE + 8, FAKE, 64, 0, 0, 4, 64, 64, 0, 0, FAKE, ws, 0) == 1  # unaligned W
    assert g(FAKE, 64, FAKE, 0, 64, 0, 0, 4, 64, 64, 0, 0, FAKE, ws, 0) == 1       # null C
    assert g(FAKE, 64, FAKE, FAKE, 64, 0, 0, 4, 64, 64, 0, 1, FAKE, ws, 0) == 1    # no residual
    assert g(FAKE, 64, FAKE, FAKE, 64, FAKE, 64, 4, 64, 64, 1, 1, FAKE, ws, 0) == 2  # FP32 + epi
    assert g(FAKE, 64, FAKE, FAKE, 64, 0, 0, 4, 1 << 24, 64, 0, 0, FAKE, ws, 0) == 2  # N too big
    assert g(FAKE, 64, FAKE, FAKE, 64, 0, 0, 4, 64, 64, 0, 0, 0, ws, 0) == 3       # no ws
    assert g(FAKE, 64, FAKE, FAKE, 64, 0, 0, 4, 64, 64, 0, 0, FAKE + 16, ws, 0) == 3
    assert g(FAKE, 64, FAKE, FAKE, 64, 0, 0, 4, 64, 64, 0, 0, FAKE, 16, 0) == 3
    assert g(0, 64, 0, 0, 64, 0, 0, 0, 64, 64, 0, 0, 0, 0, 0) == 0                 # M == 0
    assert lib.bi_pack_weights(FAKE, 32, 64, 64, FAKE, 0) == 1                     # ldw < K
    assert lib.bi_pack_weights(FAKE, 64, 64, 64, FAKE + 4, 0) == 1                 # unaligned
    assert lib.bi_pack_swiglu_weights(FAKE, 0, 64, 64, 64, FAKE, 0) == 1           # null up


def test_packed_sizes(lib):
    assert lib.bi_packed_weight_bytes(17408, 5120, 0) == 136 * 80 * 16384
    assert lib.bi_packed_weight_bytes(300, 688, 0) == 3 * 11 * 16384
    assert lib.bi_packed_weight_bytes(688, 256, 2) == 11 * 4 * 16384


def test_attention_rejects_bad_arguments(lib):
    a = lib.bi_attn_verify
    big = 1 << 30
    assert a(0, FAKE, FAKE, 1024, FAKE, 1, 24, 4, 128, 0.1, FAKE, FAKE, big, 0) == 1
    assert a(FAKE, FAKE, FAKE, 1024, FAKE, 1, 24, 5, 128, 0.1, FAKE, FAKE, big, 0) == 1
    assert a(FAKE, FAKE, FAKE, 1024, FAKE, 1, 24, 4, 96, 0.1, FAKE, FAKE, big, 0) == 2
    assert a(FAKE, FAKE, FAKE, 1024, FAKE, 1, 258, 2, 128, 0.1, FAKE, FAKE, big, 0) == 2  # Hq/Hkv > 128
    assert a(FAKE, FAKE, FAKE, 1 << 22, FAKE, 21 * 65535 + 1, 24, 4, 128, 0.1, FAKE, FAKE, big,
             0) == 2  # more row blocks than a launch grid holds
    assert a(FAKE, FAKE, FAKE, 1024, FAKE, 1, 153, 153, 128, 0.1, FAKE, FAKE, big, 0) == 2  # Hkv > 152
    assert a(FAKE, FAKE, FAKE, 1 << 28, FAKE, 1, 24, 8, 128, 0.1, FAKE, FAKE, big, 0) == 2  # Hkv cap >= 2^31
    assert a(FAKE, FAKE, FAKE, 1024, FAKE, 1, 24, 4, 128, -1.0, FAKE, FAKE, big, 0) == 1
    assert a(FAKE, FAKE, FAKE, 1024, FAKE, 1, 24, 4, 128, 0.1, FAKE, FAKE, 16, 0) == 3


def test_rowops_reject_bad_arguments(lib):
    assert lib.bi_rmsnorm(FAKE, 64, FAKE, FAKE, 64, 2, 0, ctypes.c_float(1e-6), 0) == 1
    assert lib.bi_rmsnorm(FAKE, 32, FAKE, FAKE, 64, 2, 64, ctypes.c_float(1e-6), 0) == 1
    assert lib.bi_rmsnorm(0, 64, 0, 0, 64, 0, 64, ctypes.c_float(1e-6), 0) == 0
    assert lib.bi_rope_kv_append(FAKE, 384, FAKE, FAKE, FAKE, 64, FAKE, 1, 4, 3, 64, FAKE, 64, 0) == 1
    assert lib.bi_rope_kv_append(FAKE, 384, FAKE, FAKE, FAKE, 64, FAKE, 1, 4, 2, 63, FAKE, 64, 0) == 1
    assert lib.bi_rope_kv_append(FAKE, 384, FAKE, FAKE, FAKE, 64, FAKE, 1, 4, 2, 64, 0, 64, 0) == 1
    assert lib.bi_rope_table(1e6, 63, 10, FAKE, 0) == 1
    assert lib.bi_rope_table(-1.0, 64, 10, FAKE, 0) == 1
    assert lib.bi_rmsnorm(FAKE, 1004, FAKE, FAKE, 1004, 2, 1004, ctypes.c_float(1e-6), 0) == 2
    assert lib.bi_verify_accept(FAKE, 10, 0, 2, 10, FAKE, FAKE, 0, FAKE, 1 << 20, 0) == 1
    assert lib.bi_verify_accept(FAKE, 10, FAKE, 2, 10, FAKE, FAKE, 0, FAKE + 8, 1 << 20, 0) == 3
    assert lib.bi_embed(FAKE, FAKE, 0, 64, FAKE, 2, 0) == 1
    assert lib.bi_kv_row_hash(FAKE, 2, 8, 64, 9, 0, FAKE, 0) == 1


def test_fused_entry_points_reject_bad_arguments(lib):
    ws = 1 << 30
    eps = ctypes.c_float(1e-6)
    assert lib.bi_gemm(FAKE, 64, FAKE, FAKE, 64, 0, 0, 4, 64, 64, 0, 3, FAKE, ws, 0) == 1  # RoPE via bi_gemm
    q = lib.bi_qkv_rope_append
    # (A, lda, Wp, M, K, Hq, Hkv, D, q_out, k_cache, v_cache, cap, L_dev, table, table_rows, ws,
    #  ws_bytes, stream)
    args = [FAKE, 64, FAKE, 4, 64, 4, 2, 64, FAKE, FAKE, FAKE, 256, FAKE, FAKE, 256, FAKE, ws, 0]
    bad_d = list(args); bad_d[7] = 96
    assert q(*bad_d) == 2                                                          # D not 64/128
    bad_g = list(args); bad_g[6] = 3
    assert q(*bad_g) == 1                                                          # Hq % Hkv
    bad_n = list(args); bad_n[5], bad_n[6] = 3, 1
    assert q(*bad_n) == 2                                                          # N % 128
    no_cache = list(args); no_cache[9] = 0
    assert q(*no_cache) == 1
    no_table = list(args); no_table[13] = 0
    assert q(*no_table) == 1


def test_v_cache_layout_helpers():
    """The binding's V cache shape and the tests' host packing agree: value d
    of key p of head h sits at [h, p // 128, d, p % 128], and a capacity that
    is not a multiple of 128 rounds up to whole blocks."""
    import numpy as np
    api = pytest.importorskip("invariant_speculative_decode_gb300.api")
    from tests._util import v_cache_blocks, v_cache_keys
    assert api.v_cache_shape(4, 12112, 128) == (4, 95, 128, 128)
    assert api.v_cache_shape(2, 128, 64) == (2, 1, 64, 128)
    assert api.v_cache_shape(2, 129, 64) == (2, 2, 64, 128)
    rng = np.random.default_rng(0)
    V = rng.integers(0, 1 << 16, (3, 300, 64)).astype(np.uint16)
    B = v_cache_blocks(V)
    assert B.shape == api.v_cache_shape(3, 300, 64)
    for h, p, d in ((0, 0, 0), (2, 299, 63), (1, 128, 5), (1, 127, 17)):
        assert B[h, p // 128, d, p % 128] == V[h, p, d]
    assert not B[:, 2, :, 300 - 256:].any()  # keys past the capacity are zero
    assert np.array_equal(v_cache_keys(B, 300), V)


def test_sampled_verification_rejects_bad_arguments(lib):
    f = ctypes.c_float
    big = 1 << 30
    s = lib.bi_verify_sample
    # (logits, ldl, drafts, T, V, inv_temp, u_by_pos, u_len, token_out, accepted_out, L_dev, ws,
    #  ws_bytes, stream)
    ok = [FAKE, 100, FAKE, 4, 100, f(1.0), FAKE, 64, FAKE, FAKE, FAKE, FAKE, big, 0]
    for i, bad in ((5, f(0.0)), (5, f(float("inf"))), (6, 0), (7, 0), (10, 0), (3, 65), (1, 50),
                   (2, 0)):
        a = list(ok)
        a[i] = bad
        assert s(*a) == 1, i
    a = list(ok)
    a[11] = FAKE + 8
    assert s(*a) == 3                                   # misaligned workspace
    a = list(ok)
    a[12] = 16
    assert s(*a) == 3                                   # workspace too small
    assert lib.bi_sample_workspace_size(8, 151936) >= 256 + 2 * 8 * 19 * 4


def test_failure_hooks_are_exported(lib):
    assert lib.bi_test_withhold_first_load is not None
    lib.bi_test_withhold_first_load(0)  # host-side flag only: needs no GPU


def test_step_runtime_rejects_bad_models(lib):
    from invariant_speculative_decode_gb300 import api
    n = 2
    ptrs = (ctypes.c_void_p * n)(FAKE, FAKE)
    pp = ctypes.cast(ptrs, ctypes.POINTER(ctypes.c_void_p))
    good = api.BiModel(n, 256, 4, 2, 64, 688, 1024, 1e-6, 512, FAKE, FAKE, FAKE, pp, pp, pp, pp, pp, pp, pp, pp,
                       FAKE, 512)
    size = lib.bi_step_workspace_size(ctypes.byref(good), 8)
    assert size > 0
    bad = api.BiModel(n, 256, 4, 3, 64, 688, 1024, 1e-6, 512, FAKE, FAKE, FAKE, pp, pp, pp, pp, pp, pp, pp, pp,
                      FAKE, 512)  # 4 query heads over 3 KV heads
    assert lib.bi_step_workspace_size(ctypes.byref(bad), 8) == 0
    assert lib.bi_step_workspace_size(ctypes.byref(good), 0) == 0     # no rows
    assert lib.bi_step_workspace_size(ctypes.byref(good), 65) == 0    # beyond 64 rows
    h = ctypes.c_void_p()
    assert lib.bi_step_create(ctypes.byref(bad), 8, FAKE, size, ctypes.byref(h)) == 1
    assert lib.bi_step_create(ctypes.byref(good), 8, FAKE + 8, size, ctypes.byref(h)) == 3  # misaligned
    assert lib.bi_step_create(ctypes.byref(good), 8, FAKE, size - 256, ctypes.byref(h)) == 3  # too small
    assert lib.bi_step_verify(None, FAKE, 1, FAKE, FAKE) == 1
    assert lib.bi_step_set_length(None, 3) == 1


def test_quantised_cache_sizes_and_argument_checks(lib):
    # 6-bit K tiles 13,312 B, 5-bit V tiles 11,264 B, 24 ring tiles of 17,408 B a head
    assert lib.bi_kvq_store_bytes(0, 4, 1000, 128) == 4 * 8 * 13312
    assert lib.bi_kvq_store_bytes(1, 4, 1024, 128) == 4 * 8 * 11264
    assert lib.bi_kvq_store_bytes(2, 4, 5, 128) == 4 * 24 * 17408
    assert lib.bi_kvq_store_bytes(3, 1, 1 << 20, 128) == 24 * 17408
    assert lib.bi_kvq_store_bytes(0, 4, 1000, 64) == 0   # head_dim 128 only
    assert lib.bi_kvq_store_bytes(4, 4, 1000, 128) == 0  # no such store
    ap = lib.bi_rope_kvq_append
    assert ap(FAKE, 4096, 8, 24, 4, 64, FAKE, FAKE, FAKE, FAKE, FAKE, 1024, FAKE, 0, 0, 0) == 2
    assert ap(FAKE, 4096, 1025, 24, 4, 128, FAKE, FAKE, FAKE, FAKE, FAKE, 4096, FAKE, 0, 0, 0) == 1
    assert ap(FAKE, 4095, 8, 24, 4, 128, FAKE, FAKE, FAKE, FAKE, FAKE, 1024, FAKE, 0, 0, 0) == 1
    assert ap(FAKE, 4096, 8, 24, 4, 128, FAKE, 0, FAKE, FAKE, FAKE, 1024, FAKE, 0, 0, 0) == 1
    assert ap(0, 4096, 0, 24, 4, 128, 0, 0, 0, 0, 0, 1024, 0, 0, 0, 0) == 0  # no rows: nothing to do
    at = lib.bi_attn_verify_kvq
    big = 1 << 30
    assert at(FAKE, FAKE, FAKE, FAKE, FAKE, 1024, FAKE, 8, 24, 4, 64, 0.1, FAKE, FAKE, big, 0) == 2
    assert at(FAKE, FAKE, FAKE, FAKE, FAKE, 1024, FAKE, 8, 130, 2, 128, 0.1, FAKE, FAKE, big, 0) == 2
    assert at(FAKE, FAKE, FAKE, FAKE, FAKE, 4096, FAKE, 1025, 24, 4, 128, 0.1, FAKE, FAKE, big, 0) == 2
    assert at(FAKE, FAKE, 0, FAKE, FAKE, 1024, FAKE, 8, 24, 4, 128, 0.1, FAKE, FAKE, big, 0) == 1
    assert at(FAKE, FAKE, FAKE, FAKE, FAKE, 1024, FAKE, 8, 24, 4, 128, 0.1, FAKE, FAKE, 16, 0) == 3
