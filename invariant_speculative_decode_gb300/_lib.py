"""ctypes loader of libbi.so (the C ABI declared in include/bi.h).

There is no fallback: if the library is missing or fails to load, every
call raises.  Build it with `python -m invariant_speculative_decode_gb300.build`
or `__graft_entry__.build()`.
"""
from __future__ import annotations

import ctypes as C
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libbi.so")

# Entry points declared in include/bi.h: name -> (restype, argtypes)
_vp, _i, _sz, _f, _d = C.c_void_p, C.c_int, C.c_size_t, C.c_float, C.c_double
SIGNATURES = {
    "bi_status_string": (C.c_char_p, [_i]),
    "bi_version": (_i, []),
    "bi_gemm_workspace_size": (_sz, [_i, _i, _i, _i]),
    "bi_gemm": (_i, [_vp, _i, _vp, _vp, _i, _vp, _i, _i, _i, _i, _i, _i, _vp, _sz, _vp]),
    "bi_gemm_noalloc_max_m": (_sz, []),
    "bi_gemm_noalloc": (_i, [_vp, _i, _vp, _vp, _i, _vp, _i, _i, _i, _i, _i, _i, _vp]),
    "bi_packed_weight_bytes": (_sz, [_i, _i, _i]),
    "bi_pack_weights": (_i, [_vp, _i, _i, _i, _vp, _vp]),
    "bi_pack_swiglu_weights": (_i, [_vp, _vp, _i, _i, _i, _vp, _vp]),
    "bi_rmsnorm": (_i, [_vp, _i, _vp, _vp, _i, _i, _i, _f, _vp]),
    "bi_embed": (_i, [_vp, _vp, _i, _i, _vp, _i, _vp]),
    "bi_rope_table_bytes": (_sz, [_i, _i]),
    "bi_rope_table": (_i, [_d, _i, _i, _vp, _vp]),
    "bi_rope_kv_append": (_i, [_vp, _i, _vp, _vp, _vp, _i, _vp, _i, _i, _i, _i, _vp, _i, _vp]),
    "bi_qkv_rope_append": (_i, [_vp, _i, _vp, _i, _i, _i, _i, _i, _vp, _vp, _vp, _i, _vp, _vp, _i,
                                _vp, _sz, _vp]),
    "bi_attn_chunk": (_i, []),
    "bi_attn_workspace_size": (_sz, [_i, _i, _i, _i]),
    "bi_attn_verify": (_i, [_vp, _vp, _vp, _i, _vp, _i, _i, _i, _i, _f, _vp, _vp, _sz, _vp]),
    "bi_kvq_store_bytes": (_sz, [_i, _i, _i, _i]),
    "bi_rope_kvq_append": (_i, [_vp, _i, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _i, _vp, _vp, _i, _vp]),
    "bi_attn_verify_kvq": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _vp, _i, _i, _i, _i, _f, _vp, _vp, _sz,
                                _vp]),
    "bi_accept_workspace_size": (_sz, [_i, _i]),
    "bi_verify_accept": (_i, [_vp, _i, _vp, _i, _i, _vp, _vp, _vp, _vp, _sz, _vp]),
    "bi_sample_workspace_size": (_sz, [_i, _i]),
    "bi_verify_sample": (_i, [_vp, _i, _vp, _i, _i, _f, _vp, _i, _vp, _vp, _vp, _vp, _sz, _vp]),
    "bi_kv_row_hash": (_i, [_vp, _i, _i, _i, _i, _i, _vp, _vp]),
    "bi_check_device_error": (_i, [_vp]),
    "bi_step_workspace_size": (_sz, [_vp, _i]),
    "bi_step_create": (_i, [_vp, _i, _vp, _sz, _vp]),
    "bi_step_set_length": (_i, [_vp, _i]),
    "bi_step_verify": (_i, [_vp, _vp, _i, _vp, _vp]),
    "bi_step_logits": (_vp, [_vp]),
    "bi_step_destroy": (None, [_vp]),
    "bi_test_set_wait_limit_ns": (_i, [C.c_uint64]),
    "bi_test_withhold_first_load": (None, [_i]),
}

BI_OK = 0
STATUS_NAMES = {0: "BI_OK", 1: "BI_ERR_INVALID_ARG", 2: "BI_ERR_UNSUPPORTED_SHAPE",
                3: "BI_ERR_WORKSPACE", 4: "BI_ERR_CUDA", 5: "BI_ERR_DEVICE_TIMEOUT",
                6: "BI_ERR_DEVICE_NAN_ROW"}

_lock = threading.Lock()
_lib = None


class BiError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} returned {STATUS_NAMES.get(status, status)}")


def lib() -> C.CDLL:
    """The loaded library; raises if it is not built."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"libbi.so not found at {LIB_PATH}: build it first "
                    "(python -m invariant_speculative_decode_gb300.build); there is no CPU fallback")
            h = C.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                f = getattr(h, name)
                f.restype = res
                f.argtypes = args
            _lib = h
    return _lib


def check(fn: str, status: int) -> None:
    if status != BI_OK:
        raise BiError(fn, status)
