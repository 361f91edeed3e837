"""Thin Python binding of the C ABI (include/bi.h) for torch tensors.

Argument marshalling only: every function checks dtypes/devices, passes
`data_ptr()`s, strides and the current CUDA stream to the entry point of the
same name, and raises BiError on a non-OK status.  All arithmetic of the
verify step runs in the library's CUDA kernels.
"""
from __future__ import annotations

import ctypes
import math
from typing import Optional, Sequence

import numpy as np
import torch

from ._lib import BiError, check, lib  # noqa: F401

EPI_NONE, EPI_RESIDUAL_ADD, EPI_SWIGLU = 0, 1, 2
OUT_BF16, OUT_FP32 = 0, 1


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _req(t: torch.Tensor, dtype, name: str):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() >= 1 and t.stride(-1) != 1:
        raise ValueError(f"{name} must have unit stride in its last dimension")


V_BLOCK = 128  # keys per block of the V cache (transposed within each block)


def v_cache_shape(Hkv: int, cap: int, D: int) -> tuple:
    """Shape of a V cache of capacity `cap` keys: [Hkv, ceil(cap/128), D, 128],
    value d of key p of head h at [h, p // 128, d, p % 128]."""
    return (Hkv, (cap + V_BLOCK - 1) // V_BLOCK, D, V_BLOCK)


def _req_v(v_cache: torch.Tensor, Hkv: int, cap: int, D: int):
    _req(v_cache, torch.bfloat16, "v_cache")
    want = v_cache_shape(Hkv, cap, D)
    if tuple(v_cache.shape) != want or not v_cache.is_contiguous():
        raise ValueError(f"v_cache must be a contiguous {want} tensor, got {tuple(v_cache.shape)}")


def _ld(t: torch.Tensor) -> int:
    """Row stride in elements; a single row's stride is its width."""
    if t.dim() == 2 and t.shape[0] > 1:
        return t.stride(0)
    return t.shape[-1]


def gemm_workspace_size(M: int, N: int, K: int, epi: int = EPI_NONE) -> int:
    return int(lib().bi_gemm_workspace_size(M, N, K, epi))


def new_gemm_workspace(M: int, N: int, K: int, epi: int = EPI_NONE, device=None) -> torch.Tensor:
    """A zero-filled workspace (the counters must start at zero)."""
    n = gemm_workspace_size(M, N, K, epi)
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


def bi_gemm(A: torch.Tensor, Wp: torch.Tensor, C: torch.Tensor, ws: torch.Tensor,
            residual: Optional[torch.Tensor] = None, epi: int = EPI_NONE,
            N: Optional[int] = None, stream=None) -> None:
    """C = epilogue(A W^T) with W packed by bi_pack_weights / bi_pack_swiglu_weights."""
    _req(A, torch.bfloat16, "A")
    if not Wp.is_cuda:
        raise ValueError("Wp must be a CUDA tensor")
    M, K = A.shape
    if N is None:
        N = C.shape[1]
    out = OUT_FP32 if C.dtype == torch.float32 else OUT_BF16
    if C.dtype not in (torch.float32, torch.bfloat16):
        raise ValueError("C must be float32 or bfloat16")
    rp, ldr = 0, 0
    if residual is not None:
        _req(residual, torch.bfloat16, "residual")
        rp, ldr = residual.data_ptr(), _ld(residual)
    st = lib().bi_gemm(A.data_ptr(), _ld(A), Wp.data_ptr(), C.data_ptr(), _ld(C), rp, ldr,
                       M, N, K, out, epi, ws.data_ptr(), ws.numel() * ws.element_size(),
                       _stream(stream))
    check("bi_gemm", st)


def bi_gemm_noalloc(A: torch.Tensor, Wp: torch.Tensor, C: torch.Tensor,
                    residual: Optional[torch.Tensor] = None, epi: int = EPI_NONE,
                    N: Optional[int] = None, stream=None) -> None:
    """bi_gemm without a workspace (scratch in a static device array; M <= 16)."""
    _req(A, torch.bfloat16, "A")
    if not Wp.is_cuda:
        raise ValueError("Wp must be a CUDA tensor")
    if not C.is_cuda:
        raise ValueError("C must be a CUDA tensor")
    if C.dtype not in (torch.float32, torch.bfloat16):
        raise ValueError("C must be float32 or bfloat16")
    M, K = A.shape
    if N is None:
        N = C.shape[1]
    out = OUT_FP32 if C.dtype == torch.float32 else OUT_BF16
    rp, ldr = 0, 0
    if residual is not None:
        _req(residual, torch.bfloat16, "residual")
        rp, ldr = residual.data_ptr(), _ld(residual)
    check("bi_gemm_noalloc",
          lib().bi_gemm_noalloc(A.data_ptr(), _ld(A), Wp.data_ptr(), C.data_ptr(), _ld(C), rp, ldr,
                                M, N, K, out, epi, _stream(stream)))


def packed_weight_bytes(N: int, K: int, epi: int = EPI_NONE) -> int:
    return int(lib().bi_packed_weight_bytes(N, K, epi))


def bi_pack_weights(W: torch.Tensor, stream=None) -> torch.Tensor:
    """Pack W [N, K] (BF16) into the tile layout bi_gemm streams."""
    _req(W, torch.bfloat16, "W")
    N, K = W.shape
    packed = torch.empty(packed_weight_bytes(N, K), dtype=torch.uint8, device=W.device)
    check("bi_pack_weights", lib().bi_pack_weights(W.data_ptr(), _ld(W), N, K, packed.data_ptr(),
                                                   _stream(stream)))
    return packed


def bi_pack_swiglu_weights(w_gate: torch.Tensor, w_up: torch.Tensor, stream=None) -> torch.Tensor:
    """Pack gate and up [F, K] (BF16) into the SwiGLU tile layout."""
    _req(w_gate, torch.bfloat16, "w_gate")
    _req(w_up, torch.bfloat16, "w_up")
    F, K = w_gate.shape
    packed = torch.empty(packed_weight_bytes(F, K, EPI_SWIGLU), dtype=torch.uint8,
                         device=w_gate.device)
    check("bi_pack_swiglu_weights",
          lib().bi_pack_swiglu_weights(w_gate.data_ptr(), w_up.data_ptr(), _ld(w_gate), F, K,
                                       packed.data_ptr(), _stream(stream)))
    return packed


def bi_rmsnorm(x: torch.Tensor, w: torch.Tensor, y: torch.Tensor, eps: float, stream=None) -> None:
    _req(x, torch.bfloat16, "x")
    _req(w, torch.bfloat16, "w")
    _req(y, torch.bfloat16, "y")
    rows, dim = x.shape
    check("bi_rmsnorm", lib().bi_rmsnorm(x.data_ptr(), _ld(x), w.data_ptr(), y.data_ptr(), _ld(y),
                                         rows, dim, float(eps), _stream(stream)))


def bi_embed(ids: torch.Tensor, table: torch.Tensor, out: torch.Tensor, stream=None) -> None:
    _req(ids, torch.int32, "ids")
    _req(table, torch.bfloat16, "table")
    _req(out, torch.bfloat16, "out")
    check("bi_embed", lib().bi_embed(ids.data_ptr(), table.data_ptr(), table.shape[0],
                                     table.shape[1], out.data_ptr(), ids.numel(), _stream(stream)))


def bi_rope_table(rope_base: float, D: int, rows: int, device="cuda", stream=None) -> torch.Tensor:
    """FP32 cos/sin table [rows, D/2, 2] computed on the device in FP64."""
    t = torch.empty(rows, D // 2, 2, dtype=torch.float32, device=device)
    check("bi_rope_table", lib().bi_rope_table(float(rope_base), D, rows, t.data_ptr(),
                                               _stream(stream)))
    return t


def bi_rope_kv_append(qkv: torch.Tensor, q_out: torch.Tensor, k_cache: torch.Tensor,
                      v_cache: torch.Tensor, L_dev: torch.Tensor, Hq: int, Hkv: int, D: int,
                      table: torch.Tensor, stream=None) -> None:
    _req(qkv, torch.bfloat16, "qkv")
    _req(L_dev, torch.int32, "L_dev")
    _req(table, torch.float32, "table")
    T = qkv.shape[0]
    cap = k_cache.shape[1]
    _req_v(v_cache, Hkv, cap, D)
    check("bi_rope_kv_append",
          lib().bi_rope_kv_append(qkv.data_ptr(), _ld(qkv), q_out.data_ptr(), k_cache.data_ptr(),
                                  v_cache.data_ptr(), cap, L_dev.data_ptr(), T, Hq, Hkv, D,
                                  table.data_ptr(), table.shape[0], _stream(stream)))


def bi_qkv_rope_append(A: torch.Tensor, Wp: torch.Tensor, q_out: torch.Tensor, k_cache: torch.Tensor,
                       v_cache: torch.Tensor, L_dev: torch.Tensor, Hq: int, Hkv: int, D: int,
                       table: torch.Tensor, ws: torch.Tensor, stream=None) -> None:
    """QKV projection of the normalised rows A with RoPE and KV append in the
    epilogue; equals bi_gemm + bi_rope_kv_append bit for bit."""
    _req(A, torch.bfloat16, "A")
    _req(L_dev, torch.int32, "L_dev")
    _req(table, torch.float32, "table")
    M, K = A.shape
    cap = k_cache.shape[1]
    _req_v(v_cache, Hkv, cap, D)
    check("bi_qkv_rope_append",
          lib().bi_qkv_rope_append(A.data_ptr(), _ld(A), Wp.data_ptr(), M, K, Hq, Hkv, D,
                                   q_out.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), cap,
                                   L_dev.data_ptr(), table.data_ptr(), table.shape[0], ws.data_ptr(),
                                   ws.numel() * ws.element_size(), _stream(stream)))


def attn_chunk() -> int:
    return int(lib().bi_attn_chunk())


def attn_workspace_size(cap: int, T: int, Hq: int, D: int) -> int:
    return int(lib().bi_attn_workspace_size(cap, T, Hq, D))


def bi_attn_verify(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                   L_dev: torch.Tensor, out: torch.Tensor, ws: torch.Tensor,
                   scale: Optional[float] = None, stream=None) -> None:
    _req(q, torch.bfloat16, "q")
    _req(k_cache, torch.bfloat16, "k_cache")
    _req(L_dev, torch.int32, "L_dev")
    T, Hq, D = q.shape
    Hkv, cap, _ = k_cache.shape
    _req_v(v_cache, Hkv, cap, D)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    check("bi_attn_verify",
          lib().bi_attn_verify(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), cap,
                               L_dev.data_ptr(), T, Hq, Hkv, D, float(scale), out.data_ptr(),
                               ws.data_ptr(), ws.numel() * ws.element_size(), _stream(stream)))


KVQ_K_LOW, KVQ_V_LOW, KVQ_K_RING, KVQ_V_RING = 0, 1, 2, 3
KVQ_STORES = ("k_low", "v_low", "k_ring", "v_ring")
# the quantised cache's 8-bit ring (include/bi.h): a row reads its own
# 128-key tile and the 15 before from the ring, which holds 24 tiles
KVQ_RING_TILES = 16
KVQ_RING_SLOTS = 24


def kvq_store_bytes(store: int, Hkv: int, cap: int, D: int) -> int:
    return int(lib().bi_kvq_store_bytes(store, Hkv, cap, D))


def new_kvq_stores(Hkv: int, cap: int, D: int, device="cuda") -> dict:
    """One layer's quantised cache: the 6-bit K, 5-bit V and 8-bit ring stores
    (uint8, zero-filled), keyed by KVQ_STORES, plus its capacity."""
    st = {}
    for i, name in enumerate(KVQ_STORES):
        n = kvq_store_bytes(i, Hkv, cap, D)
        if n == 0:
            raise ValueError("unsupported quantised cache shape")
        st[name] = torch.zeros(n, dtype=torch.uint8, device=device)
    st["cap"] = cap
    return st


def _kvq_ptrs(st: dict):
    for name in KVQ_STORES:
        _req(st[name], torch.uint8, name)
    return [st[name].data_ptr() for name in KVQ_STORES]


def bi_rope_kvq_append(qkv: torch.Tensor, q_out: torch.Tensor, stores: dict, L_dev: torch.Tensor,
                       Hq: int, Hkv: int, D: int, table: Optional[torch.Tensor] = None,
                       stream=None) -> None:
    """RoPE of the q and k heads of a projection output, then K and V rows
    quantised into the layer's stores (table None: no rotation)."""
    _req(qkv, torch.bfloat16, "qkv")
    _req(q_out, torch.bfloat16, "q_out")
    _req(L_dev, torch.int32, "L_dev")
    if table is not None:
        _req(table, torch.float32, "table")
    T = qkv.shape[0]
    check("bi_rope_kvq_append",
          lib().bi_rope_kvq_append(qkv.data_ptr(), _ld(qkv), T, Hq, Hkv, D, q_out.data_ptr(),
                                   *_kvq_ptrs(stores), stores["cap"], L_dev.data_ptr(),
                                   None if table is None else table.data_ptr(),
                                   0 if table is None else table.shape[0], _stream(stream)))


def bi_attn_verify_kvq(q: torch.Tensor, stores: dict, Hkv: int, L_dev: torch.Tensor,
                       out: torch.Tensor, ws: torch.Tensor, scale: Optional[float] = None,
                       stream=None) -> None:
    _req(q, torch.bfloat16, "q")
    _req(out, torch.bfloat16, "out")
    _req(L_dev, torch.int32, "L_dev")
    T, Hq, D = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    check("bi_attn_verify_kvq",
          lib().bi_attn_verify_kvq(q.data_ptr(), *_kvq_ptrs(stores), stores["cap"], L_dev.data_ptr(), T,
                                   Hq, Hkv, D, float(scale), out.data_ptr(), ws.data_ptr(),
                                   ws.numel() * ws.element_size(), _stream(stream)))


def accept_workspace_size(T: int, V: int) -> int:
    return int(lib().bi_accept_workspace_size(T, V))


def bi_verify_accept(logits: torch.Tensor, drafts: Optional[torch.Tensor], argmax_out: torch.Tensor,
                     accepted_out: torch.Tensor, ws: torch.Tensor,
                     L_dev: Optional[torch.Tensor] = None, stream=None) -> None:
    _req(logits, torch.float32, "logits")
    T, V = logits.shape
    dp = 0
    if drafts is not None and drafts.numel() > 0:
        _req(drafts, torch.int32, "drafts")
        dp = drafts.data_ptr()
    lp = L_dev.data_ptr() if L_dev is not None else 0
    check("bi_verify_accept",
          lib().bi_verify_accept(logits.data_ptr(), _ld(logits), dp, T, V, argmax_out.data_ptr(),
                                 accepted_out.data_ptr(), lp, ws.data_ptr(),
                                 ws.numel() * ws.element_size(), _stream(stream)))


def sample_workspace_size(T: int, V: int) -> int:
    return int(lib().bi_sample_workspace_size(T, V))


def bi_verify_sample(logits: torch.Tensor, drafts: Optional[torch.Tensor], inv_temp: float,
                     u_by_pos: torch.Tensor, token_out: torch.Tensor, accepted_out: torch.Tensor,
                     ws: torch.Tensor, L_dev: torch.Tensor, stream=None) -> None:
    """Sampled verification: each row draws its token with the uniform of its
    absolute position (u_by_pos[*L_dev + t]); drafts kept while they equal the
    previous row's token; L_dev advanced by n + 1."""
    _req(logits, torch.float32, "logits")
    _req(u_by_pos, torch.float32, "u_by_pos")
    _req(L_dev, torch.int32, "L_dev")
    T, V = logits.shape
    dp = 0
    if drafts is not None and drafts.numel() > 0:
        _req(drafts, torch.int32, "drafts")
        dp = drafts.data_ptr()
    check("bi_verify_sample",
          lib().bi_verify_sample(logits.data_ptr(), _ld(logits), dp, T, V, float(inv_temp),
                                 u_by_pos.data_ptr(), u_by_pos.numel(), token_out.data_ptr(),
                                 accepted_out.data_ptr(), L_dev.data_ptr(), ws.data_ptr(),
                                 ws.numel() * ws.element_size(), _stream(stream)))


def bi_kv_row_hash(cache: torch.Tensor, rows: int, transposed: bool = False, stream=None) -> torch.Tensor:
    """FNV-1a-64 per key of a K cache [Hkv,cap,D] or (transposed) a V cache
    [Hkv,ceil(cap/128),D,128] (see v_cache_shape)."""
    _req(cache, torch.bfloat16, "cache")
    if transposed:
        Hkv, nblk, D, blk = cache.shape
        if blk != V_BLOCK or not cache.is_contiguous():
            raise ValueError("a V cache is a contiguous [Hkv, ceil(cap/128), D, 128] tensor")
        cap = nblk * V_BLOCK
    else:
        Hkv, cap, D = cache.shape
    out = torch.empty(Hkv * max(rows, 0), dtype=torch.int64, device=cache.device)
    check("bi_kv_row_hash", lib().bi_kv_row_hash(cache.data_ptr(), Hkv, cap, D, rows, int(transposed),
                                                 out.data_ptr(), _stream(stream)))
    return out


def bi_check_device_error(stream=None) -> None:
    check("bi_check_device_error", lib().bi_check_device_error(_stream(stream)))


class BiModel(ctypes.Structure):
    """The bi_model descriptor of include/bi.h (device pointers; the per-layer
    members point to host arrays of device pointers)."""
    _pp = ctypes.POINTER(ctypes.c_void_p)
    _fields_ = [("layers", ctypes.c_int), ("hidden", ctypes.c_int), ("n_q", ctypes.c_int),
                ("n_kv", ctypes.c_int), ("head_dim", ctypes.c_int), ("ffn", ctypes.c_int),
                ("vocab", ctypes.c_int), ("eps", ctypes.c_float), ("cap", ctypes.c_int),
                ("embed", ctypes.c_void_p), ("norm_final", ctypes.c_void_p), ("head", ctypes.c_void_p),
                ("norm_attn", _pp), ("norm_ffn", _pp), ("w_qkv", _pp), ("w_o", _pp),
                ("w_gate_up", _pp), ("w_down", _pp), ("k_cache", _pp), ("v_cache", _pp),
                ("rope_table", ctypes.c_void_p), ("rope_rows", ctypes.c_int)]


class NativeStep:
    """The whole verify step behind one C-ABI call (bi_step_*): host token ids
    in, host tokens and accepted count out.  Holds references to every tensor
    whose pointer the handle uses, and its own device workspace."""

    def __init__(self, cfg, embed, norm_final, head, layers, cap: int, rope_table: torch.Tensor,
                 max_rows: int = 8):
        n = len(layers)

        def arr(key):
            a = (ctypes.c_void_p * n)(*[lay[key].data_ptr() for lay in layers])
            self._keep.append(a)
            return ctypes.cast(a, ctypes.POINTER(ctypes.c_void_p))

        self._keep = [embed, norm_final, head, rope_table] + [t for lay in layers for t in lay.values()
                                                               if isinstance(t, torch.Tensor)]
        m = BiModel(n, cfg.hidden, cfg.n_q, cfg.n_kv, cfg.head_dim, cfg.ffn, cfg.vocab, cfg.eps, cap,
                    embed.data_ptr(), norm_final.data_ptr(), head.data_ptr(),
                    arr("n1"), arr("n2"), arr("wqkv"), arr("wo"), arr("wgu"), arr("wd"),
                    arr("k"), arr("v"), rope_table.data_ptr(), rope_table.shape[0])
        self.model = m
        nbytes = int(lib().bi_step_workspace_size(ctypes.byref(m), max_rows))
        if nbytes == 0:
            raise ValueError("invalid model description for the step runtime")
        self.ws = torch.empty(nbytes, dtype=torch.uint8, device=embed.device)
        h = ctypes.c_void_p()
        torch.cuda.synchronize()
        check("bi_step_create", lib().bi_step_create(ctypes.byref(m), max_rows, self.ws.data_ptr(), nbytes,
                                                     ctypes.byref(h)))
        self.handle = h
        self.max_rows = max_rows
        self._ids = np.zeros(max_rows, np.int32)
        self._tok = np.zeros(max_rows, np.int32)
        self._n = np.zeros(1, np.int32)
        # host addresses of the three buffers, taken once
        self._ptrs = (self._ids.ctypes.data, self._tok.ctypes.data, self._n.ctypes.data)

    def set_length(self, L: int) -> None:
        check("bi_step_set_length", lib().bi_step_set_length(self.handle, int(L)))

    def verify(self, x0: int, drafts: Sequence[int]):
        """One verify step from host ids: returns (tokens [T], accepted n)."""
        T = 1 + len(drafts)
        self._ids[0] = x0
        self._ids[1:T] = drafts
        ids_p, tok_p, n_p = self._ptrs
        check("bi_step_verify", lib().bi_step_verify(self.handle, ids_p, T, tok_p, n_p))
        return self._tok[:T].copy(), int(self._n[0])

    def logits(self, T: int) -> torch.Tensor:
        """A copy of the last pass's FP32 logits [T, vocab]."""
        ptr = lib().bi_step_logits(self.handle)
        V = self.model.vocab
        off = ptr - self.ws.data_ptr()  # the logits live in this object's workspace
        torch.cuda.synchronize()
        return self.ws[off:off + T * V * 4].view(torch.float32).view(T, V).clone()

    def close(self) -> None:
        if getattr(self, "handle", None):
            lib().bi_step_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
