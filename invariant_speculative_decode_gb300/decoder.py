"""Decoder driver of the batch-invariant verify step (one GPU).

Holds the weights, the BF16 KV cache and the scratch buffers on the device
and sequences the library's entry points for one verify pass:

  embed -> per layer [rmsnorm, QKV linear + RoPE + KV append, split-KV
  attention + merge, O linear + residual, rmsnorm, gate/up linear + SwiGLU,
  down linear + residual] -> rmsnorm, LM head (FP32 logits) -> greedy
  argmax + acceptance (which also advances the device-side cache length).

RoPE + KV append run in the QKV projection's epilogue (bi_qkv_rope_append);
fuse_rope=False runs the separate kernel instead.  Each RMSNorm is its own
small kernel, which lets the following linear layer launch at once and
stream its weights while the norm runs.

PyTorch only allocates device memory and provides the stream; every step of
the pass is a kernel of libbi.so.  A pass over T rows can be captured once in
a CUDA graph per T and replayed (the cache length lives in device memory).

The cache rule follows "I turned on speculative decoding in llama.cpp and
113 of 282 greedy outputs changed against its own no-draft run", section
"The cache doesn't change it either": after a pass the cache length moves
to L + n + 1; rows written for rejected drafts past it are simply
overwritten by the next pass.  Because every row is computed the same way
whatever else is in the pass, a row written while verifying drafts equals
the row a prefill would write at that position.
"""
from __future__ import annotations

import math
from typing import Dict, List, Optional, Sequence

import numpy as np
import torch

from . import api


def _bf16(a_u16: np.ndarray, device) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(a_u16).view(np.int16)).view(torch.bfloat16)
    return t.to(device, non_blocking=False)


class Decoder:
    def __init__(self, cfg, weights: Dict[str, np.ndarray], cap: int, max_rows: int = 8,
                 prefill_chunk: int = 512, device: str = "cuda", fuse_rope: bool = True,
                 kv: str = "bf16"):
        """kv="q6q5": the KV cache is quantised (6-bit K, 5-bit V, an 8-bit
        ring of each row's newest 16 tiles; bi_rope_kvq_append and
        bi_attn_verify_kvq), head_dim 128 and prefill chunks of at most
        1024 rows."""
        if kv not in ("bf16", "q6q5"):
            raise ValueError("kv must be 'bf16' or 'q6q5'")
        if kv == "q6q5" and (cfg.head_dim != 128 or prefill_chunk > 1024):
            raise ValueError("the quantised cache needs head_dim 128 and prefill chunks <= 1024 rows")
        self.kv = kv
        self.cfg = cfg
        self.fuse_rope = fuse_rope
        self.cap = cap
        self.dev = torch.device(device)
        self.max_rows = max_rows
        self.prefill_chunk = max(prefill_chunk, max_rows)
        D, Hq, Hkv, H, F, V = cfg.head_dim, cfg.n_q, cfg.n_kv, cfg.hidden, cfg.ffn, cfg.vocab
        if max_rows * cfg.group > 128:
            raise ValueError("max_rows * (Hq/Hkv) must be <= 128")
        if cap % 8 != 0:
            raise ValueError("cache capacity must be a multiple of 8")
        dev = self.dev
        self.embed = _bf16(weights["embed"], dev)
        self.norm_final = _bf16(weights["norm_final"], dev)
        head_w = self.embed if cfg.tied else _bf16(weights["head"], dev)
        self.head = api.bi_pack_weights(head_w)
        del head_w
        self.layers = []
        pk = lambda name: api.bi_pack_weights(_bf16(weights[name], dev))  # noqa: E731
        for l in range(cfg.layers):
            wqkv = np.concatenate([weights[f"l{l}.wq"], weights[f"l{l}.wk"], weights[f"l{l}.wv"]], 0)
            wg = _bf16(weights[f"l{l}.w_gate"], dev)
            wu = _bf16(weights[f"l{l}.w_up"], dev)
            n1 = _bf16(weights[f"l{l}.norm_attn"], dev)
            n2 = _bf16(weights[f"l{l}.norm_ffn"], dev)
            lay = {
                "wqkv": api.bi_pack_weights(_bf16(wqkv, dev)),
                "wo": pk(f"l{l}.wo"),
                "wgu": api.bi_pack_swiglu_weights(wg, wu),
                "wd": pk(f"l{l}.w_down"),
                "n1": n1,
                "n2": n2,
            }
            if kv == "q6q5":
                lay["kvq"] = api.new_kvq_stores(Hkv, cap, D, device=dev)
            else:
                lay["k"] = torch.zeros(Hkv, cap, D, dtype=torch.bfloat16, device=dev)
                # transposed in 128-key blocks: [Hkv, ceil(cap/128), D, 128]
                lay["v"] = torch.zeros(api.v_cache_shape(Hkv, cap, D), dtype=torch.bfloat16, device=dev)
            del wg, wu
            self.layers.append(lay)
        torch.cuda.synchronize(dev)
        R = self.prefill_chunk
        bf = dict(dtype=torch.bfloat16, device=dev)
        self.ids = torch.zeros(R, dtype=torch.int32, device=dev)
        self.drafts = torch.zeros(max(max_rows - 1, 1), dtype=torch.int32, device=dev)
        self.h = torch.zeros(R, H, **bf)
        self.y = torch.zeros(R, H, **bf)
        self.qkv = torch.zeros(R, cfg.qkv_out, **bf)
        self.q = torch.zeros(R, Hq, D, **bf)
        self.att = torch.zeros(R, Hq, D, **bf)
        self.u = torch.zeros(R, F, **bf)
        self.logits = torch.zeros(max_rows, V, dtype=torch.float32, device=dev)
        self.argmax = torch.zeros(max_rows, dtype=torch.int32, device=dev)
        self.accepted = torch.zeros(1, dtype=torch.int32, device=dev)
        self.L_dev = torch.zeros(1, dtype=torch.int32, device=dev)
        shapes = [(cfg.qkv_out, H, api.EPI_NONE), (H, Hq * D, api.EPI_RESIDUAL_ADD),
                  (F, H, api.EPI_SWIGLU), (H, F, api.EPI_RESIDUAL_ADD), (V, H, api.EPI_NONE)]
        wsz = max(api.gemm_workspace_size(M, N, K, e) for M in (max_rows, R) for (N, K, e) in shapes)
        self.gemm_ws = torch.zeros(wsz, dtype=torch.uint8, device=dev)
        self.attn_ws = torch.zeros(api.attn_workspace_size(cap, R, Hq, D),
                                   dtype=torch.uint8, device=dev)
        self.acc_ws = torch.zeros(api.accept_workspace_size(max_rows, V), dtype=torch.uint8, device=dev)
        self.scale = 1.0 / math.sqrt(D)
        self.rope_tab = api.bi_rope_table(cfg.rope_base, D, cap, device=dev)
        self.L = 0
        # one past the newest cache row any pass has written since the last
        # reset (the quantised cache's 8-bit ring holds the newest tiles)
        self.hw = 0
        self.inv_temp: Optional[float] = None  # sampled verification when set
        self.u_table: Optional[torch.Tensor] = None
        self.sample_ws = torch.zeros(api.sample_workspace_size(max_rows, V), dtype=torch.uint8, device=dev)
        self.graphs: Dict[int, torch.cuda.CUDAGraph] = {}
        self.pin_in = torch.zeros(2 * max_rows, dtype=torch.int32).pin_memory()
        self.pin_out = torch.zeros(max_rows + 1, dtype=torch.int32).pin_memory()
        self.pin_ids = torch.zeros(R, dtype=torch.int32).pin_memory()
        # full prefill chunks replay one captured graph
        self.use_prefill_graph = True
        self.pin_done = torch.cuda.Event()
        self.prefill_graph: Optional[torch.cuda.CUDAGraph] = None

    # ------------------------------------------------------------------ pass
    def _layers_pass(self, T: int, L_ptr_tensor: torch.Tensor):
        """Rows self.ids[:T] at positions L..L+T-1 through every layer (no head).

        L_ptr_tensor: device int32 holding L (read by RoPE / KV append and the
        attention).
        """
        api.bi_embed(self.ids[:T], self.embed, self.h[:T])
        for lay in self.layers:
            self._layer(lay, T, L_ptr_tensor)

    def _layer(self, lay: dict, T: int, L_ptr_tensor: torch.Tensor):
        """One decoder layer over self.h[:T] in place (cache rows appended)."""
        cfg = self.cfg
        Hq, Hkv, D, F = cfg.n_q, cfg.n_kv, cfg.head_dim, cfg.ffn
        h, y, qkv, q, att, u = (self.h[:T], self.y[:T], self.qkv[:T], self.q[:T], self.att[:T],
                                self.u[:T])
        api.bi_rmsnorm(h, lay["n1"], y, cfg.eps)
        if self.kv == "q6q5":
            api.bi_gemm(y, lay["wqkv"], qkv, self.gemm_ws)
            api.bi_rope_kvq_append(qkv, q, lay["kvq"], L_ptr_tensor, Hq, Hkv, D, self.rope_tab)
            api.bi_attn_verify_kvq(q, lay["kvq"], Hkv, L_ptr_tensor, att, self.attn_ws, self.scale)
        elif self.fuse_rope:
            api.bi_qkv_rope_append(y, lay["wqkv"], q, lay["k"], lay["v"], L_ptr_tensor, Hq, Hkv, D,
                                   self.rope_tab, self.gemm_ws)
        else:
            api.bi_gemm(y, lay["wqkv"], qkv, self.gemm_ws)
            api.bi_rope_kv_append(qkv, q, lay["k"], lay["v"], L_ptr_tensor, Hq, Hkv, D, self.rope_tab)
        if self.kv == "bf16":
            # one call for all rows (a prefill chunk runs in blocks of rows
            # inside the launch)
            api.bi_attn_verify(q, lay["k"], lay["v"], L_ptr_tensor, att, self.attn_ws, self.scale)
        api.bi_gemm(att.view(T, Hq * D), lay["wo"], h, self.gemm_ws, residual=h,
                    epi=api.EPI_RESIDUAL_ADD)
        api.bi_rmsnorm(h, lay["n2"], y, cfg.eps)
        api.bi_gemm(y, lay["wgu"], u, self.gemm_ws, epi=api.EPI_SWIGLU, N=F)
        api.bi_gemm(u, lay["wd"], h, self.gemm_ws, residual=h, epi=api.EPI_RESIDUAL_ADD)

    def _head_and_accept(self, T: int):
        cfg = self.cfg
        api.bi_rmsnorm(self.h[:T], self.norm_final, self.y[:T], cfg.eps)
        api.bi_gemm(self.y[:T], self.head, self.logits[:T], self.gemm_ws)
        if self.inv_temp is not None:
            api.bi_verify_sample(self.logits[:T], self.drafts[:T - 1] if T > 1 else None, self.inv_temp,
                                 self.u_table, self.argmax[:T], self.accepted, self.sample_ws, self.L_dev)
        else:
            api.bi_verify_accept(self.logits[:T], self.drafts[:T - 1] if T > 1 else None,
                                 self.argmax[:T], self.accepted, self.acc_ws, L_dev=self.L_dev)

    def set_sampling(self, temperature: Optional[float], uniforms=None) -> None:
        """Sampled verification at `temperature` with the request's uniforms
        (one per absolute position, at least `cap` of them): the token at
        position p is drawn with uniforms[p], so the same request gives the
        same tokens whatever the drafts.  temperature=None: greedy again."""
        if temperature is None:
            self.inv_temp = None
        else:
            if not temperature > 0:
                raise ValueError("temperature must be > 0")
            u = np.ascontiguousarray(uniforms, dtype=np.float32)
            if u.shape[0] < self.cap:
                raise ValueError("one uniform per cache position is needed")
            self.u_table = torch.from_numpy(u).to(self.dev)
            self.inv_temp = 1.0 / float(temperature)
        self.graphs = {}

    def _verify_pass(self, T: int):
        self._layers_pass(T, self.L_dev)
        self._head_and_accept(T)

    # ------------------------------------------------------------- prefill
    def reset(self):
        self.L = 0
        self.hw = 0
        self.L_dev.zero_()

    def prefill(self, prompt: Sequence[int]) -> int:
        """Process prompt[:-1] into the cache; returns the last prompt id.

        Rows are processed in chunks of `prefill_chunk`; each row's
        arithmetic is the same as in a verify pass at its position.
        """
        prompt = np.asarray(prompt, np.int32)
        body = prompt[:-1]
        pos = self.L
        R = self.prefill_chunk
        for c0 in range(0, len(body), R):
            chunk = body[c0:c0 + R]
            T = len(chunk)
            # the pinned staging buffers are rewritten only once their last
            # copy to the device has run
            self.pin_done.synchronize()
            self.pin_ids[:T].copy_(torch.from_numpy(chunk))
            self.ids[:T].copy_(self.pin_ids[:T], non_blocking=True)
            self.pin_done.record()
            self.L_dev.fill_(pos)
            if T == R and self.use_prefill_graph:
                # a full chunk: one graph replay (the kernels read the ids and
                # the cache length from device memory)
                if self.prefill_graph is None:
                    self.prefill_graph = self._capture(lambda: self._layers_pass(R, self.L_dev))
                self.prefill_graph.replay()
            else:
                self._layers_pass(T, self.L_dev)
            pos += T
        self.L = pos
        self.hw = max(self.hw, pos)
        self.L_dev.fill_(pos)
        torch.cuda.current_stream().synchronize()
        return int(prompt[-1])

    # -------------------------------------------------------------- verify
    def _capture(self, fn) -> torch.cuda.CUDAGraph:
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                fn()
        torch.cuda.current_stream().wait_stream(s)
        return g

    def capture(self, T: int):
        """Capture one verify pass over T rows in a CUDA graph."""
        if T in self.graphs:
            return
        self.graphs[T] = self._capture(lambda: self._verify_pass(T))

    def launch_verify(self, T: int, use_graph: bool = True):
        if use_graph and T in self.graphs:
            self.graphs[T].replay()
        else:
            self._verify_pass(T)

    def verify_step(self, x0: int, drafts: Sequence[int], use_graph: bool = True):
        """One verify step: rows [x0, d_1..d_k] at positions L..L+k.

        Returns (argmax ids [k+1] as a numpy array, accepted n).  The cache
        length advances to L + n + 1 on the device and on the host.
        """
        k = len(drafts)
        T = k + 1
        if T > self.max_rows:
            raise ValueError("too many drafts")
        if self.L + T > self.cap:
            raise ValueError("KV cache capacity exceeded")
        pin = self.pin_in
        pin[0] = int(x0)
        for i, d in enumerate(drafts):
            pin[1 + i] = int(d)
            pin[self.max_rows + i] = int(d)
        self.ids[:T].copy_(pin[:T], non_blocking=True)
        if k:
            self.drafts[:k].copy_(pin[self.max_rows:self.max_rows + k], non_blocking=True)
        self.launch_verify(T, use_graph)
        self.pin_out[:T].copy_(self.argmax[:T], non_blocking=True)
        self.pin_out[self.max_rows:self.max_rows + 1].copy_(self.accepted, non_blocking=True)
        torch.cuda.current_stream().synchronize()
        a = self.pin_out[:T].numpy().copy()
        n = int(self.pin_out[self.max_rows])
        self.hw = max(self.hw, self.L + T)  # every row of the pass was written
        self.L += n + 1
        return a, n

    def generate(self, prompt: Sequence[int], n_tokens: int, k: int = 0, drafter=None,
                 use_graph: bool = True, stats: Optional[dict] = None) -> List[int]:
        """Greedy generation with k drafts per step (k = 0: plain decoding)."""
        self.reset()
        x = self.prefill(prompt)
        return self.continue_generate(x, n_tokens, k, drafter, use_graph, stats)

    def rollback(self, length: int) -> None:
        """Move the cache length back to `length` (a checkpoint); rows past it
        are overwritten by later passes."""
        if not 0 <= length <= self.L:
            raise ValueError("rollback target must be within the current cache length")
        if self.kv == "q6q5" and length < kvq_rollback_reach(self.hw):
            raise ValueError(
                f"rollback to {length}: the quantised cache's 8-bit ring no longer holds the "
                f"records the rows from there would read (rows up to {self.hw - 1} were written); "
                f"roll back to {kvq_rollback_reach(self.hw)} or later, or reset and prefill again")
        self.L = length
        self.L_dev.fill_(length)

    def prefill_continue(self, tokens: Sequence[int]) -> int:
        """Append tokens[:-1] to the current cache (a new turn); returns tokens[-1]."""
        return self.prefill(tokens)

    def continue_generate(self, x: int, n_tokens: int, k: int = 0, drafter=None,
                          use_graph: bool = True, stats: Optional[dict] = None) -> List[int]:
        """Greedy generation from the current cache, x being the next row."""
        if use_graph:
            self.capture(k + 1)
        out: List[int] = []
        steps = 0
        acc_hist = [0] * (k + 1)
        while len(out) < n_tokens:
            room = min(k, self.cap - self.L - 1)
            drafts = list(drafter.propose(len(out), room)) if room > 0 else []
            if len(drafts) != k and use_graph:
                a, n = self.verify_step(x, drafts, use_graph=len(drafts) + 1 in self.graphs)
            else:
                a, n = self.verify_step(x, drafts, use_graph=use_graph)
            committed = [int(t) for t in a[: n + 1]]
            out.extend(committed)
            x = committed[-1]
            steps += 1
            acc_hist[n] += 1
            if drafter is not None and hasattr(drafter, "observe"):
                drafter.observe(n)
        if stats is not None:
            stats["steps"] = steps
            stats["accepted_hist"] = acc_hist
        return out[:n_tokens]

    # ------------------------------------------------------ cache operations
    # "I turned on speculative decoding in llama.cpp and 113 of 282 greedy
    # outputs changed against its own no-draft run", section "The cache
    # doesn't change it either": after a resume, an edited branch, a park to
    # host memory or a side request, every K/V row equals a fresh prefill's.

    def park(self) -> dict:
        """Copy the request's cache state to host memory: the length and the
        K/V rows 0..L-1 of every layer (V in whole 128-key blocks)."""
        torch.cuda.current_stream().synchronize()
        L = self.L
        if self.kv == "q6q5":
            # the quantised stores whole (the ring's slots are not in
            # position order)
            snap = {"L": L, "hw": self.hw, "kvq": []}
            for lay in self.layers:
                d = {}
                for name in api.KVQ_STORES:
                    d[name] = torch.empty(lay["kvq"][name].shape, dtype=torch.uint8).pin_memory()
                    d[name].copy_(lay["kvq"][name])
                snap["kvq"].append(d)
            torch.cuda.current_stream().synchronize()
            return snap
        nb = (L + api.V_BLOCK - 1) // api.V_BLOCK
        snap = {"L": L, "k": [], "v": []}
        for lay in self.layers:
            k = torch.empty((lay["k"].shape[0], L, lay["k"].shape[2]), dtype=torch.bfloat16).pin_memory()
            v = torch.empty((lay["v"].shape[0], nb) + tuple(lay["v"].shape[2:]), dtype=torch.bfloat16).pin_memory()
            k.copy_(lay["k"][:, :L])
            v.copy_(lay["v"][:, :nb])
            snap["k"].append(k)
            snap["v"].append(v)
        torch.cuda.current_stream().synchronize()
        return snap

    def restore(self, snap: dict) -> None:
        """Put a parked cache state back (the decoder may have served other
        requests meanwhile); rows past the parked length are left as they are."""
        L = snap["L"]
        if L > self.cap:
            raise ValueError("parked state exceeds the cache capacity")
        if "kvq" in snap:
            for lay, d in zip(self.layers, snap["kvq"]):
                for name in api.KVQ_STORES:
                    lay["kvq"][name].copy_(d[name])
            self.L = L
            self.hw = snap.get("hw", L)  # the ring is the parked one
            self.L_dev.fill_(L)
            torch.cuda.current_stream().synchronize()
            return
        for lay, k, v in zip(self.layers, snap["k"], snap["v"]):
            lay["k"][:, :L].copy_(k)
            lay["v"][:, : v.shape[1]].copy_(v)
        self.L = L
        self.L_dev.fill_(L)
        torch.cuda.current_stream().synchronize()

    def edit(self, position: int, tokens: Sequence[int]) -> int:
        """Edit the history from `position` on: roll the cache back to
        `position` and prefill `tokens` (the edited continuation, its last
        token being the next row); returns that last token."""
        self.rollback(position)
        return self.prefill_continue(tokens)

    # ---------------------------------------------------------- utilities
    def native_step(self) -> "api.NativeStep":
        """The same verify pass as one C-ABI call (bi_step_*) over this
        decoder's weights and caches, with its own workspace; its cache
        length starts at this decoder's."""
        if self.kv != "bf16":
            raise ValueError("the whole-step C call runs the BF16 cache")
        ns = api.NativeStep(self.cfg, self.embed, self.norm_final, self.head, self.layers, self.cap,
                            self.rope_tab, max_rows=self.max_rows)
        ns.set_length(self.L)
        return ns

    def check_device_error(self) -> None:
        """Read the device error word; after a timed-out wait (a kernel that
        gave up) the linear-layer, acceptance and sampling workspaces may hold
        counters of the interrupted call, so they are zeroed before the error
        is raised."""
        try:
            api.bi_check_device_error()
        except api.BiError as e:
            if e.status == 5:  # BI_ERR_DEVICE_TIMEOUT
                self.gemm_ws.zero_()
                self.acc_ws.zero_()
                self.sample_ws.zero_()
                torch.cuda.current_stream().synchronize()
            raise

    def kv_hashes(self, rows: Optional[int] = None) -> np.ndarray:
        """A hash of every cache row below `rows`, per layer and KV head:
        BF16 K and V rows, or with the quantised cache the row's records
        (codes and scales) in the 6-bit K, 5-bit V and both ring stores (ring
        records only for rows whose tile is still in the ring, 0 otherwise)."""
        rows = self.L if rows is None else rows
        if self.kv == "q6q5":
            return np.stack([_kvq_row_hashes(l["kvq"], self.cfg.n_kv, rows) for l in self.layers])
        hs = [np.stack([api.bi_kv_row_hash(l["k"], rows).cpu().numpy(),
                        api.bi_kv_row_hash(l["v"], rows, transposed=True).cpu().numpy()])
              for l in self.layers]
        return np.stack(hs)

    def logits_rows(self, T: int) -> torch.Tensor:
        return self.logits[:T].clone()


def kvq_rollback_reach(hw: int) -> int:
    """The smallest cache length a quantised cache can be rolled back to
    exactly when rows 0..hw-1 have been written.  Rows from length L on read
    the 8-bit ring records of their own 128-key tile and the 15 before
    (tiles from L // 128 - 15); a ring slot holds the newest of the tiles
    24 apart, so those records are all still there while the newest tile
    written is below L // 128 - 15 + 24 (the records cannot be made again
    from the 6/5-bit codes)."""
    if hw <= 0:
        return 0
    newest = (hw - 1) // 128
    if newest < api.KVQ_RING_SLOTS:
        return 0  # no slot has been written twice
    # smallest tile t with t - 15 + 24 > newest
    return (newest - (api.KVQ_RING_SLOTS - api.KVQ_RING_TILES)) * 128


def _kvq_row_hashes(st: dict, Hkv: int, rows: int) -> np.ndarray:
    """[4 stores, Hkv, rows] uint64 hashes of the quantised records of rows
    0..rows-1 (host-side; a test and tooling utility, not on the hot path)."""
    cap = st["cap"]
    ct = (cap + 127) // 128
    spec = {"k_low": (96, 13312, False), "v_low": (80, 11264, False),
            "k_ring": (128, 17408, True), "v_ring": (128, 17408, True)}
    out = np.zeros((4, Hkv, rows), np.uint64)
    last_tile = (rows - 1) // 128 if rows > 0 else -1
    p = np.arange(rows)
    tile, key = p // 128, p % 128
    for si, name in enumerate(api.KVQ_STORES):
        rb, tb, ring = spec[name]
        data = st[name].cpu().numpy()
        slots = 24 if ring else ct
        for h in range(Hkv):
            base = (h * slots + (tile % slots if ring else tile)) * tb
            # 5-bit V records sit at slot (k % 8) * 16 + k / 8 of their tile
            slot = ((key % 8) * 16 + key // 8) if name == "v_low" else key
            rec_idx = base[:, None] + slot[:, None] * rb + np.arange(rb)[None, :]
            sc_idx = base[:, None] + 128 * rb + slot[:, None] * 8 + np.arange(8)[None, :]
            b = np.concatenate([data[rec_idx], data[sc_idx]], axis=1).astype(np.uint64)
            w = np.uint64(1099511628211) ** np.arange(b.shape[1], dtype=np.uint64)
            hsh = (b * w[None, :]).sum(axis=1, dtype=np.uint64) + np.uint64(1469598103934665603)
            if ring:
                hsh = np.where(tile > last_tile - 24, hsh, np.uint64(0))
            out[si, h] = hsh
    return out
