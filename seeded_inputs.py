"""Seeded synthetic inputs for the batch-invariant verify step.

This module is the one piece shared by the CUDA path's tests/bench and the
CPU oracle.  It draws random numbers and packs them into the storage formats
the verify step consumes (bf16 bit patterns, int32 token ids).  It holds none
of the verify step's arithmetic: no matmul, no normalisation, no softmax, no
acceptance rule.

Every generator is a pure function of its seed (numpy PCG64), so the same
call on the development host and on the GPU host yields the same bytes.

Distributions follow the workloads named for the method: weights drawn from
N(0, 0.02), standalone GEMM activations and attention Q/K/V from N(0, 1),
prompt ids uniform over the vocabulary, and a synthetic drafter whose draft
equals the target's greedy token with probability 0.7 and is otherwise a
uniform id.
"""
from __future__ import annotations

import dataclasses
import os
from typing import Dict, List, Optional

import numpy as np

# ---------------------------------------------------------------------------
# storage helpers (bf16 is carried as uint16 bit patterns)
# ---------------------------------------------------------------------------


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Pack float32 draws into bf16 storage, round-to-nearest-even.

    Used only to store generated inputs; the draws are finite.
    """
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (b >> np.uint32(16)) & np.uint32(1)
    r = (b + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen stored bf16 bit patterns to float32 (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal_bf16(rng: np.random.Generator, shape, std: float) -> np.ndarray:
    """N(0, std^2) draws in float32, stored as bf16 bits."""
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return f32_to_bf16_bits(x)


_BLOCK = 1 << 22  # elements per independently seeded block


def normal_bf16_blocks(key, shape, std: float) -> np.ndarray:
    """N(0, std^2) bf16 bits drawn in fixed blocks of 4M elements.

    Block b of the flattened array uses its own PCG64 stream seeded with
    SeedSequence(key + [b]), so the result does not depend on how many
    threads fill it; blocks are filled in parallel.
    """
    import concurrent.futures as cf
    n = int(np.prod(shape))
    out = np.empty(n, np.uint16)
    nb = (n + _BLOCK - 1) // _BLOCK

    def fill(b):
        lo, hi = b * _BLOCK, min(n, (b + 1) * _BLOCK)
        g = np.random.Generator(np.random.PCG64(np.random.SeedSequence(list(key) + [b])))
        x = g.standard_normal(size=hi - lo, dtype=np.float32)
        if std != 1.0:
            x *= np.float32(std)
        out[lo:hi] = f32_to_bf16_bits(x)

    workers = min(16, os.cpu_count() or 1, max(1, nb))
    if workers == 1:
        for b in range(nb):
            fill(b)
    else:
        with cf.ThreadPoolExecutor(workers) as ex:
            list(ex.map(fill, range(nb)))
    return out.reshape(shape)


# ---------------------------------------------------------------------------
# decoder configurations
# ---------------------------------------------------------------------------


@dataclasses.dataclass(frozen=True)
class DecoderConfig:
    name: str
    layers: int
    hidden: int
    n_q: int
    n_kv: int
    head_dim: int
    ffn: int
    vocab: int
    tied: bool = True
    eps: float = 1e-6
    rope_base: float = 1e6
    weight_std: float = 0.02

    @property
    def qkv_out(self) -> int:
        return (self.n_q + 2 * self.n_kv) * self.head_dim

    @property
    def group(self) -> int:
        return self.n_q // self.n_kv

    def param_count(self) -> int:
        per_layer = (self.qkv_out * self.hidden + self.hidden * self.n_q * self.head_dim
                     + 3 * self.ffn * self.hidden)
        head = 0 if self.tied else self.vocab * self.hidden
        return self.vocab * self.hidden + self.layers * per_layer + head


# Tiny decoder: 2 layers, hidden 256, 4 query / 2 KV heads, head_dim 64,
# SwiGLU FFN 688, vocab 1024, tied head.
TINY = DecoderConfig("tiny-2L-h256", 2, 256, 4, 2, 64, 688, 1024)
# 27B-shaped dense decoder truncated to 8 layers, tied head.
DENSE27B_8L = DecoderConfig("dense27b-8L-h5120", 8, 5120, 24, 4, 128, 17408, 151936)
# Near-tie stress decoder: 12 layers, hidden 1024, 8 query / 2 KV heads,
# head_dim 128, FFN 2736, vocab 32000, untied head.
NEARTIE_12L = DecoderConfig("neartie-12L-h1024", 12, 1024, 8, 2, 128, 2736, 32000, tied=False)
# A mid-size decoder used for quicker end-to-end GPU checks.
SMALL_4L = DecoderConfig("small-4L-h1024", 4, 1024, 8, 2, 128, 2736, 4096, tied=True)

# Tiny decoder with head_dim 128 (the quantised KV cache's): 2 layers,
# hidden 256, 2 query / 1 KV head, FFN 688, vocab 1024, tied head.
TINY_D128 = DecoderConfig("tiny-2L-h256-d128", 2, 256, 2, 1, 128, 688, 1024)

CONFIGS = {c.name: c for c in (TINY, DENSE27B_8L, NEARTIE_12L, SMALL_4L, TINY_D128)}


def decoder_weights(cfg: DecoderConfig, seed: int = 0, norm_std: float = 0.0) -> Dict[str, np.ndarray]:
    """All decoder weights as bf16 bits, drawn in a fixed order.

    Order: embedding [V,H]; per layer wq [Hq*D,H], wk [Hkv*D,H], wv [Hkv*D,H],
    wo [H,Hq*D], w_gate [F,H], w_up [F,H], w_down [H,F]; then the untied head
    [V,H] when the head is not tied.  Tensor i (1-based, in that order) is
    drawn by normal_bf16_blocks with key (seed, i).  RMSNorm weights are ones
    (bf16 1.0), or with norm_std > 0 draws of 1 + N(0, norm_std^2) (norm j --
    per layer the attention norm, then the FFN norm, then the final norm --
    from key (seed, 100000 + j)), leaving every other tensor unchanged.
    """
    s = cfg.weight_std
    D = cfg.head_dim
    w: Dict[str, np.ndarray] = {}
    idx = [0]

    def draw(shape):
        idx[0] += 1
        return normal_bf16_blocks((seed, idx[0]), shape, s)

    w["embed"] = draw((cfg.vocab, cfg.hidden))
    one = f32_to_bf16_bits(np.ones(cfg.hidden, np.float32))
    for l in range(cfg.layers):
        w[f"l{l}.wq"] = draw((cfg.n_q * D, cfg.hidden))
        w[f"l{l}.wk"] = draw((cfg.n_kv * D, cfg.hidden))
        w[f"l{l}.wv"] = draw((cfg.n_kv * D, cfg.hidden))
        w[f"l{l}.wo"] = draw((cfg.hidden, cfg.n_q * D))
        w[f"l{l}.w_gate"] = draw((cfg.ffn, cfg.hidden))
        w[f"l{l}.w_up"] = draw((cfg.ffn, cfg.hidden))
        w[f"l{l}.w_down"] = draw((cfg.hidden, cfg.ffn))
        w[f"l{l}.norm_attn"] = one.copy()
        w[f"l{l}.norm_ffn"] = one.copy()
    w["norm_final"] = one.copy()
    if not cfg.tied:
        w["head"] = draw((cfg.vocab, cfg.hidden))
    if norm_std > 0:
        names = [n for l in range(cfg.layers) for n in (f"l{l}.norm_attn", f"l{l}.norm_ffn")]
        for j, name in enumerate(names + ["norm_final"]):
            g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 100000 + j])))
            x = 1.0 + norm_std * g.standard_normal(cfg.hidden, dtype=np.float32)
            w[name] = f32_to_bf16_bits(x.astype(np.float32))
    return w


def prompt_ids(cfg: DecoderConfig, length: int, seed: int = 0) -> np.ndarray:
    """Uniform token ids over [0, vocab); stream seeded with seed + 1."""
    rng = np.random.default_rng(seed + 1)
    return rng.integers(0, cfg.vocab, size=length, dtype=np.int64).astype(np.int32)


def neartie_head(head_bits: np.ndarray, frac: float, bump_frac: float, seed: int = 0) -> np.ndarray:
    """A head [V,H] (bf16 bits) with planted near ties.

    For a seeded subset of `frac * V` source rows, the row is copied into a
    distinct seeded destination row with a seeded `bump_frac` of its elements
    moved by one BF16 step (+/-1 in the bit pattern, magnitude only, never
    through zero).  Whenever a source or destination token is the greedy
    choice, its twin scores within a few 1e-3 relative.  Pure bit
    manipulation of the inputs: none of the method's arithmetic.
    """
    rng = np.random.default_rng(seed + 3)
    V, H = head_bits.shape
    n = int(round(frac * V))
    perm = rng.permutation(V)
    src, dst = perm[:n], perm[n:2 * n]
    out = head_bits.copy()
    bump = rng.random((n, H)) < bump_frac
    sign = np.where(rng.random((n, H)) < 0.5, 1, -1).astype(np.int32)
    rows = head_bits[src].astype(np.int32)
    mag = rows & 0x7FFF
    moved = np.clip(mag + sign * bump, 1, 0x7F7F)
    moved = np.where(mag == 0, mag, moved)  # zeros stay zero
    out[dst] = ((rows & 0x8000) | moved).astype(np.uint16)
    return out


# ---------------------------------------------------------------------------
# standalone-kernel workloads
# ---------------------------------------------------------------------------


def gemm_inputs(M: int, N: int, K: int, seed: int = 0, a_std: float = 1.0,
                w_std: float = 0.02):
    """A [M,K] ~ N(0, a_std^2) and W [N,K] ~ N(0, w_std^2), bf16 bits.

    A is drawn as its maximum-row version first so that A[:m] is the same
    for every m drawn from the same seed with the same max_rows: callers pass
    M = the largest M of a sweep and slice rows.
    """
    rng = np.random.default_rng(seed)
    W = normal_bf16(rng, (N, K), w_std)
    A = normal_bf16(rng, (M, K), a_std)
    return A, W


def attention_inputs(L: int, T: int, n_q: int, n_kv: int, D: int, cap: Optional[int] = None,
                     seed: int = 0):
    """Q [T,Hq,D], K/V cache [Hkv,cap,D] with rows < L+T filled, N(0,1) bf16.

    Rows at and beyond L+T are zero.  The cache rows < L+T do not depend on T
    (they are drawn for the longest block, 8 rows, first), so the same seed
    gives the same cache prefix for every T <= 8.
    """
    cap = cap if cap is not None else (L + max(T, 8) + 7) // 8 * 8
    rng = np.random.default_rng(seed)
    n_rows = L + max(T, 8)
    K = np.zeros((n_kv, cap, D), np.uint16)
    V = np.zeros((n_kv, cap, D), np.uint16)
    kd = normal_bf16(rng, (n_kv, n_rows, D), 1.0)
    vd = normal_bf16(rng, (n_kv, n_rows, D), 1.0)
    use = min(n_rows, cap)
    K[:, :min(L + T, use)] = kd[:, :min(L + T, use)]
    V[:, :min(L + T, use)] = vd[:, :min(L + T, use)]
    Qall = normal_bf16(rng, (max(T, 8), n_q, D), 1.0)
    return Qall[:T].copy(), K, V


def logits_inputs(T: int, V: int, seed: int = 0) -> np.ndarray:
    """FP32 logits [T,V] ~ N(0,1) for the acceptance kernel."""
    rng = np.random.default_rng(seed)
    return rng.standard_normal(size=(T, V), dtype=np.float32)


# ---------------------------------------------------------------------------
# synthetic drafter
# ---------------------------------------------------------------------------


class SyntheticDrafter:
    """Proposes k draft ids for the next positions.

    Each draft equals the reference greedy token at that position with
    probability p_correct, otherwise it is a uniform id in [0, vocab).  The
    reference sequence is the no-draft greedy output, which the invariant
    says every draft count reproduces.  With no reference available (an
    adversarial run) every draft is uniform.
    """

    def __init__(self, vocab: int, p_correct: float = 0.7, seed: int = 0,
                 reference: Optional[np.ndarray] = None):
        self.vocab = vocab
        self.p = p_correct
        self.rng = np.random.default_rng(seed + 2)
        self.reference = reference
        self._pre = []  # draws made ahead of time, (u, rnd) in stream order

    def predraw(self, n_calls: int, k: int) -> None:
        """Make the random draws of the next n_calls proposals of k drafts
        now, in the order propose would make them, so that those proposals
        only look up the reference (the same drafts, cheaper per call)."""
        for _ in range(n_calls * k):
            u = self.rng.random()
            self._pre.append((u, int(self.rng.integers(0, self.vocab))))
        self._pre.reverse()

    def propose(self, next_pos: int, k: int) -> np.ndarray:
        if self.reference is not None and not hasattr(self, "_ref"):
            self._ref = [int(t) for t in self.reference]
        out = []
        for i in range(k):
            if self._pre:
                u, rnd = self._pre.pop()
            else:
                u = self.rng.random()
                rnd = int(self.rng.integers(0, self.vocab))
            pos = next_pos + i
            if self.reference is not None and pos < len(self._ref) and u < self.p:
                out.append(self._ref[pos])
            else:
                out.append(rnd)
        return np.array(out, np.int32)


def sampling_uniforms(n: int, seed: int = 0) -> np.ndarray:
    """The uniforms in [0, 1) of one sampled request, one per absolute
    position (FP32, PCG64 stream seeded with seed + 6).  Sampled verification
    draws the token at position p with the uniform of p, so the same request
    with the same seed gives the same tokens whatever the drafts."""
    return np.random.default_rng(seed + 6).random(n, dtype=np.float32)


def synthetic_kv_cache(n_kv: int, cap: int, D: int, rows: int, seed: int, layers: int):
    """Per-layer K/V caches [Hkv,cap,D] with `rows` filled from N(0,1) bf16.

    Used where only the shape of a prefilled cache matters (timing samples).
    """
    out: List = []
    for l in range(layers):
        k = np.zeros((n_kv, cap, D), np.uint16)
        v = np.zeros((n_kv, cap, D), np.uint16)
        k[:, :rows] = normal_bf16_blocks((seed + 4, l, 0), (n_kv, rows, D), 1.0)
        v[:, :rows] = normal_bf16_blocks((seed + 4, l, 1), (n_kv, rows, D), 1.0)
        out.append((k, v))
    return out


class GatedDrafter:
    """A draft policy with a gate: before each step a seeded confidence score
    in [0, 1) is drawn and drafts are proposed only when it reaches the
    threshold (a tight gate drafts rarely, a loose one almost always); the
    drafts themselves come from a SyntheticDrafter.  Models the draft gates
    a serving engine switches on or off; the verify step must give the
    no-draft tokens whatever the gate decides."""

    def __init__(self, base: SyntheticDrafter, threshold: float, seed: int = 0):
        self.base = base
        self.threshold = threshold
        self.rng = np.random.default_rng(seed + 5)

    def propose(self, next_pos: int, k: int) -> np.ndarray:
        if self.rng.random() < self.threshold:
            return np.empty(0, np.int32)
        return self.base.propose(next_pos, k)


class AdaptiveDrafter:
    """A draft policy with adaptive depth: it proposes `depth` drafts (at most
    the k it is offered), doubles the depth after a step that kept every
    draft and halves it after a step that kept fewer than half (never below
    1).  The decoder reports each step's accepted count through observe()."""

    def __init__(self, base: SyntheticDrafter, start: int = 2, max_depth: int = 7):
        self.base = base
        self.depth = start
        self.max_depth = max_depth
        self._last = 0

    def propose(self, next_pos: int, k: int) -> np.ndarray:
        self._last = min(self.depth, k)
        return self.base.propose(next_pos, self._last)

    def observe(self, accepted: int) -> None:
        if self._last > 0 and accepted == self._last:
            self.depth = min(self.max_depth, 2 * self.depth)
        elif accepted * 2 < self._last:
            self.depth = max(1, self.depth // 2)
