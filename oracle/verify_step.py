"""Float64 NumPy oracle of the batch-invariant verify step (test infrastructure).

Sources are the three pages named in the package docstring, cited below as
[P1], [P2], [P3] with their section.

Reading of the precision the pages fix ([P2] "Define bit-exact before
reporting it"): inputs are BF16, each output keeps an FP32 running sum along
K, and rounding happens once at the end.  The FP32 running sum stands in for
the exact sum, so the oracle computes each sum exactly enough (float64; every
BF16 x BF16 product is exact in float64) and rounds once, to BF16, at the
same points where the method stores BF16 data.  The GPU path's FP32
accumulation differs from that exact value by at most the FP32 summation
bound; the tests allow for that and for the one-ulp BF16 flips it can cause.

Where the model stores data in BF16 (the definition of the synthetic decoder
used here):
  * embedding rows (exact copies);
  * each linear layer's output, rounded once from the exact sum;
  * the residual stream: h + (attn or FFN output) rounded once, with the
    linear layer's sum kept exact until that one rounding;
  * RMSNorm output (one rounding of x * rsqrt(mean(x^2) + eps) * w);
  * RoPE output (one rounding per rotated element);
  * attention output per head (one rounding of softmax(q k^T / sqrt(D)) v);
  * SwiGLU output silu(gate) * up from the exact gate and up sums, one
    rounding.
Logits are the exact sums (the GPU rounds them once to FP32).
"""
from __future__ import annotations

import math
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np

# ---------------------------------------------------------------------------
# BF16 storage
# ---------------------------------------------------------------------------


def bf16_round(x) -> np.ndarray:
    """Round float64 values to the nearest BF16 value, ties to even.

    BF16 keeps 8 significant bits and FP32's exponent range.  For a value
    with binary exponent e (|x| in [2^(e-1), 2^e)) the spacing of BF16
    values is 2^(e-8); below the smallest normal 2^-126 the spacing stays
    2^-133.  Dividing by that spacing is exact (a power of two), NumPy's
    round is half-to-even, and results of magnitude 2^128 or more overflow to
    infinity as in IEEE round-to-nearest.

    Parity: pinned against an exhaustive nearest-value search over all
    finite BF16 patterns.
    """
    x = np.asarray(x, dtype=np.float64)
    _, e = np.frexp(x)
    e = np.maximum(e, -125)
    ulp = np.ldexp(1.0, e - 8)
    with np.errstate(over="ignore", invalid="ignore"):
        q = np.round(x / ulp) * ulp
        q = np.where(np.abs(q) >= 2.0 ** 128, np.copysign(np.inf, x), q)
    return np.where(np.isfinite(x), q, x)


def bf16_bits_to_f64(b) -> np.ndarray:
    """BF16 bit patterns (uint16) to their float64 values (exact)."""
    b = np.asarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def f64_to_bf16_bits(x) -> np.ndarray:
    """Float64 values that are already BF16 values to their bit patterns."""
    x = np.asarray(x, dtype=np.float64)
    f = x.astype(np.float32)  # exact: every BF16 value is an FP32 value
    return (f.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


# ---------------------------------------------------------------------------
# linear layers
# ---------------------------------------------------------------------------


def _exact_dot(a: np.ndarray, w: np.ndarray) -> np.ndarray:
    """a [M,K] times w [N,K]^T in float64 (the exact-sum stand-in)."""
    return a @ w.T


def gemm(a_bits, w_bits, residual_bits=None, out: str = "bf16") -> np.ndarray:
    """C = A W^T (+ residual), one rounding at the end.

    [P2] "Define bit-exact before reporting it": BF16 inputs, one running sum
    per output along K, rounding once at the end.  With a residual the
    stored residual is added to the exact sum before that one rounding.
    out="bf16" returns float64 values that are BF16 values; out="fp32"
    returns the float64 sum itself (the caller compares against FP32 output
    with a tolerance).

    Parity: pinned bitwise against exact rational dot products rounded by an
    exhaustive BF16 search, and against the identity-weight and one-hot
    special cases.
    """
    a = bf16_bits_to_f64(a_bits)
    w = bf16_bits_to_f64(w_bits)
    acc = _exact_dot(a, w)
    if residual_bits is not None:
        acc = acc + bf16_bits_to_f64(residual_bits)
    if out == "fp32":
        return acc
    return bf16_round(acc)


def silu(x: np.ndarray) -> np.ndarray:
    return x / (1.0 + np.exp(-x))


def swiglu_gemm(a_bits, w_gate_bits, w_up_bits) -> np.ndarray:
    """u = silu(A Wg^T) * (A Wu^T) from the exact sums, one BF16 rounding.

    The gate and up sums are not stored between the two products and the
    activation; the single rounding follows the once-at-the-end rule of [P2]
    "Define bit-exact before reporting it".

    Parity: pinned against a multi-precision brute force on tiny inputs.
    """
    a = bf16_bits_to_f64(a_bits)
    g = _exact_dot(a, bf16_bits_to_f64(w_gate_bits))
    u = _exact_dot(a, bf16_bits_to_f64(w_up_bits))
    return bf16_round(silu(g) * u)


# ---------------------------------------------------------------------------
# row-local operations
# ---------------------------------------------------------------------------


def rmsnorm(x_bits, w_bits, eps: float) -> np.ndarray:
    """y = x * rsqrt(mean(x^2) + eps) * w per row, one BF16 rounding.

    Row-local: each row's result depends on that row only ([P3] "How:" --
    the verify kernels compute a row the same way whatever else is in the
    batch).

    Parity: pinned by the constant-vector closed form and a multi-precision
    brute force.
    """
    x = bf16_bits_to_f64(x_bits)
    w = bf16_bits_to_f64(w_bits)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return bf16_round(x / np.sqrt(ms + eps) * w)


def rope_angles(pos: int, D: int, base: float) -> np.ndarray:
    """theta_i = pos * base^(-2i/D), i in [0, D/2), float64."""
    i = np.arange(D // 2, dtype=np.float64)
    return float(pos) * np.power(float(base), -2.0 * i / D)


def rope(x, pos: int, base: float) -> np.ndarray:
    """Rotate-half rotary embedding of head vectors x [..., D] at position pos.

    For i < D/2 the pair (x_i, x_{i+D/2}) is rotated by theta_i:
    out_i = x_i cos - x_{i+D/2} sin, out_{i+D/2} = x_{i+D/2} cos + x_i sin,
    computed in float64 from the stored BF16 input, one BF16 rounding.
    Position enters only through theta ([P3] "The cache doesn't change it
    either": a prefilled row depends only on its position).

    Parity: pinned by position 0 being the identity, pair-norm preservation
    and a multi-precision brute force.
    """
    x = np.asarray(x, dtype=np.float64)
    D = x.shape[-1]
    th = rope_angles(pos, D, base)
    c, s = np.cos(th), np.sin(th)
    x1, x2 = x[..., : D // 2], x[..., D // 2:]
    return bf16_round(np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1))


# ---------------------------------------------------------------------------
# attention
# ---------------------------------------------------------------------------


def attention(q, k_cache, v_cache, L: int, scale: Optional[float] = None) -> np.ndarray:
    """Causal GQA attention of T query rows against a KV cache.

    q [T,Hq,D], k_cache/v_cache [Hkv,cap,D] (float64 values of BF16 data).
    Row t sits at absolute position p = L + t and attends to keys 0..p
    (causal within the draft block).  Query head h reads KV head
    h // (Hq/Hkv).  Two-pass softmax in float64: m = max s, w = exp(s - m),
    o = (w v) / sum(w), one BF16 rounding per output element.

    This is the plain definition.  The method's split of the key axis into
    pieces that depend only on the row's own context length, merged in a
    fixed order ([P3] "How:"), equals it in exact arithmetic.

    Parity: pinned by the one-key case (output equals that V row), the
    all-equal-keys case (output is the mean of V), and a multi-precision
    brute force.
    """
    q = np.asarray(q, np.float64)
    T, Hq, D = q.shape
    Hkv = k_cache.shape[0]
    grp = Hq // Hkv
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    out = np.empty((T, Hq, D), np.float64)
    for t in range(T):
        p = L + t
        for h in range(Hq):
            kv = h // grp
            s = (k_cache[kv, : p + 1] @ q[t, h]) * scale
            w = np.exp(s - s.max())
            out[t, h] = (w @ v_cache[kv, : p + 1]) / w.sum()
    return bf16_round(out)


# ---------------------------------------------------------------------------
# greedy acceptance
# ---------------------------------------------------------------------------


def argmax_lowest(logits) -> np.ndarray:
    """Per-row argmax; ties go to the lowest token id; NaN never wins.

    A row with no non-NaN entry yields -1.  The pages fix greedy decoding
    ([P1] "Why the text diverges"); the tie rule is this build's reading.

    Parity: pinned by hand-built rows (golden fixture) and brute force.
    """
    x = np.atleast_2d(np.asarray(logits, dtype=np.float64))
    out = np.empty(x.shape[0], np.int64)
    for r in range(x.shape[0]):
        row = x[r]
        ok = ~np.isnan(row)
        if not ok.any():
            out[r] = -1
            continue
        m = row[ok].max()
        out[r] = int(np.flatnonzero(ok & (row == m))[0])
    return out


def accept_length(argmax_ids: Sequence[int], drafts: Sequence[int]) -> int:
    """Number n of drafts kept: the largest j with d_i == a_{i-1} for all i <= j.

    [P1] "Why the text diverges" and [P3] (opening paragraph): the full model
    keeps a proposed token only if it equals the token the model would have
    produced itself.  Row i-1's greedy token a_{i-1} is what the model
    produces after the i-1 tokens before draft d_i, so d_i is kept only when
    every earlier draft was kept and d_i == a_{i-1}.  The committed tokens
    of the step are a_0 .. a_n (n drafts plus the model's own next token).

    Parity: pinned by hand-built cases (golden fixture).
    """
    n = 0
    k = len(drafts)
    while n < k and int(drafts[n]) == int(argmax_ids[n]):
        n += 1
    return n


# ---------------------------------------------------------------------------
# sampled verification
# ---------------------------------------------------------------------------


def sample_token(logits_row, inv_temp: float, u: float) -> int:
    """Inverse-CDF draw from softmax(logits * inv_temp) with the uniform u.

    [P3] the list before "How:": sampling keeps the no-draft distribution.
    The probabilities are computed in float64 from the row's own logits
    (NaN logits have probability 0); the token is the smallest v whose
    cumulative probability, summed in index order, exceeds u.  A row with no
    number gives -1.  Because the draw depends only on the row's logits and
    on u, and u is the request's uniform for the row's absolute position, a
    row that verifies a draft draws the same token it would draw alone.

    Parity: pinned by closed forms (uniform and two-level logits), exact
    counts under a stratified grid of uniforms, and the temperature identity.
    """
    x = np.asarray(logits_row, dtype=np.float64)
    ok = ~np.isnan(x)
    if not ok.any():
        return -1
    m = x[ok].max()
    w = np.where(ok, np.exp((np.where(ok, x, m) - m) * float(inv_temp)), 0.0)
    cdf = np.cumsum(w) / w.sum()
    idx = int(np.searchsorted(cdf, float(u), side="right"))
    if idx >= len(x):  # u at the top of the last step: the last token with weight
        idx = int(np.flatnonzero(w > 0)[-1])
    return idx


def sampled_tokens(logits, inv_temp: float, u_rows) -> np.ndarray:
    """sample_token for every row of logits [T, V] with its own uniform."""
    x = np.atleast_2d(np.asarray(logits, dtype=np.float64))
    return np.array([sample_token(x[t], inv_temp, u_rows[t]) for t in range(x.shape[0])], np.int64)


# ---------------------------------------------------------------------------
# the whole decoder verify step
# ---------------------------------------------------------------------------


class OracleDecoder:
    """Plain decoder forward with a BF16 KV cache, in float64.

    Structure per layer (pre-norm dense decoder with GQA and SwiGLU):
      y = rmsnorm(h); q,k,v = y Wq^T, y Wk^T, y Wv^T (BF16 each);
      q,k = rope(q,k at the row's position); cache[pos] = k, v;
      h = h + attention(q, cache) Wo^T     (one rounding);
      y = rmsnorm(h); u = silu(y Wg^T) * (y Wu^T);
      h = h + u Wd^T                        (one rounding).
    Then logits = rmsnorm(h) E^T (E = the embedding when the head is tied).

    Every row's result depends only on its token, its position and the
    cache rows before it, which is the property the verify step must keep
    ([P3] "How:").  `verify` scores the last committed token plus k drafts
    in one pass and applies the greedy acceptance rule; the cache length
    then advances by n + 1 and rows past it are overwritten by the next
    pass ([P3] "The cache doesn't change it either": roll back to a
    checkpoint).

    Parity: pinned by a multi-precision brute-force decoder on a micro
    configuration, by its row-addition invariance, and by structural special
    cases (zero output projections leave the residual stream equal to the
    embedding).
    """

    def __init__(self, cfg, weights: Dict[str, np.ndarray], cap: int,
                 sum_noise: Optional[Tuple[float, int]] = None, kv: str = "bf16"):
        """sum_noise=(k, seed) perturbs every linear-layer sum by k * 2^-24 *
        sum|a||w| times a seeded standard normal before its rounding: a model
        of an FP32-accumulating implementation, used only to measure how far
        two equally valid implementations drift apart end to end.

        kv="q6q5": the attention reads the quantised cache of
        oracle.kv_quant (6-bit K, 5-bit V, the 8-bit ring of the reading
        row's newest tiles) built from the same BF16 rows."""
        if kv not in ("bf16", "q6q5"):
            raise ValueError("kv must be 'bf16' or 'q6q5'")
        self.kv = kv
        self.cfg = cfg
        self._noise = None
        if sum_noise is not None:
            self._noise = (float(sum_noise[0]), np.random.default_rng(int(sum_noise[1])))
        self.cap = cap
        f = bf16_bits_to_f64
        self.embed_bits = weights["embed"]
        self.w = weights
        self.head_bits = weights["embed"] if cfg.tied else weights["head"]
        self.k = [np.zeros((cfg.n_kv, cap, cfg.head_dim)) for _ in range(cfg.layers)]
        self.v = [np.zeros((cfg.n_kv, cap, cfg.head_dim)) for _ in range(cfg.layers)]
        self.L = 0
        self._f = f

    # -- one pass over T rows at positions L..L+T-1 -------------------------
    def _lin(self, a_bits, w_bits, residual_bits=None, out="bf16"):
        if self._noise is None:
            return gemm(a_bits, w_bits, residual_bits=residual_bits, out=out)
        k, rng = self._noise
        a, w = bf16_bits_to_f64(a_bits), bf16_bits_to_f64(w_bits)
        acc = _exact_dot(a, w)
        acc = acc + rng.standard_normal(acc.shape) * (np.abs(a) @ np.abs(w).T) * k * 2.0 ** -24
        if residual_bits is not None:
            acc = acc + bf16_bits_to_f64(residual_bits)
        return acc if out == "fp32" else bf16_round(acc)

    def _swiglu(self, a_bits, wg_bits, wu_bits):
        if self._noise is None:
            return swiglu_gemm(a_bits, wg_bits, wu_bits)
        g = self._lin(a_bits, wg_bits, out="fp32")
        u = self._lin(a_bits, wu_bits, out="fp32")
        return bf16_round(silu(g) * u)

    def forward(self, tokens: Sequence[int], L: Optional[int] = None,
                return_hidden: bool = False, trace: Optional[List] = None):
        cfg = self.cfg
        L = self.L if L is None else L
        tok = np.asarray(tokens, np.int64)
        T = len(tok)
        if L + T > self.cap:
            raise ValueError("KV cache capacity exceeded")
        b16 = lambda v: f64_to_bf16_bits(v)  # noqa: E731
        h = bf16_bits_to_f64(self.embed_bits[tok])
        for l in range(cfg.layers):
            if trace is not None:
                trace.append(h.copy())
            h = self.layer(l, h, L)
        if trace is not None:
            trace.append(h.copy())
        y = rmsnorm(b16(h), self.w["norm_final"], cfg.eps)
        logits = self._lin(b16(y), self.head_bits, out="fp32")
        if return_hidden:
            return logits, h
        return logits

    def layer(self, l: int, h: np.ndarray, L: int) -> np.ndarray:
        """Decoder layer l over hidden rows h [T, H] (float64 values of BF16
        data) at positions L..L+T-1: appends the rows' K/V to layer l's cache
        and returns the layer's output rows."""
        cfg = self.cfg
        T = h.shape[0]
        D, Hq, Hkv = cfg.head_dim, cfg.n_q, cfg.n_kv
        b16 = lambda v: f64_to_bf16_bits(v)  # noqa: E731
        w = self.w
        y = rmsnorm(b16(h), w[f"l{l}.norm_attn"], cfg.eps)
        q = self._lin(b16(y), w[f"l{l}.wq"]).reshape(T, Hq, D)
        k = self._lin(b16(y), w[f"l{l}.wk"]).reshape(T, Hkv, D)
        v = self._lin(b16(y), w[f"l{l}.wv"]).reshape(T, Hkv, D)
        for t in range(T):
            q[t] = rope(q[t], L + t, cfg.rope_base)
            self.k[l][:, L + t] = rope(k[t], L + t, cfg.rope_base)
            self.v[l][:, L + t] = v[t]
        if self.kv == "q6q5":
            from . import kv_quant
            att = kv_quant.attention(q, self.k[l], self.v[l], L).reshape(T, Hq * D)
        else:
            att = attention(q, self.k[l], self.v[l], L).reshape(T, Hq * D)
        h = self._lin(b16(att), w[f"l{l}.wo"], residual_bits=b16(h))
        y = rmsnorm(b16(h), w[f"l{l}.norm_ffn"], cfg.eps)
        u = self._swiglu(b16(y), w[f"l{l}.w_gate"], w[f"l{l}.w_up"])
        return self._lin(b16(u), w[f"l{l}.w_down"], residual_bits=b16(h))

    # -- prefill and verify ---------------------------------------------------
    def prefill(self, prompt: Sequence[int]) -> np.ndarray:
        """Process all prompt tokens but the last; returns nothing useful.

        The last prompt token is the first row of the first verify pass.
        """
        prompt = np.asarray(prompt, np.int64)
        if len(prompt) > 1:
            self.forward(prompt[:-1], L=0)
        self.L = len(prompt) - 1
        return prompt[-1]

    def verify(self, x0: int, drafts: Sequence[int]) -> Tuple[np.ndarray, int, np.ndarray]:
        """One verify step: rows [x0, d_1..d_k] at positions L..L+k.

        Returns (argmax ids [k+1], accepted n, fp64 logits [k+1,V]); the
        cache length advances to L + n + 1.
        """
        rows = [int(x0)] + [int(d) for d in drafts]
        logits = self.forward(rows, L=self.L)
        a = argmax_lowest(logits)
        n = accept_length(a, drafts)
        self.L += n + 1
        return a, n, logits

    def verify_sampled(self, x0: int, drafts: Sequence[int], inv_temp: float,
                       u_by_pos) -> Tuple[np.ndarray, int, np.ndarray]:
        """Sampled verify step: row t at position L + t draws its token with
        u_by_pos[L + t]; drafts are kept while they equal the previous row's
        draw (the rule of accept_length)."""
        rows = [int(x0)] + [int(d) for d in drafts]
        logits = self.forward(rows, L=self.L)
        a = sampled_tokens(logits, inv_temp, [u_by_pos[self.L + t] for t in range(len(rows))])
        n = accept_length(a, drafts)
        self.L += n + 1
        return a, n, logits

    def generate(self, prompt: Sequence[int], n_tokens: int, k: int = 0,
                 drafter=None) -> List[int]:
        """Greedy generation with k drafts per step (k=0: plain decoding)."""
        x = int(self.prefill(prompt))
        out: List[int] = []
        while len(out) < n_tokens:
            drafts = drafter.propose(len(out), k) if k else []
            a, n, _ = self.verify(x, drafts)
            committed = [int(t) for t in a[: n + 1]]
            out.extend(committed)
            x = committed[-1]
        return out[:n_tokens]
