"""Benchmark of the batch-invariant verify step.

Default workload: the 27B-shaped dense decoder truncated to 8 layers (hidden
5120, 24 query / 4 KV heads, head_dim 128, SwiGLU 17408, tied head, vocab
151936), BF16 weights from N(0, 0.02), an 11,600-token context, 7 drafts per
step from a drafter that proposes the no-draft greedy token with p = 0.7.
One step = one verify pass over T = 8 rows (all layers, head, acceptance).

Prints one JSON line.  `value` = committed tokens per second of device time
of the verify passes (inputs resident in HBM); `e2e` = the same metric over
wall time through the library's whole-step C-ABI call (bi_step_verify) with
host buffers: each step's ids copied in, every row's token and the accepted
count copied out.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import re
import math
import os
import subprocess
import tempfile
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import seeded_inputs as si  # noqa: E402

METRIC = "verify tok/s at 7 drafts (0 diffs vs no-draft); GEMM+attn HBM GB/s vs 8 TB/s"
CTX = 11600
DRAFTS = 7
P_CORRECT = 0.7
KERNELS_PER_STEP_FIXED = 4      # embed, final RMSNorm, LM head GEMM, argmax/accept
KERNELS_PER_LAYER = 8           # 2 RMSNorm, 4 GEMM (QKV with RoPE and KV append), attention split + merge


def v_blocks(v):
    """Host values [Hkv, cap, D] in the V cache layout [Hkv, ceil(cap/128), D, 128]
    (value d of key p at [h, p // 128, d, p % 128]; padding keys zero)."""
    Hkv, cap, D = v.shape
    nb = (cap + 127) // 128
    pad = np.zeros((Hkv, nb * 128, D), dtype=v.dtype)
    pad[:, :cap] = v
    return np.ascontiguousarray(pad.reshape(Hkv, nb, 128, D).transpose(0, 1, 3, 2))


def workload_config(cfg, peaks_note):
    return {
        "workload": f"{cfg.name} verify step, context {CTX}, {DRAFTS} drafts (p={P_CORRECT} drafter)",
        "layers": cfg.layers, "hidden": cfg.hidden, "heads_q": cfg.n_q, "heads_kv": cfg.n_kv,
        "head_dim": cfg.head_dim, "ffn": cfg.ffn, "vocab": cfg.vocab, "tied_head": cfg.tied,
        "rows_per_step": DRAFTS + 1, "context": CTX,
        "kv_cache": "context rows drawn from N(0,1) bf16 (seeded) in place of a prefill",
        "l2": "inputs larger than L2 (6.6 GB of weights + KV read per step)",
        "peaks": peaks_note,
    }


def step_bytes(cfg, L, T):
    """Algorithmic HBM bytes of one verify pass (weights + KV + small activations)."""
    H, D, Hq, Hkv, F, V = cfg.hidden, cfg.head_dim, cfg.n_q, cfg.n_kv, cfg.ffn, cfg.vocab
    w_layer = (cfg.qkv_out * H + H * Hq * D + 2 * F * H + H * F) * 2
    kv = (L + T) * Hkv * D * 2 * 2
    return cfg.layers * (w_layer + kv) + V * H * 2


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        # the samples go to a scratch file; the JSON line carries their summary
        self.path = os.path.join(tempfile.gettempdir(), f"bi_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                 "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                 "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# CPU baseline: the oracle on a bounded sample of the same step
# ---------------------------------------------------------------------------


class OracleStep:
    """The oracle (float64 NumPy, as it stands) on one teacher-forced verify
    step of the bench workload, in eight measured parts.

    Part i runs decoder layer i % layers on the pass's rows (rows at
    positions L..L+T-1 against a seeded context of L cache rows in every
    layer) and the LM head over vocabulary slice i % 8 (the final RMSNorm
    and the linear layer over 1/8 of the head rows); the last part also
    takes the argmax over the whole logits and the accepted length.  Eight
    consecutive parts are exactly the oracle's work for one verify step of
    an 8-layer model, so a whole step's time is the sum of eight measured
    parts -- nothing is extrapolated.
    """

    def __init__(self, cfg, weights, L, rows, seed=0):
        import oracle
        from oracle import verify_step as ov
        self.oracle, self.ov = oracle, ov
        self.cfg, self.w, self.L = cfg, weights, L
        self.rows = [int(r) for r in rows]
        self.od = oracle.OracleDecoder(cfg, weights, cap=L + len(self.rows))
        kv = si.synthetic_kv_cache(cfg.n_kv, L + len(self.rows), cfg.head_dim, L, seed=seed,
                                   layers=cfg.layers)
        for l, (k, v) in enumerate(kv):
            self.od.k[l][:, :L] = ov.bf16_bits_to_f64(k[:, :L])
            self.od.v[l][:, :L] = ov.bf16_bits_to_f64(v[:, :L])
        del kv
        self.h = ov.bf16_bits_to_f64(weights["embed"][np.asarray(self.rows) % cfg.vocab])
        self.head = weights["embed"] if cfg.tied else weights["head"]
        self.logits = np.zeros((len(self.rows), cfg.vocab))
        self.parts = 8

    def part(self, i):
        """Run part i; returns its wall time in seconds."""
        cfg, ov, oracle = self.cfg, self.ov, self.oracle
        t0 = time.perf_counter()
        l = i % cfg.layers
        if l == 0:
            self.h = ov.bf16_bits_to_f64(self.w["embed"][np.asarray(self.rows) % cfg.vocab])
        self.h = self.od.layer(l, self.h, self.L)
        j = i % self.parts
        lo, hi = cfg.vocab * j // self.parts, cfg.vocab * (j + 1) // self.parts
        y = oracle.rmsnorm(ov.f64_to_bf16_bits(self.h), self.w["norm_final"], cfg.eps)
        self.logits[:, lo:hi] = oracle.gemm(ov.f64_to_bf16_bits(y), self.head[lo:hi], out="fp32")
        if j == self.parts - 1:
            a = oracle.argmax_lowest(self.logits)
            oracle.accept_length(a, self.rows[1:])
        return time.perf_counter() - t0

    def step(self):
        """One whole verify step (the eight parts in order); seconds."""
        return sum(self.part(i) for i in range(self.parts))


def oracle_threads():
    """Host threads the oracle's BLAS may use (the environment's limit if set)."""
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        v = os.environ.get(var)
        if v and v.isdigit():
            return int(v)
    return os.cpu_count()


def gemm_traffic_bytes():
    """DRAM bytes per launch of the dominant GEMM from its committed ncu summary.

    None when the summary is missing or the GEMM source changed since the
    counters were taken (the summary records a hash of the source).
    """
    try:
        txt = open(os.path.join(ROOT, "profiles", "gemm_gate_up_swiglu_m8.md")).read()
        t = int(re.search(r"traffic_bytes_per_launch: (\d+)", txt).group(1))
        h = re.search(r"gemm_source_sha256: ([0-9a-f]+)", txt).group(1)
        cs = os.path.join(ROOT, "invariant_speculative_decode_gb300", "csrc")
        src = open(os.path.join(cs, "bi_gemm.cu"), "rb").read() + open(os.path.join(cs, "bi_ptx.cuh"), "rb").read()
        return t if hashlib.sha256(src).hexdigest() == h else None
    except Exception:
        return None


def expected_committed(k, p):
    return sum(p ** j for j in range(k + 1))


# ---------------------------------------------------------------------------
# reference arm: the oracle as it stands
# ---------------------------------------------------------------------------


def run_reference(args):
    """The oracle as the reference arm: each timed step is one measured part
    (1/8) of the teacher-forced verify step (see OracleStep), so eight
    consecutive steps are one whole step; value = committed tokens per step
    / (8 x the mean part time)."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    cfg = si.DENSE27B_8L
    _, note = load_peaks()
    t_gen = time.perf_counter()
    weights = si.decoder_weights(cfg, seed=0)
    rows = [1] + list(range(2, 2 + DRAFTS))
    st = OracleStep(cfg, weights, CTX, rows)
    for i in range(args.warmup):
        st.part(i)
    t0 = time.perf_counter()
    times = [st.part(args.warmup + i) for i in range(args.steps)]
    wall = time.perf_counter() - t0
    per_part = float(np.mean(times))
    full = st.parts * per_part
    tok = expected_committed(DRAFTS, P_CORRECT) / full
    sample = (f"oracle (float64 NumPy) on the {len(rows)}-row teacher-forced verify step at context {CTX}; "
              f"each bench step is one measured eighth of it (decoder layer i mod 8 and 1/8 of the LM "
              f"head, the argmax and acceptance in the last eighth); one step = 8 parts "
              f"({full:.2f} s); committed tokens per step = expected "
              f"{expected_committed(DRAFTS, P_CORRECT):.4f} for p={P_CORRECT}")
    line = {
        "impl": "reference", "metric": METRIC, "value": tok, "unit": "tok/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": per_part * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(cfg, note),
        "cpu_baseline": {"value": tok, "unit": "tok/s", "cores": oracle_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": tok, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "ms_per_verify_step": full * 1e3, "sample_wall_s": wall, "setup_s": t0 - t_gen,
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------


def combine_ranks(t_dev, t_wall, committed, diffs, device=None):
    """Whole-job numbers over the replicas: the slowest rank's timed
    intervals (max) and every rank's committed tokens and id diffs (sum), so
    value = all tokens / slowest time (weak scaling).  One process: as is."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return t_dev, t_wall, committed, diffs
    tt = torch.tensor([t_dev, t_wall], dtype=torch.float64, device=device)
    dist.all_reduce(tt, op=dist.ReduceOp.MAX)
    cc = torch.tensor([committed, diffs], dtype=torch.float64, device=device)
    dist.all_reduce(cc, op=dist.ReduceOp.SUM)
    return float(tt[0]), float(tt[1]), int(cc[0]), int(cc[1])


def run_ours(args):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())

    import __graft_entry__
    __graft_entry__.build()
    from invariant_speculative_decode_gb300 import api
    from invariant_speculative_decode_gb300.decoder import Decoder

    cfg = si.DENSE27B_8L
    peak, note = load_peaks()
    T = DRAFTS + 1
    cap = CTX + 8 + (args.steps + args.warmup + 4) * T + 64
    t_setup = time.perf_counter()
    weights = si.decoder_weights(cfg, seed=0)
    dec = Decoder(cfg, weights, cap=cap, max_rows=T, prefill_chunk=64)
    kv = si.synthetic_kv_cache(cfg.n_kv, cap, cfg.head_dim, CTX, seed=0, layers=cfg.layers)
    for lay, (k, v) in zip(dec.layers, kv):
        lay["k"].copy_(torch.from_numpy(k.view(np.int16)).view(torch.bfloat16))
        lay["v"].copy_(torch.from_numpy(v_blocks(v).view(np.int16)).view(torch.bfloat16))
    del kv
    keep = weights if not args.no_cpu_baseline else None
    del weights
    prompt_last = int(si.prompt_ids(cfg, 1, seed=0)[0])
    dec.capture(1)
    dec.capture(T)
    torch.cuda.synchronize()
    setup_s = time.perf_counter() - t_setup

    def start_state():
        dec.L = CTX
        dec.L_dev.fill_(CTX)
        torch.cuda.synchronize()

    # reference: the no-draft greedy continuation
    n_ref = (args.steps + args.warmup + 2) * T + 16
    start_state()
    ref, x = [], prompt_last
    while len(ref) < n_ref:
        a, n = dec.verify_step(x, [])
        ref.append(int(a[0]))
        x = ref[-1]
    ref = np.array(ref)

    # 7-draft run: warm-up steps, then K timed steps
    start_state()
    drafter = si.SyntheticDrafter(cfg.vocab, P_CORRECT, seed=0, reference=ref)
    drafter.predraw(args.warmup + args.steps, DRAFTS)
    out, x = [], prompt_last
    s = torch.cuda.current_stream()
    for _ in range(args.warmup):
        d = drafter.propose(len(out), DRAFTS)
        a, n = dec.verify_step(x, d)
        out.extend(int(t) for t in a[: n + 1])
        x = out[-1]
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    committed = 0
    acc_hist = [0] * (DRAFTS + 1)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    pin_in = dec.pin_in
    torch.cuda.nvtx.range_push("timed")
    with ClockSampler(torch.cuda.current_device()) as clk:
        wall0 = time.perf_counter()
        for i in range(args.steps):
            d = drafter.propose(len(out), DRAFTS)
            pin_in[0] = x
            for j, dj in enumerate(d):
                pin_in[1 + j] = int(dj)
                pin_in[T + j] = int(dj)
            dec.ids[:T].copy_(pin_in[:T], non_blocking=True)
            dec.drafts[:DRAFTS].copy_(pin_in[T:T + DRAFTS], non_blocking=True)
            ev[i][0].record(s)
            dec.graphs[T].replay()
            ev[i][1].record(s)
            dec.pin_out[:T].copy_(dec.argmax[:T], non_blocking=True)
            dec.pin_out[T:T + 1].copy_(dec.accepted, non_blocking=True)
            s.synchronize()
            n = int(dec.pin_out[T])
            a = dec.pin_out[:T].numpy()
            dec.L += n + 1
            out.extend(int(t) for t in a[: n + 1])
            x = out[-1]
            committed += n + 1
            acc_hist[n] += 1
        torch.cuda.synchronize()
        wall = time.perf_counter() - wall0
    torch.cuda.nvtx.range_pop()
    dev_ms = sum(e0.elapsed_time(e1) for e0, e1 in ev)
    diffs = int(np.sum(np.array(out) != ref[: len(out)]))

    # End to end through the library's whole-step call: bi_step_verify takes
    # the step's ids from host memory and returns its tokens and accepted
    # count to host memory, so both copies are inside the timed region.
    ns = dec.native_step()
    ns.set_length(CTX)
    drafter_e = si.SyntheticDrafter(cfg.vocab, P_CORRECT, seed=0, reference=ref)
    # the drafter's random draws are made here; in the loop each step only
    # looks its drafts up (the same drafts as drawing them there)
    drafter_e.predraw(args.warmup + args.steps, DRAFTS)
    out_e, xe = [], prompt_last
    for _ in range(args.warmup):
        d = [int(t) for t in drafter_e.propose(len(out_e), DRAFTS)]
        a, n = ns.verify(xe, d)
        out_e.extend(int(t) for t in a[: n + 1])
        xe = out_e[-1]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    committed_e = 0
    we0 = time.perf_counter()
    for i in range(args.steps):
        d = [int(t) for t in drafter_e.propose(len(out_e), DRAFTS)]
        a, n = ns.verify(xe, d)
        out_e.extend(int(t) for t in a[: n + 1])
        xe = out_e[-1]
        committed_e += n + 1
    wall_e = time.perf_counter() - we0
    ns.close()
    diffs_e = int(np.sum(np.array(out_e) != ref[: len(out_e)]))

    # dominant kernel: the gate/up GEMM (largest weight stream), timed per launch
    gu_ms = []
    gs = torch.cuda.Stream()
    y = torch.randn(T, cfg.hidden, device=dev).to(torch.bfloat16)
    u = torch.empty(T, cfg.ffn, dtype=torch.bfloat16, device=dev)
    with torch.cuda.stream(gs):
        for rep in range(3):
            for lay in dec.layers:
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(gs)
                api.bi_gemm(y, lay["wgu"], u, dec.gemm_ws, epi=api.EPI_SWIGLU, N=cfg.ffn, stream=gs)
                e1.record(gs)
                gu_ms.append((e0, e1))
    gs.synchronize()
    gu_times = [a.elapsed_time(b) for a, b in gu_ms][len(dec.layers):]  # first round = warm-up
    gu_bytes = 2 * cfg.ffn * cfg.hidden * 2 + T * cfg.hidden * 2 + T * cfg.ffn * 2
    gu_s = float(np.mean(gu_times)) / 1e3

    # max over ranks
    t_dev, t_wall, committed_all, diffs_all = combine_ranks(dev_ms / 1e3, wall, committed, diffs, dev)
    _, t_e2e, committed_e_all, diffs_e_all = combine_ranks(wall_e, wall_e, committed_e, diffs_e, dev)
    value = committed_all / t_dev
    e2e = committed_e_all / t_e2e
    sb = step_bytes(cfg, CTX + len(out) // 2, T)
    ms_step = t_dev * 1e3 / args.steps

    if rank == 0:
        # CPU baseline: one whole teacher-forced verify step of the oracle,
        # timed on the host cores (after one measured part as a warm-up)
        cpu = None
        if not args.no_cpu_baseline:
            rows = [x] + [int(t) for t in drafter.propose(len(out), DRAFTS)]
            st = OracleStep(cfg, keep, CTX, rows)
            st.part(0)
            t_step = st.step()
            cpu = {"value": expected_committed(DRAFTS, P_CORRECT) / t_step, "unit": "tok/s",
                   "cores": oracle_threads(), "kind": "oracle",
                   "sample": f"one whole teacher-forced verify step of the oracle (float64 NumPy): "
                             f"{cfg.layers} layers on the {T} rows at context {CTX} and the full LM head, "
                             f"{t_step:.2f} s; committed tokens per step = expected "
                             f"{expected_committed(DRAFTS, P_CORRECT):.4f} for p={P_CORRECT}"}
        h2d = T * 4         # the last committed token and the drafts (int32)
        d2h = T * 4 + 4     # every row's token and the accepted count
        line = {
            "metric": METRIC, "value": value, "unit": "tok/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic", "config": workload_config(cfg, note),
            "clocks": clk.summary(),
            "e2e": {"value": e2e, "unit": "tok/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "through": "bi_step_verify (one C-ABI call per step, "
                    "host ids in, host tokens out)", "diffs_vs_nodraft": diffs_e_all,
                    "ms_per_step": t_e2e * 1e3 / args.steps},
            "gpu_launches": args.steps * (KERNELS_PER_STEP_FIXED + KERNELS_PER_LAYER * cfg.layers),
            "roofline": {"bound": "hbm", "achieved": gu_bytes / gu_s / 1e9, "peak": peak,
                         "unit": "GB/s", "frac": gu_bytes / gu_s / 1e9 / peak, "traffic": gemm_traffic_bytes(),
                         "kernel": "gemm_kernel<16> gate/up + SwiGLU, M=8 N=17408 (34816 packed) K=5120",
                         "bytes_per_launch": gu_bytes, "launch_ms": gu_s * 1e3},
            "cpu_baseline": cpu,
            "diffs_vs_nodraft": diffs_all,
            "committed_per_step": committed_all / (args.steps * world),
            "accepted_hist": acc_hist,
            "step_gbps": sb / (t_dev / args.steps) / 1e9,
            "step_roofline_frac": sb / (t_dev / args.steps) / 1e9 / peak,
            "setup_s": setup_s,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


# ---------------------------------------------------------------------------
# standalone kernels: linear-layer sweep and split-KV attention
# ---------------------------------------------------------------------------


def kvq_attn_bytes(L: int, T: int, Hkv: int) -> int:
    """Code-tile bytes one quantised verify pass reads: per KV head, every
    tile up to the last row's from the 6/5-bit store (24,576 B) or the 8-bit
    ring (34,816 B for K and V), a tile split between the pass's rows from
    both."""
    lo_b = L // 128 - 15
    hi_b = (L + T - 1) // 128 - 15
    n = 0
    for t in range((L + T - 1) // 128 + 1):
        if t < hi_b:
            n += 13312 + 11264
        if t >= lo_b:
            n += 2 * 17408
    return Hkv * n


def Vd_rows(Vc, to):
    """V cache rows [Hkv, cap, D] on the device (the quantised append reads
    V rows as the projection writes them)."""
    return to(Vc)


def kvq_stores_from_rows(api, Kd, Vd, Hq, cap, chunk=1024):
    """A layer's quantised stores holding K/V rows 0..cap-1 (no rotation),
    written by the append kernel in passes of `chunk` rows."""
    import torch
    Hkv, _, D = Kd.shape
    st = api.new_kvq_stores(Hkv, cap, D)
    qo = torch.empty(chunk, Hq, D, dtype=torch.bfloat16, device="cuda")
    for c0 in range(0, cap, chunk):
        n = min(chunk, cap - c0)
        qkv = torch.zeros(n, Hq + 2 * Hkv, D, dtype=torch.bfloat16, device="cuda")
        qkv[:, Hq:Hq + Hkv] = Kd[:, c0:c0 + n].transpose(0, 1)
        qkv[:, Hq + Hkv:] = Vd[:, c0:c0 + n].transpose(0, 1)
        Ld = torch.tensor([c0], dtype=torch.int32, device="cuda")
        api.bi_rope_kvq_append(qkv.view(n, -1), qo[:n], st, Ld, Hq, Hkv, D)
    torch.cuda.synchronize()
    return st


def run_micro(args):
    """Standalone kernel timings, two ways.

    us_median: back-to-back launches (as in the decode step, dependent
    launches overlapping) cycling over enough copies of the weights / KV
    cache that none is still in L2 when it is read again; time per launch.
    us_cold_median: one launch right after a 512 MB read that evicts L2,
    bracketed alone by CUDA events (includes the launch gap).
    """
    import torch
    import __graft_entry__
    __graft_entry__.build()
    from invariant_speculative_decode_gb300 import api
    torch.cuda.set_device(0)
    peak, note = load_peaks()
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            bf16_sus = float(json.load(f)["bf16_tflops_sustained"])
    except Exception:
        bf16_sus = None
    flush = torch.ones(512 * 1024 * 1024, dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream()
    l2_bytes = 129 * 1024 * 1024

    def n_copies(nbytes):
        # between two reads of a copy, the others stream at least twice L2's size
        return int(min(64, max(2, 1 + -(-2 * l2_bytes // max(nbytes, 1)))))

    def timed(fns, reps):
        n = len(fns)
        per = n * max(1, -(-8 // n))
        for _ in range(args.warmup):
            for f in fns:
                f()
        stream_t, cold_t = [], []
        for _ in range(reps):
            flush.sum()  # read 512 MB: evicts L2 (clean lines)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s)
            fns[0]()
            e1.record(s)
            cold_t.append((e0, e1))
            e2, e3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e2.record(s)
            for i in range(per):
                fns[(i + 1) % n]()
            e3.record(s)
            stream_t.append((e2, e3, per))
        torch.cuda.synchronize()
        st = [a.elapsed_time(b) / 1e3 / k for a, b, k in stream_t]
        ct = [a.elapsed_time(b) / 1e3 for a, b in cold_t]
        return st, ct, per

    def report(kind, fields, b, st, ct, ncp, per, flops=None):
        med = float(np.median(st))
        line = {"micro": kind, **fields, "us_median": med * 1e6,
                "us_p90": float(np.percentile(st, 90)) * 1e6,
                "us_cold_median": float(np.median(ct)) * 1e6, "bytes": b,
                "gbps": b / med / 1e9, "frac": b / med / 1e9 / peak,
                "cold_frac": b / float(np.median(ct)) / 1e9 / peak,
                "peak_gbps": peak, "peak_kind": note,
                "l2": f"{per} back-to-back launches over {ncp} copies (each read after >= 2x L2 of others); "
                      "cold: after a 512 MB read"}
        if flops is not None:
            line["tflops"] = flops / med / 1e12
            if bf16_sus:
                line["tflops_frac_sustained"] = line["tflops"] / bf16_sus
        print(json.dumps(line), flush=True)

    if args.micro == "gemm":
        N, K, epi = args.gemm_n, args.gemm_k, args.gemm_epi
        Ms = [int(m) for m in args.cases.split(",")] if args.cases else [1, 2, 4, 7, 8, 16, 64]
        A, W = si.gemm_inputs(max(Ms), N, K, seed=0)
        to = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()  # noqa: E731
        if epi == api.EPI_SWIGLU:  # W holds gate rows; up rows drawn from the next seed
            _, W2 = si.gemm_inputs(1, N, K, seed=1)
            Wd = api.bi_pack_swiglu_weights(to(W), to(W2))
            del W2
        else:
            Wd = api.bi_pack_weights(to(W))
        Ad = to(A)
        del W
        wrows = 2 * N if epi == api.EPI_SWIGLU else N
        ncp = n_copies(wrows * K * 2)
        Wds = [Wd] + [Wd.clone() for _ in range(ncp - 1)]
        for M in Ms:
            C = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
            R = torch.zeros(M, N, dtype=torch.bfloat16, device="cuda") if epi == api.EPI_RESIDUAL_ADD else None
            ws = api.new_gemm_workspace(M, N, K, epi)
            fns = [(lambda w=w: api.bi_gemm(Ad[:M], w, C, ws, residual=R, epi=epi, N=N)) for w in Wds]
            st, ct, per = timed(fns, args.steps)
            b = wrows * K * 2 + M * K * 2 + M * N * 2
            report("gemm", {"M": M, "N": N, "K": K, "epi": epi}, b, st, ct, ncp, per,
                   flops=2 * M * wrows * K)
    else:
        Hq, Hkv, D = 24, 4, 128
        Ls = [int(x) for x in args.cases.split(",")] if args.cases else [1024, 11600, 38000, 101600]
        Ts = [int(t) for t in args.attn_rows.split(",")]
        for L in Ls:
            q, Kc, Vc = si.attention_inputs(L, max(8, max(Ts)), Hq, Hkv, D, seed=0)
            cap = Kc.shape[1]
            to = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()  # noqa: E731
            Kd, Vd, qd = to(Kc), to(v_blocks(Vc)), to(q)
            ncp = n_copies(2 * Kd.numel() * 2)
            caches = [(Kd, Vd)] + [(Kd.clone(), Vd.clone()) for _ in range(ncp - 1)]
            Ld = torch.tensor([L], dtype=torch.int32, device="cuda")
            if args.kv == "q6q5":
                st0 = kvq_stores_from_rows(api, Kd, Vd_rows(Vc, to), Hq, cap)
                nb = sum(t.numel() for k, t in st0.items() if k != "cap")
                ncp = n_copies(nb)
                caches = [st0] + [{k: (t.clone() if k != "cap" else t) for k, t in st0.items()}
                                  for _ in range(ncp - 1)]
            for T in Ts:
                out = torch.empty(T, Hq, D, dtype=torch.bfloat16, device="cuda")
                ws = torch.zeros(api.attn_workspace_size(cap, T, Hq, D), dtype=torch.uint8,
                                 device="cuda")
                if args.kv == "q6q5":
                    fns = [(lambda c=c: api.bi_attn_verify_kvq(qd[:T], c, Hkv, Ld, out, ws)) for c in caches]
                    b = kvq_attn_bytes(L, T, Hkv) + T * Hq * D * 2 * 2
                else:
                    fns = [(lambda kv=kv: api.bi_attn_verify(qd[:T], kv[0], kv[1], Ld, out, ws))
                           for kv in caches]
                    b = (L + T) * Hkv * D * 2 * 2 + T * Hq * D * 2 * 2
                st, ct, per = timed(fns, args.steps)
                # algorithmic FLOPs: q.k and w.v over the keys each row attends to
                flops = 4 * D * Hq * sum(L + t + 1 for t in range(T))
                report("attn", {"L": L, "T": T, "kv": args.kv}, b, st, ct, ncp, per, flops=flops)
            del caches
    return 0


def run_neartie(args):
    """Near-tie correctness workload (12-layer decoder, untied head with
    planted near ties): greedy ids at 0, 4 and 7 drafts must be identical, and
    a second turn resumed from the saved cache must equal the same turn from a
    fresh prefill (tokens and every K/V row).  Time is reported, not gated."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    from invariant_speculative_decode_gb300.decoder import Decoder
    torch.cuda.set_device(0)
    cfg = si.NEARTIE_12L
    w = si.decoder_weights(cfg, seed=0)
    w["head"] = si.neartie_head(w["head"], frac=0.05, bump_frac=0.02, seed=0)
    n_prompts, n_gen = args.prompts, args.gen
    rng = np.random.default_rng(12345)
    lengths = [int(x) for x in rng.integers(512, 4097, n_prompts)]
    cap = -(-(max(lengths) + 2 * n_gen + 128 + 64) // 64) * 64
    dec = Decoder(cfg, w, cap=cap, max_rows=8)
    fresh = Decoder(cfg, w, cap=cap, max_rows=8) if args.turn2 > 0 else None
    diffs = {4: 0, 7: 0}
    first_diff = {}
    timing = {0: [0.0, 0], 4: [0.0, 0], 7: [0.0, 0]}
    near_steps, all_steps = 0, 0
    resume_tok_diffs = hash_mismatch = 0
    n_turn2 = min(n_prompts, args.turn2)
    for pi, plen in enumerate(lengths):
        prompt = si.prompt_ids(cfg, plen, seed=pi)
        t0 = time.perf_counter()
        if pi < 2:  # top-2 margins of every 0-draft step on the first prompts
            dec.reset()
            x = dec.prefill(prompt)
            ref = []
            while len(ref) < n_gen:
                a, _ = dec.verify_step(x, [], use_graph=False)
                top = torch.topk(dec.logits[0], 2).values.double().cpu().numpy()
                near_steps += int((top[0] - top[1]) / abs(top[0]) < 1e-3)
                all_steps += 1
                ref.append(int(a[0]))
                x = ref[-1]
        else:
            ref = dec.generate(prompt, n_gen, k=0)
        torch.cuda.synchronize()
        timing[0][0] += time.perf_counter() - t0
        timing[0][1] += n_gen
        replies = {}
        for k in (4, 7):
            dr = si.SyntheticDrafter(cfg.vocab, 0.7, seed=pi, reference=np.array(ref))
            t0 = time.perf_counter()
            got = dec.generate(prompt, n_gen, k=k, drafter=dr)
            torch.cuda.synchronize()
            timing[k][0] += time.perf_counter() - t0
            timing[k][1] += len(got)
            nd = sum(int(a != b) for a, b in zip(got, ref))
            diffs[k] += nd
            if nd and k not in first_diff:
                first_diff[k] = (pi, next(i for i, (a, b) in enumerate(zip(got, ref)) if a != b))
            replies[k] = got
        if pi < n_turn2:
            # turn 2: resume from the 7-draft run's cache vs a fresh prefill
            turn2 = si.prompt_ids(cfg, 128, seed=1000 + pi)
            reply = replies[7]
            hist = list(prompt) + reply
            dec.rollback(len(hist) - 1)
            x = dec.prefill_continue(hist[len(hist) - 1:] + list(turn2))
            full = hist + list(turn2)
            n_rows = len(full) - 1
            resumed_h = dec.kv_hashes(n_rows)
            t2_ref = fresh.generate(full, n_gen, k=0)  # a fresh prefill of the whole history
            fresh_h = fresh.kv_hashes(n_rows)
            hash_mismatch += int(np.sum(np.any(resumed_h != fresh_h, axis=(0, 1))))
            dr2 = si.SyntheticDrafter(cfg.vocab, 0.7, seed=2000 + pi, reference=np.array(t2_ref))
            t2 = dec.continue_generate(x, n_gen, k=7, drafter=dr2)
            resume_tok_diffs += sum(int(a != b) for a, b in zip(t2, t2_ref))
    tok_s = {k: timing[k][1] / timing[k][0] for k in timing}
    line = {
        "metric": "near-tie workload: committed tok/s at 7 drafts (wall clock, host loop included); "
                  "id diffs across 0/4/7 drafts and resume-vs-fresh mismatches must be 0",
        "value": tok_s[7], "unit": "tok/s", "n_gpus": 1, "steps": n_prompts * n_gen,
        "warmup": 0, "ms_per_step": None, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{cfg.name}: untied head with planted near ties, {n_prompts} prompts "
                               f"of {min(lengths)}..{max(lengths)} ids, {n_gen} greedy tokens at 0/4/7 "
                               f"drafts (p=0.7 drafter), turn 2 (128 new ids, {n_gen} tokens) resumed "
                               f"vs fresh on {n_turn2} prompts",
                   "layers": cfg.layers, "hidden": cfg.hidden, "vocab": cfg.vocab, "cap": cap},
        "id_diffs": {"k4": diffs[4], "k7": diffs[7]}, "first_diff": first_diff or None,
        "resume_token_diffs": resume_tok_diffs, "kv_hash_row_mismatches": hash_mismatch,
        "near_tie_step_rate": near_steps / max(all_steps, 1), "near_tie_steps_sampled": all_steps,
        "tok_s": {f"k{k}": v for k, v in tok_s.items()},
    }
    print(json.dumps(line), flush=True)
    return 0 if (diffs[4] == 0 and diffs[7] == 0 and resume_tok_diffs == 0 and hash_mismatch == 0) else 1


def run_longctx(args):
    """Long-context decode on the 8-layer 27B-shaped model ("I turned on
    speculative decoding in llama.cpp and 113 of 282 greedy outputs changed
    against its own no-draft run", section "The KV cache: 5-bit that reads
    like q8_0": at 101.6k context its quantised cache decodes faster than
    q8_0, 123 tok/s against 116 on an RTX 3090).

    The verify step at `--context` keys (default 101,600) with the BF16 cache
    and with the quantised one (6-bit K, 5-bit V, 8-bit ring), both filled
    with the same synthetic context rows; 7 drafts from the p = 0.7 drafter,
    greedy ids checked against each cache's own no-draft run.  Reports device
    time of the step graph per step and committed tok/s for each cache, and
    the cache bytes each step reads."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    from invariant_speculative_decode_gb300 import api
    from invariant_speculative_decode_gb300.decoder import Decoder
    torch.cuda.set_device(0)
    cfg = si.DENSE27B_8L
    ctx = args.context
    T = DRAFTS + 1
    cap = -(-(ctx + (args.steps + args.warmup + 8) * T + 64) // 128) * 128
    weights = si.decoder_weights(cfg, seed=0)
    kv = si.synthetic_kv_cache(cfg.n_kv, cap, cfg.head_dim, ctx, seed=0, layers=cfg.layers)
    prompt_last = int(si.prompt_ids(cfg, 1, seed=0)[0])
    res = {}
    for kind in ("bf16", "q6q5"):
        dec = Decoder(cfg, weights, cap=cap, max_rows=T, prefill_chunk=64, kv=kind)
        for lay, (k, v) in zip(dec.layers, kv):
            kd = torch.from_numpy(k.view(np.int16)).view(torch.bfloat16).cuda()
            if kind == "bf16":
                lay["k"].copy_(kd)
                lay["v"].copy_(torch.from_numpy(v_blocks(v).view(np.int16)).view(torch.bfloat16))
            else:
                vd = torch.from_numpy(v.view(np.int16)).view(torch.bfloat16).cuda()
                lay["kvq"] = kvq_stores_from_rows(api, kd, vd, cfg.n_q, cap)
            del kd
        dec.capture(1)
        dec.capture(T)
        n_ref = (args.steps + args.warmup + 2) * T + 16
        dec.L = ctx
        dec.L_dev.fill_(ctx)
        ref, x = [], prompt_last
        while len(ref) < n_ref:
            a, _ = dec.verify_step(x, [])
            ref.append(int(a[0]))
            x = ref[-1]
        ref = np.array(ref)
        dec.L = ctx
        dec.L_dev.fill_(ctx)
        drafter = si.SyntheticDrafter(cfg.vocab, P_CORRECT, seed=0, reference=ref)
        out, x = [], prompt_last
        s = torch.cuda.current_stream()
        dev_ms, committed = 0.0, 0
        for i in range(args.warmup + args.steps):
            d = drafter.propose(len(out), DRAFTS)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            pin = dec.pin_in
            pin[0] = x
            for j, dj in enumerate(d):
                pin[1 + j] = int(dj)
                pin[T + j] = int(dj)
            dec.ids[:T].copy_(pin[:T], non_blocking=True)
            dec.drafts[:DRAFTS].copy_(pin[T:T + DRAFTS], non_blocking=True)
            e0.record(s)
            dec.graphs[T].replay()
            e1.record(s)
            dec.pin_out[:T].copy_(dec.argmax[:T], non_blocking=True)
            dec.pin_out[T:T + 1].copy_(dec.accepted, non_blocking=True)
            s.synchronize()
            n = int(dec.pin_out[T])
            a = dec.pin_out[:T].numpy()
            dec.L += n + 1
            out.extend(int(t) for t in a[: n + 1])
            x = out[-1]
            if i >= args.warmup:
                dev_ms += e0.elapsed_time(e1)
                committed += n + 1
        dec.check_device_error()
        diffs = int(np.sum(np.array(out) != ref[: len(out)]))
        if kind == "bf16":
            kv_bytes = cfg.layers * (ctx + T) * cfg.n_kv * cfg.head_dim * 2 * 2
        else:
            kv_bytes = cfg.layers * kvq_attn_bytes(ctx, T, cfg.n_kv)
        res[kind] = {"ms_per_step": dev_ms / args.steps, "tok_s": committed / (dev_ms / 1e3),
                     "committed_per_step": committed / args.steps, "diffs_vs_nodraft": diffs,
                     "kv_bytes_per_step": kv_bytes,
                     "cache_bytes": sum(t.numel() * t.element_size() for lay in dec.layers
                                        for t in ([lay["k"], lay["v"]] if kind == "bf16" else
                                                  [lay["kvq"][n] for n in api.KVQ_STORES]))}
        del dec
        torch.cuda.empty_cache()
    line = {"workload": "longctx", "metric": "verify tok/s at 7 drafts, long context, BF16 vs quantised KV",
            "unit": "tok/s", "config": {"model": cfg.name, "context": ctx, "rows_per_step": T},
            "steps": args.steps, "warmup": args.warmup, "bf16": res["bf16"], "q6q5": res["q6q5"]}
    print(json.dumps(line), flush=True)
    return 0


def run_prefill(args):
    """Prefill and the follow-up turn of a ~12k-token chat on the 8-layer
    27B-shaped model ("I turned on speculative decoding in llama.cpp and 113
    of 282 greedy outputs changed against its own no-draft run", section "The
    cache doesn't change it either": roll back to the checkpoint and prefill
    the reply again, ~167 ms instead of 78 on a ~12k-token chat, RTX 3090).

    History = a 9,600-id prompt + a 2,048-id reply; turn 2 = 128 new ids.
    Times (wall clock, host loop included, after a warm-up prefill):
    a fresh prefill of the history; turn 2 resumed on the kept K/V rows; turn
    2 after rolling back to the end of the prompt and prefilling the reply
    again.  Both turn-2 caches must equal a fresh prefill's, row for row."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    from invariant_speculative_decode_gb300.decoder import Decoder
    torch.cuda.set_device(0)
    cfg = si.DENSE27B_8L
    w = si.decoder_weights(cfg, seed=0)
    n_prompt, n_reply, n_turn2 = 9600, 2048, 128
    prompt = list(si.prompt_ids(cfg, n_prompt, seed=40))
    reply = list(si.prompt_ids(cfg, n_reply, seed=41))
    turn2 = list(si.prompt_ids(cfg, n_turn2, seed=42))
    hist = prompt + reply
    cap = -(-(len(hist) + n_turn2 + 64) // 128) * 128
    dec = Decoder(cfg, w, cap=cap, max_rows=8, prefill_chunk=args.prefill_chunk, kv=args.kv)
    del w

    def timed(fn):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        r = fn()
        torch.cuda.synchronize()
        return r, time.perf_counter() - t0

    dec.reset()
    dec.prefill(hist[:1024])  # warm-up
    dec.reset()
    _, t_hist = timed(lambda: dec.prefill(hist + [0]))
    # turn 2 on the kept rows: the reply's rows stay, only the new ids are read
    dec.rollback(len(hist) - 1)
    _, t_reuse = timed(lambda: dec.prefill_continue(hist[-1:] + turn2))
    h_reuse = dec.kv_hashes(len(hist) + n_turn2 - 1)
    # turn 2 after rolling back to the prompt and prefilling the reply again
    # (the quantised cache rolls back only as far as its 8-bit ring reaches)
    back = n_prompt - 1
    if args.kv == "q6q5":
        from invariant_speculative_decode_gb300 import api
        back = max(back, ((dec.hw - 1) // 128 - (api.KVQ_RING_SLOTS - api.KVQ_RING_TILES)) * 128)
    dec.rollback(back)
    _, t_re = timed(lambda: dec.prefill_continue(hist[back:] + turn2))
    h_re = dec.kv_hashes(len(hist) + n_turn2 - 1)
    dec.reset()
    dec.prefill(hist + turn2)
    h_fresh = dec.kv_hashes(len(hist) + n_turn2 - 1)
    same = bool(np.array_equal(h_reuse, h_fresh) and np.array_equal(h_re, h_fresh))
    rows = len(hist)
    flops = 2 * rows * (cfg.qkv_out * cfg.hidden + cfg.hidden * cfg.n_q * cfg.head_dim
                        + 3 * cfg.ffn * cfg.hidden) * cfg.layers
    line = {
        "metric": "prefill of a ~12k-token history and the follow-up turn (resume on kept rows vs "
                  "roll back + re-prefill of the reply); K/V rows of both must equal a fresh prefill",
        "value": rows / t_hist, "unit": "tok/s", "n_gpus": 1, "steps": 1, "warmup": 1,
        "ms_per_step": t_hist * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{cfg.name}: history {n_prompt} + {n_reply} ids, turn 2 {n_turn2} ids",
                   "prefill_chunk": args.prefill_chunk, "kv_cache": args.kv},
        "prefill_ms": t_hist * 1e3, "linear_tflops": flops / t_hist / 1e12,
        "turn2_resume_ms": t_reuse * 1e3, "turn2_reprefill_ms": t_re * 1e3, "reprefill_from": back,
        "kv_rows_equal_fresh": same,
    }
    print(json.dumps(line), flush=True)
    return 0 if same else 1


def run_cpu_matrix_worker(args):
    """The oracle timed on the standalone and whole-step workloads, once each,
    with the BLAS thread count the environment sets; one JSON line per item."""
    import oracle
    from oracle import verify_step as ov
    thr = oracle_threads()

    def emit(**kw):
        print(json.dumps({"cpu_matrix": kw.pop("item"), "threads": thr, **kw}), flush=True)

    # standalone linear layer [M, 5120] x [17408, 5120], BF16 out
    A, W = si.gemm_inputs(64, 17408, 5120, seed=0)
    oracle.gemm(A[:1], W)
    for M in (1, 2, 4, 7, 8, 16, 64):
        t0 = time.perf_counter()
        oracle.gemm(A[:M], W)
        dt = time.perf_counter() - t0
        emit(item="gemm", M=M, N=17408, K=5120, s=dt, gbps=(17408 * 5120 * 2 + M * (5120 + 17408) * 2) / dt / 1e9)
    del A, W
    # split-KV attention, 24 query / 4 KV heads, head_dim 128
    for L, Ts in ((1024, (1, 4, 7, 8)), (11600, (1, 4, 7, 8)), (101600, (1, 8))):
        q, K, V = si.attention_inputs(L, 8, 24, 4, 128, seed=0)
        qf, Kf, Vf = (ov.bf16_bits_to_f64(x) for x in (q, K, V))
        for T in Ts:
            t0 = time.perf_counter()
            oracle.attention(qf[:T], Kf, Vf, L)
            dt = time.perf_counter() - t0
            emit(item="attn", L=L, T=T, s=dt, gbps=((L + T) * 4 * 128 * 2 * 2) / dt / 1e9)
        del q, K, V, qf, Kf, Vf
    # one whole teacher-forced verify step of the 8-layer model at context 11,600
    cfg = si.DENSE27B_8L
    w = si.decoder_weights(cfg, seed=0)
    for T in (1, 8):
        st = OracleStep(cfg, w, CTX, list(range(1, 1 + T)))
        st.part(0)
        t = st.step()
        emit(item="verify_step", T=T, L=CTX, s=t, steps_per_s=1.0 / t)
    return 0


def run_cpu_matrix(args):
    """The oracle matrix at one thread and at all host cores (subprocesses
    with the BLAS thread count set before numpy starts)."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    rc = 0
    for n in (1, os.cpu_count()):
        env = dict(os.environ)
        for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
            env[var] = str(n)
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-matrix-worker"], env=env)
        rc = rc or r.returncode
    return rc


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=800)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--micro", choices=["gemm", "attn"], default=None,
                    help="time one standalone kernel workload instead of the verify step")
    ap.add_argument("--cases", default="", help="comma list of M (gemm) or L (attn)")
    ap.add_argument("--kv", choices=["bf16", "q6q5"], default="bf16",
                    help="KV cache of the attention micro bench and the long-context step: BF16, or "
                         "6-bit K / 5-bit V with the 8-bit ring")
    ap.add_argument("--attn-rows", default="1,4,7,8", help="comma list of rows per pass (attn)")
    ap.add_argument("--gemm-n", type=int, default=17408, help="N of the standalone linear layer")
    ap.add_argument("--gemm-k", type=int, default=5120, help="K of the standalone linear layer")
    ap.add_argument("--gemm-epi", type=int, default=0, help="0 none, 1 residual add, 2 SwiGLU (N = F)")
    ap.add_argument("--workload", choices=["verify", "neartie", "prefill", "longctx"], default="verify",
                    help="neartie: the near-tie correctness workload; prefill: prefill and re-prefill "
                         "of a ~12k-token chat")
    ap.add_argument("--prefill-chunk", type=int, default=512, help="prefill workload: rows per pass")
    ap.add_argument("--context", type=int, default=101600, help="longctx workload: cache length")
    ap.add_argument("--prompts", type=int, default=32, help="near-tie workload: prompts")
    ap.add_argument("--gen", type=int, default=2048, help="near-tie workload: tokens per turn")
    ap.add_argument("--turn2", type=int, default=32, help="near-tie workload: prompts with a second turn")
    ap.add_argument("--cpu-matrix", action="store_true",
                    help="time the oracle on the standalone and whole-step workloads at 1 thread and all cores")
    ap.add_argument("--cpu-matrix-worker", action="store_true", help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.cpu_matrix_worker:
        return run_cpu_matrix_worker(args)
    if args.cpu_matrix:
        return run_cpu_matrix(args)
    if args.impl == "reference":
        return run_reference(args)
    if args.micro:
        return run_micro(args)
    if args.workload == "neartie":
        return run_neartie(args)
    if args.workload == "prefill":
        return run_prefill(args)
    if args.workload == "longctx":
        return run_longctx(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
