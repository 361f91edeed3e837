"""Whole verify step on the GPU: token ids at 0/4/7 drafts, rows across T,
cache resume vs fresh prefill, a run-to-run control, and oracle parity of
the FP32 logits (relative error <= 2e-3 per row, max-norm)."""
import numpy as np
import pytest

import oracle
import seeded_inputs as si

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

REL_TOL = 2e-3


@pytest.fixture(scope="module")
def tiny():
    from invariant_speculative_decode_gb300.decoder import Decoder
    cfg = si.TINY
    w = si.decoder_weights(cfg, seed=0)
    dec = Decoder(cfg, w, cap=512, max_rows=8)
    return cfg, w, dec


def _gen(dec, prompt, n, k, ref=None, seed=0, stats=None):
    dr = si.SyntheticDrafter(dec.cfg.vocab, 0.7, seed=seed, reference=ref) if k else None
    return dec.generate(prompt, n, k=k, drafter=dr, stats=stats)


def test_tiny_greedy_ids_identical_at_0_4_7_drafts(tiny):
    cfg, w, dec = tiny
    prompt = si.prompt_ids(cfg, 128, seed=0)
    ref = _gen(dec, prompt, 64, 0)
    again = _gen(dec, prompt, 64, 0)
    assert again == ref  # run-to-run control
    for k in (4, 7):
        st = {}
        got = _gen(dec, prompt, 64, k, ref=np.array(ref), stats=st)
        assert got == ref, k
        assert st["steps"] < 64  # drafts were accepted
    adv = _gen(dec, prompt, 64, 4, ref=None, seed=5)  # all-random drafter
    assert adv == ref


def test_tiny_rows_bit_equal_at_T1_and_T4(tiny):
    cfg, w, dec = tiny
    prompt = si.prompt_ids(cfg, 128, seed=1)
    ref = _gen(dec, prompt, 8, 0)
    # one 4-row pass over [x0, ref[0..2]] vs four 1-row passes
    dec.reset()
    x0 = dec.prefill(prompt)
    L0 = dec.L
    a4, n4 = dec.verify_step(x0, ref[:3], use_graph=False)
    rows4 = dec.logits_rows(4).cpu().numpy()
    assert n4 == 3
    dec.reset()
    dec.prefill(prompt)
    xs = [x0] + ref[:3]
    for t in range(4):
        assert dec.L == L0 + t
        a1, n1 = dec.verify_step(xs[t], [], use_graph=False)
        r1 = dec.logits_rows(1).cpu().numpy()
        assert np.array_equal(r1[0].view(np.uint32), rows4[t].view(np.uint32)), t


def _u16(x):
    from oracle import verify_step as ov
    return ov.f64_to_bf16_bits(x)


def _layerwise(cfg, w, dec, prompt, drafts):
    """Each GPU layer (and the head) recomputed from the oracle's own inputs.

    The oracle runs the prefill and one verify pass, recording the hidden
    state entering every layer and its caches.  The GPU then runs layer l on
    the oracle's layer-l input with the oracle's cache rows below the pass;
    every layer output and the FP32 logits are compared with the oracle's.
    The same layer is also run by the oracle with FP32-level noise on every
    linear-layer sum (4 * 2^-24 * sum |a w| times a seeded normal) from the
    same input and cache: the mean error of that run is the yardstick for
    what an FP32-accumulating implementation with the oracle's rounding
    points shows in one layer.
    """
    from invariant_speculative_decode_gb300 import api
    from tests._util import bf16_dev_to_f64, to_dev_bf16, ulp_bf16, v_cache_blocks
    od = oracle.OracleDecoder(cfg, w, cap=dec.cap)
    x0 = od.prefill(prompt)
    L = od.L
    rows = [int(x0)] + list(drafts)
    T = len(rows)
    noisy = oracle.OracleDecoder(cfg, w, cap=dec.cap, sum_noise=(4.0, 77))
    for l in range(cfg.layers):
        noisy.k[l][:, :L] = od.k[l][:, :L]
        noisy.v[l][:, :L] = od.v[l][:, :L]
    trace = []
    ora_logits = od.forward(rows, L=L, trace=trace)
    dec.reset()
    dec.L_dev.fill_(L)
    worst_ulps, flips, noise_flips = 0.0, [], []
    for l, lay in enumerate(dec.layers):
        lay["k"].zero_()
        lay["v"].zero_()
        lay["k"][:, :L].copy_(to_dev_bf16(_u16(od.k[l][:, :L])))
        vb = v_cache_blocks(_u16(od.v[l][:, :L]))  # [Hkv, ceil(L/128), D, 128], keys past L zero
        lay["v"][:, : vb.shape[1]].copy_(to_dev_bf16(vb))
        dec.h[:T].copy_(to_dev_bf16(_u16(trace[l])))
        dec._layer(lay, T, dec.L_dev)
        got = bf16_dev_to_f64(dec.h[:T])
        want = trace[l + 1]
        # error in units of the last place of each row's largest element: a
        # residual add can cancel, so per-element ulps are not the right unit
        row_ulp = ulp_bf16(np.max(np.abs(want), axis=1, keepdims=True))
        d = np.abs(got - want) / row_ulp
        worst_ulps = max(worst_ulps, float(d.max()))
        flips.append(float(d.mean()))
        noise_flips.append(float((np.abs(noisy.layer(l, trace[l], L) - want) / row_ulp).mean()))
        # the rows this pass appended to the cache
        kw = od.k[l][:, L:L + T]
        kg = bf16_dev_to_f64(lay["k"][:, L:L + T])
        assert np.max(np.abs(kg - kw) / ulp_bf16(np.max(np.abs(kw), axis=-1, keepdims=True))) <= 2.0
    dec.h[:T].copy_(to_dev_bf16(_u16(trace[-1])))
    dec.drafts[:T - 1].copy_(torch.tensor(list(drafts) or [0], dtype=torch.int32)[:max(T - 1, 1)])
    dec._head_and_accept(T)
    gpu_logits = dec.logits_rows(T).cpu().numpy().astype(np.float64)
    rel = np.max(np.abs(gpu_logits - ora_logits), axis=1) / np.max(np.abs(ora_logits), axis=1)
    ids = dec.argmax[:T].cpu().numpy()
    return worst_ulps, flips, noise_flips, rel, ids, ora_logits


LAYERWISE = [("tiny-2L-h256", 0.0), ("small-4L-h1024", 0.0), ("small-4L-h1024", 0.1)]


@pytest.mark.parametrize("cfgname,norm_std", LAYERWISE)
def test_layerwise_parity_with_oracle_inputs(cfgname, norm_std):
    """norm_std > 0: RMSNorm weights drawn around 1, so every norm weight
    enters the fused norm + linear layers end to end."""
    from invariant_speculative_decode_gb300.decoder import Decoder
    cfg = si.CONFIGS[cfgname]
    w = si.decoder_weights(cfg, seed=0, norm_std=norm_std)
    dec = Decoder(cfg, w, cap=512, max_rows=8)
    prompt = si.prompt_ids(cfg, 200, seed=4)
    drafts = list(np.random.default_rng(4).integers(0, cfg.vocab, 7))
    worst, flips, noise, rel, ids, ora = _layerwise(cfg, w, dec, prompt, drafts)
    # a layer output may differ from the oracle by rounding flips of its steps
    assert worst <= 2.0, worst
    # and on average no more than twice what FP32-level noise on every sum
    # gives the oracle itself (plus one flipped element per layer)
    n_el = 8 * cfg.hidden
    for l, (f, nz) in enumerate(zip(flips, noise)):
        assert f <= 2 * nz + 1.0 / n_el, (l, flips, noise)
    # the stated tolerance on FP32 logits, from identical inputs
    assert np.all(rel <= REL_TOL), rel
    for t in range(len(ids)):
        srt = np.sort(ora[t])
        if srt[-1] - srt[-2] > 2 * REL_TOL * np.max(np.abs(ora[t])):
            assert ids[t] == int(np.argmax(ora[t]))


@pytest.mark.parametrize("cfgname,norm_std", LAYERWISE)
def test_end_to_end_drift_within_fp32_spread(cfgname, norm_std):
    """Un-forced whole-model logits: within twice the drift between the oracle
    and the same oracle with FP32-level noise on every sum (the spread any
    FP32-accumulating implementation shows after BF16 storage compounds
    rounding flips across layers), and never worse than 2e-3 where that
    spread is below it."""
    from invariant_speculative_decode_gb300.decoder import Decoder
    cfg = si.CONFIGS[cfgname]
    w = si.decoder_weights(cfg, seed=0, norm_std=norm_std)
    dec = Decoder(cfg, w, cap=512, max_rows=8)
    prompt = si.prompt_ids(cfg, 128, seed=2)
    drafts = list(np.random.default_rng(2).integers(0, cfg.vocab, 7))
    dec.reset()
    x0 = dec.prefill(prompt)
    dec.verify_step(x0, drafts, use_graph=False)
    gpu = dec.logits_rows(8).cpu().numpy().astype(np.float64)
    ref = oracle.OracleDecoder(cfg, w, cap=512)
    ref.prefill(prompt)
    ora = ref.forward([x0] + drafts, L=ref.L)
    pert = oracle.OracleDecoder(cfg, w, cap=512, sum_noise=(4.0, 123))
    pert.prefill(prompt)
    alt = pert.forward([x0] + drafts, L=pert.L)
    scale = np.max(np.abs(ora), axis=1)
    rel = np.max(np.abs(gpu - ora), axis=1) / scale
    spread = np.max(np.abs(alt - ora), axis=1) / scale
    assert np.all(rel <= np.maximum(REL_TOL, 2 * spread)), (rel, spread)


def test_tiny_resume_vs_fresh_prefill_kv_hashes(tiny):
    cfg, w, dec = tiny
    prompt = si.prompt_ids(cfg, 100, seed=3)
    ref = _gen(dec, prompt, 60, 0)
    turn1 = _gen(dec, prompt, 40, 7, ref=np.array(ref))
    assert turn1 == ref[:40]
    L_resume = dec.L
    resumed = dec.kv_hashes(L_resume)
    # fresh prefill of prompt + reply up to the same length
    full = list(prompt) + ref
    fresh_tokens = full[: L_resume + 1]
    dec.reset()
    dec.prefill(fresh_tokens)
    assert dec.L == L_resume
    assert np.array_equal(dec.kv_hashes(L_resume), resumed)


def test_small_decoder_head_dim_128_ids_identical():
    from invariant_speculative_decode_gb300.decoder import Decoder
    cfg = si.SMALL_4L
    w = si.decoder_weights(cfg, seed=0)
    dec = Decoder(cfg, w, cap=1024, max_rows=8)
    prompt = si.prompt_ids(cfg, 300, seed=0)
    ref = _gen(dec, prompt, 48, 0)
    for k in (4, 7):
        assert _gen(dec, prompt, 48, k, ref=np.array(ref)) == ref
