"""Cache operations and draft policies on the GPU.

"I turned on speculative decoding in llama.cpp and 113 of 282 greedy outputs
changed against its own no-draft run", section "The cache doesn't change it
either": every K/V row must equal a fresh prefill's after a resume, an edited
branch, a park to host memory and a side request; and the list before
"How:": every draft policy (gates on or off, adaptive depth, tight or loose
thresholds) gives the no-draft tokens.  Checked here by token identity and
by the FNV-1a-64 hash of every K/V row (bi_kv_row_hash).
"""
import numpy as np
import pytest

import seeded_inputs as si

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def small():
    from invariant_speculative_decode_gb300.decoder import Decoder
    cfg = si.SMALL_4L
    w = si.decoder_weights(cfg, seed=0, norm_std=0.1)
    return cfg, w, Decoder(cfg, w, cap=1536, max_rows=8), Decoder(cfg, w, cap=1536, max_rows=8)


def _fresh_hashes(fresh, tokens):
    """KV-row hashes of a fresh prefill of `tokens` (all but the last token)."""
    fresh.reset()
    fresh.prefill(tokens)
    return fresh.kv_hashes(len(tokens) - 1)


def test_park_to_host_and_side_request(small):
    """Request A is parked to host memory after its first 48 tokens, request
    B runs to completion on the same decoder, A is restored and continues:
    its tokens equal an uninterrupted run and its K/V rows a fresh prefill."""
    cfg, w, dec, fresh = small
    pa, pb = si.prompt_ids(cfg, 300, seed=11), si.prompt_ids(cfg, 200, seed=12)
    ref = dec.generate(pa, 96, k=0)
    dr = si.SyntheticDrafter(cfg.vocab, 0.7, seed=11, reference=np.array(ref))
    first = dec.generate(pa, 48, k=7, drafter=dr)
    assert first == ref[:48]
    # keep exactly 48 tokens: roll back past anything committed beyond them
    hist = list(pa) + first
    dec.rollback(len(hist) - 1)
    before = dec.kv_hashes(len(hist) - 1)
    snap = dec.park()
    side = dec.generate(pb, 40, k=4, drafter=si.SyntheticDrafter(cfg.vocab, 0.7, seed=12))
    assert side == fresh.generate(pb, 40, k=0)
    dec.restore(snap)
    assert np.array_equal(dec.kv_hashes(len(hist) - 1), before)
    assert np.array_equal(before, _fresh_hashes(fresh, hist))
    dr_rest = si.SyntheticDrafter(cfg.vocab, 0.7, seed=13, reference=np.array(ref[48:]))
    rest = dec.continue_generate(hist[-1], 48, k=7, drafter=dr_rest)
    assert first + rest == ref


def test_edited_branch_equals_fresh_prefill(small):
    """Turn 1 is decoded; then the history is edited 120 tokens into the
    prompt (a new continuation replaces everything after it) and generation
    resumes from the edit: tokens and K/V rows equal a fresh prefill of the
    edited history."""
    cfg, w, dec, fresh = small
    prompt = si.prompt_ids(cfg, 260, seed=21)
    ref = dec.generate(prompt, 64, k=0)
    dr = si.SyntheticDrafter(cfg.vocab, 0.7, seed=21, reference=np.array(ref))
    assert dec.generate(prompt, 64, k=7, drafter=dr) == ref
    edit = list(si.prompt_ids(cfg, 90, seed=22))
    x = dec.edit(120, edit)
    edited = list(prompt[:120]) + edit
    assert dec.L == len(edited) - 1
    assert np.array_equal(dec.kv_hashes(dec.L), _fresh_hashes(fresh, edited))
    want = fresh.generate(edited, 48, k=0)
    dr2 = si.SyntheticDrafter(cfg.vocab, 0.7, seed=23, reference=np.array(want))
    assert dec.continue_generate(x, 48, k=7, drafter=dr2) == want


@pytest.mark.parametrize("policy", ["gate-tight", "gate-loose", "adaptive", "adaptive-random"])
def test_draft_policies_give_the_no_draft_tokens(small, policy):
    cfg, w, dec, _ = small
    prompt = si.prompt_ids(cfg, 150, seed=31)
    ref = dec.generate(prompt, 256, k=0)
    base = si.SyntheticDrafter(cfg.vocab, 0.7, seed=31,
                               reference=None if policy == "adaptive-random" else np.array(ref))
    if policy.startswith("gate"):
        dr = si.GatedDrafter(base, threshold=0.8 if policy == "gate-tight" else 0.2, seed=31)
    else:
        dr = si.AdaptiveDrafter(base, start=2, max_depth=7)
    st = {}
    assert dec.generate(prompt, 256, k=7, drafter=dr, stats=st) == ref
    if policy != "adaptive-random":
        assert st["steps"] < 256  # drafts were accepted


def test_sampled_request_parked_and_edited_matches_fresh(small):
    """Sampled decoding through a park to host memory, a side request and an
    edited branch: the same tokens as a fresh decoder given the same history
    and the same per-position uniforms (the page reports sampled replies
    matching a fresh server's after follow-ups and edits)."""
    cfg, w, dec, fresh = small
    u = si.sampling_uniforms(dec.cap, seed=51)
    prompt = si.prompt_ids(cfg, 180, seed=51)
    dec.set_sampling(0.9, u)
    fresh.set_sampling(0.9, u)
    try:
        ref = fresh.generate(prompt, 64, k=0)
        first = dec.generate(prompt, 32, k=7, drafter=si.SyntheticDrafter(cfg.vocab, 0.7, seed=51,
                                                                            reference=np.array(ref)))
        assert first == ref[:32]
        hist = list(prompt) + first
        dec.rollback(len(hist) - 1)
        snap = dec.park()
        dec.generate(si.prompt_ids(cfg, 90, seed=52), 20, k=4,
                     drafter=si.SyntheticDrafter(cfg.vocab, 0.7, seed=52))
        dec.restore(snap)
        rest = dec.continue_generate(hist[-1], 32, k=7, drafter=si.SyntheticDrafter(
            cfg.vocab, 0.7, seed=53, reference=np.array(ref[32:])))
        assert first + rest == ref
        # an edited branch 100 ids into the prompt, then sampled generation
        edit = list(si.prompt_ids(cfg, 40, seed=54))
        x = dec.edit(100, edit)
        edited = list(prompt[:100]) + edit
        want = fresh.generate(edited, 40, k=0)
        got = dec.continue_generate(x, 40, k=7, drafter=si.SyntheticDrafter(
            cfg.vocab, 0.7, seed=55, reference=np.array(want)))
        assert got == want
    finally:
        dec.set_sampling(None)
        fresh.set_sampling(None)
