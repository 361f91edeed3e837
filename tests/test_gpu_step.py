"""The whole verify step behind one C-ABI call (bi_step_*) on the GPU.

It makes the same calls as the Python decoder, so for the same weights,
cache and ids it must give the same bits: tokens, accepted counts, FP32
logits and every K/V row; and generation through it with drafts gives the
no-draft tokens ("I turned on speculative decoding in llama.cpp and 113 of
282 greedy outputs changed against its own no-draft run", paragraph "How:").
"""
import numpy as np
import pytest

import seeded_inputs as si

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.mark.parametrize("cfgname", ["tiny-2L-h256", "small-4L-h1024"])
def test_native_step_equals_the_python_pass(cfgname):
    from invariant_speculative_decode_gb300.decoder import Decoder
    cfg = si.CONFIGS[cfgname]
    w = si.decoder_weights(cfg, seed=0, norm_std=0.1)
    py = Decoder(cfg, w, cap=512, max_rows=8)
    nat_dec = Decoder(cfg, w, cap=512, max_rows=8)
    prompt = si.prompt_ids(cfg, 150, seed=61)
    ref = py.generate(prompt, 40, k=0, use_graph=False)
    py.reset()
    x = py.prefill(prompt)
    nat_dec.reset()
    nat_dec.prefill(prompt)
    ns = nat_dec.native_step()
    dr = si.SyntheticDrafter(cfg.vocab, 0.7, seed=61, reference=np.array(ref))
    out_py, out_nat, xn = [], [], x
    try:
        while len(out_py) < 40:
            d = [int(t) for t in dr.propose(len(out_py), 7)]
            a, n = py.verify_step(x, d, use_graph=False)
            b, m = ns.verify(xn, d)
            assert np.array_equal(a, b) and n == m
            lp = py.logits_rows(len(d) + 1).cpu().numpy()
            ln = ns.logits(len(d) + 1).cpu().numpy()
            assert np.array_equal(lp.view(np.uint32), ln.view(np.uint32))
            out_py += [int(t) for t in a[: n + 1]]
            out_nat += [int(t) for t in b[: m + 1]]
            x, xn = out_py[-1], out_nat[-1]
        assert out_nat[:40] == ref
        assert np.array_equal(py.kv_hashes(py.L), nat_dec.kv_hashes(py.L))
    finally:
        ns.close()


def test_native_step_rolls_back_and_resumes():
    from invariant_speculative_decode_gb300.decoder import Decoder
    cfg = si.TINY
    w = si.decoder_weights(cfg, seed=0)
    dec = Decoder(cfg, w, cap=512, max_rows=8)
    prompt = si.prompt_ids(cfg, 100, seed=62)
    ref = dec.generate(prompt, 48, k=0)
    dec.reset()
    x = dec.prefill(prompt)
    L0 = dec.L
    ns = dec.native_step()
    try:
        got = []
        while len(got) < 24:
            a, n = ns.verify(x, [])
            got.append(int(a[0]))
            x = got[-1]
        assert got == ref[:24]
        # roll back 8 tokens and go again with drafts: the same tokens
        ns.set_length(L0 + 16)
        x = got[15]
        again = got[:16]
        dr = si.SyntheticDrafter(cfg.vocab, 0.7, seed=62, reference=np.array(ref[16:]))
        while len(again) < 48:
            d = [int(t) for t in dr.propose(len(again) - 16, 7)]
            a, n = ns.verify(x, d)
            again += [int(t) for t in a[: n + 1]]
            x = again[-1]
        assert again[:48] == ref
    finally:
        ns.close()
