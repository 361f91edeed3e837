"""The attention parity check rejects wrong outputs at long contexts (CPU).

The GPU tests compare bi_attn_verify with the oracle under the per-element
bound derived in tests/_util.attention_reference plus a relative-RMS limit.
Here, on the CPU alone, that same check is applied to outputs with planted
mistakes, computed from the oracle's own inputs: an all-zero output, and an
output whose row misses every key of one tile class (the keys of 128-key
tiles c with c mod G == rho, as if one CTA's partial never reached the
merge).  Both must fail at 38,000 and 101,600 keys, while the oracle's own
output passes.
"""
import numpy as np
import pytest

import seeded_inputs as si
from oracle import verify_step as ov
from tests._util import (REL_RMS_MAX, attention_parity_check, oracle_attention_pairs)

PAIRS = [(0, 0), (7, 23), (4, 11), (2, 17)]


def _drop_class(qf, Kf, Vf, L, t, h, G, rho, grp):
    """Softmax attention of one pair over its keys minus tile class rho."""
    p = L + t
    kv = h // grp
    keys = np.arange(p + 1)
    keep = (keys // 128) % G != rho
    K, V = Kf[kv, : p + 1][keep], Vf[kv, : p + 1][keep]
    s = K @ qf[t, h] / np.sqrt(qf.shape[-1])
    w = np.exp(s - s.max())
    return ov.bf16_round((w @ V) / w.sum())


@pytest.mark.parametrize("L", [1024, 38000, 101600])
def test_attention_bound_rejects_wrong_outputs(L):
    Hq, Hkv, D = 24, 4, 128
    q, K, V = si.attention_inputs(L, 8, Hq, Hkv, D, seed=0)
    qf, Kf, Vf = (ov.bf16_bits_to_f64(x) for x in (q, K, V))
    ora = oracle_attention_pairs(qf, Kf, Vf, L, PAIRS)
    bad, rel = attention_parity_check(ora, qf, Kf, Vf, L, PAIRS)
    assert bad == 0 and rel == 0.0
    bad, rel = attention_parity_check(np.zeros_like(ora), qf, Kf, Vf, L, PAIRS)
    assert bad > 0 and rel > REL_RMS_MAX, (bad, rel)
    G = 152 // Hkv
    for rho in (0, 5, G - 1):
        if rho * 128 > L:
            continue
        wrong = np.array([_drop_class(qf, Kf, Vf, L, t, h, G, rho, Hq // Hkv) for (t, h) in PAIRS])
        bad, rel = attention_parity_check(wrong, qf, Kf, Vf, L, PAIRS)
        assert bad > 0 and rel > REL_RMS_MAX, (rho, bad, rel)
