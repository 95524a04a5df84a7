"""The LSE input of snapkv_compress_with_lse, pinned on the CPU.

tests/parity.window_lse computes the window rows' log-sum-exp that the
LSE-input entry points take.  Its definition is checked here against the
oracle: summing exp(logit - lse) over the window rows and averaging over the
query heads of each KV group must reproduce the oracle's raw scores (the
window attention scores of jisaku.com glossary "SnapKV", "SnapKVの仕組み"),
and each row's probabilities over its visible keys must add up to one.
"""
import numpy as np

import synth
from tests import parity


def _logits(lay, b, h):
    g = lay.H_q // lay.H_kv
    L = int(lay.seqlens[b])
    q = synth.bf16_to_f32(lay.q_win[b, :, h * g:(h + 1) * g]).astype(np.float64)
    k = synth.bf16_to_f32(lay.k[lay.offsets[b]:lay.offsets[b] + L, h]).astype(np.float64)
    return np.einsum("imd,jd->imj", q, k) / np.sqrt(lay.d)  # [W, g, L]


def test_window_lse_reproduces_oracle_raw_scores():
    W, C = 8, 64
    lay = synth.make_inputs(31, [300, 50, 129], 8, 2, 64, W, "bf16", nspans=2)
    lse = parity.window_lse(lay, C)
    ora = parity.oracle_for(lay, 3, "avg", C)
    g = lay.H_q // lay.H_kv
    for b, L in enumerate(lay.seqlens):
        L = int(L)
        if L <= C:
            assert np.isnan(lse[b]).all()
            continue
        P = L - W
        for h in range(lay.H_kv):
            s = _logits(lay, b, h)
            lse_bh = lse[b, :, h * g:(h + 1) * g].astype(np.float64)  # [W, g]
            vis = np.arange(L)[None, None, :] <= (P + np.arange(W))[:, None, None]
            p = np.where(vis, np.exp(s - lse_bh[:, :, None]), 0.0)
            np.testing.assert_allclose(p.sum(axis=2), 1.0, rtol=1e-6)
            raw = p[:, :, :P].sum(axis=(0, 1)) / g
            np.testing.assert_allclose(raw, ora["raw"][b][h], rtol=1e-6, atol=1e-12)


def test_window_lse_zero_queries_is_log_of_visible_count():
    """q = 0 makes every logit 0, so row i's LSE is log(P + i + 1)."""
    W, C = 16, 32
    lay = synth.make_inputs(3, [100, 20, 333], 8, 4, 128, W, "bf16", nspans=1)
    lay.q_win[:] = 0
    lse = parity.window_lse(lay, C)
    for b, L in enumerate(lay.seqlens):
        L = int(L)
        if L <= C:
            continue
        want = np.log(L - W + np.arange(W) + 1.0)
        np.testing.assert_allclose(lse[b], np.repeat(want[:, None], lay.H_q, axis=1), rtol=1e-7)
