"""Oracle for one decode step of attention over a KV cache (fp64, numpy).

TEST INFRASTRUCTURE ONLY (see the package header).

After compression the generation (decode) phase attends over the compressed
cache instead of the full one (jisaku.com glossary "SnapKV", "SnapKVの仕組み",
algorithm flow step 4); the smaller cache relieves the memory-bandwidth bound
of decoding (glossary FAQ Q2; hotpaper.ai summary of "SnapKV: LLM Knows What
You are Looking for Before Generation", "주요 결과": 3.6x generation speed at
16K input).  What one decode step computes for sequence b and query head hq,
with KV head h = hq // g serving the g query heads of its group:

    o[b, hq] = sum_j softmax_j(q[b, hq] . k[b, j, h] / sqrt(d)) v[b, j, h]

over the n_b cached rows j of the sequence (no mask: a decode query sees
every cached row).  The caller appends the new token's own key and value to
the cache if it wants them attended.
"""
from __future__ import annotations

import numpy as np


def _f64(a: np.ndarray) -> np.ndarray:
    if a.dtype == np.uint16:  # bf16 bit patterns, widened exactly
        return (a.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def decode_attention(q: np.ndarray, k_rows, v_rows) -> np.ndarray:
    """q [B, H_q, d]; k_rows / v_rows: per sequence b an array [n_b, H_kv, d]
    (its cached rows, n_b >= 1).  Returns o [B, H_q, d] in fp64."""
    q = _f64(q)
    B, H_q, d = q.shape
    out = np.zeros((B, H_q, d))
    for b in range(B):
        K = _f64(np.asarray(k_rows[b]))
        V = _f64(np.asarray(v_rows[b]))
        H_kv = K.shape[1]
        g = H_q // H_kv
        for hq in range(H_q):
            h = hq // g
            s = K[:, h, :] @ q[b, hq] / np.sqrt(d)  # [n_b]
            p = np.exp(s - s.max())
            p /= p.sum()
            out[b, hq] = p @ V[:, h, :]
    return out
