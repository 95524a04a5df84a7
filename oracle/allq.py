"""Oracle for all-query ("heavy hitter") scoring, fp64 (numpy).

TEST INFRASTRUCTURE ONLY (see the package header).

A scoring variant: instead of the last W prompt queries (the observation
window), every prompt query votes -- the accumulated attention that H2O uses
to pick heavy hitters, the method the SnapKV summary compares against
(hotpaper.ai summary of "SnapKV: LLM Knows What You are Looking for Before
Generation", "주요 결과": LongBench against H2O).  For sequence b, KV head h
and prefix key j < P = L - W:

    raw[j] = (1/g) sum_{hq in group h} sum_{i = j}^{L-1} softmax_{j' <= i}(q_i . k_j' / sqrt(d))[j]

(every query row i is normalised over the keys it sees, j' <= i).  Pooling,
selection of the C - W best prefix positions and the window rows are as in
the plain compression; L <= C keeps everything.
"""
from __future__ import annotations

import numpy as np

from .decode import _f64


def scores_all_queries(q_all, k, seqlens, W: int):
    """q_all [T, H_q, d], k [T, H_kv, d] (packed); returns per sequence an
    [H_kv, P_b] array (None when P_b < 1)."""
    q_all, k = _f64(np.asarray(q_all)), _f64(np.asarray(k))
    T, H_q, d = q_all.shape
    H_kv = k.shape[1]
    g = H_q // H_kv
    out, off = [], 0
    for L in seqlens:
        L = int(L)
        P = L - W
        if P < 1:
            out.append(None)
            off += L
            continue
        raw = np.zeros((H_kv, P))
        visible = np.tril(np.ones((L, L), dtype=bool))  # row i sees keys j <= i
        for hq in range(H_q):
            h = hq // g
            s = q_all[off:off + L, hq] @ k[off:off + L, h].T / np.sqrt(d)  # [i, j]
            s = np.where(visible, s, -np.inf)
            p = np.exp(s - s.max(axis=1, keepdims=True))
            p /= p.sum(axis=1, keepdims=True)
            raw[h] += p[:, :P].sum(axis=0)
        out.append(raw / g)
        off += L
    return out


def compress_all_queries(q_all, k, v, seqlens, W: int, k_pool: int, pool_type, C: int):
    """The plain compression with all-query scores: idx [B, H_kv, C],
    out_k / out_v [B, C, H_kv, d], raw / pooled per sequence, tau [B, H_kv]."""
    from . import pool, select

    k = np.asarray(k)
    v = np.asarray(v)
    B, H_kv, d = len(seqlens), k.shape[1], k.shape[2]
    raws = scores_all_queries(q_all, k, seqlens, W)
    idx = np.full((B, H_kv, C), -1, np.int32)
    tau = np.full((B, H_kv), np.nan)
    pooleds = []
    offs = np.concatenate([[0], np.cumsum([int(L) for L in seqlens])])
    for b, L in enumerate(seqlens):
        L = int(L)
        P, n = L - W, C - W
        pb = None if raws[b] is None else np.stack([pool(raws[b][h], k_pool, pool_type)
                                                     for h in range(H_kv)])
        pooleds.append(pb)
        for h in range(H_kv):
            if L <= C:
                idx[b, h, :L] = np.arange(L)
            else:
                sel, t = select(pb[h], n)
                idx[b, h, :n] = sel
                idx[b, h, n:] = np.arange(P, L)
                tau[b, h] = t
    out_k = np.zeros((B, C, H_kv, d), k.dtype)
    out_v = np.zeros((B, C, H_kv, d), v.dtype)
    for b in range(B):
        for h in range(H_kv):
            keep = idx[b, h] >= 0
            rows = offs[b] + idx[b, h][keep]
            out_k[b, keep, h] = k[rows, h]
            out_v[b, keep, h] = v[rows, h]
    return dict(raw=raws, pooled=pooleds, tau=tau, idx=idx, out_k=out_k, out_v=out_v)
