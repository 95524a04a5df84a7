"""Oracle for Scissorhands decode-time KV-cache eviction (fp64, numpy).

TEST INFRASTRUCTURE ONLY (see the package header).

What it computes follows the abeam.tech summary of "Scissorhands: Exploiting
the Persistence of Importance Hypothesis for LLM KV Cache Compression at Test
Time", section 技術の仕組み:

* "注意の偏りと持続性を利用する": the attention output at decode step t is
  the alpha(t, i)-weighted mean of the cached values; tokens that were
  attended little so far matter little later (persistence of importance).
* "固定予算で残すトークンを選ぶ": every attention head keeps a budget of
  tokens.  When the new token's key and value push the cache past the budget,
  the attention weights of the last w steps are consulted: the more often a
  token's weight was below the average weight, the stronger a candidate for
  deletion it is.  The r most recent tokens are always kept (the page's runs
  use w = 400, r = 10).  Attention then runs over the rows that remain.
* "層ごと・ヘッドごとの予算配分": eviction is batched -- the page's setting
  drops an amount equal to half the budget at once -- and budgets may differ
  per layer (one cache object per layer here, each with its own budget).

Readings where the page leaves a step open (each restated where it is used):

R1  The average weight of a softmax row over n cached tokens is 1/n (the
    weights sum to 1); "below average" is strict: alpha < 1/n.
R2  With grouped-query attention a KV head serves g query heads; a token's
    weight for the KV head is the mean over those g heads (the same GQA mean
    the prefill scoring takes).  Decided as sum_x n * e_x / Z_x < g, with
    e_x = exp(s_x - max_x) and Z_x its row sum -- the same inequality written
    without the division by n, so that uniform attention (every e = 1, Z = n)
    decides "not below" exactly.
R3  The append comes first; if the cache then holds budget + 1 rows, m of
    them are evicted before the step's attention, which therefore always
    runs over at most `budget` rows.
R4  A token's count at an eviction during step t is the number of steps
    s in [t - w, t - 1] at which it was cached and below average.
R5  Candidates are all but the r most recent tokens; the m with the largest
    counts go, equal counts evicting the older token (earlier arrival) first.
R6  The kept tokens stay in arrival order; the new token's position is the
    next position of its sequence.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from .decode import _f64


@dataclass
class Params:
    budget: int   # tokens per head once the cache is full
    recent: int   # r: the most recent tokens, never evicted
    history: int  # w: decode steps a token's count looks back over
    evict: int    # m: tokens evicted per head in one batch

    def check(self):
        if not (self.budget >= 1 and 1 <= self.recent <= self.budget and self.history >= 1):
            raise ValueError("need budget >= 1, 1 <= recent <= budget, history >= 1")
        if not (1 <= self.evict <= self.budget + 1 - self.recent):
            raise ValueError("need 1 <= evict <= budget + 1 - recent")


@dataclass
class Token:
    pos: int
    k: np.ndarray              # [d] fp64
    v: np.ndarray              # [d] fp64
    low: list = field(default_factory=list)  # decode steps at which it was below average


class ScissorhandsCache:
    """One layer's cache: for every sequence b and KV head h an arrival-ordered
    list of tokens.  All heads of a sequence hold the same number of tokens
    (each step appends one to every head and each eviction removes m from
    every head), not the same tokens."""

    def __init__(self, params: Params, H_q: int, heads):
        params.check()
        self.p = params
        self.H_q = H_q
        self.heads = heads              # heads[b][h] -> list[Token]
        self.H_kv = len(heads[0])
        self.g = H_q // self.H_kv
        self.steps = [0] * len(heads)
        self.next_pos = [0] * len(heads)

    @classmethod
    def from_prefix(cls, params, H_q, k0, v0, pos0, lens0, next_pos0):
        """k0, v0 [B, C0, H_kv, d] (row s of head h is that head's s-th token),
        pos0 [B, H_kv, C0] positions, lens0[b] <= budget rows in use."""
        k0, v0 = _f64(np.asarray(k0)), _f64(np.asarray(v0))
        B, _, H_kv, _ = k0.shape
        if any(n > params.budget for n in lens0):
            raise ValueError("initial cache above budget")
        heads = [[[Token(int(pos0[b, h, s]), k0[b, s, h].copy(), v0[b, s, h].copy())
                   for s in range(lens0[b])] for h in range(H_kv)] for b in range(B)]
        c = cls(params, H_q, heads)
        c.next_pos = [int(x) for x in next_pos0]
        return c

    def n(self, b: int) -> int:
        return len(self.heads[b][0])

    # R4, R5: the batch eviction of one head
    def _evict(self, toks: list, t: int) -> list:
        p = self.p
        cand = len(toks) - p.recent
        lo = t - p.history
        counts = [sum(1 for s in tok.low if lo <= s <= t - 1) for tok in toks[:cand]]
        order = sorted(range(cand), key=lambda j: (-counts[j], j))
        gone = set(order[:p.evict])
        return [tok for j, tok in enumerate(toks) if j not in gone]

    def step(self, q, k_new, v_new):
        """One decode step: append, evict if over budget, attend, record the
        below-average tokens.  q [B, H_q, d]; k_new, v_new [B, H_kv, d].
        Returns (o [B, H_q, d], ratio) with ratio[b] [H_kv, n_b]: n_b times the
        group-mean weight of every cached token (below average iff < 1)."""
        q, k_new, v_new = _f64(np.asarray(q)), _f64(np.asarray(k_new)), _f64(np.asarray(v_new))
        B, _, d = q.shape
        out = np.zeros((B, self.H_q, d))
        ratio = []
        for b in range(B):
            t = self.steps[b]
            for h in range(self.H_kv):  # R3, R6
                self.heads[b][h].append(Token(self.next_pos[b], k_new[b, h].copy(),
                                              v_new[b, h].copy()))
            self.next_pos[b] += 1
            if self.n(b) > self.p.budget:
                for h in range(self.H_kv):
                    self.heads[b][h] = self._evict(self.heads[b][h], t)
            n = self.n(b)
            rb = np.zeros((self.H_kv, n))
            for h in range(self.H_kv):
                toks = self.heads[b][h]
                K = np.stack([tok.k for tok in toks])
                V = np.stack([tok.v for tok in toks])
                rel = np.zeros(n)  # sum over the group of n * e / Z (R1, R2)
                for x in range(self.g):
                    hq = h * self.g + x
                    s = K @ q[b, hq] / np.sqrt(d)
                    e = np.exp(s - s.max())
                    Z = e.sum()
                    out[b, hq] = (e / Z) @ V
                    rel += n * e / Z
                for j, tok in enumerate(toks):
                    if rel[j] < self.g:
                        tok.low.append(t)
                rb[h] = rel / self.g
            ratio.append(rb)
            self.steps[b] = t + 1
        return out, ratio

    def positions(self, b: int, h: int) -> list:
        return [tok.pos for tok in self.heads[b][h]]

    def rows(self, b: int):
        """The cached rows of sequence b as [n_b, H_kv, d] arrays (K, V)."""
        K = np.stack([np.stack([tok.k for tok in self.heads[b][h]]) for h in range(self.H_kv)], 1)
        V = np.stack([np.stack([tok.v for tok in self.heads[b][h]]) for h in range(self.H_kv)], 1)
        return K, V
