"""Pins of the Scissorhands eviction oracle (oracle/scissorhands.py), on the CPU.

Each pin fixes the oracle against something other than its own code:
* a closed form: uniform attention leaves every count at zero, so eviction
  reduces to a sliding window over the most recent tokens;
* a worked example by hand, where the history window w alone decides which
  tokens survive;
* brute force: every eviction is re-derived from a separately kept history of
  softmax weights (scipy), keyed by token position;
* the attention output against the pinned decode oracle, and the cache
  size against its closed-form recurrence.
"""
import numpy as np
import pytest
from scipy.special import softmax

import oracle
from oracle.scissorhands import Params, ScissorhandsCache


def _prefix(seed, B, C0, H_kv, d, lens0):
    rng = np.random.default_rng(seed)
    k0 = rng.standard_normal((B, C0, H_kv, d))
    v0 = rng.standard_normal((B, C0, H_kv, d))
    pos0 = np.zeros((B, H_kv, C0), dtype=np.int64)
    for b in range(B):
        for h in range(H_kv):  # each head kept its own prompt tokens
            pos0[b, h] = np.sort(rng.choice(10 * C0, size=C0, replace=False))
    return k0, v0, pos0


def _n_after(n, p):
    n += 1
    return n - p.evict if n > p.budget else n


@pytest.mark.parametrize("g", [1, 2, 4])
def test_uniform_attention_is_a_sliding_window(g):
    """q = 0: every weight is exactly 1/n, no token is ever below average, all
    counts tie at 0 and each batch evicts the m oldest -- the cache is always
    the last n tokens to arrive, and the output the mean of their values."""
    p = Params(budget=12, recent=3, history=5, evict=6)
    B, H_kv, d, lens0 = 2, 2, 8, [5, 12]
    k0, v0, pos0 = _prefix(1, B, 12, H_kv, d, lens0)
    c = ScissorhandsCache.from_prefix(p, H_kv * g, k0, v0, pos0, lens0, [1000, 2000])
    stream = [[list(pos0[b, h, :lens0[b]]) for h in range(H_kv)] for b in range(B)]
    n = list(lens0)
    rng = np.random.default_rng(2)
    for t in range(40):
        kn, vn = rng.standard_normal((B, H_kv, d)), rng.standard_normal((B, H_kv, d))
        o, ratio = c.step(np.zeros((B, H_kv * g, d)), kn, vn)
        for b in range(B):
            n[b] = _n_after(n[b], p)
            assert c.n(b) == n[b]
            np.testing.assert_array_equal(ratio[b], np.ones((H_kv, n[b])))
            K, V = c.rows(b)
            for h in range(H_kv):
                stream[b][h].append((1000, 2000)[b] + t)
                assert c.positions(b, h) == stream[b][h][-n[b]:]
                for x in range(g):
                    np.testing.assert_allclose(o[b, h * g + x], V[:, h].mean(0), rtol=1e-12,
                                               atol=1e-12)


def _hand_cache(w):
    """One head, d = 2.  Keys: A = (10, 0), D = (-10, 0), B = C = E = F = (0, 10).
    Queries (10, 0) and (-10, 0) put all weight (1 - e^-70) on A or D."""
    p = Params(budget=3, recent=1, history=w, evict=2)
    k0 = np.array([[[[10.0, 0.0]], [[0.0, 10.0]]]])  # A, B: [B=1, C0=2, H_kv=1, d=2]
    v0 = np.arange(4.0).reshape(1, 2, 1, 2)
    c = ScissorhandsCache.from_prefix(p, 1, k0, v0, np.array([[[0, 1]]]), [2], [2])
    steps = [  # (query, new key) for tokens C(2), D(3), E(4), F(5)
        ((10.0, 0.0), (0.0, 10.0)),    # t=0: cache A B C, weight on A -> B, C below
        ((-10.0, 0.0), (-10.0, 0.0)),  # t=1: + D = 4 rows -> evict 2 of A, B, C
        ((10.0, 0.0), (0.0, 10.0)),    # t=2: A D E, weight on A -> D, E below
        ((10.0, 0.0), (0.0, 10.0)),    # t=3: + F = 4 rows -> evict 2 of A, D, E
    ]
    kept = []
    for qv, kv in steps:
        c.step(np.array([[qv]]), np.array([[kv]]), np.zeros((1, 1, 2)))
        kept.append(c.positions(0, 0))
    return kept


def test_hand_example_history_window():
    # t=1, any w >= 1: counts over step 0 are A 0, B 1, C 1 -> B, C go.
    # At t=1 the weight sits on D, so A is below average at step 1.
    # t=3, w = 1: window = {2}: A 0, D 1, E 1 -> D and E go, A stays.
    # t=3, w = 2: window = {1, 2}: A 1, D 1, E 1 -> a tie; the two oldest (A, D) go.
    assert _hand_cache(1) == [[0, 1, 2], [0, 3], [0, 3, 4], [0, 5]]
    assert _hand_cache(2) == [[0, 1, 2], [0, 3], [0, 3, 4], [4, 5]]
    assert _hand_cache(3)[-1] == [4, 5]


@pytest.mark.parametrize("seed,g,p", [
    (3, 1, Params(budget=16, recent=4, history=6, evict=8)),
    (4, 4, Params(budget=10, recent=2, history=3, evict=5)),
    (5, 2, Params(budget=9, recent=9, history=20, evict=1)),   # r = budget: the oldest token goes
    (6, 8, Params(budget=24, recent=1, history=50, evict=24)),  # evict everything but the newest
])
def test_evictions_match_brute_force(seed, g, p):
    """Random keys and queries; a brute-force history of scipy softmax weights
    keyed by token position re-derives every eviction (top-m counts over the
    last w steps, ties to the older token, the r most recent exempt) and the
    oracle's output is compared with the pinned decode oracle."""
    B, H_kv, d = 2, 2, 16
    H_q = H_kv * g
    lens0 = [p.budget // 2, p.budget]
    k0, v0, pos0 = _prefix(seed, B, p.budget, H_kv, d, lens0)
    c = ScissorhandsCache.from_prefix(p, H_q, k0, v0, pos0, lens0, [500, 600])
    rng = np.random.default_rng(seed + 100)
    low = {}  # (b, h, position) -> steps below average, from scipy weights
    for t in range(3 * p.budget):
        before = [[c.positions(b, h) for h in range(H_kv)] for b in range(B)]
        q = 3.0 * rng.standard_normal((B, H_q, d))
        kn, vn = rng.standard_normal((B, H_kv, d)), rng.standard_normal((B, H_kv, d))
        o, _ = c.step(q, kn, vn)
        for b in range(B):
            K, V = c.rows(b)
            n = K.shape[0]
            assert n <= p.budget
            np.testing.assert_allclose(o[b], oracle.decode_attention(q[b:b + 1], [K], [V])[0],
                                       rtol=1e-11, atol=1e-12)
            for h in range(H_kv):
                arrived = before[b][h] + [(500, 600)[b] + t]
                now = c.positions(b, h)
                if len(arrived) > p.budget:
                    cand = arrived[:len(arrived) - p.recent]
                    cnt = {x: sum(1 for s in low.get((b, h, x), []) if t - p.history <= s < t)
                           for x in cand}
                    want_gone = sorted(cand, key=lambda x: (-cnt[x], arrived.index(x)))[:p.evict]
                    assert now == [x for x in arrived if x not in want_gone]
                else:
                    assert now == arrived
                w = softmax(K[:, h] @ q[b, h * g:(h + 1) * g].T / np.sqrt(d), axis=0).mean(1)
                for j, x in enumerate(now):
                    if w[j] < 1.0 / n:
                        low.setdefault((b, h, x), []).append(t)
                assert now[-p.recent:] == arrived[-p.recent:]  # recent tokens stay


def test_dominant_token_survives_every_eviction():
    """A key aligned with a fixed query takes nearly all the weight, is never
    below average and keeps a zero count, while every other token is below
    average from its first step on.  (The cache starts below budget: at an
    eviction with no history yet every count is zero and the oldest go.)"""
    p = Params(budget=32, recent=4, history=10, evict=16)
    B, H_kv, g, d = 1, 2, 4, 32
    k0, v0, pos0 = _prefix(7, B, 32, H_kv, d, [8])
    qdir = np.random.default_rng(8).standard_normal(d)
    qdir /= np.linalg.norm(qdir)
    k0[0, 5, 1] = 40.0 * qdir  # head 1's sixth prompt token
    planted = pos0[0, 1, 5]
    c = ScissorhandsCache.from_prefix(p, H_kv * g, k0, v0, pos0, [8], [400])
    rng = np.random.default_rng(9)
    for _ in range(120):  # 6 evictions, the first at step 24
        q = np.broadcast_to(4.0 * qdir, (B, H_kv * g, d)).copy()
        c.step(q, rng.standard_normal((B, H_kv, d)), rng.standard_normal((B, H_kv, d)))
        assert planted in c.positions(0, 1)
    assert all(x >= 400 for x in c.positions(0, 0))  # head 0 had nothing to protect


def test_cache_size_recurrence():
    p = Params(budget=7, recent=2, history=4, evict=3)
    k0, v0, pos0 = _prefix(10, 3, 7, 1, 4, [0, 3, 7])
    c = ScissorhandsCache.from_prefix(p, 2, k0, v0, pos0, [0, 3, 7], [0, 3, 7])
    n = [0, 3, 7]
    rng = np.random.default_rng(11)
    for _ in range(25):
        c.step(rng.standard_normal((3, 2, 4)), rng.standard_normal((3, 1, 4)),
               rng.standard_normal((3, 1, 4)))
        n = [_n_after(x, p) for x in n]
        assert [c.n(b) for b in range(3)] == n
        assert all(1 <= x <= p.budget for x in n)


@pytest.mark.parametrize("kw", [
    dict(budget=0, recent=1, history=1, evict=1),
    dict(budget=8, recent=0, history=1, evict=1),
    dict(budget=8, recent=9, history=1, evict=1),
    dict(budget=8, recent=2, history=0, evict=1),
    dict(budget=8, recent=2, history=4, evict=8),   # > budget + 1 - recent
    dict(budget=8, recent=2, history=4, evict=0),
])
def test_parameter_checks(kw):
    with pytest.raises(ValueError):
        Params(**kw).check()
