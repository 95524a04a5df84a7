"""Pins of the all-query scoring oracle (oracle/allq.py) on the CPU."""
import numpy as np
import torch

import oracle
import synth


def test_zero_queries_closed_form():
    """q = 0: row i is uniform over its i + 1 keys, so
    raw[j] = sum_{i=j}^{L-1} 1 / (i + 1) for every head."""
    W, L = 8, 100
    lay = synth.make_inputs(5, [L], 8, 2, 64, W, "fp32", nspans=1)
    q = np.zeros((L, 8, 64), np.float32)
    raw = oracle.scores_all_queries(q, lay.k, [L], W)[0]
    want = np.array([np.sum(1.0 / np.arange(j + 1, L + 1)) for j in range(L - W)])
    for h in range(2):
        np.testing.assert_allclose(raw[h], want, rtol=1e-13)


def test_window_rows_part_is_the_window_score():
    """The rows of the observation window contribute exactly the plain
    (window) score of the C oracle; the earlier rows add their causal softmax
    mass, computed here with torch's softmax."""
    W, L, H_q, H_kv, d = 16, 200, 8, 2, 64
    g = H_q // H_kv
    rng = np.random.default_rng(9)
    q_all = rng.standard_normal((L, H_q, d)).astype(np.float32)
    k = rng.standard_normal((L, H_kv, d)).astype(np.float32)
    v = rng.standard_normal((L, H_kv, d)).astype(np.float32)
    P = L - W
    allq = oracle.scores_all_queries(q_all, k, [L], W)[0]
    win = oracle.compress(q_all[None, P:], k, v, [L], W, 1, "avg", 64)["raw"][0]
    mask = torch.ones(L, L, dtype=torch.bool).tril()
    for h in range(H_kv):
        early = np.zeros(P)
        for m in range(g):
            Q = torch.from_numpy(q_all[:P, h * g + m].astype(np.float64))
            K = torch.from_numpy(k[:, h].astype(np.float64))
            s = (Q @ K.T / np.sqrt(d)).masked_fill(~mask[:P], float("-inf"))
            early += torch.softmax(s, dim=1)[:, :P].sum(0).numpy()
        np.testing.assert_allclose(allq[h], np.asarray(win[h]) + early / g, rtol=1e-11,
                                   atol=1e-14)


def test_compress_all_queries_keeps_window_and_orders():
    lay = synth.make_inputs(6, [300, 50], 4, 2, 64, 16, "bf16", nspans=2)
    q_all = synth.bf16_round(np.random.default_rng(1).standard_normal(
        (350, 4, 64)).astype(np.float32))
    C = 64
    out = oracle.compress_all_queries(q_all, lay.k, lay.v, lay.seqlens, lay.W, 5, "avg", C)
    idx = out["idx"]
    n = C - lay.W
    for h in range(2):
        assert idx[0, h, n:].tolist() == list(range(284, 300))
        assert (np.diff(idx[0, h, :n]) > 0).all()
        assert idx[1, h].tolist() == list(range(50)) + [-1] * 14
