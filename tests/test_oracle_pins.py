"""Pins of the CPU oracle against things other than itself.

Each test ties one part of the oracle to a closed form, a hand-derived value,
brute force with an independent library (torch fp64 full causal attention,
torch pooling, Python's sort) or an invariant of the mathematics, so that a
dropped term, a wrong sign, index, scale or mask fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import synth

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _ev(expr: str) -> float:
    return float(eval(expr, {"__builtins__": {}}, {"e": math.e}))


def _rand_layer(seed, seqlens, H_q, H_kv, d, W, dtype="fp32", scale=1.0):
    rng = np.random.default_rng(seed)
    T = int(sum(seqlens))
    q = (rng.standard_normal((len(seqlens), W, H_q, d)) * scale).astype(np.float32)
    k = rng.standard_normal((T, H_kv, d)).astype(np.float32)
    v = rng.standard_normal((T, H_kv, d)).astype(np.float32)
    if dtype == "bf16":
        return synth.bf16_round(q), synth.bf16_round(k), synth.bf16_round(v)
    return q, k, v


def _as_f64(a):
    return synth.bf16_to_f32(a).astype(np.float64) if a.dtype == np.uint16 else a.astype(np.float64)


# ---------------------------------------------------------------- scores ---

def _brute_force_raw(q_win, k, seqlens, W, b, h, seed=0):
    """Full L x L causal softmax attention in torch fp64, sliced and reduced.

    Builds a complete query matrix whose last W rows are the window queries
    (earlier rows are random and must not matter), repeats the KV head over
    its query group (kv head h serves query heads h*g .. h*g+g-1), takes the
    causal softmax of Q K^T / sqrt(d), keeps rows P..L-1 and columns < P,
    sums over rows and averages over the group.
    """
    q64 = torch.from_numpy(_as_f64(q_win))
    k64 = torch.from_numpy(_as_f64(k))
    B, _, H_q, d = q64.shape
    H_kv = k64.shape[1]
    g = H_q // H_kv
    off = int(sum(seqlens[:b]))
    L = int(seqlens[b])
    P = L - W
    gen = torch.Generator().manual_seed(seed)
    Q = torch.randn(L, H_q, d, generator=gen, dtype=torch.float64)
    Q[P:] = q64[b]
    Kx = k64[off:off + L].repeat_interleave(g, dim=1)  # [L, H_q, d]
    logits = torch.einsum("ihc,jhc->hij", Q, Kx) / math.sqrt(d)
    mask = torch.ones(L, L, dtype=torch.bool).triu(1)
    probs = torch.softmax(logits.masked_fill(mask, float("-inf")), dim=-1)
    grp = probs[h * g:(h + 1) * g, P:, :]          # [g, W, L]
    raw = grp[:, :, :P].sum(dim=(0, 1)) / g
    wmass = grp[:, :, P:].sum() / g
    return raw.numpy(), float(wmass)


@pytest.mark.parametrize("H_q,H_kv,d,W,L", [
    (1, 1, 8, 1, 5), (2, 1, 16, 3, 17), (4, 2, 8, 4, 33), (8, 1, 4, 5, 64),
    (4, 4, 64, 16, 40), (6, 3, 16, 2, 9),
])
def test_brute_force_full_attention(H_q, H_kv, d, W, L):
    seqlens = [L + 3, L]  # second sequence exercises the packed offset
    q, k, _ = _rand_layer(1000 + L, seqlens, H_q, H_kv, d, W, scale=1.5)
    for b in range(2):
        for h in range(H_kv):
            raw, wm = oracle.scores(q, k, seqlens, W, b, h)
            want, want_wm = _brute_force_raw(q, k, seqlens, W, b, h, seed=b)
            np.testing.assert_allclose(raw, want, rtol=1e-12, atol=1e-14)
            assert abs(wm - want_wm) < 1e-12


def test_brute_force_bf16_inputs():
    seqlens = [48]
    q, k, _ = _rand_layer(7, seqlens, 4, 2, 32, 6, dtype="bf16", scale=2.0)
    for h in range(2):
        raw, wm = oracle.scores(q, k, seqlens, 6, 0, h)
        want, want_wm = _brute_force_raw(q, k, seqlens, 6, 0, h)
        np.testing.assert_allclose(raw, want, rtol=1e-12, atol=1e-14)
        assert abs(wm - want_wm) < 1e-12


def test_hand_examples_scores():
    gold = json.load(open(os.path.join(GOLD, "hand_examples.json")))
    for case in gold["scores"]:
        q = np.asarray(case["q_win"], np.float32)
        k = np.asarray(case["k"], np.float32)
        W = case["W"]
        raw, wm = oracle.scores(q, k, [k.shape[0]], W, 0, 0)
        want = [_ev(x) for x in case["raw"]]
        np.testing.assert_allclose(raw, want, rtol=1e-13, err_msg=case["name"])
        assert abs(wm - _ev(case["window_mass"])) < 1e-13, case["name"]


@pytest.mark.parametrize("g", [1, 2, 4, 8])
@pytest.mark.parametrize("W,L", [(1, 2), (4, 20), (16, 100)])
def test_closed_form_zero_queries(g, W, L):
    """q = 0: row i is uniform over its P+i+1 visible keys, for any g."""
    P = L - W
    q = np.zeros((1, W, g, 8), np.float32)
    k = np.random.default_rng(3).standard_normal((L, 1, 8)).astype(np.float32)
    raw, wm = oracle.scores(q, k, [L], W, 0, 0)
    want = sum(1.0 / (P + i + 1) for i in range(W))
    np.testing.assert_allclose(raw, np.full(P, want), rtol=1e-14)
    assert abs(wm - sum((i + 1) / (P + i + 1) for i in range(W))) < 1e-13


def test_gqa_grouping_is_contiguous():
    """KV head h serves query heads h*g..h*g+g-1 (zero queries => uniform)."""
    W, L, d = 4, 30, 16
    P = L - W
    rng = np.random.default_rng(5)
    k = rng.standard_normal((L, 2, d)).astype(np.float32)
    q = np.zeros((1, W, 4, d), np.float32)
    q[0, :, 2:] = 4.0 * k[3, 1] + rng.standard_normal((W, 2, d)).astype(np.float32)
    raw0, _ = oracle.scores(q, k, [L], W, 0, 0)
    raw1, _ = oracle.scores(q, k, [L], W, 0, 1)
    uniform = sum(1.0 / (P + i + 1) for i in range(W))
    np.testing.assert_allclose(raw0, uniform, rtol=1e-14)
    assert int(np.argmax(raw1)) == 3 and raw1[3] > 2.0 * uniform


def test_key_shift_invariance():
    """Adding one vector u to every key shifts each row's logits by a constant."""
    W, L, d = 5, 40, 16
    rng = np.random.default_rng(11)
    # small integers / 8 so that k + u is exact in fp32
    k = (rng.integers(-16, 17, (L, 1, d)) / 8.0).astype(np.float32)
    u = (rng.integers(-8, 9, (d,)) / 4.0).astype(np.float32)
    q = (rng.integers(-8, 9, (1, W, 2, d)) / 8.0).astype(np.float32)
    raw_a, wm_a = oracle.scores(q, k, [L], W, 0, 0)
    raw_b, wm_b = oracle.scores(q, k + u, [L], W, 0, 0)
    np.testing.assert_allclose(raw_a, raw_b, rtol=1e-12, atol=1e-15)
    assert abs(wm_a - wm_b) < 1e-12


def test_group_permutation_and_repetition():
    W, L, d, g = 6, 50, 16, 4
    q, k, _ = _rand_layer(21, [L], g, 1, d, W, scale=2.0)
    base, _ = oracle.scores(q, k, [L], W, 0, 0)
    perm = q[:, :, [2, 0, 3, 1]]
    raw_p, _ = oracle.scores(np.ascontiguousarray(perm), k, [L], W, 0, 0)
    np.testing.assert_allclose(raw_p, base, rtol=1e-13, atol=1e-16)
    one = q[:, :, :1]
    rep = np.ascontiguousarray(np.repeat(one, g, axis=2))
    raw_rep, _ = oracle.scores(rep, k, [L], W, 0, 0)
    raw_mha, _ = oracle.scores(np.ascontiguousarray(one), k, [L], W, 0, 0)
    np.testing.assert_allclose(raw_rep, raw_mha, rtol=1e-13, atol=1e-16)


@pytest.mark.parametrize("g,W,L", [(1, 16, 200), (4, 8, 77), (8, 3, 10)])
def test_row_mass_conservation(g, W, L):
    q, k, _ = _rand_layer(31 + L, [L], g, 1, 32, W, scale=3.0)
    raw, wm = oracle.scores(q, k, [L], W, 0, 0)
    assert abs(raw.sum() + wm - W) < 1e-12
    assert (raw >= 0).all()


def test_nonfinite_inputs_rejected():
    q, k, _ = _rand_layer(1, [10], 1, 1, 4, 2)
    k[3, 0, 1] = np.inf
    with pytest.raises(RuntimeError):
        oracle.scores(q, k, [10], 2, 0, 0)


# --------------------------------------------------------------- pooling ---

def test_hand_examples_pooling_and_selection():
    gold = json.load(open(os.path.join(GOLD, "hand_examples.json")))
    for case in gold["pooling"]:
        raw = np.asarray(case["raw"], np.float64)
        for kind in ("avg", "max"):
            got = oracle.pool(raw, case["k"], kind)
            np.testing.assert_allclose(got, [_ev(x) for x in case[kind]], rtol=1e-15)
    for case in gold["selection"]:
        sel, _ = oracle.select(np.asarray(case["pooled"]), case["n"])
        assert sel.tolist() == case["sel"], case["name"]


@pytest.mark.parametrize("kp", [1, 3, 5, 7, 13])
@pytest.mark.parametrize("P", [1, 2, 6, 7, 50])
def test_pool_matches_torch(kp, P):
    raw = np.random.default_rng(kp * 100 + P).random(P)
    x = torch.from_numpy(raw)[None, None]
    want_avg = torch.nn.functional.avg_pool1d(x, kp, 1, kp // 2, count_include_pad=True)
    want_max = torch.nn.functional.max_pool1d(x, kp, 1, kp // 2)
    np.testing.assert_allclose(oracle.pool(raw, kp, "avg"), want_avg[0, 0].numpy(), rtol=1e-14)
    np.testing.assert_array_equal(oracle.pool(raw, kp, "max"), want_max[0, 0].numpy())


@pytest.mark.parametrize("pool_type", ["avg", "max"])
def test_pool_kernel_one_is_identity(pool_type):
    raw = np.random.default_rng(9).random(37)
    np.testing.assert_array_equal(oracle.pool(raw, 1, pool_type), raw)


@pytest.mark.parametrize("kp", [3, 5, 13])
def test_avg_and_max_agree_on_constant_interior(kp):
    c, P = 0.3125, 40
    r = kp // 2
    raw = np.full(P, c)
    a = oracle.pool(raw, kp, "avg")
    m = oracle.pool(raw, kp, "max")
    np.testing.assert_array_equal(m, np.full(P, c))
    np.testing.assert_allclose(a[r:P - r], m[r:P - r], rtol=1e-15)
    for j in list(range(r)) + list(range(P - r, P)):
        count = min(P - 1, j + r) - max(0, j - r) + 1
        assert abs(a[j] - c * count / kp) < 1e-15


def test_pool_rejects_even_kernel():
    with pytest.raises(RuntimeError):
        oracle.pool(np.ones(5), 4, "avg")


# ------------------------------------------------------------- selection ---

@pytest.mark.parametrize("seed", range(6))
def test_select_matches_sort(seed):
    rng = np.random.default_rng(seed)
    P = int(rng.integers(1, 300))
    pooled = rng.integers(0, 12, P).astype(np.float64) / 4.0  # many exact ties
    n = int(rng.integers(0, P + 1))
    sel, tau = oracle.select(pooled, n)
    order = sorted(range(P), key=lambda j: (-pooled[j], j))
    assert sel.tolist() == sorted(order[:n])
    if n:
        assert tau == pooled[order[n - 1]]


# -------------------------------------------------------------- compress ---

def _compress(lay, k_pool, pool, C, **kw):
    return oracle.compress(lay.q_win, lay.k, lay.v, lay.seqlens, lay.W, k_pool, pool, C, **kw)


def test_keep_all_when_budget_covers_prompt():
    lay = synth.make_inputs(1, [40, 64, 17], 4, 2, 16, 8, "bf16", nspans=2)
    C = 64
    out = _compress(lay, 5, "avg", C)
    off = 0
    for b, L in enumerate(lay.seqlens):
        for h in range(2):
            idx = out["idx"][b, h]
            assert idx[:L].tolist() == list(range(L))
            assert (idx[L:] == -1).all()
            np.testing.assert_array_equal(out["out_k"][b, :L, h], lay.k[off:off + L, h])
            np.testing.assert_array_equal(out["out_v"][b, :L, h], lay.v[off:off + L, h])
            assert (out["out_k"][b, L:, h] == 0).all() and (out["out_v"][b, L:, h] == 0).all()
        off += L


@pytest.mark.parametrize("pool", ["avg", "max"])
def test_window_rows_retained_and_rows_match_indices(pool):
    lay = synth.make_inputs(2, [300, 129, 57], 8, 2, 32, 16, "bf16", nspans=4)
    C = 48
    out = _compress(lay, 7, pool, C)
    off = 0
    for b, L in enumerate(lay.seqlens):
        P = L - 16
        for h in range(2):
            idx = out["idx"][b, h]
            if L > C:
                assert idx[C - 16:].tolist() == list(range(P, L))
                sel = idx[:C - 16]
                assert (np.diff(sel) > 0).all() and sel.min() >= 0 and sel.max() < P
            for s in range(C):
                if idx[s] >= 0:
                    np.testing.assert_array_equal(out["out_k"][b, s, h], lay.k[off + idx[s], h])
                    np.testing.assert_array_equal(out["out_v"][b, s, h], lay.v[off + idx[s], h])
        off += L


def test_compress_agrees_with_stepwise_functions():
    lay = synth.make_inputs(4, [90, 70], 4, 2, 16, 8, "fp32", nspans=3)
    out = _compress(lay, 5, "max", 30)
    for b in range(2):
        for h in range(2):
            raw, _ = oracle.scores(lay.q_win, lay.k, lay.seqlens, 8, b, h)
            pooled = oracle.pool(raw, 5, "max")
            sel, tau = oracle.select(pooled, 22)
            np.testing.assert_array_equal(out["pooled"][b][h], pooled)
            assert out["idx"][b, h, :22].tolist() == sel.tolist()
            assert out["tau"][b, h] == tau


def test_closed_form_selection_zero_queries():
    """q = 0 makes raw constant: avg keeps the interior from r, max keeps 0..n-1."""
    W, L, d, C, kp = 4, 60, 8, 20, 5
    n, r = C - W, kp // 2
    k = np.random.default_rng(0).standard_normal((L, 1, d)).astype(np.float32)
    q = np.zeros((1, W, 2, d), np.float32)
    v = k.copy()
    a = oracle.compress(q, k, v, [L], W, kp, "avg", C)
    m = oracle.compress(q, k, v, [L], W, kp, "max", C)
    assert a["idx"][0, 0, :n].tolist() == list(range(r, r + n))
    assert m["idx"][0, 0, :n].tolist() == list(range(n))


@pytest.mark.parametrize("name", ["1", "2"])
def test_planted_keys_selected(name):
    cfg = synth.CONFIGS[name]
    lay = synth.make_layer(name)
    out = _compress(lay, cfg["k_pool"], cfg["pool"], cfg["C"])
    for b in range(lay.B):
        for h in range(lay.H_kv):
            kept = set(out["idx"][b, h].tolist())
            missing = [p for p in lay.targets[b][h] if p not in kept]
            assert not missing, (b, h, missing[:10])


def test_budget_fits_planted_keys_in_every_workload():
    """W*g planted targets plus pooling spread fit in the C-W slots."""
    for name, cfg in synth.CONFIGS.items():
        g = cfg["H_q"] // cfg["H_kv"]
        assert cfg["W"] * g * cfg["k_pool"] <= cfg["C"] - cfg["W"], name


def test_threads_do_not_change_results():
    lay = synth.make_inputs(6, [120, 90, 200], 4, 2, 16, 8, "bf16", nspans=3)
    a = _compress(lay, 5, "avg", 40, nthreads=1)
    b = _compress(lay, 5, "avg", 40, nthreads=5)
    np.testing.assert_array_equal(a["idx"], b["idx"])
    np.testing.assert_array_equal(a["out_k"], b["out_k"])
    for x, y in zip(a["pooled"], b["pooled"]):
        np.testing.assert_array_equal(x, y)


def test_page_parameters_and_workloads_in_range():
    pp = json.load(open(os.path.join(GOLD, "page_parameters.json")))
    for name, cfg in synth.CONFIGS.items():
        assert pp["window_size_range"]["min"] <= cfg["W"] <= pp["window_size_range"]["max"]
        assert cfg["k_pool"] % 2 == 1
        assert cfg["pool"] + "pool" in pp["pooling_types"]["values"]


# ---- per-query-head selection (SNAPKV_PER_QUERY_HEAD) ----

def test_per_q_head_with_groups_of_one_is_the_plain_compression():
    lay = synth.make_inputs(21, [300, 90], 4, 4, 64, 16, "bf16", nspans=2)
    a = oracle.compress(lay.q_win, lay.k, lay.v, lay.seqlens, lay.W, 5, "avg", 128)
    b = oracle.compress_per_q_head(lay.q_win, lay.k, lay.v, lay.seqlens, lay.W, 5, "avg", 128)
    np.testing.assert_array_equal(a["idx"], b["idx"])
    np.testing.assert_array_equal(a["out_k"], b["out_k"])


def test_per_q_head_scores_average_to_the_group_score():
    """The g query heads' own raw scores average to their KV head's score."""
    lay = synth.make_inputs(22, [400], 8, 2, 64, 16, "bf16", nspans=2)
    C = 128
    a = oracle.compress(lay.q_win, lay.k, lay.v, lay.seqlens, lay.W, 5, "max", C)
    b = oracle.compress_per_q_head(lay.q_win, lay.k, lay.v, lay.seqlens, lay.W, 5, "max", C)
    g = 4
    for h in range(2):
        mean = np.mean([b["raw"][0][h * g + m] for m in range(g)], axis=0)
        np.testing.assert_allclose(mean, a["raw"][0][h], rtol=1e-12, atol=1e-15)
    # each query head keeps positions of its own KV head's rows
    assert b["idx"].shape == (1, 8, C)
    for hq in range(8):
        rows = b["idx"][0, hq]
        np.testing.assert_array_equal(b["out_k"][0, :, hq], lay.k[rows, hq // g])


def test_oracle_threaded_scores_are_bit_identical():
    """With fewer (sequence, KV head) units than threads the oracle spreads
    one unit's window rows and keys over the threads; the doubles must not
    change (same expressions, same summation order)."""
    lay = synth.make_inputs(61, [700, 530], 8, 2, 64, 16, "fp32", nspans=2)
    a = oracle.compress(lay.q_win, lay.k, lay.v, lay.seqlens, 16, 5, "avg", 128, nthreads=1)
    b = oracle.compress(lay.q_win, lay.k, lay.v, lay.seqlens, 16, 5, "avg", 128, nthreads=7)
    for x, y in zip(a["raw"], b["raw"]):
        assert np.array_equal(x, y)
    for x, y in zip(a["pooled"], b["pooled"]):
        assert np.array_equal(x, y)
    assert np.array_equal(a["window_mass"], b["window_mass"])
    assert np.array_equal(a["idx"], b["idx"])
