"""GPU parity of the Scissorhands step (scissorhands_step through the C ABI)
against the oracle (oracle/scissorhands.py).

Step-level parity: before every step the GPU cache (rows, positions, history
bits, state) is read back and turned into the oracle's token lists; both take
the same step from that state and everything after it is compared:
* the cache size, step count, positions and K / V bits: exactly (eviction is
  integer work on the history counts, and rows are bit copies);
* the history bit of this step: exactly wherever the oracle's n * (group-mean
  weight) is at least 1e-3 away from 1; inside that band both answers are
  valid (an fp32 weight against an fp64 one), and the GPU's answer is kept;
* the output: |gpu - oracle| <= 1e-4 max|v| + 1e-4 |oracle| (fp32 softmax
  with exp2 over at most `budget` rows; the decode kernels' bound).
Free-running checks (no read-back between steps) cover what holds whatever
the near-ties decided: uniform attention, where every decision is exact and
the cache must be a sliding window, and a CUDA-graph replay that must match
eager launches bit for bit.
"""
import numpy as np
import pytest
import torch

import synth
from oracle.scissorhands import Params, ScissorhandsCache, Token
from prefill_kv_cache_gb300 import scissorhands as SH
from prefill_kv_cache_gb300 import snapkv as S

pytestmark = pytest.mark.gpu

BAND = 1e-3


def _host(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def _dev(a: np.ndarray, dtype) -> torch.Tensor:
    if dtype == torch.bfloat16:
        return torch.from_numpy(np.ascontiguousarray(a)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _rand(rng, shape, dtype, scale=1.0):
    a = (scale * rng.standard_normal(shape)).astype(np.float32)
    return synth.bf16_round(a) if dtype == torch.bfloat16 else a


def _f64(a):
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def snapshot(c: SH.Cache):
    torch.cuda.synchronize()
    return dict(k=_host(c.k), v=_host(c.v), pos=c.pos.cpu().numpy(),
                hist=c.hist.cpu().numpy().view(np.uint32), state=c.state.cpu().numpy())


def low_steps(hist_slot: np.ndarray, t: int, w: int) -> list:
    """Steps s in [t - w, t - 1] whose bit (s mod w) is set in a slot's words."""
    out = []
    for s in range(max(0, t - w), t):
        u = s % w
        if (int(hist_slot[u // 32]) >> (u % 32)) & 1:
            out.append(s)
    return out


def to_oracle(snap, p: Params, H_q: int) -> ScissorhandsCache:
    B, _, H_kv, _ = snap["k"].shape
    heads = []
    for b in range(B):
        n, t = int(snap["state"][b, 0]), int(snap["state"][b, 1])
        heads.append([[Token(int(snap["pos"][b, h, j]), _f64(snap["k"][b, j, h]),
                             _f64(snap["v"][b, j, h]),
                             low_steps(snap["hist"][b, h, :, j], t, p.history))
                       for j in range(n)] for h in range(H_kv)])
    c = ScissorhandsCache(p, H_q, heads)
    c.steps = [int(x) for x in snap["state"][:, 1]]
    c.next_pos = [int(x) for x in snap["state"][:, 2]]
    return c


def compare_step(after, ora: ScissorhandsCache, ratio, t_before):
    """GPU state after a step against the oracle's, exempting near-average
    decisions of the step just taken."""
    B, _, H_kv, _ = after["k"].shape
    for b in range(B):
        assert int(after["state"][b, 0]) == ora.n(b)
        assert int(after["state"][b, 1]) == ora.steps[b]
        assert int(after["state"][b, 2]) == ora.next_pos[b]
        t = t_before[b]
        for h in range(H_kv):
            toks = ora.heads[b][h]
            n = len(toks)
            assert list(after["pos"][b, h, :n]) == [x.pos for x in toks], (b, h)
            np.testing.assert_array_equal(_f64(after["k"][b, :n, h]), np.stack([x.k for x in toks]))
            np.testing.assert_array_equal(_f64(after["v"][b, :n, h]), np.stack([x.v for x in toks]))
            t_after = ora.steps[b]
            for j, tok in enumerate(toks):
                got = low_steps(after["hist"][b, h, :, j], t_after, ora.p.history)
                want = [s for s in tok.low if s >= t_after - ora.p.history]
                if abs(ratio[b][h, j] - 1.0) < BAND:  # either answer is valid at step t
                    got = [s for s in got if s != t]
                    want = [s for s in want if s != t]
                assert got == want, (b, h, j, got, want)


CASES = [
    # B, H_q, H_kv, d,  dtype,          budget, recent, history, evict, lens0,      steps
    (2, 8, 2, 64, torch.float32, 24, 3, 7, 12, [5, 24], 70),
    (2, 32, 8, 128, torch.bfloat16, 32, 4, 40, 16, [32, 9], 80),
    (1, 16, 1, 128, torch.bfloat16, 40, 10, 33, 20, [17], 90),       # g = 16, two history words
    (3, 4, 4, 64, torch.bfloat16, 16, 1, 3, 16, [0, 16, 7], 50),     # g = 1, evict = budget
    (1, 8, 4, 128, torch.float32, 300, 10, 64, 150, [290], 170),     # several scan chunks
    (2, 16, 8, 64, torch.bfloat16, 12, 12, 5, 1, [12, 3], 30),       # recent = budget
]


def _prefix(rng, B, C0, H_kv, d, dtype):
    k0 = _rand(rng, (B, C0, H_kv, d), dtype)
    v0 = _rand(rng, (B, C0, H_kv, d), dtype)
    pos0 = np.stack([np.stack([np.sort(rng.choice(4 * C0 + 8, size=C0, replace=False))
                               for _ in range(H_kv)]) for _ in range(B)]).astype(np.int32)
    return k0, v0, pos0


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"B{c[0]}-g{c[1]//c[2]}-d{c[3]}-"
                         f"{str(c[4])[6:]}-bud{c[5]}-r{c[6]}-w{c[7]}-m{c[8]}")
def test_step_parity(case):
    B, H_q, H_kv, d, dtype, budget, recent, history, evict, lens0, steps = case
    p = Params(budget, recent, history, evict)
    rng = np.random.default_rng(budget * 7 + history)
    C0 = max(1, max(lens0))
    k0, v0, pos0 = _prefix(rng, B, C0, H_kv, d, dtype)
    c = SH.Cache(B, H_q, H_kv, d, dtype, SH.Params(budget, recent, history, evict))
    nxt = [4 * C0 + 8 + 5 * b for b in range(B)]
    c.init(lens0, nxt, _dev(k0, dtype), _dev(v0, dtype), torch.from_numpy(pos0).cuda())
    before = snapshot(c)
    n0 = S.kernel_launches()
    for t in range(steps):
        ora = to_oracle(before, p, H_q)
        q = _rand(rng, (B, H_q, d), dtype, 2.0)
        kn, vn = _rand(rng, (B, H_kv, d), dtype), _rand(rng, (B, H_kv, d), dtype)
        out = c.step(_dev(q, dtype), _dev(kn, dtype), _dev(vn, dtype))
        o_ref, ratio = ora.step(q, kn, vn)
        after = snapshot(c)
        o = out.cpu().numpy()
        vmax = max(np.abs(tok.v).max() for hs in ora.heads for toks in hs for tok in toks)
        err = np.abs(o - o_ref)
        assert (err <= 1e-4 * vmax + 1e-4 * np.abs(o_ref)).all(), (t, err.max())
        compare_step(after, ora, ratio, [int(x) for x in before["state"][:, 1]])
        before = after
    assert S.kernel_launches() - n0 == 4 * steps


def test_init_from_compressed_prompt():
    """The prefill compression's outputs (out_k, out_v, out_idx) load as the
    starting cache; the first steps then match the oracle."""
    lay = synth.make_inputs(31, [3000, 700], 32, 8, 128, 32, "bf16", nspans=2)
    C = 256
    q, k, v = (torch.from_numpy(x).view(torch.bfloat16).cuda() for x in (lay.q_win, lay.k, lay.v))
    out_k, out_v, out_idx, _ = S.compress(q, k, v, lay.seqlens, 32, 7, "avg", C)
    p = Params(budget=300, recent=10, history=50, evict=150)
    c = SH.Cache(2, 32, 8, 128, torch.bfloat16, SH.Params(300, 10, 50, 150))
    lens0 = [min(L, C) for L in lay.seqlens]
    c.init(lens0, lay.seqlens, out_k, out_v, out_idx)
    snap = snapshot(c)
    for b in range(2):
        n = lens0[b]
        assert list(snap["state"][b]) == [n, 0, lay.seqlens[b], 0]
        np.testing.assert_array_equal(snap["pos"][b, :, :n], out_idx[b, :, :n].cpu().numpy())
        np.testing.assert_array_equal(snap["k"][b, :n], _host(out_k[b, :n]))
        np.testing.assert_array_equal(snap["v"][b, :n], _host(out_v[b, :n]))
        assert not snap["hist"][b].any()
    rng = np.random.default_rng(32)
    for _ in range(60):  # both sequences pass the budget at step 44
        ora = to_oracle(snap, p, 32)
        qs = _rand(rng, (2, 32, 128), torch.bfloat16, 2.0)
        kn, vn = _rand(rng, (2, 8, 128), torch.bfloat16), _rand(rng, (2, 8, 128), torch.bfloat16)
        c.step(_dev(qs, torch.bfloat16), _dev(kn, torch.bfloat16), _dev(vn, torch.bfloat16))
        _, ratio = ora.step(qs, kn, vn)
        after = snapshot(c)
        compare_step(after, ora, ratio, [int(x) for x in snap["state"][:, 1]])
        snap = after


@pytest.mark.parametrize("g", [1, 4])
def test_uniform_attention_is_a_sliding_window(g):
    """q = 0: every weight is exactly 1/n on the GPU too (zero logits, exp2(0)
    = 1, integer sums), so no token is ever below average, every count is
    zero and each batch evicts the oldest: free-running, the cache must hold
    exactly the last n tokens to arrive."""
    B, H_kv, d, dtype = 2, 2, 64, torch.bfloat16
    p = SH.Params(budget=20, recent=3, history=9, evict=10)
    c = SH.Cache(B, H_kv * g, H_kv, d, dtype, p)
    rng = np.random.default_rng(40 + g)
    k0, v0, pos0 = _prefix(rng, B, 20, H_kv, d, dtype)
    c.init([20, 4], [500, 600], _dev(k0, dtype), _dev(v0, dtype), torch.from_numpy(pos0).cuda())
    stream = [[list(pos0[b, h, :(20, 4)[b]]) for h in range(H_kv)] for b in range(B)]
    zeros = torch.zeros((B, H_kv * g, d), dtype=dtype, device="cuda")
    n = [20, 4]
    for t in range(45):
        kn = _dev(_rand(rng, (B, H_kv, d), dtype), dtype)
        c.step(zeros, kn, kn)
        for b in range(B):
            n[b] += 1
            if n[b] > 20:
                n[b] -= 10
            for h in range(H_kv):
                stream[b][h].append((500, 600)[b] + t)
    snap = snapshot(c)
    for b in range(B):
        assert snap["state"][b, 0] == n[b]
        for h in range(H_kv):
            assert list(snap["pos"][b, h, :n[b]]) == stream[b][h][-n[b]:]
        assert not snap["hist"][b].any()


def test_graph_replay_matches_eager():
    """The step keeps its state on the device: a CUDA graph of several steps
    replays to the same cache, history and outputs as eager launches."""
    B, H_q, H_kv, d, dtype = 2, 32, 8, 128, torch.bfloat16
    prm = SH.Params(budget=64, recent=4, history=40, evict=32)
    rng = np.random.default_rng(50)
    k0, v0, pos0 = _prefix(rng, B, 64, H_kv, d, dtype)
    T = 8
    qs = _dev(_rand(rng, (T, B, H_q, d), dtype, 2.0), dtype)
    ks = _dev(_rand(rng, (T, B, H_kv, d), dtype), dtype)
    vs = _dev(_rand(rng, (T, B, H_kv, d), dtype), dtype)

    def fresh():
        c = SH.Cache(B, H_q, H_kv, d, dtype, prm)
        c.init([60, 30], [900, 800], _dev(k0, dtype), _dev(v0, dtype),
               torch.from_numpy(pos0).cuda())
        torch.cuda.synchronize()
        return c

    eager = fresh()
    outs_e = torch.empty((3 * T, B, H_q, d), dtype=torch.float32, device="cuda")
    for r in range(3):
        for t in range(T):
            eager.step(qs[t], ks[t], vs[t], out=outs_e[r * T + t])
    graphed = fresh()
    outs_g = torch.empty((T, B, H_q, d), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        for t in range(T):
            graphed.step(qs[t], ks[t], vs[t], out=outs_g[t], stream=s)
    # capture enqueues nothing: the cache is still at its starting state
    for r in range(3):
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(outs_g, outs_e[r * T:(r + 1) * T])
    a, b = snapshot(eager), snapshot(graphed)
    np.testing.assert_array_equal(a["state"], b["state"])
    for bb in range(B):  # slots past n hold whatever was there before
        n = int(a["state"][bb, 0])
        np.testing.assert_array_equal(a["pos"][bb, :, :n], b["pos"][bb, :, :n])
        np.testing.assert_array_equal(a["hist"][bb, :, :, :n], b["hist"][bb, :, :, :n])
        np.testing.assert_array_equal(a["k"][bb, :n], b["k"][bb, :n])
        np.testing.assert_array_equal(a["v"][bb, :n], b["v"][bb, :n])


def test_more_sequences_than_one_launch_group():
    """600 sequences (the attention runs as two launch groups): under uniform
    attention every sequence's cache must be the newest tokens, with the
    budget, the batch size and each sequence's starting length respected."""
    B, H_kv, g, d, dtype = 600, 2, 2, 64, torch.bfloat16
    c = SH.Cache(B, H_kv * g, H_kv, d, dtype, SH.Params(budget=8, recent=2, history=3, evict=4))
    rng = np.random.default_rng(70)
    k0, v0, pos0 = _prefix(rng, B, 8, H_kv, d, dtype)
    lens0 = [int(x) for x in rng.integers(0, 9, B)]
    nxt = [1000 + 7 * b for b in range(B)]
    c.init(lens0, nxt, _dev(k0, dtype), _dev(v0, dtype), torch.from_numpy(pos0).cuda())
    zeros = torch.zeros((B, H_kv * g, d), dtype=dtype, device="cuda")
    steps = 6
    for _ in range(steps):
        kn = _dev(_rand(rng, (B, H_kv, d), dtype), dtype)
        c.step(zeros, kn, kn)
    snap = snapshot(c)
    for b in range(B):
        n = lens0[b]
        stream = list(range(nxt[b], nxt[b] + steps))
        for _ in range(steps):
            n += 1
            if n > 8:
                n -= 4
        assert list(snap["state"][b, :3]) == [n, steps, nxt[b] + steps]
        for h in range(H_kv):
            arrived = list(pos0[b, h, :lens0[b]]) + stream
            assert list(snap["pos"][b, h, :n]) == arrived[-n:], (b, h)
