"""GPU parity of the LSE-input entry points (snapkv_compress_with_lse,
snapkv_score_with_lse) against the CPU oracle.

The caller's window LSE comes from tests/parity.window_lse (fp64 on the CPU,
rounded to fp32 as a prefill kernel would return it).  With it the library
runs only the column-sum sweep over K; the scores, the selection and the
gathered rows must meet the same agreement rule as snapkv_compress
(tests/parity.py), with the LSE-input tolerance parity.LSE_RTOL (an outside
LSE does not cancel the fp32 rounding of a row's dominant logit).  Sequences
kept whole get NaN LSE rows, which must never be read.
"""
import numpy as np
import pytest
import torch

import synth
from prefill_kv_cache_gb300 import snapkv as S
from tests import parity

pytestmark = pytest.mark.gpu

CASES = [
    # seqlens,              H_q, H_kv, d,  W,  C,   k, pool,  dtype   (path)
    ([1024],                  4,   4, 64, 16, 256,  5, "avg", "fp32"),  # SIMT
    ([1025, 300, 2000],       8,   2, 128, 16, 256, 7, "max", "bf16"),  # SIMT (W*g = 64)
    ([3000],                 32,   8, 128, 32, 1024, 13, "avg", "bf16"),  # tensor cores, 128 rows
    ([5000, 1100, 40],       32,   8, 128, 32, 1024, 7, "max", "bf16"),
    ([6000],                 32,   4, 128, 32, 2048, 9, "avg", "bf16"),  # 256 rows
    ([8192, 700, 3100],      32,   8, 128, 64, 1024, 5, "max", "bf16"),
    ([2049],                 16,   4, 64, 64, 512,  7, "avg", "bf16"),   # d = 64
    ([33, 17, 1],             4,   2, 64, 16, 40,   5, "avg", "bf16"),   # all keep-all
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"L{c[0]}-g{c[1]//c[2]}-d{c[3]}-W{c[4]}-C{c[5]}-{c[7]}{c[6]}-{c[8]}")
def test_small_shapes_with_lse(case):
    seqlens, H_q, H_kv, d, W, C, kp, pool, dtype = case
    lay = synth.make_inputs(177 + sum(seqlens), seqlens, H_q, H_kv, d, W, dtype, nspans=3)
    lse = parity.window_lse(lay, C)
    launches = S.kernel_launches()
    gpu = parity.run_gpu(lay, kp, pool, C, lse=lse)
    ora = parity.oracle_for(lay, kp, pool, C)
    parity.check(lay, gpu, ora, C, rtol=parity.LSE_RTOL)
    if any(L > C for L in seqlens):
        # one score launch (tensor cores, or the pass-2 kernel alone), one selection
        assert S.kernel_launches() - launches == 2


@pytest.mark.parametrize("name", ["2", "3", "4", "5a"])
def test_workload_with_lse(name):
    """Every sequence and KV head of the full-size workload, LSE-input mode,
    against the oracle."""
    cfg = synth.CONFIGS[name]
    lay = synth.make_layer(name)
    lse = parity.window_lse(lay, cfg["C"])
    gpu = parity.run_gpu(lay, cfg["k_pool"], cfg["pool"], cfg["C"], lse=lse)
    ora = parity.oracle_for(lay, cfg["k_pool"], cfg["pool"], cfg["C"])
    parity.check(lay, gpu, ora, cfg["C"], rtol=parity.LSE_RTOL)
    for b in range(lay.B):
        for h in range(lay.H_kv):
            kept = set(gpu["idx"][b, h].tolist())
            assert all(p in kept for p in lay.targets[b][h]), (b, h)


def test_score_with_lse_fills_raw_scores():
    lay = synth.make_inputs(12, [4000, 900], 32, 8, 128, 32, "bf16", nspans=2)
    C = 1024
    lse = parity.window_lse(lay, C)
    q, k = parity.to_device(lay.q_win), parity.to_device(lay.k)
    shape = S.make_shape(lay.B, lay.H_q, lay.H_kv, lay.d, q.dtype)
    ws = torch.zeros(S.workspace_size(shape, lay.seqlens, lay.W, C), dtype=torch.uint8,
                     device="cuda")
    S.score_with_lse(q, k, parity.to_device(lse), lay.seqlens, lay.W, C, ws)
    assert S.get_status(ws) == S.OK
    raw, _ = S.scores_from_workspace(ws, shape, lay.seqlens, lay.W, C)
    ora = parity.oracle_for(lay, 1, "avg", C, seqs=[0])
    got = parity.unpack_scores(raw.cpu().numpy(), lay.seqlens, lay.H_kv, lay.W, C)
    np.testing.assert_allclose(got[0], np.stack(ora["raw"][0]), rtol=parity.LSE_RTOL,
                               atol=parity.ATOL)


@pytest.mark.parametrize("n_streams,graph", [(2, False), (4, True)])
def test_layers_entry_point_with_lse(n_streams, graph):
    """snapkv_compress_layers with the caller's LSE per layer: every layer's
    outputs equal snapkv_compress_with_lse on the same layer, bit for bit,
    also replayed from a CUDA graph."""
    C, W, kp = 1024, 32, 7
    seqlens = [4000, 700, 2600]
    lays = [synth.make_inputs(60 + l, seqlens, 32, 8, 128, W, "bf16", nspans=4) for l in range(5)]
    dev = lambda x: torch.from_numpy(x).view(torch.bfloat16).cuda()
    layers = [(dev(l.q_win), dev(l.k), dev(l.v)) for l in lays]
    lses = [torch.from_numpy(parity.window_lse(l, C)).cuda() for l in lays]
    ref = [S.compress_with_lse(q, k, v, lse, seqlens, W, kp, "avg", C)[:3]
           for (q, k, v), lse in zip(layers, lses)]
    shape = S.make_shape(len(seqlens), 32, 8, 128, S.BF16)
    ws = torch.empty(S.workspace_size_layers(shape, seqlens, W, C, n_streams), dtype=torch.uint8,
                     device="cuda")
    outs = [tuple(torch.empty_like(x) for x in r) for r in ref]
    streams = [torch.cuda.Stream() for _ in range(n_streams)]
    events = [torch.cuda.Event() for _ in range(n_streams + 1)]
    if graph:
        cap = torch.cuda.Stream()
        cap.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(cap):
            with torch.cuda.graph(g, stream=cap):
                S.compress_layers(layers, seqlens, W, kp, "avg", C, outs, ws, streams, events,
                                  stream=cap, lse_wins=lses)
        for _ in range(2):
            g.replay()
    else:
        S.compress_layers(layers, seqlens, W, kp, "avg", C, outs, ws, streams, events,
                          lse_wins=lses)
    torch.cuda.synchronize()
    assert S.get_status(ws) == S.OK
    for l, (o, r) in enumerate(zip(outs, ref)):
        for a, b in zip(o, r):
            assert torch.equal(a, b), l
