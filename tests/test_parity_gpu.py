"""GPU parity: libsnapkv through its C ABI against the CPU oracle.

Small shapes are compared in full (several tiles, ragged tails, keep-all
sequences mixed in, every pooling kind and size); the named workloads run at
full size in the same launch configuration the benchmark times, and the oracle
checks every sequence and KV head of them.  The agreement rule is in
tests/parity.py.
"""
import numpy as np
import pytest
import torch

import synth
from prefill_kv_cache_gb300 import snapkv as S
from tests import parity

pytestmark = pytest.mark.gpu


def _run_and_check(lay, k_pool, pool, C, seqs=None):
    gpu = parity.run_gpu(lay, k_pool, pool, C)
    ora = parity.oracle_for(lay, k_pool, pool, C, seqs=seqs)
    return parity.check(lay, gpu, ora, C, seqs=seqs), gpu


SMALL = [
    # seqlens,              H_q, H_kv, d,  W,  C,   k, pool,  dtype
    ([1024],                  4,   4, 64, 16, 256,  5, "avg", "fp32"),
    ([1025, 300, 2000],       8,   2, 128, 16, 256, 7, "max", "bf16"),
    ([257, 256, 255, 4000],   4,   1, 64,  8, 256,  1, "avg", "bf16"),
    ([3000],                 32,   8, 128, 32, 1024, 13, "avg", "bf16"),
    ([5000, 1100],           32,   8, 128, 32, 1024, 7, "max", "bf16"),
    ([4097],                 16,   2, 128, 16, 512,  3, "max", "fp32"),
    ([2049, 33],              8,   8, 64, 32, 32,   5, "avg", "bf16"),   # C == W: no prefix kept
    ([6000],                 32,   4, 128, 32, 2048, 9, "avg", "bf16"),  # W*g = 256
    ([1500],                  2,   1, 128, 64, 600, 11, "max", "fp32"),
    ([33, 17, 1],             4,   2, 64, 16, 40,   5, "avg", "bf16"),   # all keep-all
    # W*g = 256 with fewer work items than SMs and partly masked last tiles
    ([5000],                 32,   8, 128, 64, 1024, 13, "avg", "bf16"),
    ([8192, 700, 3100],      32,   8, 128, 64, 1024, 5, "max", "bf16"),
    ([2049],                 16,   4, 64, 64, 512,  7, "avg", "bf16"),
]


@pytest.mark.parametrize("case", SMALL, ids=lambda c: f"L{c[0]}-g{c[1]//c[2]}-d{c[3]}-W{c[4]}-C{c[5]}-{c[7]}{c[6]}-{c[8]}")
def test_small_shapes(case):
    seqlens, H_q, H_kv, d, W, C, kp, pool, dtype = case
    lay = synth.make_inputs(77 + sum(seqlens), seqlens, H_q, H_kv, d, W, dtype, nspans=3)
    _run_and_check(lay, kp, pool, C)


@pytest.mark.parametrize("L", [3000, 20000])
@pytest.mark.parametrize("pool", ["avg", "max"])
def test_exact_ties_zero_queries(pool, L):
    """q = 0 makes every raw score equal: the tie rule alone decides.  At
    L = 20000 the threshold's first-digit bin holds more values than one CTA
    gathers, so the select runs all three digits over the cluster."""
    W, C, kp = 16, 512, 5
    lay = synth.make_inputs(5, [L, L + 7], 8, 2, 128, W, "bf16", nspans=2)
    lay.q_win[:] = 0
    gpu = parity.run_gpu(lay, kp, pool, C)
    n, r = C - W, kp // 2
    want = list(range(r, r + n)) if pool == "avg" else list(range(n))
    for b in range(2):
        for h in range(2):
            assert gpu["idx"][b, h, :n].tolist() == want


@pytest.mark.parametrize("seqlens", [[12000, 9000], [30000]])
def test_near_uniform_scores(seqlens):
    """Tiny queries make the attention nearly uniform: all scores share one
    first-digit bin far beyond what one CTA gathers, and the cluster-wide
    digits decide among values a few ulps apart (checked against the oracle)."""
    W, C, kp = 32, 2048, 7
    lay = synth.make_inputs(31, seqlens, 16, 4, 128, W, "bf16", nspans=0)
    lay.q_win[:] = synth.bf16_round(synth.bf16_to_f32(lay.q_win) * np.float32(1e-3))
    gpu = parity.run_gpu(lay, kp, "avg", C)
    ora = parity.oracle_for(lay, kp, "avg", C)
    parity.check(lay, gpu, ora, C)


@pytest.mark.parametrize("name", ["1", "2"])
def test_workload_full(name):
    cfg = synth.CONFIGS[name]
    lay = synth.make_layer(name)
    _, gpu = _run_and_check(lay, cfg["k_pool"], cfg["pool"], cfg["C"])
    _assert_planted(lay, gpu)


def _assert_planted(lay, gpu):
    for b in range(lay.B):
        for h in range(lay.H_kv):
            kept = set(gpu["idx"][b, h].tolist())
            missing = [p for p in lay.targets[b][h] if p not in kept]
            assert not missing, (b, h, missing[:8])


@pytest.mark.parametrize("name,layer", [
    ("3", 0),      # all 8 prompts of 32768 tokens
    ("4", 0),
    ("4", 31),
    ("5a", 0),     # all 16 ragged prompts
    ("5b", 0),
])
def test_workload_full_size(name, layer):
    """Every sequence and KV head of the full-size workload against the oracle."""
    cfg = synth.CONFIGS[name]
    lay = synth.make_layer(name, layer)
    gpu = parity.run_gpu(lay, cfg["k_pool"], cfg["pool"], cfg["C"])
    _assert_planted(lay, gpu)
    ora = parity.oracle_for(lay, cfg["k_pool"], cfg["pool"], cfg["C"])
    parity.check(lay, gpu, ora, cfg["C"])


def test_repeated_calls_reuse_workspace():
    lay = synth.make_inputs(9, [5000, 2000], 32, 8, 128, 32, "bf16", nspans=4)
    q, k, v = (parity.to_device(x) for x in (lay.q_win, lay.k, lay.v))
    a = S.compress(q, k, v, lay.seqlens, 32, 7, "max", 1024)
    b = S.compress(q, k, v, lay.seqlens, 32, 7, "max", 1024, workspace=a[3])
    for x, y in zip(a[:3], b[:3]):
        assert torch.equal(x, y)


@pytest.mark.parametrize("pinned_v", [True, False])
def test_host_buffer_entry_point_matches_device(pinned_v):
    """Page-locked V is read in place by the gather (only the kept rows cross
    the link); pageable V is uploaded whole.  Both match the device call."""
    lay = synth.make_inputs(10, [4000, 700], 32, 8, 128, 32, "bf16", nspans=4)
    C = 1024
    gpu = parity.run_gpu(lay, 7, "avg", C)
    q, k, v = (torch.from_numpy(x).view(torch.bfloat16).pin_memory()
               for x in (lay.q_win, lay.k, lay.v))
    if not pinned_v:
        v = torch.from_numpy(lay.v.copy()).view(torch.bfloat16)
    B, H_kv, d = lay.B, lay.H_kv, lay.d
    ok = torch.empty((B, C, H_kv, d), dtype=torch.bfloat16).pin_memory()
    ov = torch.empty_like(ok)
    oi = torch.empty((B, H_kv, C), dtype=torch.int32).pin_memory()
    shape = S.make_shape(B, lay.H_q, H_kv, d, S.BF16)
    staging = torch.empty(S.host_staging_size(shape, lay.seqlens, 32, C), dtype=torch.uint8,
                          device="cuda")
    S.compress_host(q, k, v, lay.seqlens, 32, 7, "avg", C, ok, ov, oi, staging)
    np.testing.assert_array_equal(oi.numpy(), gpu["idx"])
    np.testing.assert_array_equal(ok.view(torch.int16).numpy().view(np.uint16), gpu["out_k"])
    np.testing.assert_array_equal(ov.view(torch.int16).numpy().view(np.uint16), gpu["out_v"])


def test_argument_errors_enqueue_nothing():
    lay = synth.make_inputs(11, [3000], 8, 2, 64, 16, "bf16", nspans=2)
    q, k, v = (parity.to_device(x) for x in (lay.q_win, lay.k, lay.v))
    with pytest.raises(S.SnapKVError) as e:
        S.compress(q, k, v, lay.seqlens, 16, 4, "avg", 256)
    assert e.value.code == S.ERR_INVALID_ARG
    with pytest.raises(S.SnapKVError) as e:
        S.compress(q, k, v, lay.seqlens, 16, 5, "avg", 256,
                   workspace=torch.empty(64, dtype=torch.uint8, device="cuda"))
    assert e.value.code == S.ERR_WORKSPACE


@pytest.mark.parametrize("H_q,H_kv,d,W,dtype,tc", [
    (32, 8, 128, 32, "bf16", True),    # W*g = 128: tensor cores
    (32, 8, 128, 64, "bf16", True),    # W*g = 256: tensor cores
    (16, 8, 64, 64, "bf16", True),     # d = 64
    (4, 4, 64, 16, "fp32", False),     # fp32 stays on CUDA cores
    (8, 8, 128, 16, "bf16", False),    # W*g = 16: CUDA cores
])
def test_score_path_selection(H_q, H_kv, d, W, dtype, tc):
    """bf16 with W*g in {128, 256} runs the single tcgen05 kernel; else 3 CUDA-core kernels."""
    lay = synth.make_inputs(12, [3000], H_q, H_kv, d, W, dtype, nspans=2)
    q, k = parity.to_device(lay.q_win), parity.to_device(lay.k)
    shape = S.make_shape(1, H_q, H_kv, d, q.dtype)
    ws = torch.empty(S.workspace_size(shape, [3000], W, 512), dtype=torch.uint8, device="cuda")
    n0 = S.kernel_launches()
    paths0 = [S.score_path_launches(x) for x in (S.SCORE_PATH_TENSOR_CORES,
                                                 S.SCORE_PATH_CUDA_CORES)]
    S.score(q, k, [3000], W, 512, ws)
    torch.cuda.synchronize()
    assert S.kernel_launches() - n0 == (1 if tc else 3)
    paths = [S.score_path_launches(x) - y for x, y in zip((S.SCORE_PATH_TENSOR_CORES,
                                                           S.SCORE_PATH_CUDA_CORES), paths0)]
    assert paths == ([1, 0] if tc else [0, 1])
    assert S.get_status(ws) == S.OK


def test_many_kv_heads_stay_on_tensor_cores():
    """136 KV heads of 131072 tokens in one launch group: more than one
    launch's queue can describe (128 groups of whole heads), so the call is
    split into two tensor-core launches instead of leaving the tensor cores.
    The first and the last prompt are compared with the oracle."""
    seqlens = [131072] * 17
    lay = synth.make_inputs(13, seqlens, 32, 8, 64, 32, "bf16", nspans=4)
    paths0 = [S.score_path_launches(x) for x in (S.SCORE_PATH_TENSOR_CORES,
                                                 S.SCORE_PATH_CUDA_CORES)]
    gpu = parity.run_gpu(lay, 7, "max", 1024)
    paths = [S.score_path_launches(x) - y for x, y in zip((S.SCORE_PATH_TENSOR_CORES,
                                                           S.SCORE_PATH_CUDA_CORES), paths0)]
    assert paths == [2, 0]
    ora = parity.oracle_for(lay, 7, "max", 1024, seqs=[0, 16])
    parity.check(lay, gpu, ora, 1024, seqs=[0, 16])


@pytest.mark.parametrize("pinned_v", [True, False])
def test_host_layers_entry_point_matches_device(pinned_v):
    """snapkv_compress_host_layers overlaps each layer's upload with the
    previous layer's compression; every layer's outputs must equal the device
    entry point's on the same inputs, bit for bit."""
    C, W = 1024, 32
    lays = [synth.make_inputs(20 + l, [4000, 700], 32, 8, 128, W, "bf16", nspans=4)
            for l in range(3)]
    ref = [parity.run_gpu(lay, 7, "avg", C) for lay in lays]
    pin = lambda x: torch.from_numpy(x).view(torch.bfloat16).pin_memory()
    layers = [(pin(l.q_win), pin(l.k), pin(l.v) if pinned_v
               else torch.from_numpy(l.v.copy()).view(torch.bfloat16)) for l in lays]
    B, H_kv, d = 2, 8, 128
    outs = [(torch.empty((B, C, H_kv, d), dtype=torch.bfloat16).pin_memory(),
             torch.empty((B, C, H_kv, d), dtype=torch.bfloat16).pin_memory(),
             torch.empty((B, H_kv, C), dtype=torch.int32).pin_memory()) for _ in lays]
    shape = S.make_shape(B, 32, H_kv, d, S.BF16)
    staging = torch.empty(S.host_staging_size_layers(shape, lays[0].seqlens, W, C),
                          dtype=torch.uint8, device="cuda")
    events = [torch.cuda.Event() for _ in range(4)]
    S.compress_host_layers(layers, lays[0].seqlens, W, 7, "avg", C, outs, staging,
                           torch.cuda.current_stream(), torch.cuda.Stream(), events)
    for (ok, ov, oi), r in zip(outs, ref):
        np.testing.assert_array_equal(oi.numpy(), r["idx"])
        np.testing.assert_array_equal(ok.view(torch.int16).numpy().view(np.uint16), r["out_k"])
        np.testing.assert_array_equal(ov.view(torch.int16).numpy().view(np.uint16), r["out_v"])


@pytest.mark.parametrize("n_layers,n_streams,graph",
                         [(1, 2, False), (5, 2, False), (4, 2, True), (7, 3, False),
                          (6, 4, True), (3, 1, False), (9, 8, False)])
def test_layers_entry_point_matches_single_calls(n_layers, n_streams, graph):
    """snapkv_compress_layers runs consecutive layers on n_streams streams,
    each with its own workspace part; every layer's outputs must equal
    snapkv_compress on the same layer, bit for bit, also when the call is
    captured in a CUDA graph and replayed."""
    C, W, kp = 1024, 32, 7
    seqlens = [4000, 700, 2600]
    lays = [synth.make_inputs(40 + l, seqlens, 32, 8, 128, W, "bf16", nspans=4)
            for l in range(n_layers)]
    dev = lambda x: torch.from_numpy(x).view(torch.bfloat16).cuda()
    layers = [(dev(l.q_win), dev(l.k), dev(l.v)) for l in lays]
    B, H_kv, d = len(seqlens), 8, 128
    new_outs = lambda: [(torch.empty((B, C, H_kv, d), dtype=torch.bfloat16, device="cuda"),
                         torch.empty((B, C, H_kv, d), dtype=torch.bfloat16, device="cuda"),
                         torch.empty((B, H_kv, C), dtype=torch.int32, device="cuda"))
                        for _ in lays]
    ref = []
    for q, k, v in layers:
        ok, ov, oi, _ = S.compress(q, k, v, seqlens, W, kp, "avg", C)
        ref.append((ok, ov, oi))
    shape = S.make_shape(B, 32, H_kv, d, S.BF16)
    ws = torch.empty(S.workspace_size_layers(shape, seqlens, W, C, n_streams),
                     dtype=torch.uint8, device="cuda")
    outs = new_outs()
    streams = [torch.cuda.Stream() for _ in range(n_streams)]
    events = [torch.cuda.Event() for _ in range(n_streams + 1)]
    if graph:
        cap = torch.cuda.Stream()
        cap.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(cap):
            with torch.cuda.graph(g, stream=cap):
                S.compress_layers(layers, seqlens, W, kp, "avg", C, outs, ws, streams, events,
                                  stream=cap)
        for _ in range(2):
            g.replay()
    else:
        S.compress_layers(layers, seqlens, W, kp, "avg", C, outs, ws, streams, events)
    torch.cuda.synchronize()
    assert S.get_status(ws) == S.OK
    for l, ((ok, ov, oi), (rk, rv, ri)) in enumerate(zip(outs, ref)):
        assert torch.equal(oi, ri), l
        assert torch.equal(ok, rk), l
        assert torch.equal(ov, rv), l
