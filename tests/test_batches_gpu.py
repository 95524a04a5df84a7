"""GPU parity with batches larger than one planning group (64 sequences for
compression, 512 for the decode step), so the per-group launches, the
cumulative score / row offsets and the reused work-queue counters are all
exercised.  Agreement rules as in tests/parity.py and tests/test_decode_gpu.py."""
import numpy as np
import pytest

import oracle
import synth
from prefill_kv_cache_gb300 import snapkv as S
from tests import parity

pytestmark = pytest.mark.gpu


def _lens(seed, n, lo, hi):
    return [int(x) for x in np.random.default_rng(seed).integers(lo, hi, n)]


@pytest.mark.parametrize("dtype,H_q,H_kv,d,W,C", [
    ("bf16", 16, 4, 128, 32, 512),   # tensor-core scoring (W*g = 128)
    ("fp32", 8, 4, 64, 16, 256),     # FFMA scoring
])
def test_compress_150_sequences(dtype, H_q, H_kv, d, W, C):
    lens = _lens(150, 150, 16, 2500)
    lay = synth.make_inputs(150, lens, H_q, H_kv, d, W, dtype, nspans=2)
    gpu = parity.run_gpu(lay, 5, "avg", C)
    ora = parity.oracle_for(lay, 5, "avg", C)
    parity.check(lay, gpu, ora, C)


def test_compress_with_lse_130_sequences():
    lens = _lens(130, 130, 16, 3000)
    C = 512
    lay = synth.make_inputs(130, lens, 16, 4, 128, 32, "bf16", nspans=2)
    lse = parity.window_lse(lay, C)
    gpu = parity.run_gpu(lay, 7, "max", C, lse=lse)
    ora = parity.oracle_for(lay, 7, "max", C)
    parity.check(lay, gpu, ora, C, rtol=parity.LSE_RTOL)


def test_decode_600_sequences():
    lens = _lens(600, 600, 1, 400)
    H_q, H_kv, d = 8, 2, 64
    rng = np.random.default_rng(6)
    k = synth.bf16_round(rng.standard_normal((sum(lens), H_kv, d)).astype(np.float32))
    v = synth.bf16_round(rng.standard_normal((sum(lens), H_kv, d)).astype(np.float32))
    q = synth.bf16_round((2.0 * rng.standard_normal((600, H_q, d))).astype(np.float32))
    offs = np.concatenate([[0], np.cumsum(lens)])
    o = S.decode_attention(parity.to_device(q), parity.to_device(k), parity.to_device(v), lens,
                           S.CACHE_PACKED)
    ref = oracle.decode_attention(q, [k[offs[b]:offs[b + 1]] for b in range(600)],
                                  [v[offs[b]:offs[b + 1]] for b in range(600)])
    vmax = np.abs(synth.bf16_to_f32(v)).max()
    err = np.abs(o.cpu().numpy() - ref)
    assert (err <= 1e-4 * vmax + 1e-4 * np.abs(ref)).all(), err.max()


EDGE = [
    # seqlens,                  H_q, H_kv, d,  W,  C,   k, pool,  dtype   what
    ([1024, 1025, 1026],         16,   4, 128, 32, 1024, 5, "avg", "bf16"),  # L = C, C+1, C+2
    ([40, 41, 300],               4,   4, 64,  1, 40,   3, "max", "bf16"),   # W = 1
    ([300],                       8,   2, 128, 16, 290, 13, "avg", "fp32"),  # P = 284 > n, wide pool
    ([60, 61],                   16,   4, 128, 32, 58,  31, "max", "bf16"),  # pool wider than P
    ([2000],                     32,   8, 128, 32, 1024, 1, "avg", "bf16"),  # k = 1: pooled = raw
]


@pytest.mark.parametrize("case", EDGE, ids=lambda c: f"L{c[0]}-W{c[4]}-C{c[5]}-k{c[6]}-{c[8]}")
def test_edge_shapes(case):
    seqlens, H_q, H_kv, d, W, C, kp, pool, dtype = case
    lay = synth.make_inputs(991 + sum(seqlens), seqlens, H_q, H_kv, d, W, dtype, nspans=1)
    gpu = parity.run_gpu(lay, kp, pool, C)
    ora = parity.oracle_for(lay, kp, pool, C)
    parity.check(lay, gpu, ora, C)
    if kp == 1:  # no pooling: pooled scores are the raw scores, bit for bit
        np.testing.assert_array_equal(gpu["pooled"], gpu["raw"])
