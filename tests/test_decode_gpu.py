"""GPU parity of snapkv_decode_attention against the decode oracle.

Tolerance: the output is a convex combination of V rows, so |o| <= max|v|;
each weight carries the fp32 rounding of its logit and the exp2
approximation (a few 1e-7 relative), and the fp32 sums run over at most
2^17 keys in chunks merged by their maxima.  The test allows
|gpu - oracle| <= 1e-4 * max|v| + 1e-4 * |oracle|.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from prefill_kv_cache_gb300 import snapkv as S
from tests import parity

pytestmark = pytest.mark.gpu


def _cache(seed, lens, H_kv, d, dtype):
    rng = np.random.default_rng(seed)
    k = rng.standard_normal((sum(lens), H_kv, d)).astype(np.float32)
    v = rng.standard_normal((sum(lens), H_kv, d)).astype(np.float32)
    if dtype == "bf16":
        k, v = synth.bf16_round(k), synth.bf16_round(v)
    return k, v


def _q(seed, B, H_q, d, dtype):
    q = (2.0 * np.random.default_rng(seed).standard_normal((B, H_q, d))).astype(np.float32)
    return synth.bf16_round(q) if dtype == "bf16" else q


def _check(o_gpu, o_ref, vmax):
    err = np.abs(o_gpu - o_ref)
    bound = 1e-4 * vmax + 1e-4 * np.abs(o_ref)
    assert (err <= bound).all(), f"max err {err.max():.3g}, at {np.unravel_index(err.argmax(), err.shape)}"


CASES = [
    # lens,                  H_q, H_kv, d,  dtype
    ([1, 31, 33, 1000],        8,   8, 64,  "fp32"),
    ([5000, 17],              32,   8, 128, "bf16"),
    ([4096],                  32,   8, 128, "bf16"),
    ([300, 2049, 7],          16,   1, 128, "bf16"),
    ([129],                    2,   2, 128, "fp32"),
    ([777, 12000],            16,   8, 64,  "bf16"),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"L{c[0]}-g{c[1]//c[2]}-d{c[3]}-{c[4]}")
@pytest.mark.parametrize("layout", [S.CACHE_PACKED, S.CACHE_SLOTS])
def test_decode_matches_oracle(case, layout):
    lens, H_q, H_kv, d, dtype = case
    k, v = _cache(sum(lens), lens, H_kv, d, dtype)
    q = _q(len(lens), len(lens), H_q, d, dtype)
    offs = np.concatenate([[0], np.cumsum(lens)])
    ks = [k[offs[b]:offs[b + 1]] for b in range(len(lens))]
    vs = [v[offs[b]:offs[b + 1]] for b in range(len(lens))]
    C = max(lens) + 3
    if layout == S.CACHE_SLOTS:  # rows of sequence b in slots 0..lens[b]-1, garbage after
        kc = np.full((len(lens), C, H_kv, d), 7, dtype=k.dtype)
        vc = np.full((len(lens), C, H_kv, d), 7, dtype=v.dtype)
        for b in range(len(lens)):
            kc[b, :lens[b]] = ks[b]
            vc[b, :lens[b]] = vs[b]
    else:
        kc, vc = k, v
    launches = S.kernel_launches()
    o = S.decode_attention(parity.to_device(q), parity.to_device(kc), parity.to_device(vc), lens,
                           layout, C)
    torch.cuda.synchronize()
    assert S.kernel_launches() - launches == 2
    ref = oracle.decode_attention(q, ks, vs)
    vmax = max(np.abs(synth.bf16_to_f32(x) if x.dtype == np.uint16 else x).max() for x in vs)
    _check(o.cpu().numpy(), ref, vmax)


def test_decode_over_compressed_cache_equals_decode_over_kept_rows():
    """snapkv_compress, then a decode step over its output slots: the same
    as attending over the kept rows of the full cache."""
    lay = synth.make_inputs(41, [6000, 700, 3000], 32, 8, 128, 32, "bf16", nspans=4)
    C = 1024
    gpu = parity.run_gpu(lay, 7, "max", C)
    q = _q(3, lay.B, lay.H_q, lay.d, "bf16")
    lens = [min(int(L), C) for L in lay.seqlens]
    o = S.decode_attention(parity.to_device(q), parity.to_device(gpu["out_k"]),
                           parity.to_device(gpu["out_v"]), lens, S.CACHE_SLOTS, C)
    ks, vs = [], []
    for b in range(lay.B):
        # the kept positions are the same for every head only by chance: gather per head
        idx = gpu["idx"][b]  # [H_kv, C]
        n = lens[b]
        kb = np.stack([lay.k[lay.offsets[b] + idx[h, :n], h] for h in range(lay.H_kv)], axis=1)
        vb = np.stack([lay.v[lay.offsets[b] + idx[h, :n], h] for h in range(lay.H_kv)], axis=1)
        ks.append(kb)
        vs.append(vb)
    ref = oracle.decode_attention(q, ks, vs)
    _check(o.cpu().numpy(), ref, max(np.abs(synth.bf16_to_f32(x)).max() for x in vs))


@pytest.mark.parametrize("layout", [S.CACHE_PACKED, S.CACHE_SLOTS])
def test_decode_full_size_128k(layout):
    """The 128K Llama-3-8B layer: full packed cache and its compressed cache."""
    lay = synth.make_layer("4", 0)
    q = _q(11, 1, lay.H_q, lay.d, "bf16")
    if layout == S.CACHE_PACKED:
        kc, vc, lens, C = lay.k, lay.v, [int(lay.seqlens[0])], 0
        ks, vs = [lay.k], [lay.v]
    else:
        C = 4096
        kc = np.ascontiguousarray(lay.k[None, -C:])  # a C-slot cache holding the last C rows
        vc = np.ascontiguousarray(lay.v[None, -C:])
        lens = [C]
        ks, vs = [lay.k[-C:]], [lay.v[-C:]]
    o = S.decode_attention(parity.to_device(q), parity.to_device(kc), parity.to_device(vc), lens,
                           layout, C)
    ref = oracle.decode_attention(q, ks, vs)
    _check(o.cpu().numpy(), ref, np.abs(synth.bf16_to_f32(vs[0])).max())


@pytest.mark.parametrize("layout", [S.CACHE_PACKED, S.CACHE_SLOTS])
def test_decode_more_sequences_than_one_launch_group(layout):
    """1100 sequences: three launch groups of at most 512 sequences run in
    turn and share one workspace."""
    lens = [int(x) for x in np.random.default_rng(61).integers(1, 48, 1100)]
    H_q, H_kv, d = 8, 2, 64
    k, v = _cache(62, lens, H_kv, d, "bf16")
    q = _q(63, len(lens), H_q, d, "bf16")
    offs = np.concatenate([[0], np.cumsum(lens)])
    ks = [k[offs[b]:offs[b + 1]] for b in range(len(lens))]
    vs = [v[offs[b]:offs[b + 1]] for b in range(len(lens))]
    C = 48
    if layout == S.CACHE_SLOTS:
        kc = np.zeros((len(lens), C, H_kv, d), dtype=k.dtype)
        vc = np.zeros((len(lens), C, H_kv, d), dtype=v.dtype)
        for b in range(len(lens)):
            kc[b, :lens[b]] = ks[b]
            vc[b, :lens[b]] = vs[b]
    else:
        kc, vc = k, v
    launches = S.kernel_launches()
    o = S.decode_attention(parity.to_device(q), parity.to_device(kc), parity.to_device(vc), lens,
                           layout, C)
    torch.cuda.synchronize()
    assert S.kernel_launches() - launches == 2 * 3
    ref = oracle.decode_attention(q, ks, vs)
    _check(o.cpu().numpy(), ref, max(np.abs(synth.bf16_to_f32(x)).max() for x in vs))
