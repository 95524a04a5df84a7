"""Pins of the decode-attention oracle (oracle/decode.py), on the CPU.

Each pin fixes the oracle against something other than its own formula: a
closed form, a library routine (torch's scaled-dot-product attention in
fp64), or an invariant of softmax attention.
"""
import numpy as np
import pytest
import torch

import oracle


def _rand(seed, B, H_q, H_kv, d, lens):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, H_q, d))
    ks = [rng.standard_normal((n, H_kv, d)) for n in lens]
    vs = [rng.standard_normal((n, H_kv, d)) for n in lens]
    return q, ks, vs


def test_zero_query_is_the_mean_of_the_values():
    q, ks, vs = _rand(1, 3, 8, 2, 64, [5, 17, 1])
    q[:] = 0
    o = oracle.decode_attention(q, ks, vs)
    for b in range(3):
        for hq in range(8):
            np.testing.assert_allclose(o[b, hq], vs[b][:, hq // 4].mean(axis=0), rtol=1e-13,
                                       atol=1e-13)


def test_single_row_returns_its_value():
    q, ks, vs = _rand(2, 2, 4, 4, 32, [1, 1])
    o = oracle.decode_attention(q, ks, vs)
    for b in range(2):
        np.testing.assert_array_equal(o[b], vs[b][0])


@pytest.mark.parametrize("H_q,H_kv,d", [(8, 8, 64), (32, 8, 128), (16, 2, 64)])
def test_matches_torch_sdpa(H_q, H_kv, d):
    lens = [7, 300, 64]
    q, ks, vs = _rand(3 + H_q, len(lens), H_q, H_kv, d, lens)
    o = oracle.decode_attention(q, ks, vs)
    g = H_q // H_kv
    for b, n in enumerate(lens):
        K = torch.from_numpy(ks[b]).permute(1, 0, 2).repeat_interleave(g, dim=0)  # [H_q, n, d]
        V = torch.from_numpy(vs[b]).permute(1, 0, 2).repeat_interleave(g, dim=0)
        Q = torch.from_numpy(q[b])[:, None, :]                                     # [H_q, 1, d]
        ref = torch.nn.functional.scaled_dot_product_attention(Q, K, V)[:, 0, :].numpy()
        np.testing.assert_allclose(o[b], ref, rtol=1e-12, atol=1e-12)


def test_key_shift_leaves_the_output_unchanged():
    q, ks, vs = _rand(4, 2, 8, 2, 64, [50, 9])
    o = oracle.decode_attention(q, ks, vs)
    u = np.random.default_rng(5).standard_normal(64)
    o2 = oracle.decode_attention(q, [k + u for k in ks], vs)
    np.testing.assert_allclose(o2, o, rtol=1e-10, atol=1e-12)


def test_dominant_key_selects_its_value():
    q, ks, vs = _rand(6, 1, 4, 1, 64, [40])
    ks[0][17, 0] = 50.0 * q[0, 0] / np.linalg.norm(q[0, 0])  # logit ~ 50 |q| / 8 for head 0
    o = oracle.decode_attention(q, ks, vs)
    np.testing.assert_allclose(o[0, 0], vs[0][17, 0], atol=1e-6)


def test_bf16_bits_are_widened_exactly():
    q, ks, vs = _rand(7, 1, 2, 1, 64, [8])
    to_bf16 = lambda a: (a.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    back = lambda h: (h.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    qb, kb, vb = to_bf16(q), [to_bf16(ks[0])], [to_bf16(vs[0])]
    o = oracle.decode_attention(qb, kb, vb)
    o_ref = oracle.decode_attention(back(qb), [back(kb[0])], [back(vb[0])])
    np.testing.assert_array_equal(o, o_ref)
