"""GPU parity of all-query scoring (snapkv_compress_all_queries) against the
oracle (oracle/allq.py), with the agreement rule of tests/parity.py.  The
caller's per-row LSE is computed here in fp64 on the CPU (rounded to fp32)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from prefill_kv_cache_gb300 import snapkv as S
from tests import parity

pytestmark = pytest.mark.gpu


def _all_lse(q_all, k, seqlens, g):
    """[T, H_q] natural-log LSE of every query row over its keys j <= i."""
    q = torch.from_numpy(synth.bf16_to_f32(q_all) if q_all.dtype == np.uint16 else q_all)
    kk = torch.from_numpy(synth.bf16_to_f32(k) if k.dtype == np.uint16 else k)
    T, H_q, d = q.shape
    out = np.zeros((T, H_q), np.float32)
    off = 0
    for L in seqlens:
        L = int(L)
        mask = torch.ones(L, L, dtype=torch.bool).tril()
        for hq in range(H_q):
            s = q[off:off + L, hq].double() @ kk[off:off + L, hq // g].double().T / np.sqrt(d)
            out[off:off + L, hq] = torch.logsumexp(s.masked_fill(~mask, float("-inf")), 1).numpy()
        off += L
    return out


CASES = [
    # seqlens,          H_q, H_kv, d,  W,  C,  k, pool,  dtype
    ([700, 130],          8,   2, 128, 16, 128, 5, "avg", "bf16"),
    ([1500],              8,   8, 64,  32, 256, 7, "max", "fp32"),
    ([900, 40, 1200],    16,   4, 64,  16, 200, 3, "avg", "bf16"),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"L{c[0]}-g{c[1]//c[2]}-d{c[3]}-{c[8]}")
def test_all_queries_matches_oracle(case):
    seqlens, H_q, H_kv, d, W, C, kp, pool, dtype = case
    lay = synth.make_inputs(77 + sum(seqlens), seqlens, H_q, H_kv, d, W, dtype, nspans=2)
    rng = np.random.default_rng(sum(seqlens))
    q_all = (1.5 * rng.standard_normal((sum(seqlens), H_q, d))).astype(np.float32)
    if dtype == "bf16":
        q_all = synth.bf16_round(q_all)
    lse = _all_lse(q_all, lay.k, seqlens, H_q // H_kv)
    ok, ov, oi, ws = S.compress_all_queries(parity.to_device(q_all), parity.to_device(lay.k),
                                            parity.to_device(lay.v), parity.to_device(lse),
                                            seqlens, W, kp, pool, C)
    assert S.get_status(ws) == S.OK
    shape = S.make_shape(lay.B, H_q, H_kv, d, ok.dtype)
    raw, pooled = S.scores_from_workspace(ws, shape, seqlens, W, C)
    torch.cuda.synchronize()

    def host(t):
        t = t.cpu()
        return t.view(torch.int16).numpy().view(np.uint16) if t.dtype == torch.bfloat16 else t.numpy()

    gpu = dict(out_k=host(ok), out_v=host(ov), idx=oi.cpu().numpy(), raw=raw.cpu().numpy(),
               pooled=pooled.cpu().numpy())
    ora = oracle.compress_all_queries(q_all, lay.k, lay.v, seqlens, W, kp, pool, C)
    parity.check(lay, gpu, ora, C)
