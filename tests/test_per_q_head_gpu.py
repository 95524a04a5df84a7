"""GPU parity of per-query-head selection (snapkv_compress_ex with
SNAPKV_PER_QUERY_HEAD) against the oracle: the GPU runs on the layer itself,
the oracle and the agreement rule (tests/parity.py) on the same layer with
each KV head repeated for its query heads (tests/parity.expand_heads)."""
import numpy as np
import pytest

import synth
from prefill_kv_cache_gb300 import snapkv as S
from tests import parity

pytestmark = pytest.mark.gpu

CASES = [
    # seqlens,              H_q, H_kv, d,  W,  C,   k, pool,  dtype   (score path)
    ([3000, 700],             32,   8, 128, 32, 1024, 7, "max", "bf16"),  # tensor cores, g = 4
    ([5000],                  32,   4, 128, 32, 2048, 5, "avg", "bf16"),  # tensor cores, g = 8
    ([2049, 40],               8,   4, 64,  64, 512, 13, "avg", "bf16"),  # tensor cores, g = 2
    ([1500, 333],              8,   2, 64,  16, 256,  5, "max", "fp32"),  # FFMA, g = 4
    ([900],                    4,   4, 128, 16, 300,  3, "avg", "bf16"),  # g = 1
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"L{c[0]}-g{c[1]//c[2]}-d{c[3]}-W{c[4]}-{c[8]}")
def test_per_q_head_matches_oracle(case):
    seqlens, H_q, H_kv, d, W, C, kp, pool, dtype = case
    lay = synth.make_inputs(333 + sum(seqlens), seqlens, H_q, H_kv, d, W, dtype, nspans=3)
    gpu = parity.run_gpu(lay, kp, pool, C, flags=S.PER_QUERY_HEAD)
    lx = parity.expand_heads(lay)
    ora = parity.oracle_for(lx, kp, pool, C)
    parity.check(lx, gpu, ora, C)


def test_per_q_head_full_size_sampled():
    """The Mistral-7B 8 x 32K layer (g = 4) at full size; the oracle checks
    two sequences."""
    cfg = synth.CONFIGS["3"]
    lay = synth.make_layer("3", 0)
    gpu = parity.run_gpu(lay, cfg["k_pool"], cfg["pool"], cfg["C"], flags=S.PER_QUERY_HEAD)
    lx = parity.expand_heads(lay)
    ora = parity.oracle_for(lx, cfg["k_pool"], cfg["pool"], cfg["C"], seqs=[0, 5])
    parity.check(lx, gpu, ora, cfg["C"], seqs=[0, 5])
