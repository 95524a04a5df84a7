"""Failure detection without a GPU fault: a bounded device-side wait on a flag
that nothing sets runs out, the status word reports it, and the context stays
usable for the next compression."""
import pytest
import torch

import synth
from prefill_kv_cache_gb300 import snapkv as S
from tests import parity

pytestmark = pytest.mark.gpu


def test_unset_flag_times_out_and_context_survives():
    ws = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    assert S.selftest_wait(ws, set_flag=True) == S.OK
    assert S.selftest_wait(ws, set_flag=False) == S.ERR_TIMEOUT
    # the context is still usable: a compression right after is correct
    lay = synth.make_inputs(3, [3000, 500], 32, 8, 128, 32, "bf16", nspans=2)
    gpu = parity.run_gpu(lay, 5, "avg", 1024)
    ora = parity.oracle_for(lay, 5, "avg", 1024)
    parity.check(lay, gpu, ora, 1024)
    assert S.selftest_wait(ws, set_flag=True) == S.OK
