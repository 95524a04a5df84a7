"""The no-allocation entry point, snapkv_compress_noalloc.

Callers that cannot call cudaMalloc (an engine plugin whose device memory is
all owned by the engine's pool, or a path that cannot pay cudaMalloc's
device-wide synchronisation) use this entry point: the library's built-in
scratch array replaces the workspace.  It must give exactly what
snapkv_compress gives on the same inputs -- indices and K/V bytes are
compared bit for bit, as everywhere in these tests -- and it must do so on
consecutive calls, since every call reuses the same scratch.

This file is collected last on purpose.
"""
import ctypes

import pytest
import torch

import synth
from prefill_kv_cache_gb300 import snapkv as S
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("seqlens,H_q,H_kv,d,W,C,kp,pool,dtype", [
    ([16384], 32, 8, 128, 32, 1024, 7, "max", "bf16"),        # tensor-core score path
    ([5000, 700, 3100], 32, 8, 128, 64, 1024, 13, "avg", "bf16"),
    ([2000, 1500], 4, 4, 64, 16, 256, 5, "avg", "fp32"),      # CUDA-core score path
])
def test_noalloc_matches_compress_on_consecutive_calls(seqlens, H_q, H_kv, d, W, C, kp, pool,
                                                        dtype):
    lay = synth.make_inputs(31 + len(seqlens), seqlens, H_q, H_kv, d, W, dtype, nspans=4)
    q, k, v = (parity.to_device(x) for x in (lay.q_win, lay.k, lay.v))
    ref_k, ref_v, ref_i, _ = S.compress(q, k, v, lay.seqlens, W, kp, pool, C)
    for _ in range(2):
        ok = torch.full_like(ref_k, 7)
        ov = torch.full_like(ref_v, 7)
        oi = torch.full_like(ref_i, 7)
        S.compress_noalloc(q, k, v, lay.seqlens, W, kp, pool, C, ok, ov, oi)
        assert S.noalloc_get_status() == S.OK  # synchronizes the stream
        assert torch.equal(oi, ref_i)
        assert torch.equal(ok.view(torch.int16) if ok.dtype == torch.bfloat16 else ok,
                           ref_k.view(torch.int16) if ref_k.dtype == torch.bfloat16 else ref_k)
        assert torch.equal(ov.view(torch.int16) if ov.dtype == torch.bfloat16 else ov,
                           ref_v.view(torch.int16) if ref_v.dtype == torch.bfloat16 else ref_v)


def test_noalloc_rejects_problems_beyond_its_scratch():
    # one 380000-token prompt needs ~25 MB of workspace, above the 16 MiB limit;
    # the call returns before touching any buffer (these pointers are never used)
    shape = S.make_shape(1, 32, 8, 128, S.BF16)
    sl = (ctypes.c_int32 * 1)(380000)
    assert S.workspace_size(shape, [380000], 32, 1024) > (16 << 20)
    fake = 0x10000
    rc = S.load().snapkv_compress_noalloc(ctypes.byref(shape), fake, fake, fake, sl, 32, 7,
                                          S.POOL_MAX, 1024, fake, fake, fake, None)
    assert rc == S.ERR_WORKSPACE
    bad = S.load().snapkv_compress_noalloc(ctypes.byref(shape), fake, fake, fake, sl, 0, 7,
                                           S.POOL_MAX, 1024, fake, fake, fake, None)
    assert bad == S.ERR_INVALID_ARG


def test_noalloc_binding_checks_its_arguments():
    """The binding refuses what the C entry point cannot see: a window size
    that disagrees with q_win, strided views and mis-shaped outputs."""
    lay = synth.make_inputs(41, [3000], 32, 8, 128, 32, "bf16", nspans=2)
    q, k, v = (parity.to_device(x) for x in (lay.q_win, lay.k, lay.v))
    ok = torch.empty((1, 1024, 8, 128), dtype=torch.bfloat16, device="cuda")
    ov = torch.empty_like(ok)
    oi = torch.empty((1, 8, 1024), dtype=torch.int32, device="cuda")
    with pytest.raises(ValueError):
        S.compress_noalloc(q, k, v, [3000], 16, 7, "max", 1024, ok, ov, oi)
    with pytest.raises(ValueError):
        S.compress_noalloc(q, k, v, [3000], 32, 7, "max", 1024, ok.transpose(2, 3), ov, oi)
    with pytest.raises(ValueError):
        S.compress_noalloc(q, k, v, [3000], 32, 7, "max", 1024, ok, ov, oi[:, :4])
