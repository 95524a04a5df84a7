"""The C ABI without a GPU: exports, argument checks, workspace sizing.

No call here reaches the CUDA runtime's compute paths: every invalid case is
rejected by the library before anything is enqueued, and valid-looking cases
use fake (never dereferenced) pointers only where the library must reject
them first.
"""
import ctypes
import json
import os
import re

import pytest

from prefill_kv_cache_gb300 import snapkv as S

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
FAKE = 0x10000  # aligned, never dereferenced


def header_functions():
    text = open(os.path.join(ROOT, "include", "snapkv.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(snapkv_[a-z_]+)\s*\(", text)))


def test_library_exports_every_declared_function():
    lib = S.load()
    names = header_functions()
    assert set(names) == set(S.EXPORTED)
    for n in names:
        assert hasattr(lib, n), n
    assert S.load().snapkv_version() >= 0x000100


def shape(B=1, Hq=32, Hkv=8, d=128, dtype=S.BF16):
    return S.make_shape(B, Hq, Hkv, d, dtype)


def compress_rc(sh, seqlens, W=32, k=5, pool=0, C=1024, ptrs=None, ws_bytes=1 << 30,
                q=FAKE, kk=FAKE, v=FAKE, ok=FAKE, ov=FAKE, oi=FAKE, ws=FAKE):
    arr = (ctypes.c_int32 * len(seqlens))(*seqlens) if seqlens is not None else None
    return S.load().snapkv_compress(ctypes.byref(sh) if sh is not None else None, q, kk, v, arr,
                                    W, k, pool, C, ok, ov, oi, ws, ws_bytes, None)


@pytest.mark.parametrize("kw", [
    dict(q=None), dict(kk=None), dict(v=None), dict(ok=None), dict(ov=None), dict(oi=None),
    dict(ws=None), dict(W=0), dict(C=31), dict(k=0), dict(k=4), dict(k=-3), dict(pool=2),
    dict(q=FAKE + 8), dict(kk=FAKE + 4), dict(ok=FAKE + 2), dict(ws=FAKE + 16),
])
def test_invalid_arguments(kw):
    assert compress_rc(shape(), [4096], **kw) == S.ERR_INVALID_ARG


def lse_rc(sh, seqlens, lse=FAKE, score_only=False, W=32, C=1024, ws_bytes=1 << 30, q=FAKE):
    arr = (ctypes.c_int32 * len(seqlens))(*seqlens)
    lib = S.load()
    if score_only:
        return lib.snapkv_score_with_lse(ctypes.byref(sh), q, FAKE, lse, arr, W, C, FAKE,
                                         ws_bytes, None)
    return lib.snapkv_compress_with_lse(ctypes.byref(sh), q, FAKE, FAKE, lse, arr, W, 5, 0, C,
                                        FAKE, FAKE, FAKE, FAKE, ws_bytes, None)


@pytest.mark.parametrize("score_only", [False, True])
def test_lse_entry_points_check_arguments(score_only):
    sh = shape()
    assert lse_rc(sh, [4096], lse=None, score_only=score_only) == S.ERR_INVALID_ARG
    assert lse_rc(sh, [4096], lse=FAKE + 2, score_only=score_only) == S.ERR_INVALID_ARG
    assert lse_rc(sh, [4096], q=None, score_only=score_only) == S.ERR_INVALID_ARG
    assert lse_rc(sh, [4096], W=0, score_only=score_only) == S.ERR_INVALID_ARG
    assert lse_rc(shape(d=96), [4096], score_only=score_only) == S.ERR_UNSUPPORTED
    need = S.workspace_size(sh, [20000], 32, 1024)
    assert lse_rc(sh, [20000], ws_bytes=need - 1, score_only=score_only) == S.ERR_WORKSPACE


def test_lse_binding_checks_tensor_shape():
    import torch
    q = torch.zeros(2, 4, 8, 64)
    k = torch.zeros(100, 2, 64)
    ws = torch.zeros(16, dtype=torch.uint8)
    with pytest.raises(ValueError):
        S.score_with_lse(q, k, torch.zeros(2, 4, 7), [50, 50], 4, 32, ws)
    with pytest.raises(ValueError):
        S.score_with_lse(q, k, torch.zeros(2, 4, 8, dtype=torch.float64), [50, 50], 4, 32, ws)


def test_invalid_shapes():
    assert compress_rc(None, [4096]) == S.ERR_INVALID_ARG
    assert compress_rc(shape(), None) == S.ERR_INVALID_ARG
    assert compress_rc(shape(B=0), [4096]) == S.ERR_INVALID_ARG
    assert compress_rc(shape(B=5000), [4096] * 5000) == S.ERR_INVALID_ARG
    assert compress_rc(shape(Hq=30), [4096]) == S.ERR_INVALID_ARG
    assert compress_rc(shape(dtype=7), [4096]) == S.ERR_INVALID_ARG
    assert compress_rc(shape(B=2), [4096, 0]) == S.ERR_INVALID_ARG


def test_unsupported_shapes():
    assert compress_rc(shape(d=96), [4096]) == S.ERR_UNSUPPORTED
    assert compress_rc(shape(Hq=64, Hkv=4), [4096], W=32) == S.ERR_UNSUPPORTED  # W*g = 512


def test_workspace_too_small():
    sh = shape()
    need = S.workspace_size(sh, [20000], 32, 1024)
    assert need > 0
    assert compress_rc(sh, [20000], ws_bytes=need - 1) == S.ERR_WORKSPACE


def test_workspace_size_invalid_is_zero_and_monotone():
    sh = shape()
    assert S.workspace_size(sh, [4096], 0, 1024) == 0
    assert S.workspace_size(shape(d=96), [4096], 32, 1024) == 0
    sizes = [S.workspace_size(sh, [L], 32, 1024) for L in (100, 1024, 1025, 5000, 131072)]
    assert sizes == sorted(sizes)
    # sequences that fit the budget need no score space
    assert S.workspace_size(sh, [1024], 32, 1024) == S.workspace_size(sh, [10], 32, 1024)


def test_score_offsets_count():
    sh = shape(B=3)
    seqlens = [5000, 800, 3000]
    r, p, c = S.score_offsets(sh, seqlens, 32, 1024)
    assert c == 8 * (5000 - 32) + 8 * (3000 - 32)
    assert r % 256 == 0 and p % 256 == 0 and p >= r + 4 * c


def test_host_staging_size_covers_buffers():
    sh = shape()
    st = S.host_staging_size(sh, [16384], 32, 1024)
    kv = 16384 * 8 * 128 * 2
    assert st >= 2 * kv + S.workspace_size(sh, [16384], 32, 1024)


def test_status_strings():
    for code in range(6):
        assert S.status_string(code)
    assert S.status_string(99) == "unknown status"


def test_binding_defaults_follow_page_example():
    gold = json.load(open(os.path.join(ROOT, "tests", "golden", "page_parameters.json")))
    d = gold["api_defaults"]
    cfg = S.SnapKVConfig()
    assert (cfg.window_size, cfg.max_capacity_prompt, cfg.kernel_size, cfg.pooling) == (
        d["window_size"], d["max_capacity_prompt"], d["kernel_size"], d["pooling"])
    assert S.pool_code("avgpool") == S.POOL_AVG and S.pool_code("maxpool") == S.POOL_MAX


def decode_rc(sh, lens, layout=0, C=0, q=FAKE, k=FAKE, v=FAKE, out=FAKE, ws=FAKE, ws_bytes=1 << 30):
    arr = (ctypes.c_int32 * len(lens))(*lens)
    return S.load().snapkv_decode_attention(ctypes.byref(sh), q, k, v, layout, arr, C, out, ws,
                                            ws_bytes, None)


@pytest.mark.parametrize("kw", [
    dict(q=None), dict(k=None), dict(v=None), dict(out=None), dict(ws=None), dict(q=FAKE + 8),
    dict(out=FAKE + 4), dict(layout=2), dict(layout=-1),
])
def test_decode_invalid_arguments(kw):
    assert decode_rc(shape(), [100], **kw) == S.ERR_INVALID_ARG


def test_decode_invalid_and_unsupported_shapes():
    assert decode_rc(shape(B=2), [100, 0]) == S.ERR_INVALID_ARG
    assert decode_rc(shape(), [100], layout=S.CACHE_SLOTS, C=64) == S.ERR_INVALID_ARG  # lens > C
    assert decode_rc(shape(), [100], layout=S.CACHE_SLOTS, C=0) == S.ERR_INVALID_ARG
    assert decode_rc(shape(Hq=30), [100]) == S.ERR_INVALID_ARG
    assert decode_rc(shape(d=96), [100]) == S.ERR_UNSUPPORTED
    assert decode_rc(shape(Hq=24, Hkv=8), [100]) == S.ERR_UNSUPPORTED  # group of 3
    assert decode_rc(shape(Hq=64, Hkv=2), [100]) == S.ERR_UNSUPPORTED  # group of 32


def test_decode_workspace():
    sh = shape(B=3)
    assert S.decode_workspace_size(sh, [0, 5, 5], S.CACHE_PACKED) == 0
    need = S.decode_workspace_size(sh, [1000, 5, 70000], S.CACHE_PACKED)
    assert need > 0
    assert S.decode_workspace_size(sh, [1000, 5, 80000], S.CACHE_PACKED) >= need
    assert decode_rc(sh, [1000, 5, 70000], ws_bytes=need - 1) == S.ERR_WORKSPACE


def test_selftest_wait_checks_arguments():
    lib = S.load()
    assert lib.snapkv_selftest_wait(None, 4096, 0, None) == S.ERR_INVALID_ARG
    assert lib.snapkv_selftest_wait(FAKE, 256, 0, None) == S.ERR_INVALID_ARG
    assert lib.snapkv_selftest_wait(FAKE + 16, 4096, 0, None) == S.ERR_INVALID_ARG


def test_compress_ex_flags():
    lib = S.load()
    arr = (ctypes.c_int32 * 1)(4096)

    def rc(flags, sh):
        return lib.snapkv_compress_ex(ctypes.byref(sh), FAKE, FAKE, FAKE, arr, 32, 5, 0, 1024,
                                      FAKE, FAKE, FAKE, FAKE, 1 << 30, None, flags)
    assert rc(2, shape()) == S.ERR_INVALID_ARG
    assert rc(S.PER_QUERY_HEAD, shape(Hq=32, Hkv=2)) == S.ERR_UNSUPPORTED  # group of 16
    assert rc(S.PER_QUERY_HEAD, shape(d=96)) == S.ERR_UNSUPPORTED
    sh = shape(Hq=32, Hkv=8)
    plain = S.workspace_size(sh, [20000], 32, 1024)
    per_q = S.workspace_size(sh, [20000], 32, 1024, S.PER_QUERY_HEAD)
    assert per_q > plain  # four times the score vectors
    assert S.workspace_size(shape(Hq=8, Hkv=8), [20000], 32, 1024, S.PER_QUERY_HEAD) == \
        S.workspace_size(shape(Hq=8, Hkv=8), [20000], 32, 1024)
    r0, p0, c0 = S.score_offsets(sh, [20000], 32, 1024)
    r1, p1, c1 = S.score_offsets(sh, [20000], 32, 1024, S.PER_QUERY_HEAD)
    assert c1 == 4 * c0


def test_host_layers_entry_point_checks_arguments():
    """Argument errors return before any CUDA call (so this runs without a GPU)."""
    lib = S.load()
    shape = S.make_shape(1, 8, 2, 64, S.BF16)
    sl = (ctypes.c_int32 * 1)(3000)
    one = S.host_staging_size_layers(shape, [3000], 16, 256)
    assert one >= 2 * S.host_staging_size(shape, [3000], 16, 256)
    fake = 0x10000
    ptrs = (ctypes.c_void_p * 1)(fake)
    ev = (ctypes.c_void_p * 4)(fake, fake, fake, fake)
    call = lambda n, events: lib.snapkv_compress_host_layers(
        ctypes.byref(shape), n, ptrs, ptrs, ptrs, sl, 16, 5, 0, 256, ptrs, ptrs, ptrs, 0x10000,
        one, None, None, events)
    assert call(0, ev) == S.ERR_INVALID_ARG
    assert call(1, None) == S.ERR_INVALID_ARG
    ev0 = (ctypes.c_void_p * 4)(fake, fake, None, fake)
    assert call(1, ev0) == S.ERR_INVALID_ARG


def test_layers_entry_point_checks_arguments():
    """snapkv_compress_layers: argument errors and a short workspace return
    before any CUDA call (so this runs without a GPU)."""
    lib = S.load()
    shape = S.make_shape(1, 8, 2, 64, S.BF16)
    sl = (ctypes.c_int32 * 1)(3000)
    single = S.workspace_size(shape, [3000], 16, 256)
    for ns in range(1, S.MAX_LAYER_STREAMS + 1):
        size = S.workspace_size_layers(shape, [3000], 16, 256, ns)
        assert size >= ns * single and size % 256 == 0
    assert S.workspace_size_layers(shape, [3000], 16, 256, 0) == 0
    assert S.workspace_size_layers(shape, [3000], 16, 256, S.MAX_LAYER_STREAMS + 1) == 0
    both = S.workspace_size_layers(shape, [3000], 16, 256, 2)
    fake = 0x10000
    ptrs = (ctypes.c_void_p * 2)(fake, fake)
    sts = (ctypes.c_void_p * 2)(0x100, 0x200)
    ev = (ctypes.c_void_p * 3)(fake, fake, fake)

    def call(n, streams=sts, events=ev, ws_bytes=both, p=ptrs, ns=2, lse=None):
        return lib.snapkv_compress_layers(ctypes.byref(shape), n, p, p, p, lse, sl, 16, 5, 0, 256,
                                          p, p, p, 0x10000, ws_bytes, None, ns, streams, events)

    assert call(0) == S.ERR_INVALID_ARG
    assert call(1, ns=0) == S.ERR_INVALID_ARG
    assert call(1, ns=S.MAX_LAYER_STREAMS + 1) == S.ERR_INVALID_ARG
    assert call(1, streams=None) == S.ERR_INVALID_ARG
    assert call(1, events=None) == S.ERR_INVALID_ARG
    assert call(1, streams=(ctypes.c_void_p * 2)(0x100, 0x100)) == S.ERR_INVALID_ARG
    assert call(1, streams=(ctypes.c_void_p * 2)(0x100, None)) == S.ERR_INVALID_ARG
    assert call(1, events=(ctypes.c_void_p * 3)(fake, None, fake)) == S.ERR_INVALID_ARG
    assert call(2, p=(ctypes.c_void_p * 2)(fake, None)) == S.ERR_INVALID_ARG
    assert call(2, ws_bytes=both - 256) == S.ERR_WORKSPACE
    # an LSE array must hold a 4-byte-aligned pointer for every layer
    assert call(2, lse=(ctypes.c_void_p * 2)(fake, None)) == S.ERR_INVALID_ARG
    assert call(2, lse=(ctypes.c_void_p * 2)(fake, fake + 2)) == S.ERR_INVALID_ARG
    assert call(2, lse=(ctypes.c_void_p * 2)(fake, fake), ws_bytes=both - 256) == S.ERR_WORKSPACE
    # three streams want three workspace parts and four events
    three = S.workspace_size_layers(shape, [3000], 16, 256, 3)
    sts3 = (ctypes.c_void_p * 3)(0x100, 0x200, 0x300)
    ev4 = (ctypes.c_void_p * 4)(fake, fake, fake, None)
    assert call(1, streams=sts3, events=ev4, ws_bytes=three, ns=3) == S.ERR_INVALID_ARG
    ev4 = (ctypes.c_void_p * 4)(fake, fake, fake, fake)
    assert call(1, streams=sts3, events=ev4, ws_bytes=three - 256, ns=3) == S.ERR_WORKSPACE
    # unsupported head size, before anything else
    bad = S.make_shape(1, 8, 2, 96, S.BF16)
    assert lib.snapkv_compress_layers(ctypes.byref(bad), 1, ptrs, ptrs, ptrs, None, sl, 16, 5, 0,
                                      256, ptrs, ptrs, ptrs, 0x10000, both, None, 2, sts,
                                      ev) == S.ERR_UNSUPPORTED
    assert S.workspace_size_layers(bad, [3000], 16, 256, 2) == 0


def test_layers_binding_checks_arguments():
    """compress_layers (Python binding) rejects bad arguments before any CUDA
    call: counts of outputs, streams and events; CPU or strided tensors;
    layers of different shapes."""
    import torch

    def lay(L=3000, W=16, dev="cpu"):
        q = torch.zeros((1, W, 8, 64), dtype=torch.bfloat16, device=dev)
        k = torch.zeros((L, 2, 64), dtype=torch.bfloat16, device=dev)
        return q, k, k.clone()

    def outs(C=256):
        return (torch.zeros((1, C, 2, 64), dtype=torch.bfloat16),
                torch.zeros((1, C, 2, 64), dtype=torch.bfloat16),
                torch.zeros((1, 2, C), dtype=torch.int32))

    ws = torch.zeros(16, dtype=torch.uint8)
    one = [lay()]
    with pytest.raises(ValueError):  # no output triple for the layer
        S.compress_layers(one, [3000], 16, 5, "avg", 256, [], ws, [object()] * 2, [object()] * 3)
    with pytest.raises(ValueError):  # events: one more than streams
        S.compress_layers(one, [3000], 16, 5, "avg", 256, [outs()], ws, [object()] * 2,
                          [object()] * 2)
    with pytest.raises(ValueError):  # too many streams
        S.compress_layers(one, [3000], 16, 5, "avg", 256, [outs()], ws,
                          [object()] * (S.MAX_LAYER_STREAMS + 1),
                          [object()] * (S.MAX_LAYER_STREAMS + 2))
    with pytest.raises(ValueError):  # window size disagrees with q_win
        S.compress_layers(one, [3000], 32, 5, "avg", 256, [outs()], ws, [object()] * 2,
                          [object()] * 3)
    with pytest.raises(ValueError):  # CPU tensors
        S.compress_layers(one, [3000], 16, 5, "avg", 256, [outs()], ws, [object()] * 2,
                          [object()] * 3)
