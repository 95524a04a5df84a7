"""The Scissorhands C ABI without a GPU: exports, argument checks, sizes.

Every call here is rejected by the library before anything is enqueued;
pointers are fake and never dereferenced.
"""
import ctypes
import os
import re

import pytest

from prefill_kv_cache_gb300 import scissorhands as SH
from prefill_kv_cache_gb300 import snapkv as S

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
FAKE = 0x10000


def test_library_exports_every_declared_function():
    text = open(os.path.join(ROOT, "include", "scissorhands.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = sorted(set(re.findall(r"\b(scissorhands_[a-z_]+)\s*\(", text)))
    assert set(names) == set(SH.EXPORTED)
    lib = SH.load()
    for n in names:
        assert hasattr(lib, n), n


def _shape(B=2, Hq=32, Hkv=8, d=128, dtype=S.BF16):
    return S.make_shape(B, Hq, Hkv, d, dtype)


def _prm(budget=64, recent=4, history=40, evict=32):
    return SH.scissorhands_params(budget, recent, history, evict)


def test_buffer_sizes_follow_the_layout():
    sh, p = _shape(), _prm()
    cap, hw = 65, 2
    lib = SH.load()
    size = lambda w: lib.scissorhands_buffer_bytes(ctypes.byref(sh), ctypes.byref(p), w)
    assert size(SH.BUF_K) == size(SH.BUF_V) == 2 * cap * 8 * 128 * 2
    assert size(SH.BUF_POS) == 2 * 8 * cap * 4
    assert size(SH.BUF_HIST) == 2 * 8 * hw * cap * 4
    assert size(SH.BUF_STATE) == 2 * 4 * 4
    assert size(5) == 0
    ws = lib.scissorhands_workspace_size(ctypes.byref(sh), ctypes.byref(p))
    assert ws >= 2 * 32 * cap * 4 + 256  # at least the logits and the counter


@pytest.mark.parametrize("kw", [
    dict(budget=0), dict(budget=16384), dict(recent=0), dict(recent=65), dict(history=0),
    dict(history=1025), dict(evict=0), dict(evict=62),  # > budget + 1 - recent
])
def test_invalid_parameters(kw):
    args = dict(budget=64, recent=4, history=40, evict=32)
    args.update(kw)
    sh, p = _shape(), _prm(**args)
    lib = SH.load()
    assert lib.scissorhands_workspace_size(ctypes.byref(sh), ctypes.byref(p)) == 0
    for w in range(5):
        assert lib.scissorhands_buffer_bytes(ctypes.byref(sh), ctypes.byref(p), w) == 0
    assert _step_rc(sh=sh, p=p) == S.ERR_INVALID_ARG
    assert _init_rc(sh=sh, p=p) == S.ERR_INVALID_ARG


def _cache(**kw):
    f = dict(k=FAKE, v=FAKE, pos=FAKE, hist=FAKE, state=FAKE)
    f.update(kw)
    return SH.scissorhands_cache(f["k"], f["v"], f["pos"], f["hist"], f["state"])


def _step_rc(sh=None, p=None, c=None, q=FAKE, kn=FAKE, vn=FAKE, out=FAKE, ws=FAKE,
             ws_bytes=1 << 30):
    sh = sh or _shape()
    p = p or _prm()
    c = c or _cache()
    return SH.load().scissorhands_step(ctypes.byref(sh), ctypes.byref(p), ctypes.byref(c), q,
                                       kn, vn, out, ws, ws_bytes, None)


def _init_rc(sh=None, p=None, c=None, k0=FAKE, v0=FAKE, C0=64, pos0=None, lens=(10, 20),
             nxt=(100, 200)):
    sh = sh or _shape()
    p = p or _prm()
    c = c or _cache()
    la = (ctypes.c_int32 * len(lens))(*lens)
    na = (ctypes.c_int32 * len(nxt))(*nxt)
    return SH.load().scissorhands_init(ctypes.byref(sh), ctypes.byref(p), ctypes.byref(c), k0,
                                       v0, C0, pos0, la, na, None)


@pytest.mark.parametrize("kw", [
    dict(q=None), dict(kn=None), dict(vn=None), dict(out=None), dict(ws=None),
    dict(q=FAKE + 8), dict(kn=FAKE + 4), dict(out=FAKE + 2), dict(ws=FAKE + 16),
    dict(c=_cache(k=None)), dict(c=_cache(hist=None)), dict(c=_cache(state=FAKE + 4)),
])
def test_step_invalid_arguments(kw):
    assert _step_rc(**kw) == S.ERR_INVALID_ARG


def test_step_workspace_too_small():
    sh, p = _shape(), _prm()
    need = SH.load().scissorhands_workspace_size(ctypes.byref(sh), ctypes.byref(p))
    assert _step_rc(ws_bytes=need - 1) == S.ERR_WORKSPACE


@pytest.mark.parametrize("kw,code", [
    (dict(sh=_shape(d=96)), S.ERR_UNSUPPORTED),
    (dict(sh=_shape(Hq=24, Hkv=8)), S.ERR_UNSUPPORTED),   # g = 3
    (dict(sh=_shape(Hq=30, Hkv=8)), S.ERR_INVALID_ARG),
    (dict(sh=_shape(dtype=7)), S.ERR_INVALID_ARG),
    (dict(sh=_shape(B=0)), S.ERR_INVALID_ARG),
])
def test_shapes(kw, code):
    assert _step_rc(**kw) == code


@pytest.mark.parametrize("kw", [
    dict(lens=(10, 65)),          # above budget
    dict(lens=(10, -1)),
    dict(C0=8),                   # lens above C0
    dict(nxt=(-1, 0)),
    dict(k0=None),                # rows to load but no source
    dict(v0=FAKE + 8),
    dict(c=_cache(pos=None)),
])
def test_init_invalid_arguments(kw):
    assert _init_rc(**kw) == S.ERR_INVALID_ARG


def test_binding_default_parameters_follow_the_page():
    p = SH.Params(budget=1024).c()
    assert (p.budget, p.recent, p.history, p.evict) == (1024, 10, 400, 512)
