"""CPU oracle for SnapKV prefill-time KV-cache compression (ctypes wrapper).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg use this package.  The CUDA library never imports,
links or runs it, and it shares no code with the CUDA library.  The arithmetic
lives in ``snapkv_ref.c`` (plain C, fp64; compression), ``decode.py``
(numpy, fp64; one decode step of attention over a cache), ``allq.py``
(numpy, fp64; all-query scoring) and ``scissorhands.py`` (numpy, fp64;
Scissorhands decode-time eviction); this module only
marshals numpy arrays and builds the shared object with gcc.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

from .decode import decode_attention  # noqa: F401
from .allq import compress_all_queries, scores_all_queries  # noqa: F401
from . import scissorhands  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "snapkv_ref.c")
_LIBDIR = os.path.join(_HERE, "_lib")
_LIB = os.path.join(_LIBDIR, "libsnapkv_ref.so")

BF16, FP32 = 0, 1
POOL_AVG, POOL_MAX = 0, 1
_ERR = {1: "invalid argument", 2: "non-finite logit", 3: "out of memory"}

_lib = None


def build(force: bool = False) -> str:
    """Compile snapkv_ref.c with gcc into oracle/_lib (plain -O2, no fast-math)."""
    os.makedirs(_LIBDIR, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".{os.getpid()}.tmp"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-o", tmp, _SRC, "-lm"]
        )
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i = ctypes.c_int
        ll = ctypes.c_longlong
        lib.ref_scores_unit.argtypes = [P, P, i, i, i, i, i, i, i, i, ll, P, P]
        lib.ref_pool.argtypes = [P, i, i, i, P]
        lib.ref_select.argtypes = [P, i, i, P, P]
        lib.ref_compress.argtypes = [P, P, P, i, i, i, i, i, i, P, P, P, i, i, i,
                                     P, P, P, P, P, P, P, i]
        for f in (lib.ref_scores_unit, lib.ref_pool, lib.ref_select, lib.ref_compress):
            f.restype = ctypes.c_int
        _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int) -> None:
    if rc:
        raise RuntimeError(f"oracle: {_ERR.get(rc, rc)}")


def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.uint16:
        return BF16
    if a.dtype == np.float32:
        return FP32
    raise TypeError(f"unsupported element type {a.dtype}")


def pool_code(pool) -> int:
    if pool in (POOL_AVG, "avg", "avgpool"):
        return POOL_AVG
    if pool in (POOL_MAX, "max", "maxpool"):
        return POOL_MAX
    raise ValueError(pool)


def scores(q_win: np.ndarray, k: np.ndarray, seqlens, W: int, b: int, h: int):
    """raw[j], j < P, and the window mass of unit (b, h) (fp64)."""
    lib = _load()
    q_win = np.ascontiguousarray(q_win)
    k = np.ascontiguousarray(k)
    B, Wq, H_q, d = q_win.shape
    assert Wq == W
    H_kv = k.shape[1]
    seqlens = [int(x) for x in seqlens]
    off = int(sum(seqlens[:b]))
    L = seqlens[b]
    raw = np.zeros(max(L - W, 1), np.float64)
    wm = np.zeros(1, np.float64)
    _check(lib.ref_scores_unit(_ptr(q_win), _ptr(k), _dtype_code(k), W, H_q, H_kv, d, b, h,
                               L, off, _ptr(raw), _ptr(wm)))
    return raw[: L - W], float(wm[0])


def pool(raw: np.ndarray, k_pool: int, pool_type) -> np.ndarray:
    lib = _load()
    raw = np.ascontiguousarray(raw, dtype=np.float64)
    out = np.zeros(max(len(raw), 1), np.float64)
    _check(lib.ref_pool(_ptr(raw), len(raw), int(k_pool), pool_code(pool_type), _ptr(out)))
    return out[: len(raw)]


def select(pooled: np.ndarray, n: int):
    """(ascending positions of the n best, score of the n-th best)."""
    lib = _load()
    pooled = np.ascontiguousarray(pooled, dtype=np.float64)
    sel = np.zeros(max(n, 1), np.int32)
    tau = np.zeros(1, np.float64)
    _check(lib.ref_select(_ptr(pooled), len(pooled), int(n), _ptr(sel), _ptr(tau)))
    return sel[:n], float(tau[0])


def score_offsets(seqlens, H_kv: int, W: int) -> tuple[np.ndarray, int]:
    """Offsets of each (b, h)'s P_b scores in a packed [sum_b H_kv*P_b] vector."""
    offs = []
    cur = 0
    for L in seqlens:
        P = max(int(L) - W, 0)
        for _ in range(H_kv):
            offs.append(cur)
            cur += P
    return np.asarray(offs, np.int64), cur


def compress(q_win, k, v, seqlens, W: int, k_pool: int, pool_type, C: int,
             nthreads: int | None = None) -> dict:
    """The whole compression of one layer (fp64 scores, bit-copied K/V rows).

    Returns dict with raw / pooled (lists per sequence of [H_kv, P_b] fp64),
    tau [B, H_kv], window_mass [B, H_kv], idx [B, H_kv, C] int32 and
    out_k / out_v [B, C, H_kv, d] in the input element type.
    """
    lib = _load()
    q_win = np.ascontiguousarray(q_win)
    k = np.ascontiguousarray(k)
    v = np.ascontiguousarray(v)
    B, Wq, H_q, d = q_win.shape
    assert Wq == W
    H_kv = k.shape[1]
    sl = np.asarray([int(x) for x in seqlens], np.int32)
    offs = np.concatenate([[0], np.cumsum(sl)[:-1]]).astype(np.int64)
    soffs, total = score_offsets(sl, H_kv, W)
    raw = np.zeros(max(total, 1), np.float64)
    pooled = np.zeros(max(total, 1), np.float64)
    tau = np.full(B * H_kv, np.nan)
    wm = np.zeros(B * H_kv)
    out_k = np.zeros((B, C, H_kv, d), dtype=k.dtype)
    out_v = np.zeros((B, C, H_kv, d), dtype=k.dtype)
    idx = np.zeros((B, H_kv, C), np.int32)
    nthreads = nthreads or (os.cpu_count() or 1)
    _check(lib.ref_compress(_ptr(q_win), _ptr(k), _ptr(v), _dtype_code(k), B, W, H_q, H_kv,
                            d, _ptr(sl), _ptr(offs), _ptr(soffs), int(k_pool),
                            pool_code(pool_type), int(C), _ptr(raw), _ptr(pooled), _ptr(tau),
                            _ptr(wm), _ptr(out_k), _ptr(out_v), _ptr(idx), int(nthreads)))
    raws, pooleds = [], []
    for b in range(B):
        P = max(int(sl[b]) - W, 0)
        o = int(soffs[b * H_kv])
        raws.append(raw[o:o + H_kv * P].reshape(H_kv, P))
        pooleds.append(pooled[o:o + H_kv * P].reshape(H_kv, P))
    return dict(raw=raws, pooled=pooleds, tau=tau.reshape(B, H_kv),
                window_mass=wm.reshape(B, H_kv), idx=idx, out_k=out_k, out_v=out_v)


def compress_per_q_head(q_win, k, v, seqlens, W: int, k_pool: int, pool_type, C: int,
                        nthreads=None):
    """Per-query-head selection: every query head hq scores (its own window
    sum, no group mean), pools and selects on its own over the rows of KV
    head hq // g (the pages select "for each attention head": hotpaper.ai
    summary, abstract).  That is the group-averaged compression of an MHA
    layer whose KV head hq is a copy of KV head hq // g, since a group of one
    query head has the identity as its mean; the outputs have H_q heads."""
    g = q_win.shape[2] // k.shape[1]
    kx = np.ascontiguousarray(np.repeat(k, g, axis=1))
    vx = np.ascontiguousarray(np.repeat(v, g, axis=1))
    return compress(q_win, kx, vx, seqlens, W, k_pool, pool_type, C, nthreads=nthreads)
