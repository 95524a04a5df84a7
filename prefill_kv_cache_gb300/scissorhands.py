"""Python binding of the Scissorhands entry points of libsnapkv (ctypes;
argument marshalling only).

Decode-time KV-cache eviction after the abeam.tech summary of "Scissorhands:
Exploiting the Persistence of Importance Hypothesis for LLM KV Cache
Compression at Test Time" (section 技術の仕組み).  Every step runs in the
library's CUDA kernels; this module allocates the caller-owned buffers with
torch and passes pointers.  There is no Python or CPU fallback.
"""
from __future__ import annotations

import ctypes
import dataclasses

import torch

from . import snapkv as S

BUF_K, BUF_V, BUF_POS, BUF_HIST, BUF_STATE = range(5)

EXPORTED = (
    "scissorhands_buffer_bytes",
    "scissorhands_workspace_size",
    "scissorhands_init",
    "scissorhands_step",
)


class scissorhands_params(ctypes.Structure):
    _fields_ = [("budget", ctypes.c_int32), ("recent", ctypes.c_int32),
                ("history", ctypes.c_int32), ("evict", ctypes.c_int32)]


class scissorhands_cache(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("pos", ctypes.c_void_p),
                ("hist", ctypes.c_void_p), ("state", ctypes.c_void_p)]


_done = False


def load() -> ctypes.CDLL:
    global _done
    lib = S.load()
    if not _done:
        vp, sz, i32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32
        shp = ctypes.POINTER(S.snapkv_shape)
        prm = ctypes.POINTER(scissorhands_params)
        cch = ctypes.POINTER(scissorhands_cache)
        lib.scissorhands_buffer_bytes.argtypes = [shp, prm, i32]
        lib.scissorhands_buffer_bytes.restype = sz
        lib.scissorhands_workspace_size.argtypes = [shp, prm]
        lib.scissorhands_workspace_size.restype = sz
        lib.scissorhands_init.argtypes = [shp, prm, cch, vp, vp, i32, vp, vp, vp, vp]
        lib.scissorhands_init.restype = ctypes.c_int
        lib.scissorhands_step.argtypes = [shp, prm, cch, vp, vp, vp, vp, vp, sz, vp]
        lib.scissorhands_step.restype = ctypes.c_int
        _done = True
    return lib


@dataclasses.dataclass
class Params:
    """budget per KV head; recent r kept; history w steps; evict m per batch
    (the page's runs: w = 400, r = 10, m = budget / 2)."""
    budget: int
    recent: int = 10
    history: int = 400
    evict: int | None = None

    def c(self) -> scissorhands_params:
        m = self.budget // 2 if self.evict is None else self.evict
        return scissorhands_params(int(self.budget), int(self.recent), int(self.history), int(m))


def buffer_bytes(shape: S.snapkv_shape, params: Params, which: int) -> int:
    p = params.c()
    return int(load().scissorhands_buffer_bytes(ctypes.byref(shape), ctypes.byref(p), int(which)))


def workspace_size(shape: S.snapkv_shape, params: Params) -> int:
    p = params.c()
    return int(load().scissorhands_workspace_size(ctypes.byref(shape), ctypes.byref(p)))


class Cache:
    """One layer's device buffers (include/scissorhands.h, scissorhands_cache)
    plus the step workspace, allocated with torch on `device`."""

    def __init__(self, B, H_q, H_kv, d, dtype, params: Params, device="cuda"):
        self.shape = S.make_shape(B, H_q, H_kv, d, dtype)
        self.params = params
        self.dtype = dtype
        sizes = [buffer_bytes(self.shape, params, w) for w in range(5)]
        ws = workspace_size(self.shape, params)
        if min(sizes) == 0 or ws == 0:
            raise S.SnapKVError(S.ERR_INVALID_ARG, "scissorhands_buffer_bytes")
        cap = params.budget + 1
        hw = (params.history + 31) // 32
        self.k = torch.empty((B, cap, H_kv, d), dtype=dtype, device=device)
        self.v = torch.empty_like(self.k)
        self.pos = torch.empty((B, H_kv, cap), dtype=torch.int32, device=device)
        self.hist = torch.empty((B, H_kv, hw, cap), dtype=torch.int32, device=device)
        self.state = torch.empty((B, 4), dtype=torch.int32, device=device)
        self.workspace = torch.empty(ws, dtype=torch.uint8, device=device)
        for t, n in zip((self.k, self.v, self.pos, self.hist, self.state), sizes):
            assert t.numel() * t.element_size() == n
        self._c = scissorhands_cache(self.k.data_ptr(), self.v.data_ptr(), self.pos.data_ptr(),
                                     self.hist.data_ptr(), self.state.data_ptr())
        self._p = params.c()

    def init(self, lens0, next_pos0, k0=None, v0=None, pos0=None, stream=None):
        """scissorhands_init: k0 / v0 [B, C0, H_kv, d] (e.g. snapkv compress's
        out_k / out_v), pos0 int32 [B, H_kv, C0] or None."""
        B = self.shape.batch
        lens, _ = S._seqlens_array(lens0)
        nxt, _ = S._seqlens_array(next_pos0)
        if len(lens) != B or len(nxt) != B:
            raise ValueError("lens0 and next_pos0 need one entry per sequence")
        C0 = 0 if k0 is None else k0.shape[1]
        for name, t in (("k0", k0), ("v0", v0), ("pos0", pos0)):
            if t is not None and not t.is_contiguous():
                raise ValueError(f"{name} must be contiguous")
        if pos0 is not None and pos0.dtype != torch.int32:
            raise ValueError("pos0 must be int32")
        ptr = lambda t: None if t is None else t.data_ptr()
        rc = load().scissorhands_init(ctypes.byref(self.shape), ctypes.byref(self._p),
                                      ctypes.byref(self._c), ptr(k0), ptr(v0), C0, ptr(pos0),
                                      lens, nxt, S._stream_handle(stream))
        if rc:
            raise S.SnapKVError(rc, "scissorhands_init")

    def step(self, q, k_new, v_new, out=None, stream=None) -> torch.Tensor:
        """scissorhands_step: q [B, H_q, d], k_new / v_new [B, H_kv, d] in the
        cache dtype.  Returns fp32 [B, H_q, d]."""
        if out is None:
            out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
        for name, t in (("q", q), ("k_new", k_new), ("v_new", v_new), ("out", out)):
            if not t.is_contiguous():
                raise ValueError(f"{name} must be contiguous")
        rc = load().scissorhands_step(ctypes.byref(self.shape), ctypes.byref(self._p),
                                      ctypes.byref(self._c), q.data_ptr(), k_new.data_ptr(),
                                      v_new.data_ptr(), out.data_ptr(), self.workspace.data_ptr(),
                                      self.workspace.numel(), S._stream_handle(stream))
        if rc:
            raise S.SnapKVError(rc, "scissorhands_step")
        return out
