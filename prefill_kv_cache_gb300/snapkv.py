"""Python binding of libsnapkv (ctypes; argument marshalling only).

Every step of the compression runs in the library's CUDA kernels; this module
only turns torch tensors into pointers, sizes and a stream handle.  If the
shared library is missing it raises: there is no Python or CPU fallback.

Keyword names follow the SnapKV usage example on the jisaku.com glossary page
"SnapKV" (section "実装と統合"): window_size, max_capacity_prompt, kernel_size,
pooling ("avgpool" / "maxpool").
"""
from __future__ import annotations

import ctypes
import dataclasses
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libsnapkv.so")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_WORKSPACE, ERR_CUDA, ERR_TIMEOUT = range(6)
POOL_AVG, POOL_MAX = 0, 1
BF16, FP32 = 0, 1

EXPORTED = (
    "snapkv_workspace_size",
    "snapkv_compress",
    "snapkv_score",
    "snapkv_compress_with_lse",
    "snapkv_score_with_lse",
    "snapkv_decode_workspace_size",
    "snapkv_decode_attention",
    "snapkv_selftest_wait",
    "snapkv_workspace_size_ex",
    "snapkv_score_offsets_ex",
    "snapkv_compress_ex",
    "snapkv_compress_all_queries",
    "snapkv_score_offsets",
    "snapkv_get_status",
    "snapkv_host_staging_size",
    "snapkv_compress_host",
    "snapkv_host_staging_size_layers",
    "snapkv_compress_host_layers",
    "snapkv_workspace_size_layers",
    "snapkv_compress_layers",
    "snapkv_compress_noalloc",
    "snapkv_noalloc_get_status",
    "snapkv_kernel_launches",
    "snapkv_score_path_launches",
    "snapkv_status_string",
    "snapkv_version",
)


class SnapKVError(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        self.code = code
        super().__init__(f"{what}: {status_string(code)} ({code})" if what else status_string(code))


class snapkv_shape(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("dtype", ctypes.c_int32)]


_lib = None


def load() -> ctypes.CDLL:
    """Load libsnapkv.so (built by __graft_entry__.build()); raise if absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"libsnapkv.so is not built ({LIB_PATH}); run __graft_entry__.build()")
    lib = ctypes.CDLL(LIB_PATH)
    vp, sz, i32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32
    shp = ctypes.POINTER(snapkv_shape)
    lib.snapkv_workspace_size.argtypes = [shp, vp, i32, i32]
    lib.snapkv_workspace_size.restype = sz
    lib.snapkv_compress.argtypes = [shp, vp, vp, vp, vp, i32, i32, i32, i32, vp, vp, vp, vp, sz, vp]
    lib.snapkv_compress.restype = ctypes.c_int
    lib.snapkv_score.argtypes = [shp, vp, vp, vp, i32, i32, vp, sz, vp]
    lib.snapkv_score.restype = ctypes.c_int
    lib.snapkv_compress_with_lse.argtypes = [shp, vp, vp, vp, vp, vp, i32, i32, i32, i32, vp, vp,
                                             vp, vp, sz, vp]
    lib.snapkv_compress_with_lse.restype = ctypes.c_int
    lib.snapkv_score_with_lse.argtypes = [shp, vp, vp, vp, vp, i32, i32, vp, sz, vp]
    lib.snapkv_score_with_lse.restype = ctypes.c_int
    lib.snapkv_decode_workspace_size.argtypes = [shp, vp, i32, i32]
    lib.snapkv_decode_workspace_size.restype = sz
    lib.snapkv_decode_attention.argtypes = [shp, vp, vp, vp, i32, vp, i32, vp, vp, sz, vp]
    lib.snapkv_decode_attention.restype = ctypes.c_int
    lib.snapkv_selftest_wait.argtypes = [vp, sz, i32, vp]
    lib.snapkv_selftest_wait.restype = ctypes.c_int
    lib.snapkv_workspace_size_ex.argtypes = [shp, vp, i32, i32, i32]
    lib.snapkv_workspace_size_ex.restype = sz
    lib.snapkv_score_offsets_ex.argtypes = [shp, vp, i32, i32, i32, ctypes.POINTER(sz),
                                            ctypes.POINTER(sz), ctypes.POINTER(sz)]
    lib.snapkv_score_offsets_ex.restype = ctypes.c_int
    lib.snapkv_compress_ex.argtypes = [shp, vp, vp, vp, vp, i32, i32, i32, i32, vp, vp, vp, vp,
                                       sz, vp, i32]
    lib.snapkv_compress_ex.restype = ctypes.c_int
    lib.snapkv_compress_all_queries.argtypes = [shp, vp, vp, vp, vp, vp, i32, i32, i32, i32, vp,
                                                vp, vp, vp, sz, vp]
    lib.snapkv_compress_all_queries.restype = ctypes.c_int
    lib.snapkv_kernel_launches.argtypes = []
    lib.snapkv_kernel_launches.restype = ctypes.c_uint64
    lib.snapkv_score_path_launches.argtypes = [i32]
    lib.snapkv_score_path_launches.restype = ctypes.c_uint64
    lib.snapkv_score_offsets.argtypes = [shp, vp, i32, i32, ctypes.POINTER(sz),
                                         ctypes.POINTER(sz), ctypes.POINTER(sz)]
    lib.snapkv_score_offsets.restype = ctypes.c_int
    lib.snapkv_get_status.argtypes = [vp, sz, vp]
    lib.snapkv_get_status.restype = ctypes.c_int
    lib.snapkv_host_staging_size.argtypes = [shp, vp, i32, i32]
    lib.snapkv_host_staging_size.restype = sz
    lib.snapkv_compress_host.argtypes = [shp, vp, vp, vp, vp, i32, i32, i32, i32, vp, vp, vp,
                                         vp, sz, vp]
    lib.snapkv_compress_host.restype = ctypes.c_int
    lib.snapkv_host_staging_size_layers.argtypes = [shp, vp, i32, i32]
    lib.snapkv_host_staging_size_layers.restype = sz
    lib.snapkv_compress_host_layers.argtypes = [shp, i32, vp, vp, vp, vp, i32, i32, i32, i32,
                                                vp, vp, vp, vp, sz, vp, vp, vp]
    lib.snapkv_compress_host_layers.restype = ctypes.c_int
    lib.snapkv_workspace_size_layers.argtypes = [shp, vp, i32, i32, i32]
    lib.snapkv_workspace_size_layers.restype = sz
    lib.snapkv_compress_layers.argtypes = [shp, i32, vp, vp, vp, vp, vp, i32, i32, i32, i32, vp,
                                           vp, vp, vp, sz, vp, i32, vp, vp]
    lib.snapkv_compress_layers.restype = ctypes.c_int
    lib.snapkv_compress_noalloc.argtypes = [shp, vp, vp, vp, vp, i32, i32, i32, i32, vp, vp, vp,
                                            vp]
    lib.snapkv_compress_noalloc.restype = ctypes.c_int
    lib.snapkv_noalloc_get_status.argtypes = [vp]
    lib.snapkv_noalloc_get_status.restype = ctypes.c_int
    lib.snapkv_status_string.argtypes = [ctypes.c_int]
    lib.snapkv_status_string.restype = ctypes.c_char_p
    lib.snapkv_version.argtypes = []
    lib.snapkv_version.restype = ctypes.c_int
    _lib = lib
    return lib


def status_string(code: int) -> str:
    return load().snapkv_status_string(int(code)).decode()


def pool_code(pooling) -> int:
    if pooling in ("avgpool", "avg", POOL_AVG):
        return POOL_AVG
    if pooling in ("maxpool", "max", POOL_MAX):
        return POOL_MAX
    raise ValueError(f"unknown pooling {pooling!r}")


def dtype_code(dtype) -> int:
    if dtype == torch.bfloat16:
        return BF16
    if dtype == torch.float32:
        return FP32
    raise TypeError(f"unsupported dtype {dtype}")


@dataclasses.dataclass
class SnapKVConfig:
    """The four knobs of the pages' usage example, with its default values."""
    window_size: int = 32
    max_capacity_prompt: int = 4096
    kernel_size: int = 5
    pooling: str = "avgpool"


def _seqlens_array(seqlens):
    vals = [int(x) for x in seqlens]
    arr = (ctypes.c_int32 * len(vals))(*vals)
    return arr, len(vals)


def make_shape(batch, num_q_heads, num_kv_heads, head_dim, dtype) -> snapkv_shape:
    return snapkv_shape(int(batch), int(num_q_heads), int(num_kv_heads), int(head_dim),
                        dtype if isinstance(dtype, int) else dtype_code(dtype))


PER_QUERY_HEAD = 1  # flag of the _ex entry points (include/snapkv.h)


def workspace_size(shape: snapkv_shape, seqlens, window_size: int, max_capacity_prompt: int,
                   flags: int = 0) -> int:
    arr, _ = _seqlens_array(seqlens)
    if flags:
        return int(load().snapkv_workspace_size_ex(ctypes.byref(shape), arr, int(window_size),
                                                   int(max_capacity_prompt), int(flags)))
    return int(load().snapkv_workspace_size(ctypes.byref(shape), arr, int(window_size),
                                            int(max_capacity_prompt)))


def score_offsets(shape: snapkv_shape, seqlens, window_size: int, max_capacity_prompt: int,
                  flags: int = 0):
    arr, _ = _seqlens_array(seqlens)
    r, p, c = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    rc = load().snapkv_score_offsets_ex(ctypes.byref(shape), arr, int(window_size),
                                        int(max_capacity_prompt), int(flags), ctypes.byref(r),
                                        ctypes.byref(p), ctypes.byref(c))
    if rc:
        raise SnapKVError(rc, "snapkv_score_offsets")
    return r.value, p.value, c.value


def _stream_handle(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def compress(q_win: torch.Tensor, k: torch.Tensor, v: torch.Tensor, seqlens,
             window_size: int, kernel_size: int, pooling, max_capacity_prompt: int,
             out_k: torch.Tensor | None = None, out_v: torch.Tensor | None = None,
             out_idx: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
             stream=None, lse_win: torch.Tensor | None = None, flags: int = 0):
    """Compress one layer (see include/snapkv.h, snapkv_compress).

    q_win [B, W, H_q, d], k / v [T, H_kv, d] (packed, bf16 or fp32, CUDA);
    seqlens: B host integers.  Returns (out_k, out_v, out_idx, workspace);
    outputs that are not given are allocated here with torch.  With lse_win
    (fp32 [B, W, H_q], the window rows' natural-log LSE) the call goes to
    snapkv_compress_with_lse; with flags (PER_QUERY_HEAD) to snapkv_compress_ex,
    whose outputs have H_q heads.
    """
    B, W, H_q, d = q_win.shape
    H_kv = k.shape[1]
    C = int(max_capacity_prompt)
    if W != int(window_size):
        raise ValueError("q_win's second dimension must equal window_size")
    shape = make_shape(B, H_q, H_kv, d, q_win.dtype)
    H_out = H_q if flags & PER_QUERY_HEAD else H_kv
    if lse_win is not None and flags:
        raise ValueError("lse_win and flags cannot be combined")
    if out_k is None:
        out_k = torch.empty((B, C, H_out, d), dtype=k.dtype, device=k.device)
    if out_v is None:
        out_v = torch.empty((B, C, H_out, d), dtype=k.dtype, device=k.device)
    if out_idx is None:
        out_idx = torch.empty((B, H_out, C), dtype=torch.int32, device=k.device)
    ws_bytes = workspace_size(shape, seqlens, W, C, flags)
    if ws_bytes == 0:
        raise SnapKVError(ERR_INVALID_ARG, "snapkv_workspace_size")
    if workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=k.device)
    for name, t in (("q_win", q_win), ("k", k), ("v", v), ("out_k", out_k), ("out_v", out_v),
                    ("out_idx", out_idx), ("workspace", workspace)):
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    arr, _ = _seqlens_array(seqlens)
    if lse_win is not None:
        _check_lse(lse_win, B, W, H_q)
    ws_args = (workspace.data_ptr(), workspace.numel() * workspace.element_size(),
               _stream_handle(stream))
    if flags:
        rc = load().snapkv_compress_ex(ctypes.byref(shape), q_win.data_ptr(), k.data_ptr(),
                                       v.data_ptr(), arr, W, int(kernel_size), pool_code(pooling),
                                       C, out_k.data_ptr(), out_v.data_ptr(), out_idx.data_ptr(),
                                       *ws_args, int(flags))
        name = "snapkv_compress_ex"
    elif lse_win is None:
        rc = load().snapkv_compress(ctypes.byref(shape), q_win.data_ptr(), k.data_ptr(),
                                    v.data_ptr(), arr, W, int(kernel_size), pool_code(pooling), C,
                                    out_k.data_ptr(), out_v.data_ptr(), out_idx.data_ptr(),
                                    *ws_args)
        name = "snapkv_compress"
    else:
        rc = load().snapkv_compress_with_lse(ctypes.byref(shape), q_win.data_ptr(), k.data_ptr(),
                                             v.data_ptr(), lse_win.data_ptr(), arr, W,
                                             int(kernel_size), pool_code(pooling), C,
                                             out_k.data_ptr(), out_v.data_ptr(),
                                             out_idx.data_ptr(), *ws_args)
        name = "snapkv_compress_with_lse"
    if rc:
        raise SnapKVError(rc, name)
    return out_k, out_v, out_idx, workspace


def _check_lse(lse_win: torch.Tensor, B: int, W: int, H_q: int) -> None:
    if lse_win.dtype != torch.float32 or tuple(lse_win.shape) != (B, W, H_q) or \
            not lse_win.is_contiguous():
        raise ValueError(f"lse_win must be a contiguous float32 tensor of shape {(B, W, H_q)}")


def compress_with_lse(q_win: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                      lse_win: torch.Tensor, seqlens, window_size: int, kernel_size: int, pooling,
                      max_capacity_prompt: int, **kw):
    """snapkv_compress_with_lse (include/snapkv.h): the caller gives the window
    rows' log-sum-exp, so only the column-sum sweep over K runs."""
    return compress(q_win, k, v, seqlens, window_size, kernel_size, pooling, max_capacity_prompt,
                    lse_win=lse_win, **kw)


def score(q_win: torch.Tensor, k: torch.Tensor, seqlens, window_size: int,
          max_capacity_prompt: int, workspace: torch.Tensor, stream=None,
          lse_win: torch.Tensor | None = None) -> None:
    """Scoring step only (include/snapkv.h, snapkv_score, or snapkv_score_with_lse
    when lse_win is given); raw scores stay in workspace."""
    B, W, H_q, d = q_win.shape
    shape = make_shape(B, H_q, k.shape[1], d, q_win.dtype)
    arr, _ = _seqlens_array(seqlens)
    if lse_win is not None:
        _check_lse(lse_win, B, W, H_q)
    tail = (W, int(max_capacity_prompt), workspace.data_ptr(),
            workspace.numel() * workspace.element_size(), _stream_handle(stream))
    if lse_win is None:
        rc = load().snapkv_score(ctypes.byref(shape), q_win.data_ptr(), k.data_ptr(), arr, *tail)
        name = "snapkv_score"
    else:
        rc = load().snapkv_score_with_lse(ctypes.byref(shape), q_win.data_ptr(), k.data_ptr(),
                                          lse_win.data_ptr(), arr, *tail)
        name = "snapkv_score_with_lse"
    if rc:
        raise SnapKVError(rc, name)


def score_with_lse(q_win: torch.Tensor, k: torch.Tensor, lse_win: torch.Tensor, seqlens,
                   window_size: int, max_capacity_prompt: int, workspace: torch.Tensor,
                   stream=None) -> None:
    """snapkv_score_with_lse (include/snapkv.h)."""
    score(q_win, k, seqlens, window_size, max_capacity_prompt, workspace, stream, lse_win=lse_win)


def kernel_launches() -> int:
    return int(load().snapkv_kernel_launches())


SCORE_PATH_TENSOR_CORES, SCORE_PATH_CUDA_CORES = 0, 1


def score_path_launches(path: int) -> int:
    """snapkv_score_path_launches (include/snapkv.h)."""
    return int(load().snapkv_score_path_launches(int(path)))


def get_status(workspace: torch.Tensor, stream=None) -> int:
    return int(load().snapkv_get_status(workspace.data_ptr(),
                                        workspace.numel() * workspace.element_size(),
                                        _stream_handle(stream)))


def scores_from_workspace(workspace: torch.Tensor, shape: snapkv_shape, seqlens,
                          window_size: int, max_capacity_prompt: int, flags: int = 0):
    """(raw, pooled) fp32 views into the workspace after a compress call."""
    r, p, c = score_offsets(shape, seqlens, window_size, max_capacity_prompt, flags)
    raw = workspace[r:r + 4 * c].view(torch.float32)
    pooled = workspace[p:p + 4 * c].view(torch.float32)
    return raw, pooled


def host_staging_size(shape: snapkv_shape, seqlens, window_size: int,
                      max_capacity_prompt: int) -> int:
    arr, _ = _seqlens_array(seqlens)
    return int(load().snapkv_host_staging_size(ctypes.byref(shape), arr, int(window_size),
                                               int(max_capacity_prompt)))


def compress_host(q_win: torch.Tensor, k: torch.Tensor, v: torch.Tensor, seqlens,
                  window_size: int, kernel_size: int, pooling, max_capacity_prompt: int,
                  out_k: torch.Tensor, out_v: torch.Tensor, out_idx: torch.Tensor,
                  staging: torch.Tensor, stream=None) -> None:
    """Host-buffer variant (include/snapkv.h, snapkv_compress_host).

    All tensors but `staging` are CPU tensors (pinned for speed); `staging`
    is a CUDA uint8 tensor of at least host_staging_size bytes.  Returns when
    the outputs are complete.
    """
    B, W, H_q, d = q_win.shape
    shape = make_shape(B, H_q, k.shape[1], d, q_win.dtype)
    arr, _ = _seqlens_array(seqlens)
    rc = load().snapkv_compress_host(ctypes.byref(shape), q_win.data_ptr(), k.data_ptr(),
                                     v.data_ptr(), arr, W, int(kernel_size), pool_code(pooling),
                                     int(max_capacity_prompt), out_k.data_ptr(), out_v.data_ptr(),
                                     out_idx.data_ptr(), staging.data_ptr(), staging.numel(),
                                     _stream_handle(stream))
    if rc:
        raise SnapKVError(rc, "snapkv_compress_host")


def host_staging_size_layers(shape: snapkv_shape, seqlens, window_size: int,
                             max_capacity_prompt: int) -> int:
    arr, _ = _seqlens_array(seqlens)
    return int(load().snapkv_host_staging_size_layers(ctypes.byref(shape), arr,
                                                      int(window_size),
                                                      int(max_capacity_prompt)))


def compress_host_layers(layers, seqlens, window_size: int, kernel_size: int, pooling,
                         max_capacity_prompt: int, outs, staging: torch.Tensor, stream,
                         copy_stream, events) -> None:
    """snapkv_compress_host_layers (include/snapkv.h): layers = [(q_win, k, v)]
    and outs = [(out_k, out_v, out_idx)] of CPU tensors (pinned for speed);
    staging a CUDA uint8 tensor; stream / copy_stream two torch CUDA streams;
    events four torch.cuda.Event.  Returns when every layer is complete."""
    n = len(layers)
    if n < 1 or len(outs) != n or len(events) != 4:
        raise ValueError("one output triple per layer and four events")
    q0, k0, _ = layers[0]
    B, W, H_q, d = q0.shape
    shape = make_shape(B, H_q, k0.shape[1], d, q0.dtype)
    arr, _ = _seqlens_array(seqlens)
    ptrs = lambda ts: (ctypes.c_void_p * n)(*[t.data_ptr() for t in ts])
    for t in [x for lay in layers for x in lay] + [x for o in outs for x in o]:
        if not t.is_contiguous():
            raise ValueError("every layer tensor must be contiguous")
    for e in events:  # torch creates an event's CUDA handle when it is first recorded
        if not e.cuda_event:
            e.record(stream)
    ev = (ctypes.c_void_p * 4)(*[e.cuda_event for e in events])
    rc = load().snapkv_compress_host_layers(
        ctypes.byref(shape), n, ptrs([l[0] for l in layers]), ptrs([l[1] for l in layers]),
        ptrs([l[2] for l in layers]), arr, int(window_size), int(kernel_size),
        pool_code(pooling), int(max_capacity_prompt), ptrs([o[0] for o in outs]),
        ptrs([o[1] for o in outs]), ptrs([o[2] for o in outs]), staging.data_ptr(),
        staging.numel(), _stream_handle(stream), _stream_handle(copy_stream), ev)
    if rc:
        raise SnapKVError(rc, "snapkv_compress_host_layers")


MAX_LAYER_STREAMS = 8


def workspace_size_layers(shape: snapkv_shape, seqlens, window_size: int,
                          max_capacity_prompt: int, n_streams: int = 2) -> int:
    arr, _ = _seqlens_array(seqlens)
    return int(load().snapkv_workspace_size_layers(ctypes.byref(shape), arr, int(window_size),
                                                   int(max_capacity_prompt), int(n_streams)))


def compress_layers(layers, seqlens, window_size: int, kernel_size: int, pooling,
                    max_capacity_prompt: int, outs, workspace: torch.Tensor, layer_streams,
                    events, stream=None, lse_wins=None) -> None:
    """snapkv_compress_layers (include/snapkv.h): layers = [(q_win, k, v)] and
    outs = [(out_k, out_v, out_idx)] of CUDA tensors, one triple per layer;
    layer_streams 1 .. MAX_LAYER_STREAMS torch CUDA streams; workspace a CUDA
    uint8 tensor of workspace_size_layers(..., len(layer_streams)) bytes;
    events len(layer_streams) + 1 torch.cuda.Event.  Asynchronous on
    `stream` (default: the current stream).  lse_wins: None, or one fp32
    [B, W, H_q] CUDA tensor per layer (the window rows' natural-log LSE, as
    compress's lse_win), which skips pass 1."""
    n = len(layers)
    ns = len(layer_streams)
    if n < 1 or len(outs) != n or not 1 <= ns <= MAX_LAYER_STREAMS or len(events) != ns + 1:
        raise ValueError("one output triple per layer, 1 .. 8 layer streams and one event "
                         "more than streams")
    q0, k0, _ = layers[0]
    B, W, H_q, d = q0.shape
    H_kv = k0.shape[1]
    if W != int(window_size):
        raise ValueError("q_win's second dimension must equal window_size")
    C = int(max_capacity_prompt)
    shape = make_shape(B, H_q, H_kv, d, q0.dtype)
    for (q, k, v), (ok, ov, oi) in zip(layers, outs):
        for name, t in (("q_win", q), ("k", k), ("v", v), ("out_k", ok), ("out_v", ov),
                        ("out_idx", oi)):
            if not t.is_cuda or not t.is_contiguous():
                raise ValueError(f"every layer's {name} must be a contiguous CUDA tensor")
        if tuple(q.shape) != (B, W, H_q, d) or tuple(k.shape) != tuple(k0.shape) or \
                tuple(v.shape) != tuple(k0.shape):
            raise ValueError("every layer must have the first layer's shapes")
        if tuple(ok.shape) != (B, C, H_kv, d) or tuple(ov.shape) != (B, C, H_kv, d) or \
                tuple(oi.shape) != (B, H_kv, C):
            raise ValueError("output shapes must be [B, C, H_kv, d] and [B, H_kv, C]")
        if q.dtype != q0.dtype or k.dtype != q0.dtype or v.dtype != q0.dtype or \
                ok.dtype != q0.dtype or ov.dtype != q0.dtype or oi.dtype != torch.int32:
            raise ValueError("inputs and out_k / out_v share one dtype; out_idx is int32")
    if lse_wins is not None:
        if len(lse_wins) != n:
            raise ValueError("one lse_win per layer")
        for t in lse_wins:
            if not t.is_cuda:
                raise ValueError("every lse_win must be a CUDA tensor")
            _check_lse(t, B, W, H_q)
    st = torch.cuda.current_stream() if stream is None else stream
    for e in events:  # torch creates an event's CUDA handle when it is first recorded
        if not e.cuda_event:
            e.record(st)
    arr, _ = _seqlens_array(seqlens)
    ptrs = lambda ts: (ctypes.c_void_p * n)(*[t.data_ptr() for t in ts])
    sts = (ctypes.c_void_p * ns)(*[s.cuda_stream for s in layer_streams])
    ev = (ctypes.c_void_p * (ns + 1))(*[e.cuda_event for e in events])
    lse_arr = None if lse_wins is None else ptrs(lse_wins)
    rc = load().snapkv_compress_layers(
        ctypes.byref(shape), n, ptrs([l[0] for l in layers]), ptrs([l[1] for l in layers]),
        ptrs([l[2] for l in layers]), lse_arr, arr, int(window_size), int(kernel_size),
        pool_code(pooling), C, ptrs([o[0] for o in outs]), ptrs([o[1] for o in outs]),
        ptrs([o[2] for o in outs]), workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), _stream_handle(st), ns, sts, ev)
    if rc:
        raise SnapKVError(rc, "snapkv_compress_layers")


def compress_noalloc(q_win: torch.Tensor, k: torch.Tensor, v: torch.Tensor, seqlens,
                     window_size: int, kernel_size: int, pooling, max_capacity_prompt: int,
                     out_k: torch.Tensor, out_v: torch.Tensor, out_idx: torch.Tensor,
                     stream=None) -> None:
    """snapkv_compress_noalloc (include/snapkv.h): no workspace argument.

    For callers that cannot allocate device memory; the library's built-in
    16 MiB scratch serves as workspace.  All buffers are the caller's.
    """
    B, W, H_q, d = q_win.shape
    H_kv = k.shape[1]
    C = int(max_capacity_prompt)
    if W != int(window_size):
        raise ValueError("q_win's second dimension must equal window_size")
    for name, t in (("q_win", q_win), ("k", k), ("v", v), ("out_k", out_k), ("out_v", out_v),
                    ("out_idx", out_idx)):
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    for name, t, want in (("out_k", out_k, (B, C, H_kv, d)), ("out_v", out_v, (B, C, H_kv, d)),
                          ("out_idx", out_idx, (B, H_kv, C))):
        if tuple(t.shape) != want:
            raise ValueError(f"{name} must have shape {want}")
    if out_idx.dtype != torch.int32 or out_k.dtype != k.dtype or out_v.dtype != k.dtype:
        raise ValueError("out_idx must be int32 and out_k / out_v of k's dtype")
    shape = make_shape(B, H_q, H_kv, d, q_win.dtype)
    arr, _ = _seqlens_array(seqlens)
    rc = load().snapkv_compress_noalloc(ctypes.byref(shape), q_win.data_ptr(), k.data_ptr(),
                                        v.data_ptr(), arr, W, int(kernel_size),
                                        pool_code(pooling), int(max_capacity_prompt),
                                        out_k.data_ptr(), out_v.data_ptr(), out_idx.data_ptr(),
                                        _stream_handle(stream))
    if rc:
        raise SnapKVError(rc, "snapkv_compress_noalloc")


def noalloc_get_status(stream=None) -> int:
    """snapkv_noalloc_get_status (include/snapkv.h): synchronize the stream and
    read the status word of the last snapkv_compress_noalloc."""
    return int(load().snapkv_noalloc_get_status(_stream_handle(stream)))


# ---- decode step over a KV cache (include/snapkv.h, snapkv_decode_attention) ----

CACHE_PACKED, CACHE_SLOTS = 0, 1


def decode_workspace_size(shape: snapkv_shape, lens, layout: int, C: int = 0) -> int:
    arr, _ = _seqlens_array(lens)
    return int(load().snapkv_decode_workspace_size(ctypes.byref(shape), arr, int(layout), int(C)))


def decode_attention(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, lens,
                     layout: int, C: int = 0, out: torch.Tensor | None = None,
                     workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """One decode step of attention (include/snapkv.h, snapkv_decode_attention).

    q [B, H_q, d]; k_cache / v_cache [sum(lens), H_kv, d] (CACHE_PACKED) or
    [B, C, H_kv, d] (CACHE_SLOTS, rows 0..lens[b]-1 of each sequence); bf16 or
    fp32, CUDA.  Returns fp32 [B, H_q, d].
    """
    B, H_q, d = q.shape
    H_kv = k_cache.shape[-2]
    shape = make_shape(B, H_q, H_kv, d, q.dtype)
    arr, _ = _seqlens_array(lens)
    if out is None:
        out = torch.empty((B, H_q, d), dtype=torch.float32, device=q.device)
    ws_bytes = decode_workspace_size(shape, lens, layout, C)
    if ws_bytes == 0:
        raise SnapKVError(ERR_INVALID_ARG, "snapkv_decode_workspace_size")
    if workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    for name, t in (("q", q), ("k_cache", k_cache), ("v_cache", v_cache), ("out", out)):
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    rc = load().snapkv_decode_attention(ctypes.byref(shape), q.data_ptr(), k_cache.data_ptr(),
                                        v_cache.data_ptr(), int(layout), arr, int(C),
                                        out.data_ptr(), workspace.data_ptr(),
                                        workspace.numel() * workspace.element_size(),
                                        _stream_handle(stream))
    if rc:
        raise SnapKVError(rc, "snapkv_decode_attention")
    return out


def selftest_wait(workspace: torch.Tensor, set_flag: bool, stream=None) -> int:
    """snapkv_selftest_wait (include/snapkv.h), then snapkv_get_status: returns
    SNAPKV_ERR_TIMEOUT when the flag was left unset, SNAPKV_OK otherwise."""
    rc = load().snapkv_selftest_wait(workspace.data_ptr(),
                                     workspace.numel() * workspace.element_size(),
                                     1 if set_flag else 0, _stream_handle(stream))
    if rc:
        raise SnapKVError(rc, "snapkv_selftest_wait")
    return get_status(workspace, stream)


def compress_all_queries(q_all: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                         lse_all: torch.Tensor, seqlens, window_size: int, kernel_size: int,
                         pooling, max_capacity_prompt: int, stream=None):
    """snapkv_compress_all_queries (include/snapkv.h): every prompt query
    votes.  q_all [T, H_q, d] like k; lse_all fp32 [T, H_q].  Returns
    (out_k, out_v, out_idx, workspace)."""
    T, H_q, d = q_all.shape
    B = len(seqlens)
    H_kv = k.shape[1]
    C, W = int(max_capacity_prompt), int(window_size)
    if lse_all.dtype != torch.float32 or tuple(lse_all.shape) != (T, H_q) or \
            not lse_all.is_contiguous():
        raise ValueError(f"lse_all must be a contiguous float32 tensor of shape {(T, H_q)}")
    shape = make_shape(B, H_q, H_kv, d, q_all.dtype)
    out_k = torch.empty((B, C, H_kv, d), dtype=k.dtype, device=k.device)
    out_v = torch.empty((B, C, H_kv, d), dtype=k.dtype, device=k.device)
    out_idx = torch.empty((B, H_kv, C), dtype=torch.int32, device=k.device)
    workspace = torch.empty(workspace_size(shape, seqlens, W, C), dtype=torch.uint8,
                            device=k.device)
    arr, _ = _seqlens_array(seqlens)
    rc = load().snapkv_compress_all_queries(
        ctypes.byref(shape), q_all.data_ptr(), k.data_ptr(), v.data_ptr(), lse_all.data_ptr(),
        arr, W, int(kernel_size), pool_code(pooling), C, out_k.data_ptr(), out_v.data_ptr(),
        out_idx.data_ptr(), workspace.data_ptr(), workspace.numel(), _stream_handle(stream))
    if rc:
        raise SnapKVError(rc, "snapkv_compress_all_queries")
    return out_k, out_v, out_idx, workspace
