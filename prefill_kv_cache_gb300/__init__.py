"""SnapKV prefill-time KV-cache compression for GB300 (sm_103a).

The compute lives in libsnapkv.so (hand-written CUDA, C ABI in
include/snapkv.h and include/scissorhands.h); ``snapkv`` (compression,
scoring, decode steps) and ``scissorhands`` (decode-time eviction) are its
thin ctypes bindings.
"""
from . import scissorhands, snapkv  # noqa: F401
from .snapkv import SnapKVConfig, compress, compress_host, load  # noqa: F401

__version__ = "0.2.0"
