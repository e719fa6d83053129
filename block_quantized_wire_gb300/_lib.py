"""ctypes loader for libbq.so (the C ABI declared in include/bq.h).

There is no fallback: if the library is missing or does not load, every codec call
raises. Build it with ``block_quantized_wire_gb300.build.build_library()`` (or
``__graft_entry__.build()``).
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import threading

from . import build as _build

_lock = threading.Lock()
_lib = None

ABI_VERSION = 5
BQ_OK = 0
STATUS_NAMES = {0: "BQ_OK", 1: "BQ_ERR_NULL", 2: "BQ_ERR_SHAPE", 3: "BQ_ERR_ALIGN", 4: "BQ_ERR_ALIAS",
                5: "BQ_ERR_CUDA", 6: "BQ_ERR_UNSUPPORTED"}

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_PROTOS = {
    "bq_abi_version": ([], ctypes.c_int),
    "bq_status_string": ([ctypes.c_int], ctypes.c_char_p),
    "bq_wire_bytes": ([_I64], _I64),
    "bq_quant_i8": ([_P, _I64, _P, _P, _P], ctypes.c_int),
    "bq_dequant_i8": ([_P, _P, _I64, _P, _P], ctypes.c_int),
    "bq_dequant_accum_i8": ([_P, _P, ctypes.c_int, _I64, _P, _P, _P, _P], ctypes.c_int),
    "bq_ring_hop_i8": ([_P, _P, _P, _I64, _P, _P, _P, _P], ctypes.c_int),
    "bq_quant_mx": ([_P, _I64, _I64, _I64, _P, _I64, _P, _I64, _P], ctypes.c_int),
    "bq_dequant_mx": ([_P, _I64, _P, _I64, _I64, _I64, _P, _I64, _P], ctypes.c_int),
    "bq_dequant_accum_mx": ([_P, _P, ctypes.c_int, _I64, _P, _P, _P, _P], ctypes.c_int),
    "bq_ring_hop_mx": ([_P, _P, _P, _I64, _P, _P, _P, _P], ctypes.c_int),
    "bq_quant_mx_f16": ([_P, _I64, _I64, _I64, _P, _I64, _P, _I64, _P], ctypes.c_int),
    "bq_quant_mx_tiled": ([_P, ctypes.c_int, _I64, _I64, _I64, _P, _I64, _P, _I64, _I64, _P], ctypes.c_int),
    "bq_mx_tiled_scale_bytes": ([_I64, _I64], _I64),
    "bq_quant_mx_slices": ([_P, ctypes.c_int, ctypes.c_int, _I64, _P, _I64, _P, _I64, _P], ctypes.c_int),
    "bq_reduce_quant_i8": ([_P, ctypes.c_int, _I64, _P, _P, _P, _P], ctypes.c_int),
    "bq_quant_e4m3": ([_P, _I64, _P, _P, _P], ctypes.c_int),
    "bq_dequant_e4m3": ([_P, _P, _I64, _P, _P], ctypes.c_int),
    "bq_reduce_quant_e4m3": ([_P, ctypes.c_int, _I64, _P, _P, _P, _P], ctypes.c_int),
    "bq_take_wait_timeouts": ([_P], ctypes.c_int),
    "bq_take_wait_unlanded": ([_P], ctypes.c_int),
    "bq_take_index_errors": ([_P], ctypes.c_int),
    "bq_debug_build": ([], ctypes.c_int),
    "bq_selftest_index_check": ([_P, _I64, _P], ctypes.c_int),
    "bq_selftest_wait_timeout": ([_P], ctypes.c_int),
}


class BQError(RuntimeError):
    """A bq_* call returned a non-OK status."""

    def __init__(self, func: str, status: int, message: str):
        super().__init__(f"{func}: {STATUS_NAMES.get(status, status)} ({message})")
        self.func = func
        self.status = status


def library_path() -> str:
    return _build.LIB


def _open(path: str):
    if not os.path.exists(path):
        raise ImportError(f"{os.path.basename(path)} is not built ({path}); run "
                          "block_quantized_wire_gb300.build.build_library()")
    lib = ctypes.CDLL(path)
    for name, (args, res) in _PROTOS.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    if lib.bq_abi_version() != ABI_VERSION:
        raise ImportError(f"{path}: ABI version {lib.bq_abi_version()} != {ABI_VERSION}")
    return lib


def load():
    """Load libbq.so once; raise if it is not built or does not load."""
    global _lib
    with _lock:
        if _lib is None:
            _lib = _open(library_path())
    return _lib


@contextlib.contextmanager
def use_library(path: str):
    """Route every call of this package to another build of the same sources (the
    tests run the compile-time alternatives of the kernels through it). Not for
    concurrent use with other calls."""
    global _lib
    alt = _open(path)
    with _lock:
        saved = _lib
        _lib = alt
    try:
        yield alt
    finally:
        with _lock:
            _lib = saved


def check(func: str, status: int) -> None:
    if status != BQ_OK:
        msg = load().bq_status_string(status).decode()
        raise BQError(func, status, msg)
