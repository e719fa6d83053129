"""CPU oracle for the block-quantized wire codec (numpy arrays in, numpy arrays out).

TEST INFRASTRUCTURE ONLY. The test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` are the only callers. The product path (the CUDA
library and its Python binding) never imports this package, and this package never
imports the product path: the two share no code.

The arithmetic lives in ``bq_oracle.c`` (plain C, built with gcc, no fused
multiply-add, no fast-math); this module builds it on first use and marshals numpy
arrays. BF16 tensors are passed as ``uint16`` arrays of their bit patterns.

Each function follows the pull-request pages on the wire codec:

* ``quant_i8`` / ``dequant_i8`` / ``dequant_accum_i8`` / ``ring_hop_i8``:
  "feat(pcie_dma): add block-INT8 wire modes for AG, ring, and A2A", Summary and
  Implementation.
* ``quant_mx`` / ``dequant_mx`` / ``e8m0_scale`` / ``e4m3_*``:
  "feat(pcie_dma): add INT8 and MXFP8 wire modes", Summary and the review comment
  on ``mxfp8_scale_byte``; slices per "[II] Support staged MXFP8 linear inputs",
  Behavior and Compatibility.
* ``dequant_accum_mx`` / ``ring_hop_mx``: the mx_a2a and mx_ring modes of the MXFP8
  page's Summary, on flat MX wires (E4M3 [n] then E8M0 [n/32]).
* ``quant_mx(..., fmt="f16")``: FP16 slices, "[II] Support staged MXFP8 linear
  inputs", Behavior.
* ``reduce_quant_i8`` / ``reduce_quant_e4m3``: the BF16 reduce-scatter of the i8 mode
  (and of the E4M3 all-gather mode) fused with its all-gather payload, block-INT8
  page, Summary.
* ``quant_e4m3`` / ``dequant_e4m3``: the legacy E4M3 codec the block-INT8 page
  compares against (Summary and Why: one E4M3 byte per value, FP32 scale per 128).
* ``mx_scales_to_tiled``: the tiled E8M0 layout block-scaled GEMMs read. The
  staged-input page names scale layouts for its GEMM but prints none; the tests pin
  this one to PyTorch's independent statements of cuBLAS's block-scaling-factor
  layout (``to_blocked`` / ``from_blocked``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "bq_oracle.c")
_LIB = os.path.join(_HERE, "libbq_oracle.so")
_CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]

BLOCK_I8 = 128
GROUP_MX = 32

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``bq_oracle.c`` into ``libbq_oracle.so`` with gcc (if stale)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".%d.tmp" % os.getpid()
        subprocess.run(["gcc", *_CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I64 = ctypes.c_int64
            for name, args in {
                "bqo_quant_i8": [P, I64, P, P],
                "bqo_dequant_i8": [P, P, I64, P],
                "bqo_dequant_accum_i8": [P, P, ctypes.c_int, I64, P, P, P],
                "bqo_ring_hop_i8": [P, P, P, I64, P, P, P],
                "bqo_quant_mx": [P, I64, I64, I64, P, I64, P, I64],
                "bqo_dequant_mx": [P, I64, P, I64, I64, I64, P, I64],
                "bqo_dequant_accum_mx": [P, P, ctypes.c_int, I64, P, P, P],
                "bqo_ring_hop_mx": [P, P, P, I64, P, P, P],
                "bqo_quant_mx_f16": [P, I64, I64, I64, P, I64, P, I64],
                "bqo_reduce_quant_i8": [P, ctypes.c_int, I64, P, P, P],
                "bqo_reduce_quant_e4m3": [P, ctypes.c_int, I64, P, P, P],
                "bqo_quant_e4m3": [P, I64, P, P],
                "bqo_dequant_e4m3": [P, P, I64, P],
                "bqo_mx_scales_to_tiled": [P, I64, I64, I64, P],
            }.items():
                fn = getattr(lib, name)
                fn.argtypes = args
                fn.restype = ctypes.c_int
            lib.bqo_bf16_round.argtypes = [ctypes.c_double]
            lib.bqo_bf16_round.restype = ctypes.c_uint16
            lib.bqo_e4m3_encode.argtypes = [ctypes.c_double]
            lib.bqo_e4m3_encode.restype = ctypes.c_uint8
            lib.bqo_e4m3_decode.argtypes = [ctypes.c_uint8]
            lib.bqo_e4m3_decode.restype = ctypes.c_double
            lib.bqo_e8m0_scale.argtypes = [ctypes.c_float]
            lib.bqo_e8m0_scale.restype = ctypes.c_uint8
            lib.bqo_mx_tiled_scale_offset.argtypes = [I64, I64, I64]
            lib.bqo_mx_tiled_scale_offset.restype = I64
            lib.bqo_f16_to_float.argtypes = [ctypes.c_uint16]
            lib.bqo_f16_to_float.restype = ctypes.c_float
            lib.bqo_wire_bytes.argtypes = [I64]
            lib.bqo_wire_bytes.restype = I64
            _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"] or a.ndim <= 1
    return a.ctypes.data


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise ValueError(f"oracle {what}: invalid shape or stride")


def wire_bytes(n: int) -> int:
    """Bytes on the wire for n values: 132 per 128 (both codecs)."""
    return int(_load().bqo_wire_bytes(n))


# ---------------------------------------------------------------- block INT8
def quant_i8(x_bits: np.ndarray):
    """BF16 bits [n] -> (payload int8 [n], scales float32 [n/128])."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16).reshape(-1)
    n = x.size
    q = np.empty(n, np.int8)
    s = np.empty(n // BLOCK_I8 if n % BLOCK_I8 == 0 else 0, np.float32)
    _check(_load().bqo_quant_i8(_ptr(x), n, _ptr(q), _ptr(s)), "quant_i8")
    return q, s


def dequant_i8(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    """payload [n] + scales [n/128] -> BF16 bits [n]."""
    q = np.ascontiguousarray(q, dtype=np.int8).reshape(-1)
    s = np.ascontiguousarray(s, dtype=np.float32).reshape(-1)
    if s.size * BLOCK_I8 != q.size:
        raise ValueError("oracle dequant_i8: scale count does not match payload")
    out = np.empty(q.size, np.uint16)
    _check(_load().bqo_dequant_i8(_ptr(q), _ptr(s), q.size, _ptr(out)), "dequant_i8")
    return out


def dequant_accum_i8(qs, ss, materialize: bool = True):
    """W payloads + scales -> (payload, scales, BF16 bits or None).

    Accumulates in source order 0..W-1 in FP32, requantizes, and (when asked)
    materializes the new payload as the owner would.
    """
    W = len(qs)
    if W != len(ss) or W < 1:
        raise ValueError("oracle dequant_accum_i8: need W >= 1 matching sources")
    qs = [np.ascontiguousarray(q, dtype=np.int8).reshape(-1) for q in qs]
    ss = [np.ascontiguousarray(s, dtype=np.float32).reshape(-1) for s in ss]
    n = qs[0].size
    for q, s in zip(qs, ss):
        if q.size != n or s.size * BLOCK_I8 != n:
            raise ValueError("oracle dequant_accum_i8: sources differ in size")
    qp = (ctypes.c_void_p * W)(*[_ptr(q) for q in qs])
    sp = (ctypes.c_void_p * W)(*[_ptr(s) for s in ss])
    q_out = np.empty(n, np.int8)
    s_out = np.empty(n // BLOCK_I8, np.float32)
    out = np.empty(n, np.uint16) if materialize else None
    rc = _load().bqo_dequant_accum_i8(
        ctypes.cast(qp, ctypes.c_void_p), ctypes.cast(sp, ctypes.c_void_p), W, n,
        _ptr(q_out), _ptr(s_out), _ptr(out) if materialize else None)
    _check(rc, "dequant_accum_i8")
    return q_out, s_out, out


def ring_hop_i8(q_in, s_in, x_local_bits, materialize: bool = False):
    """Incoming payload + local BF16 shard -> (payload, scales, BF16 bits or None)."""
    q_in = np.ascontiguousarray(q_in, dtype=np.int8).reshape(-1)
    s_in = np.ascontiguousarray(s_in, dtype=np.float32).reshape(-1)
    x = np.ascontiguousarray(x_local_bits, dtype=np.uint16).reshape(-1)
    n = q_in.size
    if x.size != n or s_in.size * BLOCK_I8 != n:
        raise ValueError("oracle ring_hop_i8: operand sizes differ")
    q_out = np.empty(n, np.int8)
    s_out = np.empty(n // BLOCK_I8, np.float32)
    out = np.empty(n, np.uint16) if materialize else None
    rc = _load().bqo_ring_hop_i8(_ptr(q_in), _ptr(s_in), _ptr(x), n, _ptr(q_out), _ptr(s_out),
                                 _ptr(out) if materialize else None)
    _check(rc, "ring_hop_i8")
    return q_out, s_out, out


# ---------------------------------------------------------------- MXFP8
def _quant_mx_fn(fmt: str):
    if fmt not in ("bf16", "f16"):
        raise ValueError(f"oracle quant_mx: input format {fmt!r} is not bf16 or f16")
    return _load().bqo_quant_mx if fmt == "bf16" else _load().bqo_quant_mx_f16


def quant_mx(x_bits: np.ndarray, fmt: str = "bf16"):
    """BF16 (or FP16) bits [rows, cols] -> (E4M3 codes [rows, cols], E8M0 bytes [rows, cols/32])."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    rows, cols = x.shape
    q = np.empty((rows, cols), np.uint8)
    s = np.empty((rows, cols // GROUP_MX), np.uint8)
    _check(_quant_mx_fn(fmt)(_ptr(x), rows, cols, cols, _ptr(q), cols, _ptr(s), cols // GROUP_MX), "quant_mx")
    return q, s


def quant_mx_into(x_bits: np.ndarray, q_buf: np.ndarray, s_buf: np.ndarray, col0: int, fmt: str = "bf16") -> None:
    """Quantize a [rows, cols] slice into columns [col0, col0+cols) of wider buffers.

    ``q_buf`` is uint8 [rows, C], ``s_buf`` uint8 [rows, C/32]; col0 % 128 == 0.
    """
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    rows, cols = x.shape
    if col0 % 128 or q_buf.shape[0] != rows or col0 + cols > q_buf.shape[1]:
        raise ValueError("oracle quant_mx_into: bad slice")
    assert q_buf.flags["C_CONTIGUOUS"] and s_buf.flags["C_CONTIGUOUS"]
    ld_q = q_buf.shape[1]
    ld_s = s_buf.shape[1]
    rc = _quant_mx_fn(fmt)(_ptr(x), rows, cols, cols, q_buf.ctypes.data + col0, ld_q,
                           s_buf.ctypes.data + col0 // GROUP_MX, ld_s)
    _check(rc, "quant_mx_into")


def dequant_mx(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    """E4M3 codes [rows, cols] + E8M0 bytes [rows, cols/32] -> BF16 bits [rows, cols]."""
    q = np.ascontiguousarray(q, dtype=np.uint8)
    s = np.ascontiguousarray(s, dtype=np.uint8)
    rows, cols = q.shape
    if s.shape != (rows, cols // GROUP_MX):
        raise ValueError("oracle dequant_mx: scale shape does not match")
    out = np.empty((rows, cols), np.uint16)
    _check(_load().bqo_dequant_mx(_ptr(q), cols, _ptr(s), cols // GROUP_MX, rows, cols, _ptr(out), cols),
           "dequant_mx")
    return out


def dequant_accum_mx(qs, ss, materialize: bool = True):
    """W flat MX wires (codes uint8 [n], E8M0 uint8 [n/32]) -> (codes, E8M0, BF16 bits or None).

    Decodes every source exactly to FP32, sums in source order 0..W-1 in FP32,
    requantizes per 32-value group and (when asked) materializes the new payload.
    """
    W = len(qs)
    if W != len(ss) or W < 1:
        raise ValueError("oracle dequant_accum_mx: need W >= 1 matching sources")
    qs = [np.ascontiguousarray(q, dtype=np.uint8).reshape(-1) for q in qs]
    ss = [np.ascontiguousarray(s, dtype=np.uint8).reshape(-1) for s in ss]
    n = qs[0].size
    for q, s in zip(qs, ss):
        if q.size != n or s.size * GROUP_MX != n:
            raise ValueError("oracle dequant_accum_mx: sources differ in size")
    qp = (ctypes.c_void_p * W)(*[_ptr(q) for q in qs])
    sp = (ctypes.c_void_p * W)(*[_ptr(s) for s in ss])
    q_out = np.empty(n, np.uint8)
    s_out = np.empty(n // GROUP_MX, np.uint8)
    out = np.empty(n, np.uint16) if materialize else None
    rc = _load().bqo_dequant_accum_mx(
        ctypes.cast(qp, ctypes.c_void_p), ctypes.cast(sp, ctypes.c_void_p), W, n,
        _ptr(q_out), _ptr(s_out), _ptr(out) if materialize else None)
    _check(rc, "dequant_accum_mx")
    return q_out, s_out, out


def ring_hop_mx(q_in, s_in, x_local_bits, materialize: bool = False):
    """Incoming flat MX wire + local BF16 shard -> (codes, E8M0, BF16 bits or None)."""
    q_in = np.ascontiguousarray(q_in, dtype=np.uint8).reshape(-1)
    s_in = np.ascontiguousarray(s_in, dtype=np.uint8).reshape(-1)
    x = np.ascontiguousarray(x_local_bits, dtype=np.uint16).reshape(-1)
    n = q_in.size
    if x.size != n or s_in.size * GROUP_MX != n:
        raise ValueError("oracle ring_hop_mx: operand sizes differ")
    q_out = np.empty(n, np.uint8)
    s_out = np.empty(n // GROUP_MX, np.uint8)
    out = np.empty(n, np.uint16) if materialize else None
    rc = _load().bqo_ring_hop_mx(_ptr(q_in), _ptr(s_in), _ptr(x), n, _ptr(q_out), _ptr(s_out),
                                 _ptr(out) if materialize else None)
    _check(rc, "ring_hop_mx")
    return q_out, s_out, out


def quant_mx_flat(x_bits: np.ndarray):
    """BF16 bits [n] -> flat MX wire (codes [n], E8M0 [n/32]); n % 128 == 0."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16).reshape(1, -1)
    q, s = quant_mx(x)
    return q.reshape(-1), s.reshape(-1)


def dequant_mx_flat(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    """Flat MX wire -> BF16 bits [n]."""
    return dequant_mx(np.asarray(q, np.uint8).reshape(1, -1), np.asarray(s, np.uint8).reshape(1, -1)).reshape(-1)


# ---------------------------------------------------------------- BF16 reduce + quantize, legacy E4M3
def _reduce_quant(fn, what, x_srcs, materialize, qtype):
    W = len(x_srcs)
    if W < 1:
        raise ValueError(f"oracle {what}: need W >= 1 sources")
    xs = [np.ascontiguousarray(x, dtype=np.uint16).reshape(-1) for x in x_srcs]
    n = xs[0].size
    if any(x.size != n for x in xs):
        raise ValueError(f"oracle {what}: sources differ in size")
    xp = (ctypes.c_void_p * W)(*[_ptr(x) for x in xs])
    q = np.empty(n, qtype)
    s = np.empty(n // BLOCK_I8 if n % BLOCK_I8 == 0 else 0, np.float32)
    out = np.empty(n, np.uint16) if materialize else None
    _check(fn(ctypes.cast(xp, ctypes.c_void_p), W, n, _ptr(q), _ptr(s), _ptr(out) if materialize else None), what)
    return q, s, out


def reduce_quant_i8(x_srcs, materialize: bool = False):
    """W BF16 shards -> (payload, scales, BF16 bits or None): binary32 sum in rank
    order, rounded once to BF16, then quant_i8."""
    return _reduce_quant(_load().bqo_reduce_quant_i8, "reduce_quant_i8", x_srcs, materialize, np.int8)


def reduce_quant_e4m3(x_srcs, materialize: bool = False):
    """As reduce_quant_i8 with the legacy E4M3 codec."""
    return _reduce_quant(_load().bqo_reduce_quant_e4m3, "reduce_quant_e4m3", x_srcs, materialize, np.uint8)


def quant_e4m3(x_bits: np.ndarray):
    """BF16 bits [n] -> (E4M3 codes uint8 [n], scales float32 [n/128])."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16).reshape(-1)
    n = x.size
    q = np.empty(n, np.uint8)
    s = np.empty(n // BLOCK_I8 if n % BLOCK_I8 == 0 else 0, np.float32)
    _check(_load().bqo_quant_e4m3(_ptr(x), n, _ptr(q), _ptr(s)), "quant_e4m3")
    return q, s


def dequant_e4m3(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    """E4M3 codes [n] + scales [n/128] -> BF16 bits [n]."""
    q = np.ascontiguousarray(q, dtype=np.uint8).reshape(-1)
    s = np.ascontiguousarray(s, dtype=np.float32).reshape(-1)
    if s.size * BLOCK_I8 != q.size:
        raise ValueError("oracle dequant_e4m3: scale count does not match payload")
    out = np.empty(q.size, np.uint16)
    _check(_load().bqo_dequant_e4m3(_ptr(q), _ptr(s), q.size, _ptr(out)), "dequant_e4m3")
    return out


def mx_tiled_scale_bytes(rows: int, g: int) -> int:
    """Bytes of the tiled layout for [rows, g] scales (rows padded to 128, g % 4 == 0)."""
    return ((rows + 127) // 128) * (g // 4) * 512


def mx_scales_to_tiled(s: np.ndarray, fill: int = 0) -> np.ndarray:
    """Row-major E8M0 [rows, g] -> the tiled layout (uint8, padding rows = fill)."""
    s = np.ascontiguousarray(s, dtype=np.uint8)
    rows, g = s.shape
    out = np.full(mx_tiled_scale_bytes(rows, g), fill, np.uint8)
    _check(_load().bqo_mx_scales_to_tiled(_ptr(s), rows, g, g, _ptr(out)), "mx_scales_to_tiled")
    return out


def mx_tiled_scale_offset(row: int, gcol: int, g: int) -> int:
    return int(_load().bqo_mx_tiled_scale_offset(row, gcol, g))


# ---------------------------------------------------------------- scalar helpers (for pins)
def f16_to_float(bits: int) -> float:
    return float(_load().bqo_f16_to_float(int(bits)))

def bf16_round(v: float) -> int:
    """Round a real (given exactly as a double) to a BF16 bit pattern, ties to even."""
    return int(_load().bqo_bf16_round(float(v)))


def e4m3_encode(y: float) -> int:
    return int(_load().bqo_e4m3_encode(float(y)))


def e4m3_decode(code: int) -> float:
    return float(_load().bqo_e4m3_decode(int(code)))


def e8m0_scale(amax: float) -> int:
    return int(_load().bqo_e8m0_scale(float(np.float32(amax))))
