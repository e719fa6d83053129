"""Python binding of the codec calls: torch tensors in, C ABI call out.

Every function only checks dtypes/devices/strides, reads pointers and the current
CUDA stream, and calls the same-named ``bq_*`` entry point of libbq.so; all
arithmetic runs in the library's kernels. Outputs are caller-owned tensors written in
place; nothing is allocated here except by the explicit ``empty_*`` helpers.

Wire layout (include/bq.h): an n-value INT8 wire is ``q`` (int8 [n]) followed by
``scales`` (float32 [n/128]); an MXFP8 tensor [rows, cols] is ``q`` (uint8 E4M3
[rows, cols]) and ``s`` (uint8 E8M0 [rows, cols/32]); a flat MXFP8 wire of n values
(the all-reduce shard of the mx_a2a / mx_ring modes) is ``q`` (uint8 [n]) followed by
``s`` (uint8 [n/32]).
"""
from __future__ import annotations

import ctypes
from typing import Optional, Sequence

import torch

from ._lib import check, load

BLOCK_I8 = 128
GROUP_MX = 32


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        cur = torch.cuda.current_device()
        if stream.device.index != cur:
            raise ValueError(f"stream belongs to {stream.device}, but the current CUDA device is cuda:{cur}")
        return stream.cuda_stream
    return int(stream)


def _on_current_device(t: torch.Tensor, name: str) -> None:
    """The library launches on the current device, so every tensor must live there (a
    pointer into another device's memory would be dereferenced by the wrong GPU)."""
    cur = torch.cuda.current_device()
    if t.device.index != cur:
        raise ValueError(f"{name}: tensor is on {t.device}, but the current CUDA device is cuda:{cur} "
                         f"(run the call under torch.cuda.device({t.device.index}))")


def _flat(t: torch.Tensor, dtype: torch.dtype, name: str) -> int:
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name}: expected a CUDA tensor")
    _on_current_device(t, name)
    if not t.is_contiguous():
        raise ValueError(f"{name}: expected a contiguous tensor")
    return t.data_ptr()


def _rows(t: torch.Tensor, dtype: torch.dtype, name: str):
    """(pointer, rows, cols, leading dimension in elements) of a row-major 2-D view."""
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name}: expected a CUDA tensor")
    _on_current_device(t, name)
    if t.dim() != 2 or (t.shape[1] > 1 and t.stride(1) != 1):
        raise ValueError(f"{name}: expected a 2-D row-major view with unit column stride")
    ld = t.stride(0) if t.shape[0] > 1 else t.shape[1]
    return t.data_ptr(), t.shape[0], t.shape[1], ld


# ---------------------------------------------------------------- allocation helpers
def wire_bytes(n: int) -> int:
    """132 bytes per 128 values (bq_wire_bytes)."""
    r = load().bq_wire_bytes(n)
    if r < 0:
        raise ValueError(f"wire_bytes: n={n} is not a non-negative multiple of 128")
    return r


def empty_wire_i8(n: int, device="cuda"):
    """One contiguous n-value INT8 wire buffer, returned as (buffer, q view, scales view)."""
    nbytes = wire_bytes(n)
    buf = torch.empty(nbytes, dtype=torch.uint8, device=device)
    q = buf[:n].view(torch.int8)
    s = buf[n:].view(torch.float32)
    return buf, q, s


def empty_wire_mx(n: int, device="cuda"):
    """One contiguous n-value flat MXFP8 wire buffer: (buffer, E4M3 codes [n], E8M0 [n/32])."""
    nbytes = wire_bytes(n)
    buf = torch.empty(nbytes, dtype=torch.uint8, device=device)
    return buf, buf[:n], buf[n:]


def empty_mx(rows: int, cols: int, device="cuda"):
    """(E4M3 values [rows, cols], E8M0 scales [rows, cols/32]) for an MXFP8 tensor."""
    return (torch.empty((rows, cols), dtype=torch.uint8, device=device),
            torch.empty((rows, cols // GROUP_MX), dtype=torch.uint8, device=device))


# ---------------------------------------------------------------- block INT8
def quant_i8(x: torch.Tensor, q: torch.Tensor, scales: torch.Tensor, stream=None) -> None:
    """BF16 x [n] -> payload q [n] (int8) + scales [n/128] (float32)."""
    n = x.numel()
    if q.numel() != n or scales.numel() * BLOCK_I8 != n:
        raise ValueError("quant_i8: output sizes do not match x")
    check("bq_quant_i8", load().bq_quant_i8(
        _flat(x, torch.bfloat16, "x"), n, _flat(q, torch.int8, "q"), _flat(scales, torch.float32, "scales"),
        _stream(stream)))


def dequant_i8(q: torch.Tensor, scales: torch.Tensor, out: torch.Tensor, stream=None) -> None:
    """payload q [n] + scales [n/128] -> BF16 out [n]."""
    n = q.numel()
    if out.numel() != n or scales.numel() * BLOCK_I8 != n:
        raise ValueError("dequant_i8: sizes do not match")
    check("bq_dequant_i8", load().bq_dequant_i8(
        _flat(q, torch.int8, "q"), _flat(scales, torch.float32, "scales"), n, _flat(out, torch.bfloat16, "out"),
        _stream(stream)))


def dequant_accum_i8(q_srcs: Sequence[torch.Tensor], scale_srcs: Sequence[torch.Tensor], q_out: torch.Tensor,
                     scales_out: torch.Tensor, out: Optional[torch.Tensor] = None, stream=None) -> None:
    """Sum W dequantized sources in FP32 in list order, requantize into q_out/scales_out;
    optionally materialize the new payload into out (BF16)."""
    W = len(q_srcs)
    if W != len(scale_srcs):
        raise ValueError("dequant_accum_i8: q_srcs and scale_srcs differ in length")
    n = q_out.numel()
    for q, s in zip(q_srcs, scale_srcs):
        if q.numel() != n or s.numel() * BLOCK_I8 != n:
            raise ValueError("dequant_accum_i8: a source's size differs from the output's")
    if scales_out.numel() * BLOCK_I8 != n or (out is not None and out.numel() != n):
        raise ValueError("dequant_accum_i8: output sizes do not match")
    qp = (ctypes.c_void_p * max(W, 1))(*[_flat(q, torch.int8, "q_srcs[]") for q in q_srcs])
    sp = (ctypes.c_void_p * max(W, 1))(*[_flat(s, torch.float32, "scale_srcs[]") for s in scale_srcs])
    check("bq_dequant_accum_i8", load().bq_dequant_accum_i8(
        ctypes.cast(qp, ctypes.c_void_p), ctypes.cast(sp, ctypes.c_void_p), W, n,
        _flat(q_out, torch.int8, "q_out"), _flat(scales_out, torch.float32, "scales_out"),
        _flat(out, torch.bfloat16, "out") if out is not None else None, _stream(stream)))


def ring_hop_i8(q_in: torch.Tensor, s_in: torch.Tensor, x_local: torch.Tensor, q_out: torch.Tensor,
                s_out: torch.Tensor, out: Optional[torch.Tensor] = None, stream=None) -> None:
    """Fused hop: requant(dequant(q_in, s_in) + x_local) -> q_out/s_out; optional BF16 out."""
    n = q_in.numel()
    if x_local.numel() != n or q_out.numel() != n or s_in.numel() * BLOCK_I8 != n or \
            s_out.numel() * BLOCK_I8 != n or (out is not None and out.numel() != n):
        raise ValueError("ring_hop_i8: sizes do not match")
    check("bq_ring_hop_i8", load().bq_ring_hop_i8(
        _flat(q_in, torch.int8, "q_in"), _flat(s_in, torch.float32, "s_in"),
        _flat(x_local, torch.bfloat16, "x_local"), n, _flat(q_out, torch.int8, "q_out"),
        _flat(s_out, torch.float32, "s_out"), _flat(out, torch.bfloat16, "out") if out is not None else None,
        _stream(stream)))


# ---------------------------------------------------------------- MXFP8
def quant_mx(x: torch.Tensor, q: torch.Tensor, s: torch.Tensor, stream=None) -> None:
    """BF16 or FP16 x [rows, cols] -> E4M3 q [rows, cols] + E8M0 s [rows, cols/32].

    Any of the three may be a column slice of a wider row-major buffer, e.g.
    ``q_buf[:, c0:c0+cols]`` and ``s_buf[:, c0//32:(c0+cols)//32]`` with c0 % 128 == 0.
    The input's dtype selects bq_quant_mx (BF16) or bq_quant_mx_f16 (FP16).
    """
    f16 = x.dtype == torch.float16
    xp, rows, cols, ld_x = _rows(x, torch.float16 if f16 else torch.bfloat16, "x")
    qp, qr, qc, ld_q = _rows(q, torch.uint8, "q")
    sp, sr, sc, ld_s = _rows(s, torch.uint8, "s")
    if (qr, qc) != (rows, cols) or (sr, sc) != (rows, cols // GROUP_MX):
        raise ValueError("quant_mx: output shapes do not match x")
    name = "bq_quant_mx_f16" if f16 else "bq_quant_mx"
    check(name, getattr(load(), name)(xp, rows, cols, ld_x, qp, ld_q, sp, ld_s, _stream(stream)))


def dequant_mx(q: torch.Tensor, s: torch.Tensor, out: torch.Tensor, stream=None) -> None:
    """E4M3 q [rows, cols] + E8M0 s [rows, cols/32] -> BF16 out [rows, cols]."""
    qp, rows, cols, ld_q = _rows(q, torch.uint8, "q")
    sp, sr, sc, ld_s = _rows(s, torch.uint8, "s")
    op, orr, oc, ld_o = _rows(out, torch.bfloat16, "out")
    if (sr, sc) != (rows, cols // GROUP_MX) or (orr, oc) != (rows, cols):
        raise ValueError("dequant_mx: shapes do not match")
    check("bq_dequant_mx", load().bq_dequant_mx(qp, ld_q, sp, ld_s, rows, cols, op, ld_o, _stream(stream)))


def mx_tiled_scale_bytes(rows: int, g_total: int) -> int:
    """Bytes of the tiled GEMM scale layout for rows x g_total E8M0 scales."""
    r = load().bq_mx_tiled_scale_bytes(rows, g_total)
    if r < 0:
        raise ValueError(f"mx_tiled_scale_bytes: g_total={g_total} is not a non-negative multiple of 4")
    return r


class _MxSlice(ctypes.Structure):
    _fields_ = [("x", ctypes.c_void_p), ("cols", ctypes.c_int64), ("ld_x", ctypes.c_int64)]


def quant_mx_slices(xs: Sequence[torch.Tensor], q: torch.Tensor, s: torch.Tensor, stream=None) -> None:
    """Quantize several staged slices (all BF16 or all FP16, each [rows, cols_i]) in one
    launch into q [rows, sum cols_i] and s [rows, sum cols_i / 32], slice i at the columns
    after slice i-1's: the bytes of quant_mx called once per slice (bq_quant_mx_slices)."""
    if not 1 <= len(xs) <= 16:
        raise ValueError("quant_mx_slices: 1 to 16 slices")
    f16 = xs[0].dtype == torch.float16
    dt = torch.float16 if f16 else torch.bfloat16
    arr = (_MxSlice * len(xs))()
    rows = None
    total = 0
    for i, x in enumerate(xs):
        xp, r, c, ld = _rows(x, dt, f"xs[{i}]")
        if rows is None:
            rows = r
        elif r != rows:
            raise ValueError("quant_mx_slices: every slice must have the same number of rows")
        arr[i] = _MxSlice(xp, c, ld)
        total += c
    qp, qr, qc, ld_q = _rows(q, torch.uint8, "q")
    sp, sr, sc, ld_s = _rows(s, torch.uint8, "s")
    if (qr, qc) != (rows, total) or (sr, sc) != (rows, total // GROUP_MX):
        raise ValueError("quant_mx_slices: q and s must cover the slices' rows and total columns")
    check("bq_quant_mx_slices", load().bq_quant_mx_slices(arr, len(xs), int(f16), rows, qp, ld_q, sp, ld_s,
                                                          _stream(stream)))


def quant_mx_tiled(x: torch.Tensor, q: torch.Tensor, s_tiled: torch.Tensor, g_total: int, g0: int = 0,
                   stream=None) -> None:
    """BF16 or FP16 x [rows, cols] -> E4M3 q [rows, cols] and E8M0 scales written into the
    tiled GEMM layout of a tensor with g_total scale columns, starting at scale column g0
    (the slice's column offset / 32). The pages do not print the layout; it is the
    block-scaled GEMM operand layout described in include/bq.h (bq_quant_mx_tiled)."""
    f16 = x.dtype == torch.float16
    xp, rows, cols, ld_x = _rows(x, torch.float16 if f16 else torch.bfloat16, "x")
    qp, qr, qc, ld_q = _rows(q, torch.uint8, "q")
    if (qr, qc) != (rows, cols):
        raise ValueError("quant_mx_tiled: q's shape does not match x")
    if s_tiled.numel() < mx_tiled_scale_bytes(rows, g_total):
        raise ValueError("quant_mx_tiled: the tiled scale buffer is too small")
    check("bq_quant_mx_tiled", load().bq_quant_mx_tiled(
        xp, int(f16), rows, cols, ld_x, qp, ld_q, _flat(s_tiled, torch.uint8, "s_tiled"), g_total, g0,
        _stream(stream)))


# ---------------------------------------------------------------- flat MXFP8 wires
def quant_mx_flat(x: torch.Tensor, q: torch.Tensor, s: torch.Tensor, stream=None) -> None:
    """BF16 x [n] -> flat MX wire q [n] + s [n/32] (bq_quant_mx on one row of n values)."""
    n = x.numel()
    quant_mx(x.reshape(1, n), q.reshape(1, n), s.reshape(1, n // GROUP_MX), stream)


def dequant_mx_flat(q: torch.Tensor, s: torch.Tensor, out: torch.Tensor, stream=None) -> None:
    """Flat MX wire q [n] + s [n/32] -> BF16 out [n] (bq_dequant_mx on one row)."""
    n = q.numel()
    dequant_mx(q.reshape(1, n), s.reshape(1, n // GROUP_MX), out.reshape(1, n), stream)


def dequant_accum_mx(q_srcs: Sequence[torch.Tensor], s_srcs: Sequence[torch.Tensor], q_out: torch.Tensor,
                     s_out: torch.Tensor, out: Optional[torch.Tensor] = None, stream=None) -> None:
    """Sum W decoded flat MX wires in FP32 in list order, requantize into q_out/s_out;
    optionally materialize the new wire into out (BF16)."""
    W = len(q_srcs)
    if W != len(s_srcs):
        raise ValueError("dequant_accum_mx: q_srcs and s_srcs differ in length")
    n = q_out.numel()
    for q, sc in zip(q_srcs, s_srcs):
        if q.numel() != n or sc.numel() * GROUP_MX != n:
            raise ValueError("dequant_accum_mx: a source's size differs from the output's")
    if s_out.numel() * GROUP_MX != n or (out is not None and out.numel() != n):
        raise ValueError("dequant_accum_mx: output sizes do not match")
    qp = (ctypes.c_void_p * max(W, 1))(*[_flat(q, torch.uint8, "q_srcs[]") for q in q_srcs])
    sp = (ctypes.c_void_p * max(W, 1))(*[_flat(sc, torch.uint8, "s_srcs[]") for sc in s_srcs])
    check("bq_dequant_accum_mx", load().bq_dequant_accum_mx(
        ctypes.cast(qp, ctypes.c_void_p), ctypes.cast(sp, ctypes.c_void_p), W, n,
        _flat(q_out, torch.uint8, "q_out"), _flat(s_out, torch.uint8, "s_out"),
        _flat(out, torch.bfloat16, "out") if out is not None else None, _stream(stream)))


def ring_hop_mx(q_in: torch.Tensor, s_in: torch.Tensor, x_local: torch.Tensor, q_out: torch.Tensor,
                s_out: torch.Tensor, out: Optional[torch.Tensor] = None, stream=None) -> None:
    """Fused MX hop: decode(q_in, s_in) + x_local in FP32, requantized into q_out/s_out."""
    n = q_in.numel()
    if (x_local.numel() != n or q_out.numel() != n or s_in.numel() * GROUP_MX != n
            or s_out.numel() * GROUP_MX != n or (out is not None and out.numel() != n)):
        raise ValueError("ring_hop_mx: sizes do not match")
    check("bq_ring_hop_mx", load().bq_ring_hop_mx(
        _flat(q_in, torch.uint8, "q_in"), _flat(s_in, torch.uint8, "s_in"), _flat(x_local, torch.bfloat16, "x_local"),
        n, _flat(q_out, torch.uint8, "q_out"), _flat(s_out, torch.uint8, "s_out"),
        _flat(out, torch.bfloat16, "out") if out is not None else None, _stream(stream)))


# ---------------------------------------------------------------- reduce + quantize, legacy E4M3
def _reduce_quant(name, x_srcs, q, scales, out, stream, qtype):
    W = len(x_srcs)
    n = q.numel()
    for x in x_srcs:
        if x.numel() != n:
            raise ValueError(f"{name}: a source's size differs from the payload's")
    if scales.numel() * BLOCK_I8 != n or (out is not None and out.numel() != n):
        raise ValueError(f"{name}: output sizes do not match")
    xp = (ctypes.c_void_p * max(W, 1))(*[_flat(x, torch.bfloat16, "x_srcs[]") for x in x_srcs])
    check(name, getattr(load(), name)(
        ctypes.cast(xp, ctypes.c_void_p), W, n, _flat(q, qtype, "q"), _flat(scales, torch.float32, "scales"),
        _flat(out, torch.bfloat16, "out") if out is not None else None, _stream(stream)))


def reduce_quant_i8(x_srcs: Sequence[torch.Tensor], q: torch.Tensor, scales: torch.Tensor,
                    out: Optional[torch.Tensor] = None, stream=None) -> None:
    """The i8 mode's BF16 reduce fused with quant_i8: W BF16 shards summed in list (rank)
    order in FP32, rounded once to BF16, quantized into q/scales; optionally the
    owner's materialization into out."""
    _reduce_quant("bq_reduce_quant_i8", x_srcs, q, scales, out, stream, torch.int8)


def empty_wire_e4m3(n: int, device="cuda"):
    """One contiguous n-value legacy E4M3 wire: (buffer, codes uint8 [n], scales float32 [n/128])."""
    nbytes = wire_bytes(n)
    buf = torch.empty(nbytes, dtype=torch.uint8, device=device)
    return buf, buf[:n], buf[n:].view(torch.float32)


def quant_e4m3(x: torch.Tensor, q: torch.Tensor, scales: torch.Tensor, stream=None) -> None:
    """BF16 x [n] -> legacy E4M3 codes q [n] (uint8) + FP32 scales [n/128]."""
    n = x.numel()
    if q.numel() != n or scales.numel() * BLOCK_I8 != n:
        raise ValueError("quant_e4m3: output sizes do not match x")
    check("bq_quant_e4m3", load().bq_quant_e4m3(
        _flat(x, torch.bfloat16, "x"), n, _flat(q, torch.uint8, "q"), _flat(scales, torch.float32, "scales"),
        _stream(stream)))


def dequant_e4m3(q: torch.Tensor, scales: torch.Tensor, out: torch.Tensor, stream=None) -> None:
    """Legacy E4M3 codes q [n] + scales [n/128] -> BF16 out [n]."""
    n = q.numel()
    if out.numel() != n or scales.numel() * BLOCK_I8 != n:
        raise ValueError("dequant_e4m3: sizes do not match")
    check("bq_dequant_e4m3", load().bq_dequant_e4m3(
        _flat(q, torch.uint8, "q"), _flat(scales, torch.float32, "scales"), n, _flat(out, torch.bfloat16, "out"),
        _stream(stream)))


def reduce_quant_e4m3(x_srcs: Sequence[torch.Tensor], q: torch.Tensor, scales: torch.Tensor,
                      out: Optional[torch.Tensor] = None, stream=None) -> None:
    """reduce_quant_i8 with the legacy E4M3 codec (the E4M3 all-gather mode)."""
    _reduce_quant("bq_reduce_quant_e4m3", x_srcs, q, scales, out, stream, torch.uint8)


# ---------------------------------------------------------------- bounded waits
def take_wait_timeouts() -> int:
    """Waits inside codec kernels on the current device that ran out (1 s limit) since
    the previous call. Synchronizes with the device."""
    n = ctypes.c_int64(0)
    check("bq_take_wait_timeouts", load().bq_take_wait_timeouts(ctypes.byref(n)))
    return int(n.value)


def take_index_errors() -> int:
    """Accesses a debug build's checks declined on the current device since the previous
    call (always 0 in the default build)."""
    n = ctypes.c_int64(0)
    check("bq_take_index_errors", load().bq_take_index_errors(ctypes.byref(n)))
    return int(n.value)


def debug_build() -> bool:
    """True if the loaded library is the debug build (BQ_DEBUG=1)."""
    return bool(load().bq_debug_build())


def selftest_index_check(buf: torch.Tensor, stream=None) -> None:
    """Debug build: one deliberately declined load against a 1 KB device buffer."""
    check("bq_selftest_index_check", load().bq_selftest_index_check(_flat(buf, torch.uint8, "buf"), buf.numel(),
                                                                    _stream(stream)))


def take_wait_unlanded() -> int:
    """Bulk copies that had not landed within the limit after an abandoned wait, since
    the previous call (each may have written a finished block's shared memory)."""
    n = ctypes.c_int64(0)
    check("bq_take_wait_unlanded", load().bq_take_wait_unlanded(ctypes.byref(n)))
    return int(n.value)


def selftest_wait_timeout(stream=None) -> None:
    """Run one deliberately unsatisfied 20 ms bounded wait (the count grows by one)."""
    check("bq_selftest_wait_timeout", load().bq_selftest_wait_timeout(_stream(stream)))
