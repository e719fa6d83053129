"""The C ABI without a GPU: libbq.so loads, exports every entry point include/bq.h
declares, and rejects invalid arguments before any CUDA call.

Every call here carries at least one invalid argument, so the library returns an error
status before it would touch the device; the fake pointers are never dereferenced.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "bq.h")

OK, NULL, SHAPE, ALIGN, ALIAS, CUDA = range(6)
A = 0x7F0000000000  # a 256-byte-aligned fake device address, never dereferenced


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"BQ_API\s+[\w\s\*]*?\b(bq_\w+)\s*\(", text)))


def test_header_declares_the_calls():
    names = declared_functions()
    for want in ("bq_quant_i8", "bq_dequant_i8", "bq_dequant_accum_i8", "bq_ring_hop_i8", "bq_quant_mx",
                 "bq_dequant_mx", "bq_dequant_accum_mx", "bq_ring_hop_mx", "bq_quant_mx_f16", "bq_reduce_quant_i8",
                 "bq_quant_e4m3", "bq_dequant_e4m3", "bq_reduce_quant_e4m3", "bq_quant_mx_tiled", "bq_quant_mx_slices",
                 "bq_mx_tiled_scale_bytes", "bq_wire_bytes", "bq_status_string",
                 "bq_abi_version", "bq_take_wait_timeouts", "bq_take_wait_unlanded", "bq_selftest_wait_timeout",
                 "bq_take_index_errors", "bq_debug_build", "bq_selftest_index_check"):
        assert want in names


def test_library_exports_every_declared_symbol(bq_lib):
    for name in declared_functions():
        assert hasattr(bq_lib, name), name
    assert bq_lib.bq_abi_version() == 5


def test_wire_bytes_and_status_strings(bq_lib):
    assert bq_lib.bq_wire_bytes(0) == 0
    assert bq_lib.bq_wire_bytes(128) == 132
    assert bq_lib.bq_wire_bytes(512 * 7168) == 3784704
    assert bq_lib.bq_wire_bytes(65536 * 7168) == 484442112
    assert bq_lib.bq_wire_bytes(100) == -1
    assert bq_lib.bq_wire_bytes(-128) == -1
    for s in range(6):
        assert bq_lib.bq_status_string(s)
    assert bq_lib.bq_status_string(99) == b"unknown status"


def _srcs(ptrs):
    arr = (ctypes.c_void_p * len(ptrs))(*ptrs)
    return ctypes.cast(arr, ctypes.c_void_p), arr


def test_quant_i8_rejections(bq_lib):
    f = bq_lib.bq_quant_i8
    n = 1024
    assert f(A, 100, A + 0x100000, A + 0x200000, None) == SHAPE
    assert f(A, -128, A + 0x100000, A + 0x200000, None) == SHAPE
    assert f(None, 0, None, None, None) == OK  # empty input: nothing to do, no launch
    assert f(None, n, A + 0x100000, A + 0x200000, None) == NULL
    assert f(A, n, None, A + 0x200000, None) == NULL
    assert f(A, n, A + 0x100000, None, None) == NULL
    assert f(A + 8, n, A + 0x100000, A + 0x200000, None) == ALIGN
    assert f(A, n, A + 0x100004, A + 0x200000, None) == ALIGN
    assert f(A, n, A + 0x100000, A + 0x200002, None) == ALIGN
    assert f(A, n, A + 1024, A + 0x200000, None) == ALIAS  # payload inside x (x spans 2n bytes)
    assert f(A, n, A + 0x100000, A + 0x100000 + n - 4, None) == ALIAS  # scales overlap payload


def test_dequant_i8_rejections(bq_lib):
    f = bq_lib.bq_dequant_i8
    n = 2048
    assert f(A, A + 0x100000, 129, A + 0x200000, None) == SHAPE
    assert f(A, A + 0x100000, 0, None, None) == OK
    assert f(A, None, n, A + 0x200000, None) == NULL
    assert f(A, A + 0x100000, n, A + 0x200008, None) == ALIGN
    assert f(A, A + 0x100000, n, A + 0x100000 - 64, None) == ALIAS


def test_accum_i8_rejections(bq_lib):
    f = bq_lib.bq_dequant_accum_i8
    n = 4096
    q = [A + k * 0x100000 for k in range(4)]
    s = [A + 0x1000000 + k * 0x10000 for k in range(4)]
    qp, qa = _srcs(q)
    sp, sa = _srcs(s)
    out_q, out_s, out_b = A + 0x2000000, A + 0x3000000, A + 0x4000000
    assert f(qp, sp, 0, n, out_q, out_s, None, None) == SHAPE
    assert f(qp, sp, 17, n, out_q, out_s, None, None) == SHAPE
    assert f(qp, sp, 4, n + 64, out_q, out_s, None, None) == SHAPE
    assert f(qp, sp, 4, 0, out_q, out_s, None, None) == OK
    assert f(None, sp, 4, n, out_q, out_s, None, None) == NULL
    qn, qna = _srcs([q[0], None, q[2], q[3]])
    assert f(qn, sp, 4, n, out_q, out_s, None, None) == NULL
    qm, qma = _srcs([q[0], q[1] + 4, q[2], q[3]])
    assert f(qm, sp, 4, n, out_q, out_s, None, None) == ALIGN
    assert f(qp, sp, 4, n, out_q, out_s, out_b + 2, None) == ALIGN
    assert f(qp, sp, 4, n, q[2], out_s, None, None) == ALIAS  # output payload is a source
    assert f(qp, sp, 4, n, out_q, s[3] + 16, None, None) == ALIAS
    assert f(qp, sp, 4, n, out_q, out_s, out_q + 1024, None) == ALIAS  # BF16 out over payload out


def test_ring_hop_rejections(bq_lib):
    f = bq_lib.bq_ring_hop_i8
    n = 4096
    qi, si, x, qo, so, ob = (A + k * 0x100000 for k in range(6))
    assert f(qi, si, x, 96, qo, so, None, None) == SHAPE
    assert f(qi, si, x, 0, qo, so, None, None) == OK
    assert f(qi, si, None, n, qo, so, None, None) == NULL
    assert f(qi, si + 2, x, n, qo, so, None, None) == ALIGN
    assert f(qi, si, x, n, x + 16, so, None, None) == ALIAS
    assert f(qi, si, x, n, qo, so, qi, None) == ALIAS


def test_accum_mx_rejections(bq_lib):
    f = bq_lib.bq_dequant_accum_mx
    n = 4096
    q = [A + k * 0x100000 for k in range(4)]
    s = [A + 0x1000000 + k * 0x10000 for k in range(4)]
    qp, qa = _srcs(q)
    sp, sa = _srcs(s)
    out_q, out_s, out_b = A + 0x2000000, A + 0x3000000, A + 0x4000000
    assert f(qp, sp, 0, n, out_q, out_s, None, None) == SHAPE
    assert f(qp, sp, 17, n, out_q, out_s, None, None) == SHAPE
    assert f(qp, sp, 4, n + 32, out_q, out_s, None, None) == SHAPE  # groups of 32 but not blocks of 128
    assert f(qp, sp, 4, 0, out_q, out_s, None, None) == OK
    assert f(qp, None, 4, n, out_q, out_s, None, None) == NULL
    sn, sna = _srcs([s[0], s[1], None, s[3]])
    assert f(qp, sn, 4, n, out_q, out_s, None, None) == NULL
    sm, sma = _srcs([s[0], s[1] + 2, s[2], s[3]])
    assert f(qp, sm, 4, n, out_q, out_s, None, None) == ALIGN  # scale words are 4-byte aligned
    assert f(qp, sp, 4, n, out_q + 8, out_s, None, None) == ALIGN
    assert f(qp, sp, 4, n, out_q, out_s + 1, None, None) == ALIGN
    assert f(qp, sp, 4, n, q[1], out_s, None, None) == ALIAS
    assert f(qp, sp, 4, n, out_q, s[0] + 64, None, None) == ALIAS  # E8M0 run spans n/32 bytes
    assert f(qp, sp, 4, n, out_q, out_s, out_s - 64, None) == ALIAS


def test_ring_hop_mx_rejections(bq_lib):
    f = bq_lib.bq_ring_hop_mx
    n = 4096
    qi, si, x, qo, so, ob = (A + k * 0x100000 for k in range(6))
    assert f(qi, si, x, 160, qo, so, None, None) == SHAPE
    assert f(qi, si, x, 0, qo, so, None, None) == OK
    assert f(qi, None, x, n, qo, so, None, None) == NULL
    assert f(qi, si + 1, x, n, qo, so, None, None) == ALIGN
    assert f(qi, si, x + 8, n, qo, so, None, None) == ALIGN
    assert f(qi, si, x, n, qo, so, ob + 2, None) == ALIGN
    assert f(qi, si, x, n, x + 2 * n - 16, so, None, None) == ALIAS
    assert f(qi, si, x, n, qo, si + n // 32 - 4, None, None) == ALIAS
    assert f(qi, si, x, n, qo, so, qo + n - 16, None) == ALIAS


@pytest.mark.parametrize("name", ["bq_reduce_quant_i8", "bq_reduce_quant_e4m3"])
def test_reduce_quant_rejections(bq_lib, name):
    f = getattr(bq_lib, name)
    n = 4096
    x = [A + k * 0x100000 for k in range(4)]
    xp, xa = _srcs(x)
    q, s, o = A + 0x2000000, A + 0x3000000, A + 0x4000000
    assert f(xp, 0, n, q, s, None, None) == SHAPE
    assert f(xp, 17, n, q, s, None, None) == SHAPE
    assert f(xp, 4, n + 64, q, s, None, None) == SHAPE
    assert f(xp, 4, 0, q, s, None, None) == OK
    assert f(None, 4, n, q, s, None, None) == NULL
    xn, xna = _srcs([x[0], x[1], None, x[3]])
    assert f(xn, 4, n, q, s, None, None) == NULL
    xm, xma = _srcs([x[0], x[1] + 2, x[2], x[3]])
    assert f(xm, 4, n, q, s, None, None) == ALIGN
    assert f(xp, 4, n, q + 8, s, None, None) == ALIGN
    assert f(xp, 4, n, q, s + 2, None, None) == ALIGN
    assert f(xp, 4, n, q, s, o + 8, None) == ALIGN
    assert f(xp, 4, n, x[3] + 2 * n - 16, s, None, None) == ALIAS  # payload over a source
    assert f(xp, 4, n, q, s, q + n - 16, None) == ALIAS


def test_e4m3_rejections(bq_lib):
    fq, fd = bq_lib.bq_quant_e4m3, bq_lib.bq_dequant_e4m3
    n = 1024
    assert fq(A, 100, A + 0x100000, A + 0x200000, None) == SHAPE
    assert fq(None, 0, None, None, None) == OK
    assert fq(A, n, None, A + 0x200000, None) == NULL
    assert fq(A, n, A + 0x100004, A + 0x200000, None) == ALIGN
    assert fq(A, n, A + 0x100000, A + 0x200001, None) == ALIGN
    assert fq(A, n, A + 512, A + 0x200000, None) == ALIAS
    assert fd(A, A + 0x100000, 129, A + 0x200000, None) == SHAPE
    assert fd(A, A + 0x100000, n, None, None) == NULL
    assert fd(A, A + 0x100000, n, A + 0x200004, None) == ALIGN
    assert fd(A, A + 0x100000, n, A + 0x100000 - 16, None) == ALIAS


def test_quant_mx_f16_rejections(bq_lib):
    f = bq_lib.bq_quant_mx_f16
    assert f(A, 4, 100, 100, A + 0x100000, 100, A + 0x200000, 4, None) == SHAPE
    assert f(A, 4, 128, 64, A + 0x100000, 128, A + 0x200000, 4, None) == SHAPE  # ld_x < cols
    assert f(A, 0, 128, 128, None, 128, None, 4, None) == OK
    assert f(None, 4, 128, 128, A + 0x100000, 128, A + 0x200000, 4, None) == NULL
    assert f(A + 2, 4, 128, 128, A + 0x100000, 128, A + 0x200000, 4, None) == ALIGN
    assert f(A, 4, 128, 132, A + 0x100000, 128, A + 0x200000, 4, None) == ALIGN  # ld_x % 8
    assert f(A, 4, 128, 128, A + 512, 128, A + 0x200000, 4, None) == ALIAS


def test_quant_mx_tiled_rejections(bq_lib):
    f = bq_lib.bq_quant_mx_tiled
    x, q, s = A, A + 0x1000000, A + 0x2000000
    assert f(x, 0, 256, 100, 256, q, 256, s, 8, 0, None) == SHAPE      # cols % 128
    assert f(x, 0, 256, 256, 256, q, 256, s, 6, 0, None) == SHAPE      # g_total % 4
    assert f(x, 0, 256, 256, 256, q, 256, s, 8, 2, None) == SHAPE      # g0 % 4
    assert f(x, 0, 256, 256, 256, q, 256, s, 8, 4, None) == SHAPE      # g0 + cols/32 > g_total
    assert f(x, 0, 0, 256, 256, None, 256, None, 8, 0, None) == OK     # empty
    assert f(None, 0, 256, 256, 256, q, 256, s, 8, 0, None) == NULL
    assert f(x, 0, 256, 256, 256, q, 256, s + 2, 8, 0, None) == ALIGN
    assert f(x, 1, 256, 256, 260, q, 256, s, 8, 0, None) == ALIGN     # ld_x % 8 != 0 (FP16 too)
    assert f(x, 0, 256, 256, 256, q, 256, x + 512, 8, 0, None) == ALIAS
    assert bq_lib.bq_mx_tiled_scale_bytes(256, 8) == 2 * 2 * 512
    assert bq_lib.bq_mx_tiled_scale_bytes(300, 1344) == 3 * 336 * 512
    assert bq_lib.bq_mx_tiled_scale_bytes(1, 6) == -1


def test_quant_mx_slices_rejections(bq_lib):
    from block_quantized_wire_gb300.codec import _MxSlice
    f = bq_lib.bq_quant_mx_slices
    q, s = A + 0x10000000, A + 0x20000000

    def sl(*specs):
        arr = (_MxSlice * len(specs))()
        for i, (x, cols, ld) in enumerate(specs):
            arr[i] = _MxSlice(x, cols, ld)
        return arr

    two = sl((A, 256, 256), (A + 0x1000000, 128, 128))
    assert f(two, 0, 0, 64, q, 384, s, 12, None) == SHAPE                   # no slices
    assert f(sl(*[(A, 128, 128)] * 17), 17, 0, 64, q, 17 * 128, s, 68, None) == SHAPE  # too many
    assert f(None, 2, 0, 64, q, 384, s, 12, None) == NULL
    assert f(two, 2, 0, -1, q, 384, s, 12, None) == SHAPE
    assert f(sl((A, 200, 256)), 1, 0, 64, q, 256, s, 8, None) == SHAPE    # cols % 128
    assert f(sl((A, 256, 128)), 1, 0, 64, q, 256, s, 8, None) == SHAPE    # ld_x < cols
    assert f(two, 2, 0, 0, None, 384, None, 12, None) == OK               # no rows: nothing to do
    assert f(sl((A, 0, 0), (None, 0, 0)), 2, 0, 64, None, 0, None, 0, None) == OK  # no columns
    assert f(two, 2, 0, 64, q, 256, s, 12, None) == SHAPE                 # ld_q < total columns
    assert f(two, 2, 0, 64, q, 384, s, 8, None) == SHAPE                  # ld_s < total / 32
    assert f(two, 2, 0, 64, None, 384, s, 12, None) == NULL
    assert f(sl((A, 256, 256), (None, 128, 128)), 2, 0, 64, q, 384, s, 12, None) == NULL
    assert f(sl((A, 256, 256), (None, 0, 0)), 2, 0, 0, q, 384, s, 12, None) == OK  # empty slice skipped
    assert f(sl((A + 8, 256, 256)), 1, 1, 64, q, 256, s, 8, None) == ALIGN  # x 16-byte aligned
    assert f(sl((A, 256, 260)), 1, 0, 64, q, 256, s, 8, None) == ALIGN      # ld_x % 8
    assert f(two, 2, 0, 64, q, 392, s, 12, None) == ALIGN                 # ld_q % 16
    assert f(two, 2, 0, 64, q, 384, s + 2, 12, None) == ALIGN
    assert f(two, 2, 0, 64, A + 0x1000000 + 512, 384, s, 12, None) == ALIAS  # q over slice 1
    assert f(two, 2, 0, 64, q, 384, A + 64, 12, None) == ALIAS              # s over slice 0
    assert f(two, 2, 0, 64, q, 384, q + 256, 12, None) == ALIAS             # s over q


def test_mx_rejections(bq_lib):
    fq = bq_lib.bq_quant_mx
    fd = bq_lib.bq_dequant_mx
    x, q, s, o = A, A + 0x1000000, A + 0x2000000, A + 0x3000000
    rows, cols = 64, 256
    assert fq(x, rows, 200, 256, q, 256, s, 8, None) == SHAPE  # cols % 128
    assert fq(x, -1, cols, cols, q, cols, s, 8, None) == SHAPE
    assert fq(x, 0, cols, cols, q, cols, s, 8, None) == OK
    assert fq(x, rows, cols, 128, q, cols, s, 8, None) == SHAPE  # ld_x < cols
    assert fq(x, rows, cols, cols, q, cols, s, 4, None) == SHAPE  # ld_s < cols/32
    assert fq(None, rows, cols, cols, q, cols, s, 8, None) == NULL
    assert fq(x, rows, cols, cols + 4, q, cols, s, 8, None) == ALIGN  # ld_x % 8
    assert fq(x, rows, cols, cols, q, cols + 8, s, 8, None) == ALIGN  # ld_q % 16
    assert fq(x, rows, cols, cols, q, cols, s + 2, 8, None) == ALIGN  # s 4-byte aligned
    assert fq(x, rows, cols, cols, q, cols, s, 10, None) == ALIGN  # ld_s % 4
    assert fq(x, rows, cols, cols, x + 2 * cols * (rows - 1), cols, s, 8, None) == ALIAS
    assert fq(x, rows, cols, cols, q, cols, q + cols * rows - 4, 8, None) == ALIAS
    assert fd(q, cols, s, 8, rows, 100, o, cols, None) == SHAPE
    assert fd(q, cols, s, 8, 0, cols, o, cols, None) == OK
    assert fd(q, cols, s, 8, rows, cols, None, cols, None) == NULL
    assert fd(q, cols, s, 8, rows, cols, o, cols + 2, None) == ALIGN
    assert fd(q, cols, s, 8, rows, cols, q - 2 * cols, cols, None) == ALIAS


def test_binding_without_library_fails_loudly(tmp_path, monkeypatch):
    # the binding never falls back: a missing library raises instead of computing
    from block_quantized_wire_gb300 import _lib, build
    monkeypatch.setattr(build, "LIB", str(tmp_path / "missing_libbq.so"))
    monkeypatch.setattr(_lib, "_lib", None)
    with pytest.raises(ImportError):
        _lib.load()


class _FakeCudaTensor:
    """Just enough of a CUDA tensor for the binding's argument checks (no memory)."""

    def __init__(self, dtype, n, device_index):
        import torch
        self.dtype = dtype
        self.is_cuda = True
        self.device = torch.device("cuda", device_index)
        self._n = n

    def is_contiguous(self):
        return True

    def numel(self):
        return self._n

    def data_ptr(self):
        return A


def test_binding_rejects_tensors_on_another_device(monkeypatch):
    # launches go to the current device, so a tensor on another device is refused
    # before the library is called
    import torch
    from block_quantized_wire_gb300 import codec
    monkeypatch.setattr(torch.cuda, "current_device", lambda: 0)
    called = []
    monkeypatch.setattr(codec, "check", lambda *a: called.append(a))
    n = 1024
    x = _FakeCudaTensor(torch.bfloat16, n, 1)
    q = _FakeCudaTensor(torch.int8, n, 0)
    s = _FakeCudaTensor(torch.float32, n // 128, 0)
    with pytest.raises(ValueError, match="current CUDA device"):
        codec.quant_i8(x, q, s, stream=0)
    x0 = _FakeCudaTensor(torch.bfloat16, n, 0)
    q1 = _FakeCudaTensor(torch.int8, n, 1)
    with pytest.raises(ValueError, match="current CUDA device"):
        codec.quant_i8(x0, q1, s, stream=0)
    assert not called


def test_use_library_routes_calls_and_restores_the_default(bq_lib):
    from block_quantized_wire_gb300 import _lib, build
    main = _lib.load()
    with _lib.use_library(build.LIB) as other:
        assert _lib.load() is other and other is not main
        assert other.bq_abi_version() == _lib.ABI_VERSION
    assert _lib.load() is main
    with pytest.raises(ImportError):
        with _lib.use_library(os.path.join(os.path.dirname(build.LIB), "no_such_library.so")):
            pass
    assert _lib.load() is main


def test_alternative_build_flags_name_existing_switches():
    # a misspelt switch would build the defaults again under the alternative's name
    from block_quantized_wire_gb300 import build
    src = "".join(open(os.path.join(build.CSRC, f)).read() for f in build.SOURCES + build.HEADERS)
    for flag in build.ALT_FLAGS:
        m = re.fullmatch(r"-D(BQ_[A-Z0-9_]+)=0", flag)
        assert m, flag
        assert f"#ifndef {m.group(1)}" in src and f"#define {m.group(1)} 1" in src, flag


def test_default_build_has_no_debug_checks(bq_lib):
    # the default build compiles the access checks away and refuses the debug self-test
    # before touching the device
    assert bq_lib.bq_debug_build() == 0
    assert bq_lib.bq_selftest_index_check(None, 0, None) == 6  # BQ_ERR_UNSUPPORTED
    assert bq_lib.bq_status_string(6).decode().startswith("the call needs the debug build")
