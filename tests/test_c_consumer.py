"""libbq.so used from plain C (tests/c_consumer/bq_c_demo.c): it compiles and links
with gcc against include/bq.h on any machine, and on a GPU its outputs equal the
oracle's for the same input bits."""
import glob
import os
import subprocess

import numpy as np
import pytest

import oracle
from block_quantized_wire_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c_consumer", "bq_c_demo.c")


def _cuda_dirs():
    root = os.path.dirname(os.path.dirname(build.nvcc()))
    libs = [d for d in [os.path.join(root, "lib64")] + glob.glob(os.path.join(root, "targets", "*", "lib"))
            if os.path.exists(os.path.join(d, "libcudart.so"))]
    return os.path.join(root, "include"), libs[0]


def _compile(out_path):
    build.build_library()
    inc, lib = _cuda_dirs()
    libdir = os.path.dirname(build.LIB)
    cmd = ["gcc", "-O2", "-std=c11", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"), "-I", inc,
           SRC, "-o", out_path, "-L", libdir, "-lbq", "-L", lib, "-lcudart", f"-Wl,-rpath,{libdir}",
           f"-Wl,-rpath,{lib}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return out_path


def test_c_consumer_compiles_and_links(tmp_path):
    exe = _compile(str(tmp_path / "bq_c_demo"))
    assert os.path.exists(exe)


@pytest.mark.gpu
def test_c_consumer_outputs_equal_the_oracle(tmp_path):
    exe = _compile(str(tmp_path / "bq_c_demo"))
    rng = np.random.default_rng(71)
    n = 128 * 1003
    x = (rng.standard_normal(n) * 10.0 ** rng.uniform(-3, 3, n)).astype(np.float32)
    x[:128] = 0.0
    bits = (x.view(np.uint32) >> 16).astype(np.uint16)  # truncation is fine: any BF16 bits
    inp, out = tmp_path / "x.bf16", tmp_path / "out.bin"
    bits.tofile(inp)
    r = subprocess.run([exe, str(inp), str(out)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    raw = np.fromfile(out, np.uint8)
    o = 0
    payload = raw[o:o + n].view(np.int8); o += n
    scales = raw[o:o + 4 * (n // 128)].view(np.float32); o += 4 * (n // 128)
    mat = raw[o:o + 2 * n].view(np.uint16); o += 2 * n
    codes = raw[o:o + n]; o += n
    e8 = raw[o:o + n // 32]; o += n // 32
    assert o == raw.size
    q, s = oracle.quant_i8(bits)
    assert np.array_equal(payload, q) and np.array_equal(scales.view(np.uint32), s.view(np.uint32))
    assert np.array_equal(mat, oracle.dequant_i8(q, s))
    qm, sm = oracle.quant_mx_flat(bits)
    assert np.array_equal(codes, qm) and np.array_equal(e8, sm)
