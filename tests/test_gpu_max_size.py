"""Sizes past 2^31 elements: every kernel indexes with 64-bit offsets, so a tensor larger
than any 32-bit element count must come out as bit-exact as a small one.

One BF16 tensor of 2^31 + 2^20 + 384 values (4.3 GB; the tail is a ragged, partial
chunk) goes through quant_i8, dequant_i8, dequant_accum_i8 (two sources),
ring_hop_i8 and the E4M3 codec; one BF16 matrix of 299,600 x 7168 values (rows x
cols past 2^31) goes through quant_mx and dequant_mx. The oracle recomputes sampled
blocks (MX: rows) from the same input bits: the first ones, the ones around element
2^31, the last ones, and a random sample in between.
"""
import numpy as np
import pytest
import torch

import oracle
from block_quantized_wire_gb300 import codec
from tests.helpers import bits

pytestmark = pytest.mark.gpu

N = 2 ** 31 + 2 ** 20 + 3 * 128
NBLK = N // 128


@pytest.fixture(scope="module", autouse=True)
def _lib(bq_lib):
    return bq_lib


def _randn_bf16(n: int, seed: int, shape=None) -> torch.Tensor:
    g = torch.Generator(device="cuda").manual_seed(seed)
    out = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    step = 1 << 28  # draw in pieces to bound the FP32 temporary
    for lo in range(0, n, step):
        hi = min(n, lo + step)
        out[lo:hi] = torch.randn(hi - lo, generator=g, device="cuda").mul_(0.02).to(torch.bfloat16)
    return out.view(shape) if shape is not None else out


def _sample_blocks(nblk: int, seed: int) -> np.ndarray:
    edge = 2 ** 31 // 128
    picks = [np.arange(0, 8), np.arange(edge - 8, edge + 8), np.arange(nblk - 8, nblk),
             np.random.default_rng(seed).choice(nblk, 2048, replace=False)]
    return np.unique(np.concatenate(picks))


def _gather(t: torch.Tensor, blk: np.ndarray, width: int) -> np.ndarray:
    idx = torch.from_numpy(blk).cuda()
    return bits(t.view(-1, width)[idx]).reshape(-1)


def _same(got: np.ndarray, want: np.ndarray, what: str):
    g, w = got.reshape(-1), np.asarray(want).reshape(-1)
    if not np.array_equal(g.view(np.uint8), w.view(np.uint8)):
        bad = np.nonzero(g.view(w.dtype) != w)[0]
        raise AssertionError(f"{what}: {bad.size} mismatches, first at sampled element {bad[0]}")


def test_int8_and_e4m3_paths_past_2_pow_31_elements():
    torch.cuda.empty_cache()
    x0 = _randn_bf16(N, 31)
    _, q0, s0 = codec.empty_wire_i8(N)
    codec.quant_i8(x0, q0, s0)
    blk = _sample_blocks(NBLK, 1)
    xb0 = _gather(x0, blk, 128)
    rq0, rs0 = oracle.quant_i8(xb0)
    _same(_gather(q0, blk, 128), rq0, "quant_i8 payload")
    _same(bits(s0[torch.from_numpy(blk).cuda()]).view(np.uint32), rs0.view(np.uint32), "quant_i8 scales")

    out = torch.empty(N, dtype=torch.bfloat16, device="cuda")
    codec.dequant_i8(q0, s0, out)
    _same(_gather(out, blk, 128), oracle.dequant_i8(rq0, rs0), "dequant_i8")

    x1 = _randn_bf16(N, 32)
    xb1 = _gather(x1, blk, 128)
    _, q1, s1 = codec.empty_wire_i8(N)
    codec.quant_i8(x1, q1, s1)
    rq1, rs1 = oracle.quant_i8(xb1)
    _, qa, sa = codec.empty_wire_i8(N)
    codec.dequant_accum_i8([q0, q1], [s0, s1], qa, sa, out)  # with the owner output
    aq, as_, ao = oracle.dequant_accum_i8([rq0, rq1], [rs0, rs1])
    _same(_gather(qa, blk, 128), aq, "dequant_accum_i8 payload")
    _same(bits(sa[torch.from_numpy(blk).cuda()]).view(np.uint32), as_.view(np.uint32), "dequant_accum_i8 scales")
    _same(_gather(out, blk, 128), ao, "dequant_accum_i8 owner BF16")
    del q1, s1

    _, qh, sh = codec.empty_wire_i8(N)
    codec.ring_hop_i8(q0, s0, x1, qh, sh, None)
    hq, hs, _ = oracle.ring_hop_i8(rq0, rs0, xb1)
    _same(_gather(qh, blk, 128), hq, "ring_hop_i8 payload")
    _same(bits(sh[torch.from_numpy(blk).cuda()]).view(np.uint32), hs.view(np.uint32), "ring_hop_i8 scales")
    del qh, sh, qa, sa

    _, qe, se = codec.empty_wire_e4m3(N)
    codec.quant_e4m3(x1, qe, se)
    eq, es = oracle.quant_e4m3(xb1)
    _same(_gather(qe, blk, 128), eq, "quant_e4m3 codes")
    _same(bits(se[torch.from_numpy(blk).cuda()]).view(np.uint32), es.view(np.uint32), "quant_e4m3 scales")
    codec.dequant_e4m3(qe, se, out)
    _same(_gather(out, blk, 128), oracle.dequant_e4m3(eq, es), "dequant_e4m3")
    torch.cuda.synchronize()


def test_mx_past_2_pow_31_elements():
    torch.cuda.empty_cache()
    rows, cols = 299_600, 7168  # rows * cols = 2,147,532,800 > 2^31
    x = _randn_bf16(rows * cols, 33, (rows, cols))
    q, s = codec.empty_mx(rows, cols)
    codec.quant_mx(x, q, s)
    out = torch.empty_like(x)
    codec.dequant_mx(q, s, out)
    edge_row = 2 ** 31 // cols
    picks = [np.arange(0, 2), np.arange(edge_row - 2, edge_row + 3), np.arange(rows - 2, rows),
             np.random.default_rng(2).choice(rows, 64, replace=False)]
    r = np.unique(np.concatenate(picks))
    idx = torch.from_numpy(r).cuda()
    xr = bits(x[idx])
    rq, rs = oracle.quant_mx(xr)
    _same(bits(q[idx]), rq, "quant_mx codes")
    _same(bits(s[idx]), rs, "quant_mx E8M0")
    _same(bits(out[idx]), oracle.dequant_mx(rq, rs), "dequant_mx")
    # the same matrix as two strided half-width slices quantized by one call: the bytes of
    # the single call, every one of them (the destination holds more than 2^31 values)
    del out
    q2, s2 = codec.empty_mx(rows, cols)
    codec.quant_mx_slices([x[:, :cols // 2], x[:, cols // 2:]], q2, s2)
    assert torch.equal(q2, q) and torch.equal(s2, s)
