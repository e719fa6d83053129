"""Whole-tensor parity at full size, in the launch configuration the benchmark times.

The benchmark's own step (four 65536x7168 BF16 buffers through quant_i8 x4,
dequant_accum_i8 (W=4), dequant_i8 and ring_hop_i8; six 4096x7168 slices staged by
quant_mx into one 4096x43008 buffer, then dequant_mx) runs once on the GPU. Then the
oracle recomputes every output byte from the same BF16 input bits. It runs on row
ranges in host threads (blocks are independent, so the bytes are those of one call),
and the oracle chains its own results: it never sees a value the GPU produced. Every
payload byte, scale word and BF16 output is compared. Each range copies only its own
rows from the device, which bounds host memory.

The kernels beyond the step (the MX wire reductions, the fused reduce + quantize of
the all-gather modes, the legacy E4M3 codec, FP16 slices with row-major and tiled
scales) get the same whole-tensor comparison on the same full-size inputs.
"""
import numpy as np
import pytest
import torch

import bench
import oracle
from block_quantized_wire_gb300 import codec, inputs
from oracle import shards
from tests.helpers import bits
from tests.step_check import compare_step, diff

pytestmark = pytest.mark.gpu

ROWS, SLICE_ROWS = 65536, 4096  # the benchmark's buffers and slices


@pytest.fixture(scope="module", autouse=True)
def _lib(bq_lib):
    return bq_lib


def test_prefill_step_whole_tensors_bitexact():
    torch.cuda.empty_cache()
    pipe = bench.Pipeline(ROWS, SLICE_ROWS, torch.device("cuda"))
    pipe.run()
    torch.cuda.synchronize()
    # 1024-row ranges: about 0.2 GB of host memory per thread at a time
    errs = compare_step(pipe, shards.host_cores())
    assert not errs, "\n".join(errs[:20])


def test_next_rows_whole_tensors_bitexact():
    # The kernels beyond the step, on the benchmark's full-size inputs and in the calls
    # its next_rows section times: flat MX wires of the four prefill buffers,
    # dequant_accum_mx (W=4) and ring_hop_mx over them, reduce_quant_i8 and
    # reduce_quant_e4m3 of the four buffers, quant_e4m3 + dequant_e4m3 of buffer 2, and
    # the six FP16 slices staged by quant_mx into row-major and tiled scales.
    torch.cuda.empty_cache()
    H, W = bench.HIDDEN, bench.W_SRC
    n = ROWS * H
    xs = [inputs.prefill_buffer(w, device="cuda", rows=ROWS) for w in range(W)]
    flat = [x.view(-1) for x in xs]
    mw = [codec.empty_wire_mx(n) for _ in range(W)]
    for w in range(W):
        codec.quant_mx_flat(flat[w], mw[w][1], mw[w][2])
    _, qa, sa = codec.empty_wire_mx(n)
    codec.dequant_accum_mx([m[1] for m in mw], [m[2] for m in mw], qa, sa, None)
    _, qh, sh = codec.empty_wire_mx(n)
    codec.ring_hop_mx(mw[0][1], mw[0][2], flat[1], qh, sh, None)
    _, qr, sr = codec.empty_wire_i8(n)
    codec.reduce_quant_i8(flat, qr, sr, None)
    _, qe, se = codec.empty_wire_e4m3(n)
    codec.reduce_quant_e4m3(flat, qe, se, None)
    _, q4, s4 = codec.empty_wire_e4m3(n)
    codec.quant_e4m3(flat[2], q4, s4)
    d4 = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    codec.dequant_e4m3(q4, s4, d4)

    f16 = inputs.mx_slices_4096(device="cuda", rows=SLICE_ROWS, dtype=torch.float16)
    C = H * len(f16)
    g_total = C // 32
    mq, ms = codec.empty_mx(SLICE_ROWS, C)
    tq = torch.empty_like(mq)
    tiled = torch.empty(codec.mx_tiled_scale_bytes(SLICE_ROWS, g_total), dtype=torch.uint8, device="cuda")
    for i, x in enumerate(f16):
        c0 = i * H
        codec.quant_mx(x, mq[:, c0:c0 + H], ms[:, c0 // 32:(c0 + H) // 32])
        codec.quant_mx_tiled(x, tq[:, c0:c0 + H], tiled, g_total, c0 // 32)
    torch.cuda.synchronize()

    def flat_range(lo, hi):
        e0, e1 = lo * H, hi * H
        g0, g1, b0, b1 = e0 // 32, e1 // 32, e0 // 128, e1 // 128
        xb = [bits(x[lo:hi]).reshape(-1) for x in xs]
        errs = []
        ref = [oracle.quant_mx_flat(b) for b in xb]
        for w in range(W):
            errs.append(diff(bits(mw[w][1][e0:e1]), ref[w][0], f"quant_mx flat {w} codes", e0))
            errs.append(diff(bits(mw[w][2][g0:g1]), ref[w][1], f"quant_mx flat {w} E8M0", g0))
        aq, as_, _ = oracle.dequant_accum_mx([r[0] for r in ref], [r[1] for r in ref], materialize=False)
        errs.append(diff(bits(qa[e0:e1]), aq, "dequant_accum_mx codes", e0))
        errs.append(diff(bits(sa[g0:g1]), as_, "dequant_accum_mx E8M0", g0))
        hq, hs, _ = oracle.ring_hop_mx(ref[0][0], ref[0][1], xb[1])
        errs.append(diff(bits(qh[e0:e1]), hq, "ring_hop_mx codes", e0))
        errs.append(diff(bits(sh[g0:g1]), hs, "ring_hop_mx E8M0", g0))
        rq, rs, _ = oracle.reduce_quant_i8(xb)
        errs.append(diff(bits(qr[e0:e1]), rq, "reduce_quant_i8 payload", e0))
        errs.append(diff(bits(sr[b0:b1]).view(np.uint32), rs.view(np.uint32), "reduce_quant_i8 scales", b0))
        eq, es, _ = oracle.reduce_quant_e4m3(xb)
        errs.append(diff(bits(qe[e0:e1]), eq, "reduce_quant_e4m3 codes", e0))
        errs.append(diff(bits(se[b0:b1]).view(np.uint32), es.view(np.uint32), "reduce_quant_e4m3 scales", b0))
        cq, cs = oracle.quant_e4m3(xb[2])
        errs.append(diff(bits(q4[e0:e1]), cq, "quant_e4m3 codes", e0))
        errs.append(diff(bits(s4[b0:b1]).view(np.uint32), cs.view(np.uint32), "quant_e4m3 scales", b0))
        errs.append(diff(bits(d4[e0:e1]), oracle.dequant_e4m3(cq, cs), "dequant_e4m3 BF16", e0))
        return [e for e in errs if e]

    tile_row_bytes = (g_total // 4) * 512  # one 128-row band of the tiled layout

    def f16_range(lo, hi):  # lo, hi multiples of 128
        qb = np.empty((hi - lo, C), np.uint8)
        sb = np.empty((hi - lo, g_total), np.uint8)
        for i, x in enumerate(f16):
            oracle.quant_mx_into(x[lo:hi].contiguous().view(torch.int16).cpu().numpy().view(np.uint16), qb, sb,
                                 i * H, fmt="f16")
        errs = [diff(bits(mq[lo:hi]), qb, "quant_mx f16 codes", lo * C),
                diff(bits(ms[lo:hi]), sb, "quant_mx f16 E8M0", lo * g_total),
                diff(bits(tq[lo:hi]), qb, "quant_mx_tiled codes", lo * C),
                diff(bits(tiled[lo // 128 * tile_row_bytes:hi // 128 * tile_row_bytes]),
                     oracle.mx_scales_to_tiled(sb), "quant_mx_tiled scales", lo // 128 * tile_row_bytes)]
        return [e for e in errs if e]

    T = shards.host_cores()
    errs = shards.run(flat_range, ROWS, T, parts=ROWS // 1024)
    bands = SLICE_ROWS // 128
    errs += shards.run(lambda lo, hi: f16_range(lo * 128, hi * 128), bands, T, parts=min(bands, 16))
    flat_errs = [e for part in errs for e in part]
    assert not flat_errs, "\n".join(flat_errs[:20])
