"""Whole-step comparison against the oracle, used by the full-size GPU test and checked
on the CPU with a step built from the oracle itself.

`compare_step(step, threads, rows_per_part, slice_rows_per_part)` recomputes every
output of one benchmark step (quant_i8 of the W buffers, dequant_accum_i8 in source
order, dequant_i8 of the accumulated wire, ring_hop_i8 of wire 0 with buffer 1, quant_mx
of the staged slices and dequant_mx of the assembled buffer) from the step's BF16 input
bits. It runs on row ranges in host threads (blocks are independent, so the bytes are
those of one call), and the oracle chains its own results: it never sees a produced
value. Each range copies only its own rows of the step's tensors to the host. Returns
the mismatch descriptions, empty when every byte agrees. No codec arithmetic lives here.
"""
from __future__ import annotations

import numpy as np

import oracle
from oracle import shards
from tests.helpers import bits


def diff(got: np.ndarray, want: np.ndarray, what: str, base: int):
    """None if the bytes agree, else a description of the first mismatch."""
    g, w = got.reshape(-1), np.asarray(want).reshape(-1)
    assert g.view(np.uint8).size == w.view(np.uint8).size, what
    if np.array_equal(g.view(np.uint8), w.view(np.uint8)):
        return None
    gv = g.view(w.dtype)
    bad = np.nonzero(gv != w)[0]
    return f"{what}: {bad.size} mismatches, first at element {base + bad[0]}: got {gv[bad[0]]} want {w[bad[0]]}"


def compare_step(step, threads: int, rows_per_part: int = 1024, slice_rows_per_part: int = 256):
    """`step` has the benchmark pipeline's tensors: xs (W BF16 [rows, H]), wires (W
    (buffer, payload, scales)), acc, hop (the same triple), out (BF16 [rows, H]), slices
    (BF16 [slice_rows, H]), mx_q / mx_s / mx_out ([slice_rows, C], [slice_rows, C/32],
    [slice_rows, C]), and rows, slice_rows."""
    H = step.xs[0].shape[1]
    per_row = H // 128
    W = len(step.xs)

    def int8_range(lo, hi):
        errs = []
        e0, e1, b0, b1 = lo * H, hi * H, lo * per_row, hi * per_row
        xb = [bits(x[lo:hi]).reshape(-1) for x in step.xs]
        ref = [oracle.quant_i8(b) for b in xb]
        for w in range(W):
            _, q, s = step.wires[w]
            errs.append(diff(bits(q[e0:e1]), ref[w][0], f"quant_i8 source {w} payload", e0))
            errs.append(diff(bits(s[b0:b1]).view(np.uint32), ref[w][1].view(np.uint32),
                             f"quant_i8 source {w} scales", b0))
        qa, sa, _ = oracle.dequant_accum_i8([r[0] for r in ref], [r[1] for r in ref], materialize=False)
        errs.append(diff(bits(step.acc[1][e0:e1]), qa, "dequant_accum_i8 payload", e0))
        errs.append(diff(bits(step.acc[2][b0:b1]).view(np.uint32), sa.view(np.uint32),
                         "dequant_accum_i8 scales", b0))
        errs.append(diff(bits(step.out[lo:hi]), oracle.dequant_i8(qa, sa), "dequant_i8 BF16", e0))
        qh, sh, _ = oracle.ring_hop_i8(ref[0][0], ref[0][1], xb[1])
        errs.append(diff(bits(step.hop[1][e0:e1]), qh, "ring_hop_i8 payload", e0))
        errs.append(diff(bits(step.hop[2][b0:b1]).view(np.uint32), sh.view(np.uint32), "ring_hop_i8 scales", b0))
        return [e for e in errs if e]

    def mx_range(lo, hi):
        errs = []
        C = step.mx_q.shape[1]
        qb = np.empty((hi - lo, C), np.uint8)
        sb = np.empty((hi - lo, C // 32), np.uint8)
        for i, sl in enumerate(step.slices):
            oracle.quant_mx_into(bits(sl[lo:hi]), qb, sb, i * H)
        errs.append(diff(bits(step.mx_q[lo:hi]), qb, "quant_mx codes", lo * C))
        errs.append(diff(bits(step.mx_s[lo:hi]), sb, "quant_mx E8M0", lo * (C // 32)))
        errs.append(diff(bits(step.mx_out[lo:hi]), oracle.dequant_mx(qb, sb), "dequant_mx BF16", lo * C))
        return [e for e in errs if e]

    errs = shards.run(int8_range, step.rows, threads, parts=max(1, step.rows // rows_per_part))
    errs += shards.run(mx_range, step.slice_rows, threads, parts=max(1, step.slice_rows // slice_rows_per_part))
    return [e for part in errs for e in part]
