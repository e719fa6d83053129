"""The pages' wire topologies, simulated on one GPU, for both codecs.

W "ranks" are W buffers resident in one GPU's memory; moving a payload from one rank
to another is handing over the same device tensor, so there is no transport and no
collective. Each topology is a host loop over the codec calls of ``codec``; it adds no
kernels of its own.

From "feat(pcie_dma): add block-INT8 wire modes for AG, ring, and A2A", Summary:
``i8`` (BF16 reduce-scatter, INT8 all-gather: here the quantize -> materialize round
trip of one shard), ``i8_ring`` (INT8 reduce-scatter ring: the fused hop at every
step, then an INT8 all-gather), ``i8_a2a`` (each rank quantizes once, the shard owner
accumulates all sources in FP32 and requantizes, then an INT8 broadcast); in every
topology the owner materializes from the same final payload it forwards.

From "feat(pcie_dma): add INT8 and MXFP8 wire modes", Summary: ``mx``, ``mx_ring`` and
``mx_a2a`` are the same topologies with the MXFP8 codec on flat MX wires.

``i8_ag`` and ``e4m3_ag`` are the all-gather modes whole: for every shard, its owner
reduces the W ranks' BF16 copies (binary32 in rank order, one rounding to BF16) and
quantizes the result in the same kernel; every rank then materializes all W payloads.
"""
from __future__ import annotations

from typing import Callable, List, NamedTuple, Sequence

import torch

from . import codec


class Wire(NamedTuple):
    """The codec calls one topology needs, on flat wires of n values."""
    empty: Callable
    quant: Callable
    dequant: Callable
    accum: Callable
    hop: Callable


I8 = Wire(codec.empty_wire_i8, codec.quant_i8, codec.dequant_i8, codec.dequant_accum_i8, codec.ring_hop_i8)
MX = Wire(codec.empty_wire_mx, codec.quant_mx_flat, codec.dequant_mx_flat, codec.dequant_accum_mx, codec.ring_hop_mx)


def roundtrip(wire: Wire, x: torch.Tensor, stream=None):
    """Quantize one BF16 tensor and materialize it: (payload, scales, BF16)."""
    n = x.numel()
    _, q, s = wire.empty(n, x.device)
    out = torch.empty_like(x)
    wire.quant(x, q, s, stream)
    wire.dequant(q, s, out, stream)
    return q, s, out


def a2a(wire: Wire, xs: Sequence[torch.Tensor], stream=None):
    """Quantize-once all-to-all for one owner: every source is quantized, the owner sums
    the W payloads in source order and requantizes (the broadcast payload), and
    materializes it. Returns (payload, scales, owner BF16, per-source payloads)."""
    n = xs[0].numel()
    srcs = []
    for x in xs:
        _, q, s = wire.empty(n, x.device)
        wire.quant(x, q, s, stream)
        srcs.append((q, s))
    _, q_out, s_out = wire.empty(n, xs[0].device)
    owner = torch.empty_like(xs[0])
    wire.accum([q for q, _ in srcs], [s for _, s in srcs], q_out, s_out, owner, stream)
    return q_out, s_out, owner, srcs


def ring_order(shard: int, W: int) -> List[int]:
    """Ranks visited by shard `shard`'s reduce-scatter chain: it starts at the rank after
    the owner, which quantizes its own copy, and every later rank adds its copy with a
    fused hop; the last hop runs on the owner (rank `shard`)."""
    return [(shard + 1 + k) % W for k in range(W)]


def ring(wire: Wire, xs: Sequence[torch.Tensor], stream=None):
    """Quantized reduce-scatter ring + quantized all-gather over W rank buffers.

    Every buffer [rows, cols] is split into W contiguous row shards. For shard c the
    chain of ring_order(c, W) runs one quantize and W-1 fused hops, the last (at the
    owner c) also materializing the owner's BF16. Then every rank materializes all W
    final payloads into its own full-size output (the all-gather).
    Returns (per-rank BF16 outputs, final payloads [(q, s)] per shard, owner BF16 per shard).
    """
    W = len(xs)
    rows = xs[0].shape[0]
    if rows % W:
        raise ValueError("ring: rows must divide evenly into W shards")
    shard_rows = rows // W
    shards = [[x[c * shard_rows:(c + 1) * shard_rows] for c in range(W)] for x in xs]
    n = shards[0][0].numel()
    finals, owners = [], []
    for c in range(W):
        chain = ring_order(c, W)
        _, q, s = wire.empty(n, xs[0].device)
        wire.quant(shards[chain[0]][c], q, s, stream)
        owner = torch.empty_like(shards[0][c])
        for step, rank in enumerate(chain[1:], start=1):
            _, q2, s2 = wire.empty(n, xs[0].device)
            last = step == W - 1
            wire.hop(q, s, shards[rank][c], q2, s2, owner if last else None, stream)
            q, s = q2, s2
        finals.append((q, s))
        owners.append(owner)
    outs = []
    for _rank in range(W):
        out = torch.empty_like(xs[0])
        for c in range(W):
            wire.dequant(finals[c][0], finals[c][1], out[c * shard_rows:(c + 1) * shard_rows], stream)
        outs.append(out)
    return outs, finals, owners


# the pages' mode names
def i8_roundtrip(x, stream=None):
    return roundtrip(I8, x, stream)


def i8_a2a(xs, stream=None):
    return a2a(I8, xs, stream)


def i8_ring(xs, stream=None):
    return ring(I8, xs, stream)


def mx_roundtrip(x, stream=None):
    return roundtrip(MX, x, stream)


def mx_a2a(xs, stream=None):
    return a2a(MX, xs, stream)


def mx_ring(xs, stream=None):
    return ring(MX, xs, stream)


def _allgather(reduce_quant, empty, dequant, xs, stream=None):
    """BF16 reduce-scatter fused with quantization, then the quantized all-gather.
    Returns (per-rank BF16 outputs, payload (q, s) per shard, owner BF16 per shard)."""
    W = len(xs)
    rows = xs[0].shape[0]
    if rows % W:
        raise ValueError("all-gather mode: rows must divide evenly into W shards")
    sr = rows // W
    n = xs[0][:sr].numel()
    finals, owners = [], []
    for c in range(W):
        _, q, s = empty(n, xs[0].device)
        owner = torch.empty_like(xs[0][c * sr:(c + 1) * sr])
        reduce_quant([x[c * sr:(c + 1) * sr] for x in xs], q, s, owner, stream)
        finals.append((q, s))
        owners.append(owner)
    outs = []
    for _rank in range(W):
        out = torch.empty_like(xs[0])
        for c in range(W):
            dequant(finals[c][0], finals[c][1], out[c * sr:(c + 1) * sr], stream)
        outs.append(out)
    return outs, finals, owners


def i8_ag(xs, stream=None):
    """The ``i8`` mode: BF16 reduce-scatter + INT8 all-gather."""
    return _allgather(codec.reduce_quant_i8, codec.empty_wire_i8, codec.dequant_i8, xs, stream)


def e4m3_ag(xs, stream=None):
    """The E4M3 all-gather mode with the legacy E4M3 codec."""
    return _allgather(codec.reduce_quant_e4m3, codec.empty_wire_e4m3, codec.dequant_e4m3, xs, stream)


# Mode selection by name ("feat(pcie_dma): add INT8 and MXFP8 wire modes", Modes:
# names are matched after trimming surrounding whitespace and ignoring case; an empty
# name keeps the uncompressed BF16 path; any other unknown name is an error rather than
# a silent fallback).
MODES = {
    "i8": i8_roundtrip,     # per-shard quantize -> materialize of the INT8 all-gather
    "i8_ring": i8_ring,
    "i8_a2a": i8_a2a,
    "i8_ag": i8_ag,         # BF16 reduce-scatter fused with the INT8 all-gather payload
    "mx": mx_roundtrip,
    "mx_ring": mx_ring,
    "mx_a2a": mx_a2a,
    "e4m3_ag": e4m3_ag,
}


def select_mode(name):
    """The topology function for a wire-mode name, or None for the BF16 path (empty or
    whitespace-only name). Raises ValueError for any other unknown name."""
    if name is None:
        return None
    key = str(name).strip().lower()
    if not key:
        return None
    try:
        return MODES[key]
    except KeyError:
        raise ValueError(f"unknown wire mode {name!r}; expected one of {sorted(MODES)} or empty for BF16") from None
