"""The whole-step comparison on the CPU: a step assembled from whole-tensor oracle
calls passes it, and a single wrong byte planted in any output is reported with its
tensor and element index. This checks the harness the full-size GPU test relies on
(its row ranges, offsets and chaining), not the codec."""
import types

import numpy as np
import pytest
import torch

import oracle
from tests.step_check import compare_step

H, W, NS = 7168, 4, 6


def _t(a: np.ndarray, dtype=None) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(a))
    return t.view(dtype) if dtype is not None else t


def _bf16(bits_: np.ndarray) -> torch.Tensor:
    return _t(bits_.view(np.int16), torch.bfloat16)


def _wire(q: np.ndarray, s: np.ndarray):
    return (None, _t(q), _t(s))


def _oracle_step(rows: int, slice_rows: int):
    g = torch.Generator().manual_seed(11)
    xs = [(torch.randn(rows, H, generator=g) * 0.02).to(torch.bfloat16) for _ in range(W)]
    slices = [(torch.randn(slice_rows, H, generator=g) * 0.02).to(torch.bfloat16) for _ in range(NS)]
    xb = [x.view(torch.int16).numpy().view(np.uint16).reshape(-1) for x in xs]
    qs = [oracle.quant_i8(b) for b in xb]
    qa, sa, _ = oracle.dequant_accum_i8([q for q, _ in qs], [s for _, s in qs], materialize=False)
    qh, sh, _ = oracle.ring_hop_i8(qs[0][0], qs[0][1], xb[1])
    C = H * NS
    mq = np.empty((slice_rows, C), np.uint8)
    ms = np.empty((slice_rows, C // 32), np.uint8)
    for i, s in enumerate(slices):
        oracle.quant_mx_into(s.view(torch.int16).numpy().view(np.uint16), mq, ms, i * H)
    return types.SimpleNamespace(
        rows=rows, slice_rows=slice_rows, xs=xs, slices=slices,
        wires=[_wire(q, s) for q, s in qs], acc=_wire(qa, sa), hop=_wire(qh, sh),
        out=_bf16(oracle.dequant_i8(qa, sa)).view(rows, H),
        mx_q=_t(mq), mx_s=_t(ms), mx_out=_bf16(oracle.dequant_mx(mq, ms)))


@pytest.fixture(scope="module")
def step():
    return _oracle_step(rows=24, slice_rows=12)


def test_oracle_step_passes(step):
    assert compare_step(step, threads=3, rows_per_part=5, slice_rows_per_part=5) == []


@pytest.mark.parametrize("target,index,what", [
    ("wires.2.q", 3 * H + 17, "quant_i8 source 2 payload"),
    ("acc.s", 24 * H // 128 - 1, "dequant_accum_i8 scales"),
    ("out", 7 * H + 128, "dequant_i8 BF16"),
    ("hop.q", 23 * H + H - 1, "ring_hop_i8 payload"),
    ("mx_s", 11 * (H * NS // 32) + 5, "quant_mx E8M0"),
    ("mx_out", 6 * H * NS + 2 * H + 1, "dequant_mx BF16"),
])
def test_planted_byte_is_reported(step, target, index, what):
    parts = target.split(".")
    if parts[0] == "wires":
        t = step.wires[int(parts[1])][1 if parts[2] == "q" else 2]
    elif parts[0] in ("acc", "hop"):
        t = getattr(step, parts[0])[1 if parts[1] == "q" else 2]
    else:
        t = getattr(step, parts[0])
    flat = t.view(-1)
    raw = flat.view(torch.uint8) if flat.element_size() == 1 else flat.view(torch.int16 if flat.element_size() == 2
                                                                             else torch.int32)
    old = raw[index].clone()
    raw[index] = raw[index] ^ 1
    try:
        errs = compare_step(step, threads=3, rows_per_part=5, slice_rows_per_part=5)
    finally:
        raw[index] = old
    assert len(errs) == 1, errs
    assert errs[0].startswith(what + ": 1 mismatches, first at element " + str(index) + ":"), errs[0]
