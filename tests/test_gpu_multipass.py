"""Parity at sizes where every warp of a launch walks several chunks and a ragged tail
follows: the grid-stride loops, the two-stage per-lane async copies of the
accumulates (each stage refilled several times) and the one-CTA-per-SM launches are
exercised beyond their first pass. Bit-exact against the oracle; outputs framed by
guard bands.

Operations: "feat(pcie_dma): add block-INT8 wire modes for AG, ring, and A2A",
Implementation (quantize, materialize, multi-source accumulate, ring hop) and Summary
(the i8 all-gather mode, whose BF16 reduce is fused with quantization here, and the
legacy E4M3 codec it is compared against), and "feat(pcie_dma): add INT8 and MXFP8 wire
modes", Summary (the same topologies on MX wires)."""
import numpy as np
import pytest
import torch

import oracle
from block_quantized_wire_gb300 import codec
from tests.helpers import Guarded, adversarial_blocks, bits, from_bits_bf16

pytestmark = pytest.mark.gpu


def multipass_nblk() -> int:
    """Three passes of 32 warps per SM over 8-block chunks, then a 5-block tail (a
    512-thread launch of 16 warps per SM makes six passes)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    return 3 * sms * 32 * 8 + 5


def source_bits(seed: int, nblk: int) -> np.ndarray:
    """BF16 bits [nblk * 128]: normal values with a magnitude per block across 2^-40..2^40,
    and adversarial blocks (subnormal, tie-heavy, near-maximum, zero) at both ends."""
    rng = np.random.default_rng(seed)
    mag = np.exp2(rng.integers(-40, 41, nblk)).astype(np.float64)
    v = (rng.standard_normal((nblk, 128)) * mag[:, None]).astype(np.float32)
    xb = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()
    k = 45
    xb[:k] = adversarial_blocks(rng, k, max_abs=1.0e37)
    xb[-k:] = adversarial_blocks(rng, k, max_abs=1.0e37)
    return xb.reshape(-1)


def same(got: torch.Tensor, want: np.ndarray, what: str):
    """Byte-for-byte equality of a device result with the oracle's array."""
    g = bits(got).reshape(-1).view(np.uint8)
    w = np.ascontiguousarray(want).reshape(-1).view(np.uint8)
    assert g.size == w.size, f"{what}: {g.size} bytes against {w.size}"
    if not np.array_equal(g, w):
        bad = np.flatnonzero(g != w)
        raise AssertionError(f"{what}: {bad.size} bytes differ, first at byte {bad[0]}")


@pytest.fixture(scope="module")
def i8_sources():
    nblk = multipass_nblk()
    xs = [source_bits(900 + i, nblk) for i in range(5)]
    refs = [oracle.quant_i8(x) for x in xs]
    return nblk, xs, refs


def test_quant_dequant_multipass(i8_sources):
    nblk, xs, refs = i8_sources
    n = nblk * 128
    gq, gs, go = Guarded(n), Guarded(4 * nblk), Guarded(2 * n)
    codec.quant_i8(from_bits_bf16(xs[0]), gq.view(torch.int8), gs.view(torch.float32))
    same(gq.view(torch.int8), refs[0][0], "payload")
    same(gs.view(torch.float32), refs[0][1], "scales")
    codec.dequant_i8(gq.view(torch.int8), gs.view(torch.float32), go.view(torch.bfloat16))
    same(go.view(torch.bfloat16), oracle.dequant_i8(*refs[0]), "materialized")
    assert gq.bands_intact() and gs.bands_intact() and go.bands_intact()


@pytest.mark.parametrize("owner", [False, True])
def test_ring_hop_multipass(i8_sources, owner):
    nblk, xs, refs = i8_sources
    n = nblk * 128
    gq, gs, go = Guarded(n), Guarded(4 * nblk), Guarded(2 * n)
    qi, si = torch.from_numpy(refs[0][0]).cuda(), torch.from_numpy(refs[0][1]).cuda()
    codec.ring_hop_i8(qi, si, from_bits_bf16(xs[1]), gq.view(torch.int8), gs.view(torch.float32),
                      go.view(torch.bfloat16) if owner else None)
    qh, sh, oh = oracle.ring_hop_i8(refs[0][0], refs[0][1], xs[1], materialize=owner)
    same(gq.view(torch.int8), qh, "hop payload")
    same(gs.view(torch.float32), sh, "hop scales")
    if owner:
        same(go.view(torch.bfloat16), oh, "hop materialized")
    else:
        assert (go.raw == Guarded.SENTINEL).all().item()
    assert gq.bands_intact() and gs.bands_intact() and go.bands_intact()


@pytest.mark.parametrize("owner", [False, True])
@pytest.mark.parametrize("W", [1, 2, 3, 4, 5])
def test_accumulate_multipass(i8_sources, W, owner):
    # W <= 4 without the owner output: the per-lane async copy kernel; the rest: direct loads
    nblk, _, refs = i8_sources
    n = nblk * 128
    qd = [torch.from_numpy(r[0]).cuda() for r in refs[:W]]
    sd = [torch.from_numpy(r[1]).cuda() for r in refs[:W]]
    gq, gs, go = Guarded(n), Guarded(4 * nblk), Guarded(2 * n)
    codec.dequant_accum_i8(qd, sd, gq.view(torch.int8), gs.view(torch.float32),
                           go.view(torch.bfloat16) if owner else None)
    qa, sa, oa = oracle.dequant_accum_i8([r[0] for r in refs[:W]], [r[1] for r in refs[:W]], materialize=owner)
    same(gq.view(torch.int8), qa, "accumulated payload")
    same(gs.view(torch.float32), sa, "accumulated scales")
    if owner:
        same(go.view(torch.bfloat16), oa, "accumulated materialized")
    assert gq.bands_intact() and gs.bands_intact() and go.bands_intact()


@pytest.mark.parametrize("W", [1, 2, 4])
def test_mx_accumulate_multipass(W):
    nblk = multipass_nblk()
    n = nblk * 128
    xs = [source_bits(950 + i, nblk) for i in range(W)]
    refs = [oracle.quant_mx_flat(x) for x in xs]
    qd = [torch.from_numpy(r[0]).cuda() for r in refs]
    sd = [torch.from_numpy(r[1]).cuda() for r in refs]
    gq, gs = Guarded(n), Guarded(n // 32)
    codec.dequant_accum_mx(qd, sd, gq.view(torch.uint8), gs.view(torch.uint8), None)
    qa, sa, _ = oracle.dequant_accum_mx([r[0] for r in refs], [r[1] for r in refs], materialize=False)
    same(gq.view(torch.uint8), qa, "MX accumulated codes")
    same(gs.view(torch.uint8), sa, "MX accumulated scales")
    assert gq.bands_intact() and gs.bands_intact()


@pytest.mark.parametrize("owner", [False, True])
@pytest.mark.parametrize("W", [1, 2, 4, 5])
@pytest.mark.parametrize("codec_name", ["i8", "e4m3"])
def test_reduce_quant_multipass(i8_sources, codec_name, W, owner):
    # W <= 4: the per-lane async copy kernel of exactly W sources; 5: groups of four
    nblk, xs, _ = i8_sources
    n = nblk * 128
    xd = [from_bits_bf16(x) for x in xs[:W]]
    gq, gs, go = Guarded(n), Guarded(4 * nblk), Guarded(2 * n)
    qt = torch.int8 if codec_name == "i8" else torch.uint8
    run = codec.reduce_quant_i8 if codec_name == "i8" else codec.reduce_quant_e4m3
    run(xd, gq.view(qt), gs.view(torch.float32), go.view(torch.bfloat16) if owner else None)
    ref = oracle.reduce_quant_i8 if codec_name == "i8" else oracle.reduce_quant_e4m3
    qr, sr, orr = ref(xs[:W], materialize=owner)
    same(gq.view(qt), qr, f"{codec_name} reduced payload")
    same(gs.view(torch.float32), sr, f"{codec_name} reduced scales")
    if owner:
        same(go.view(torch.bfloat16), orr, f"{codec_name} reduced materialized")
    else:
        assert (go.raw == Guarded.SENTINEL).all().item()
    assert gq.bands_intact() and gs.bands_intact() and go.bands_intact()


def test_e4m3_quant_dequant_multipass(i8_sources):
    nblk, xs, _ = i8_sources
    n = nblk * 128
    gq, gs, go = Guarded(n), Guarded(4 * nblk), Guarded(2 * n)
    codec.quant_e4m3(from_bits_bf16(xs[2]), gq.view(torch.uint8), gs.view(torch.float32))
    qr, sr = oracle.quant_e4m3(xs[2])
    same(gq.view(torch.uint8), qr, "E4M3 codes")
    same(gs.view(torch.float32), sr, "E4M3 scales")
    codec.dequant_e4m3(gq.view(torch.uint8), gs.view(torch.float32), go.view(torch.bfloat16))
    same(go.view(torch.bfloat16), oracle.dequant_e4m3(qr, sr), "E4M3 materialized")
    assert gq.bands_intact() and gs.bands_intact() and go.bands_intact()
