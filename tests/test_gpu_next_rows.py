"""The all-gather modes' fused BF16 reduce + quantize (i8 and E4M3), the legacy E4M3
codec, and FP16 MX slices, vs the CPU oracle, bit for bit, through the C ABI.

Pages: "feat(pcie_dma): add block-INT8 wire modes for AG, ring, and A2A", Summary and
Why (the i8 mode, the E4M3 codec it compares against); "[II] Support staged MXFP8
linear inputs", Behavior (BF16 or FP16 slices). Expected values come only from the
oracle run on the same input bits.
"""
import numpy as np
import pytest
import torch

import oracle
from block_quantized_wire_gb300 import codec, inputs, topology
from block_quantized_wire_gb300._lib import BQError
from tests.helpers import Guarded, adversarial_blocks, bits, from_bits_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(bq_lib):
    return bq_lib


def assert_same(got: torch.Tensor, want: np.ndarray, what: str):
    g = bits(got).reshape(-1)
    w = np.asarray(want).reshape(-1)
    if not np.array_equal(g.view(np.uint8), w.view(np.uint8)):
        g2 = g.view(w.dtype)
        bad = np.nonzero(g2 != w)[0]
        raise AssertionError(f"{what}: {bad.size} mismatches, first at {bad[0]}: got {g2[bad[0]]} want {w[bad[0]]}")


def f16_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


CODECS = {
    "i8": (codec.reduce_quant_i8, codec.empty_wire_i8, oracle.reduce_quant_i8, oracle.dequant_i8, torch.int8),
    "e4m3": (codec.reduce_quant_e4m3, codec.empty_wire_e4m3, oracle.reduce_quant_e4m3, oracle.dequant_e4m3,
             torch.uint8),
}


# ------------------------------------------------------------------ reduce + quantize
@pytest.mark.parametrize("name", list(CODECS))
def test_allgather_mode_bitexact(name):
    xs = [x.cuda() for x in inputs.a2a_3072(rows=1024)]
    W = len(xs)
    outs, finals, owners = (topology.i8_ag if name == "i8" else topology.e4m3_ag)(xs)
    _, _, ref_rq, ref_deq, _ = CODECS[name]
    xb = [bits(x).reshape(W, -1) for x in xs]
    sr = xs[0].shape[0] // W
    for c in range(W):
        q, s, o = ref_rq([xb[w][c] for w in range(W)], materialize=True)
        assert_same(finals[c][0], q, f"shard {c} payload")
        assert_same(finals[c][1], s, f"shard {c} scales")
        assert_same(owners[c], o, f"shard {c} owner")
    for o in outs[1:]:
        assert torch.equal(o, outs[0])
    for c in range(W):
        assert torch.equal(owners[c], outs[0][c * sr:(c + 1) * sr])


@pytest.mark.parametrize("name", list(CODECS))
@pytest.mark.parametrize("nblk", [1, 2, 3, 5, 8, 9, 17, 63, 65, 1027, 4099])
def test_reduce_quant_ragged(name, nblk):
    rq, _, ref_rq, _, qtype = CODECS[name]
    rng = np.random.default_rng(800 + nblk)
    W = 3
    xs = [adversarial_blocks(rng, nblk, max_abs=1.0e37).reshape(-1) for _ in range(W)]
    xs[1][:256] = xs[0][:256] ^ 0x8000  # cancellations to +0 and tiny sums
    n = nblk * 128
    gq, gs, go = Guarded(n), Guarded(4 * nblk), Guarded(2 * n)
    rq([from_bits_bf16(x) for x in xs], gq.view(qtype), gs.view(torch.float32), go.view(torch.bfloat16))
    q, s, o = ref_rq(xs, materialize=True)
    assert_same(gq.view(qtype), q, "payload")
    assert_same(gs.view(torch.float32), s, "scales")
    assert_same(go.view(torch.bfloat16), o, "materialized")
    assert gq.bands_intact() and gs.bands_intact() and go.bands_intact()


@pytest.mark.parametrize("name", list(CODECS))
@pytest.mark.parametrize("W", [1, 2, 3, 4, 5, 8, 9, 16])
def test_reduce_quant_any_width(name, W):
    rq, empty, ref_rq, _, _ = CODECS[name]
    rng = np.random.default_rng(900 + W)
    nblk = 41
    xs = [adversarial_blocks(rng, nblk, max_abs=1.0e36).reshape(-1) for _ in range(W)]
    for w in range(W):  # a block of negative zeros in every source (-0 + ... + -0 = -0)
        xs[w][128:256] = 0x8000
    xs[0][128] = 0x0000
    n = nblk * 128
    _, q, s = empty(n)
    rq([from_bits_bf16(x) for x in xs], q, s, None)
    qr, sr, _ = ref_rq(xs)
    assert_same(q, qr, "payload")
    assert_same(s, sr, "scales")


@pytest.mark.parametrize("name", list(CODECS))
def test_reduce_quant_prefill_sampled(name):
    # full-size launch (4 x 65536 x 7168, as the benchmark times it); 4096 sampled blocks
    rq, empty, ref_rq, ref_deq, _ = CODECS[name]
    torch.cuda.empty_cache()
    xs = inputs.prefill_65536()
    n = xs[0].numel()
    _, q, s = empty(n)
    out = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    rq([x.reshape(-1) for x in xs], q, s, out)
    torch.cuda.synchronize()
    rng = np.random.default_rng(9)
    blk = np.sort(rng.choice(n // 128, 4096, replace=False))
    blk[-1] = n // 128 - 1
    idx = torch.from_numpy(blk).cuda()
    xb = [bits(x.reshape(-1, 128)[idx]) for x in xs]
    qr, sr, orr = ref_rq(xb, materialize=True)
    assert_same(q.reshape(-1, 128)[idx], qr, "payload")
    assert_same(s[idx], sr, "scales")
    assert_same(out.reshape(-1, 128)[idx], orr, "materialized")


def test_reduce_quant_errors():
    n = 256
    x = torch.zeros(n, dtype=torch.bfloat16, device="cuda")
    _, q, s = codec.empty_wire_i8(n)
    with pytest.raises(BQError) as ei:
        codec.reduce_quant_i8([x] * 17, q, s)
    assert ei.value.status == 2
    with pytest.raises(BQError) as ei:  # a payload that overlaps a source
        codec.reduce_quant_i8([x], x.view(torch.int8)[:n], s)
    assert ei.value.status == 4
    e = torch.empty(0, dtype=torch.bfloat16, device="cuda")
    codec.reduce_quant_i8([e], torch.empty(0, dtype=torch.int8, device="cuda"),
                          torch.empty(0, dtype=torch.float32, device="cuda"))


# ------------------------------------------------------------------ legacy E4M3 codec
@pytest.mark.parametrize("workload", ["roundtrip_512", "mixed_3072"])
def test_e4m3_codec_workloads(workload):
    x = getattr(inputs, workload)().cuda()
    n = x.numel()
    _, q, s = codec.empty_wire_e4m3(n)
    out = torch.empty_like(x)
    codec.quant_e4m3(x.reshape(-1), q, s)
    codec.dequant_e4m3(q, s, out.reshape(-1))
    qr, sr = oracle.quant_e4m3(bits(x))
    assert_same(q, qr, "codes")
    assert_same(s, sr, "scales")
    assert_same(out, oracle.dequant_e4m3(qr, sr), "materialized")


@pytest.mark.parametrize("nblk", [1, 2, 3, 7, 8, 9, 15, 16, 17, 63, 64, 65, 1001, 4099])
def test_e4m3_ragged_and_adversarial(nblk):
    rng = np.random.default_rng(1000 + nblk)
    xb = adversarial_blocks(rng, nblk).reshape(-1)
    n = xb.size
    gq, gs, go = Guarded(n), Guarded(4 * nblk), Guarded(2 * n)
    codec.quant_e4m3(from_bits_bf16(xb), gq.view(torch.uint8), gs.view(torch.float32))
    codec.dequant_e4m3(gq.view(torch.uint8), gs.view(torch.float32), go.view(torch.bfloat16))
    qr, sr = oracle.quant_e4m3(xb)
    assert_same(gq.view(torch.uint8), qr, "codes")
    assert_same(gs.view(torch.float32), sr, "scales")
    assert_same(go.view(torch.bfloat16), oracle.dequant_e4m3(qr, sr), "materialized")
    assert gq.bands_intact() and gs.bands_intact() and go.bands_intact()


def test_e4m3_input_aligned_to_16_but_not_32_bytes():
    # 32-byte-aligned BF16 input takes 256-bit loads, other 16-byte-aligned input two
    # 16-byte loads: the same codes and scales
    rng = np.random.default_rng(91)
    nblk = 45
    xb = adversarial_blocks(rng, nblk).reshape(-1)
    n = xb.size
    qr, sr = oracle.quant_e4m3(xb)
    for off in (0, 8):
        raw = torch.empty(n + 16, dtype=torch.bfloat16, device="cuda")
        x = raw[off:off + n]
        x.copy_(from_bits_bf16(xb))
        assert x.data_ptr() % 32 == 2 * off
        _, q, s = codec.empty_wire_e4m3(n)
        codec.quant_e4m3(x, q, s)
        assert_same(q, qr, f"codes, offset {off}")
        assert_same(s, sr, f"scales, offset {off}")


def test_e4m3_scales_across_the_exact_division_cutoff():
    # s = amax / 448 >= 2^-90 exactly when amax >= 448 * 2^-90 = 2^-81.19, BF16 bits
    # 0x16e0 and up: every BF16 amax from 0x1600 to 0x1700 straddles the cutoff between
    # per-element division and the reciprocal path; also the smallest amaxes (subnormal
    # scales, saturating quotients) and the largest. Other elements: random magnitudes
    # up to the amax with random signs.
    a_bits = np.concatenate([np.arange(0x0001, 0x0100), np.arange(0x1600, 0x1700), np.arange(0x7F00, 0x7F80)])
    rng = np.random.default_rng(1100)
    blocks = np.zeros((a_bits.size, 128), np.uint16)
    for i, a in enumerate(a_bits):
        signs = (rng.integers(0, 2, 128) << 15).astype(np.uint16)
        blocks[i] = rng.integers(0, int(a) + 1, 128).astype(np.uint16) | signs
        blocks[i, rng.integers(0, 128)] = a
    xb = blocks.reshape(-1)
    _, q, s = codec.empty_wire_e4m3(xb.size)
    codec.quant_e4m3(from_bits_bf16(xb), q, s)
    qr, sr = oracle.quant_e4m3(xb)
    assert_same(q, qr, "codes")
    assert_same(s, sr, "scales")


def test_e4m3_dequant_arbitrary_codes_and_scales():
    rng = np.random.default_rng(1200)
    nblk = 512
    codes = rng.integers(0, 256, nblk * 128).astype(np.uint8)
    codes[:256] = np.arange(256)
    codes[(codes & 0x7F) == 0x7F] = 0x7E  # NaN codes are not inputs
    sc = np.abs((rng.standard_normal(nblk) * 10.0 ** rng.uniform(-44, 35, nblk)).astype(np.float32))
    sc[:4] = [0.0, np.float32(2.0 ** -149), np.float32(1.5e-39), np.float32(3.0e35)]
    out = torch.empty(codes.size, dtype=torch.bfloat16, device="cuda")
    codec.dequant_e4m3(torch.from_numpy(codes).cuda(), torch.from_numpy(sc).cuda(), out)
    assert_same(out, oracle.dequant_e4m3(codes, sc), "materialized")


# ------------------------------------------------------------------ FP16 MX slices
def test_mx_f16_staged_slices_bitexact_and_equal_to_concatenated():
    slices = inputs.mx_slices_4096(rows=512, n_slices=3, dtype=torch.float16)
    rows, cols = slices[0].shape
    q_buf, s_buf = codec.empty_mx(rows, 3 * cols)
    for i, x in enumerate(slices):
        codec.quant_mx(x, q_buf[:, i * cols:(i + 1) * cols], s_buf[:, i * cols // 32:(i + 1) * cols // 32])
    cat = torch.cat(slices, dim=1)
    q_cat, s_cat = codec.empty_mx(rows, 3 * cols)
    codec.quant_mx(cat, q_cat, s_cat)
    assert torch.equal(q_buf, q_cat) and torch.equal(s_buf, s_cat)
    qr, sr = oracle.quant_mx(f16_bits(cat), fmt="f16")
    assert_same(q_buf, qr, "codes")
    assert_same(s_buf, sr, "scales")


def test_mx_f16_every_value_and_ragged_rows():
    # every finite FP16 pattern once, in groups with varied amax; then 4099 blocks
    bits_all = np.arange(0, 0x10000, dtype=np.uint32)
    bits_all = bits_all[((bits_all >> 10) & 0x1F) != 0x1F].astype(np.uint16)
    rng = np.random.default_rng(1300)
    rng.shuffle(bits_all)
    pad = (-bits_all.size) % 128
    xb = np.concatenate([bits_all, np.zeros(pad, np.uint16)]).reshape(-1, 128)
    x = torch.from_numpy(xb.view(np.int16)).cuda().view(torch.float16)
    q, s = codec.empty_mx(*xb.shape)
    codec.quant_mx(x, q, s)
    qr, sr = oracle.quant_mx(xb, fmt="f16")
    assert_same(q, qr, "codes")
    assert_same(s, sr, "scales")
    y = (rng.standard_normal((4099, 128)) * 10.0 ** rng.uniform(-7, 4, (4099, 1))).astype(np.float16)
    yt = torch.from_numpy(y).cuda()
    q2, s2 = codec.empty_mx(4099, 128)
    codec.quant_mx(yt, q2, s2)
    qr2, sr2 = oracle.quant_mx(y.view(np.uint16), fmt="f16")
    assert_same(q2, qr2, "codes")
    assert_same(s2, sr2, "scales")


# ------------------------------------------------------------------ tiled scale layout (pinned on the CPU to torch's to_blocked)
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_mx_tiled_scales_staged_slices(dtype):
    # six staged slices of 300 rows (a ragged last tile row) into one tiled scale buffer;
    # codes equal the row-major call's, scales equal the oracle's scales placed by the
    # oracle's tiled layout, and the padding rows of the last tile row stay untouched
    slices = inputs.mx_slices_4096(rows=300, n_slices=6, dtype=dtype)
    rows, cols = slices[0].shape
    C = 6 * cols
    g_total = C // 32
    q, s_rm = codec.empty_mx(rows, C)
    q_t = torch.empty_like(q)
    tiled = torch.full((codec.mx_tiled_scale_bytes(rows, g_total),), 0xA5, dtype=torch.uint8, device="cuda")
    for i, x in enumerate(slices):
        c0 = i * cols
        codec.quant_mx(x, q[:, c0:c0 + cols], s_rm[:, c0 // 32:(c0 + cols) // 32])
        codec.quant_mx_tiled(x, q_t[:, c0:c0 + cols], tiled, g_total, c0 // 32)
    assert torch.equal(q, q_t)
    fmt = "f16" if dtype == torch.float16 else "bf16"
    qr, sr = oracle.quant_mx((torch.cat(slices, dim=1).contiguous().view(torch.int16).cpu().numpy().view(np.uint16)),
                             fmt=fmt)
    assert_same(q, qr, "codes")
    want = oracle.mx_scales_to_tiled(sr, fill=0xA5)
    assert_same(tiled, want, "tiled scales")


def test_mx_tiled_scales_feed_a_block_scaled_gemm():
    # The layout's consumer: a block-scaled MXFP8 GEMM (PyTorch's _scaled_mm with E8M0
    # scales, cuBLASLt underneath) reads E4M3 codes and tiled scales that this library
    # wrote, A staged from two slices at scale-column offsets 0 and 8. Its result must
    # equal the float64 product of the two operands' materializations up to the GEMM's
    # FP32 accumulation and its BF16 output rounding; a misplaced scale would scale
    # whole 32-value groups by powers of two and miss by far more.
    if not hasattr(torch, "float8_e8m0fnu"):
        pytest.skip("this torch has no float8_e8m0fnu")
    M, N, K = 256, 256, 512
    g = torch.Generator(device="cuda")
    g.manual_seed(77)
    a = torch.randn((M, K), generator=g, device="cuda").to(torch.bfloat16)
    b = (torch.randn((N, K), generator=g, device="cuda") * 3).to(torch.bfloat16)
    qa = torch.empty((M, K), dtype=torch.uint8, device="cuda")
    qb = torch.empty((N, K), dtype=torch.uint8, device="cuda")
    sa = torch.zeros((codec.mx_tiled_scale_bytes(M, K // 32),), dtype=torch.uint8, device="cuda")
    sb = torch.zeros((codec.mx_tiled_scale_bytes(N, K // 32),), dtype=torch.uint8, device="cuda")
    for c0 in (0, K // 2):
        codec.quant_mx_tiled(a[:, c0:c0 + K // 2], qa[:, c0:c0 + K // 2], sa, K // 32, c0 // 32)
    codec.quant_mx_tiled(b, qb, sb, K // 32, 0)
    try:
        c = torch._scaled_mm(qa.view(torch.float8_e4m3fn), qb.view(torch.float8_e4m3fn).t(),
                             sa.view(torch.float8_e8m0fnu), sb.view(torch.float8_e8m0fnu), out_dtype=torch.bfloat16)
    except (RuntimeError, TypeError, ValueError, NotImplementedError) as e:
        pytest.skip(f"no MXFP8 block-scaled GEMM in this torch/cuBLAS on this GPU: {str(e).splitlines()[0][:160]}")
    torch.cuda.synchronize()
    # the operands' values: row-major scales from the same kernel body, materialized
    qr, sr = codec.empty_mx(M, K)
    qc, sc = codec.empty_mx(N, K)
    codec.quant_mx(a, qr, sr)
    codec.quant_mx(b, qc, sc)
    assert torch.equal(qr, qa) and torch.equal(qc, qb)
    da = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
    db = torch.empty((N, K), dtype=torch.bfloat16, device="cuda")
    codec.dequant_mx(qr, sr, da)
    codec.dequant_mx(qc, sc, db)
    ref = da.double() @ db.double().t()
    mag = da.double().abs() @ db.double().abs().t()
    err = (c.double() - ref).abs()
    bound = ref.abs() * 2.0 ** -8 + mag * K * 2.0 ** -23 + 1e-30
    assert bool((err <= bound).all()), f"max err {err.max().item()}, worst ratio {(err / bound).max().item()}"
    assert err.max().item() < 0.05 * ref.abs().max().item()
