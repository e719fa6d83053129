"""MXFP8 kernels vs the CPU oracle, bit for bit, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
from block_quantized_wire_gb300 import codec, inputs
from tests.helpers import Guarded, adversarial_blocks, bits, from_bits_bf16
from tests.test_gpu_i8 import assert_same

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(bq_lib):
    return bq_lib


def gpu_quant_mx(x: torch.Tensor):
    rows, cols = x.shape
    q, s = codec.empty_mx(rows, cols)
    codec.quant_mx(x, q, s)
    return q, s


def gpu_dequant_mx(q, s):
    out = torch.empty(q.shape, dtype=torch.bfloat16, device="cuda")
    codec.dequant_mx(q, s, out)
    return out


def test_mixed_3072_mx_bitexact():
    x = inputs.mixed_3072().cuda()
    q, s = gpu_quant_mx(x)
    out = gpu_dequant_mx(q, s)
    q_ref, s_ref = oracle.quant_mx(bits(x))
    assert_same(q, q_ref, "E4M3 codes")
    assert_same(s, s_ref, "E8M0 scales")
    assert_same(out, oracle.dequant_mx(q_ref, s_ref), "materialized")


def test_every_bf16_amax_scale_byte():
    # one group per positive finite BF16 amax (with its negation beside it)
    a = np.arange(1, 0x7F80, dtype=np.uint16)
    ng = ((a.size + 3) // 4) * 4
    g = np.zeros((ng, 32), np.uint16)
    g[: a.size, 0] = a
    g[: a.size, 17] = a | 0x8000
    g[: a.size, 3] = a >> 2
    x = g.reshape(-1, 128)
    q, s = gpu_quant_mx(from_bits_bf16(x))
    q_ref, s_ref = oracle.quant_mx(x)
    assert_same(s, s_ref, "E8M0 scales")
    assert_same(q, q_ref, "E4M3 codes")
    out = gpu_dequant_mx(q, s)
    assert_same(out, oracle.dequant_mx(q_ref, s_ref), "materialized")


@pytest.mark.parametrize("shift", [-127, -20, -9, 0, 7, 100, 119])
def test_every_bf16_value_as_e4m3_input(shift):
    # all BF16 magnitudes below 448 * 2^shift, each in a group whose amax is 448 * 2^shift
    # (so the E8M0 scale is 2^shift exactly and y = x * 2^-shift spans [0, 448])
    top = np.float32(448.0 * 2.0 ** shift)
    top_bits = np.array([top], np.float32).view(np.uint32)[0] >> 16
    vals = np.arange(0, top_bits + 1, dtype=np.uint16)
    vals = np.concatenate([vals, vals | 0x8000])
    per = 31
    ng = (vals.size + per - 1) // per
    ng = ((ng + 3) // 4) * 4
    g = np.zeros((ng, 32), np.uint16)
    flat = np.zeros(ng * per, np.uint16)
    flat[: vals.size] = vals
    g[:, 1:] = flat.reshape(ng, per)
    g[:, 0] = top_bits
    x = g.reshape(-1, 128)
    q, s = gpu_quant_mx(from_bits_bf16(x))
    q_ref, s_ref = oracle.quant_mx(x)
    assert np.all(s_ref == 127 + shift)
    assert_same(s, s_ref, "E8M0 scales")
    assert_same(q, q_ref, "E4M3 codes")


def test_dequant_every_code_and_scale():
    codes = np.tile(np.arange(256, dtype=np.uint8), 2)  # 512 columns = 16 groups
    rows = 32
    q = np.tile(codes, (rows, 1))
    e = np.array([0, 1, 2, 100, 119, 126, 127, 128, 140, 200, 240, 247, 250, 253, 254, 127], np.uint8)
    s = np.tile(e, (rows, 1))
    s[1:] = np.roll(e, 5)[None, :]
    q[:, 0x7F] = 0  # NaN codes: their BF16 bit pattern is not specified
    q[:, 0xFF] = 0
    q[:, 0x17F] = 0
    q[:, 0x1FF] = 0
    out = gpu_dequant_mx(torch.from_numpy(q).cuda(), torch.from_numpy(s).cuda())
    want = oracle.dequant_mx(q, s)
    assert_same(out, want, "materialized")


def test_staged_slices_4096_bitexact_and_equal_to_concatenated():
    # six 4096 x 7168 BF16 slices quantized into one 4096 x 43008 MXFP8 buffer at
    # columns 7168 * i; bitwise equal to quantizing the concatenation in one call
    # ("[II] Support staged MXFP8 linear inputs", Validation)
    slices = inputs.mx_slices_4096()
    rows, w = slices[0].shape
    C = w * len(slices)
    gq, gs = Guarded(rows * C), Guarded(rows * C // 32)
    qb, sb = gq.view(torch.uint8, (rows, C)), gs.view(torch.uint8, (rows, C // 32))
    for i, x in enumerate(slices):
        c0 = i * w
        codec.quant_mx(x, qb[:, c0:c0 + w], sb[:, c0 // 32:(c0 + w) // 32])
    assert gq.bands_intact() and gs.bands_intact()
    cat = torch.cat(slices, dim=1)
    q_cat, s_cat = gpu_quant_mx(cat)
    assert torch.equal(qb, q_cat) and torch.equal(sb, s_cat)
    # oracle on sampled rows of every slice
    rng = np.random.default_rng(3)
    pick = np.sort(rng.choice(rows, 96, replace=False))
    pick[-1] = rows - 1
    idx = torch.from_numpy(pick).cuda()
    for i, x in enumerate(slices):
        q_ref, s_ref = oracle.quant_mx(bits(x[idx]))
        c0 = i * w
        assert_same(qb[idx, c0:c0 + w], q_ref, f"slice {i} codes")
        assert_same(sb[idx, c0 // 32:(c0 + w) // 32], s_ref, f"slice {i} scales")
    out = gpu_dequant_mx(qb, sb)
    refs = [oracle.quant_mx(bits(x[idx])) for x in slices]  # the oracle's own codes
    q_all = np.concatenate([r[0] for r in refs], axis=1)
    s_all = np.concatenate([r[1] for r in refs], axis=1)
    assert_same(out[idx], oracle.dequant_mx(q_all, s_all), "materialized")


@pytest.mark.parametrize("rows,cols,pad_x,pad_q,pad_s", [
    (1, 128, 0, 0, 0), (3, 256, 8, 16, 4), (17, 384, 24, 48, 12), (5, 1152, 0, 128, 0), (64, 128, 128, 0, 60),
])
def test_strided_shapes(rows, cols, pad_x, pad_q, pad_s):
    rng = np.random.default_rng(rows * 1000 + cols)
    nblk = rows * cols // 128
    xb = adversarial_blocks(rng, nblk).reshape(rows, cols)
    ld_x, ld_q, ld_s = cols + pad_x, cols + pad_q, cols // 32 + pad_s
    xfull = torch.zeros((rows, ld_x), dtype=torch.bfloat16, device="cuda")
    xfull[:, :cols] = from_bits_bf16(xb)
    gq, gs = Guarded(rows * ld_q), Guarded(rows * ld_s)
    qv = gq.view(torch.uint8, (rows, ld_q))[:, :cols]
    sv = gs.view(torch.uint8, (rows, ld_s))[:, : cols // 32]
    codec.quant_mx(xfull[:, :cols], qv, sv)
    q_ref, s_ref = oracle.quant_mx(xb)
    assert_same(qv, q_ref, "codes")
    assert_same(sv, s_ref, "scales")
    # untouched padding columns keep their sentinel
    if pad_q:
        assert bool((gq.view(torch.uint8, (rows, ld_q))[:, cols:] == Guarded.SENTINEL).all())
    if pad_s:
        assert bool((gs.view(torch.uint8, (rows, ld_s))[:, cols // 32:] == Guarded.SENTINEL).all())
    assert gq.bands_intact() and gs.bands_intact()
    go = Guarded(rows * (cols + pad_x) * 2)
    ov = go.view(torch.bfloat16, (rows, cols + pad_x))[:, :cols]
    codec.dequant_mx(qv, sv, ov)
    assert_same(ov, oracle.dequant_mx(q_ref, s_ref), "materialized")
    assert go.bands_intact()


def test_mx_empty_is_noop():
    x = torch.empty((0, 128), dtype=torch.bfloat16, device="cuda")
    q, s = codec.empty_mx(0, 128)
    codec.quant_mx(x, q, s)
    codec.dequant_mx(q, s, torch.empty((0, 128), dtype=torch.bfloat16, device="cuda"))
    torch.cuda.synchronize()


# ------------------------------------------------------------------ several slices in one call
def _slices_vs_oracle(widths, rows, dtype, seed, ld_pad=0, col_off=0):
    """Slices of the given widths (views into wider tensors when ld_pad > 0) quantized by
    one bq_quant_mx_slices call into a destination that starts at column col_off of a
    guarded wider buffer; compared with the oracle on the concatenation and with one
    bq_quant_mx call per slice."""
    rng = np.random.default_rng(seed)
    xs = []
    for w in widths:
        xf = (rng.standard_normal((rows, w + ld_pad)) * 0.02).astype(np.float32)
        xf[rng.random(xf.shape) < 0.002] *= 100
        full = torch.from_numpy(xf).to(dtype).cuda()
        xs.append(full[:, :w])
    total = sum(widths)
    C = col_off + total + 128
    gq = Guarded(rows * C)
    gs = Guarded(rows * (C // 32))
    q_all = gq.view(torch.uint8, (rows, C))
    s_all = gs.view(torch.uint8, (rows, C // 32))
    q = q_all[:, col_off:col_off + total]
    s = s_all[:, col_off // 32:(col_off + total) // 32]
    codec.quant_mx_slices(xs, q, s)
    torch.cuda.synchronize()
    assert gq.bands_intact() and gs.bands_intact()
    untouched_q = torch.cat([q_all[:, :col_off], q_all[:, col_off + total:]], dim=1)
    assert bool((untouched_q == Guarded.SENTINEL).all())
    fmt = "f16" if dtype == torch.float16 else "bf16"
    cat = torch.cat([x.contiguous() for x in xs if x.shape[1]], dim=1)
    q_ref, s_ref = oracle.quant_mx(cat.view(torch.int16).cpu().numpy().view(np.uint16), fmt=fmt)
    assert_same(q.contiguous(), q_ref, "E4M3 codes")
    assert_same(s.contiguous(), s_ref, "E8M0 scales")
    # the same bytes as one quant_mx call per slice
    q1, s1 = codec.empty_mx(rows, total)
    c = 0
    for x in xs:
        w = x.shape[1]
        if w:
            codec.quant_mx(x, q1[:, c:c + w], s1[:, c // 32:(c + w) // 32])
        c += w
    assert torch.equal(q1, q) and torch.equal(s1, s)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_slices_in_one_call_ragged_widths(dtype):
    # unequal widths, strided views, a destination offset, rows that end mid-chunk
    _slices_vs_oracle([128, 384, 256, 1024, 128, 640], rows=300, dtype=dtype, seed=41, ld_pad=64, col_off=256)


def test_slices_in_one_call_sixteen_narrow_slices_and_an_empty_one():
    _slices_vs_oracle([128] * 7 + [0] + [128] * 8, rows=37, dtype=torch.bfloat16, seed=42)


def test_slices_in_one_call_single_slice_and_single_row():
    _slices_vs_oracle([7168], rows=1, dtype=torch.bfloat16, seed=43)
    _slices_vs_oracle([256, 128], rows=5, dtype=torch.float16, seed=44, ld_pad=8)


def test_slices_in_one_call_staged_workload():
    # the staged workload at full size: six 4096 x 7168 slices into 4096 x 43008 in one
    # call equal six bq_quant_mx calls byte for byte; sampled rows against the oracle
    slices = inputs.mx_slices_4096()
    rows, cols = slices[0].shape
    C = len(slices) * cols
    q, s = codec.empty_mx(rows, C)
    codec.quant_mx_slices(slices, q, s)
    q1, s1 = codec.empty_mx(rows, C)
    for i, x in enumerate(slices):
        codec.quant_mx(x, q1[:, i * cols:(i + 1) * cols], s1[:, i * cols // 32:(i + 1) * cols // 32])
    assert torch.equal(q, q1) and torch.equal(s, s1)
    pick = torch.tensor([0, 1, 2047, 4094, 4095], device="cuda")
    cat = torch.cat([x[pick] for x in slices], dim=1)
    q_ref, s_ref = oracle.quant_mx(bits(cat))
    assert_same(q[pick], q_ref, "E4M3 codes")
    assert_same(s[pick], s_ref, "E8M0 scales")


def test_slices_in_one_call_graph_replay_is_bit_identical():
    # stream-ordered and allocation-free: the call captures into a CUDA graph, and a
    # replay writes the bytes of the eager call
    slices = inputs.mx_slices_4096(rows=256, n_slices=3)
    rows, cols = slices[0].shape
    q, s = codec.empty_mx(rows, 3 * cols)
    codec.quant_mx_slices(slices, q, s)
    torch.cuda.synchronize()
    q_eager, s_eager = q.clone(), s.clone()
    q.fill_(0)
    s.fill_(0)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        codec.quant_mx_slices(slices, q, s)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(q, q_eager) and torch.equal(s, s_eager)
