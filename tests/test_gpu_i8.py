"""Block-INT8 kernels vs the CPU oracle, bit for bit, through the C ABI.

Expected values come only from the oracle run on the same input bits; the oracle
never sees a value the GPU produced (for chained steps it recomputes the chain).
"""
import numpy as np
import pytest
import torch

import oracle
from block_quantized_wire_gb300 import codec, inputs, topology
from block_quantized_wire_gb300._lib import BQError
from tests.helpers import Guarded, adversarial_blocks, bits, from_bits_bf16, near_half_blocks

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(bq_lib):
    return bq_lib


def gpu_quant(x: torch.Tensor):
    n = x.numel()
    _, q, s = codec.empty_wire_i8(n)
    codec.quant_i8(x.reshape(-1), q, s)
    return q, s


def gpu_dequant(q, s):
    out = torch.empty(q.numel(), dtype=torch.bfloat16, device="cuda")
    codec.dequant_i8(q, s, out)
    return out


def assert_same(got: torch.Tensor, want: np.ndarray, what: str):
    g = bits(got).reshape(-1)
    w = np.asarray(want).reshape(-1)
    assert g.dtype == w.dtype or g.view(np.uint8).size == w.view(np.uint8).size
    gv, wv = g.view(np.uint8), w.view(np.uint8)
    if not np.array_equal(gv, wv):
        bad = np.nonzero(g.view(w.dtype) != w)[0]
        raise AssertionError(f"{what}: {bad.size} mismatches, first at {bad[0]}: got {g.view(w.dtype)[bad[0]]} "
                             f"want {w[bad[0]]}")


# ------------------------------------------------------------------ workloads
def test_roundtrip_512_bitexact():
    x = inputs.roundtrip_512().cuda()
    q, s = gpu_quant(x)
    out = gpu_dequant(q, s)
    q_ref, s_ref = oracle.quant_i8(bits(x))
    assert_same(q, q_ref, "payload")
    assert_same(s, s_ref, "scales")
    assert_same(out, oracle.dequant_i8(q_ref, s_ref), "materialized")
    assert (s == 0).sum().item() == 573  # the 2% zero blocks


def test_mixed_3072_bitexact():
    x = inputs.mixed_3072().cuda()
    q, s = gpu_quant(x)
    out = gpu_dequant(q, s)
    q_ref, s_ref = oracle.quant_i8(bits(x))
    assert_same(q, q_ref, "payload")
    assert_same(s, s_ref, "scales")
    assert_same(out, oracle.dequant_i8(q_ref, s_ref), "materialized")


def test_a2a_3072_bitexact():
    xs = [x.cuda() for x in inputs.a2a_3072()]
    q_out, s_out, owner, srcs = topology.i8_a2a(xs)
    refs = [oracle.quant_i8(bits(x)) for x in xs]
    for (q, s), (qr, sr) in zip(srcs, refs):
        assert_same(q, qr, "source payload")
        assert_same(s, sr, "source scales")
    qa, sa, oa = oracle.dequant_accum_i8([r[0] for r in refs], [r[1] for r in refs], materialize=True)
    assert_same(q_out, qa, "accumulated payload")
    assert_same(s_out, sa, "accumulated scales")
    assert_same(owner, oa, "owner materialization")
    # the same call without the fused BF16 output gives the same payload
    _, q2, s2 = codec.empty_wire_i8(q_out.numel())
    codec.dequant_accum_i8([q for q, _ in srcs], [s for _, s in srcs], q2, s2, None)
    assert torch.equal(q2, q_out) and torch.equal(s2, s_out)


def test_ring_16384_chain_bitexact():
    xs = [x.cuda() for x in inputs.ring_16384()]
    W = len(xs)
    outs, finals, owners = topology.i8_ring(xs)
    xb = [bits(x).reshape(W, -1) for x in xs]  # [shard, n]
    rng = np.random.default_rng(0)
    shard_rows = xs[0].shape[0] // W
    for c in range(W):
        chain = topology.ring_order(c, W)
        q, s = oracle.quant_i8(xb[chain[0]][c])
        for rank in chain[1:]:
            q, s, _ = oracle.ring_hop_i8(q, s, xb[rank][c])
        assert_same(finals[c][0], q, f"shard {c} final payload")
        assert_same(finals[c][1], s, f"shard {c} final scales")
        # owner materialization and all-gather, on sampled rows of the shard
        rows = rng.choice(shard_rows, 64, replace=False)
        cols = xs[0].shape[1]
        for r in rows:
            lo, hi = r * cols, (r + 1) * cols
            want = oracle.dequant_i8(q[lo:hi], s[lo // 128:hi // 128])
            assert_same(owners[c].reshape(-1)[lo:hi], want, f"shard {c} owner row {r}")
    for o in outs[1:]:
        assert torch.equal(o, outs[0])  # every rank materializes identical BF16
    for c in range(W):
        assert torch.equal(owners[c], outs[0][c * shard_rows:(c + 1) * shard_rows])


def test_prefill_65536_sampled_bitexact():
    # Largest workload: the whole pipeline runs at full size on the GPU; the oracle
    # recomputes 4096 sampled blocks from the same BF16 bits.
    torch.cuda.empty_cache()
    xs = inputs.prefill_65536()
    n = xs[0].numel()
    nblk = n // 128
    qs = [gpu_quant(x) for x in xs]
    _, qa, sa = codec.empty_wire_i8(n)
    codec.dequant_accum_i8([q for q, _ in qs], [s for _, s in qs], qa, sa, None)
    out = gpu_dequant(qa, sa)
    _, qh, sh = codec.empty_wire_i8(n)
    codec.ring_hop_i8(qs[0][0], qs[0][1], xs[1].reshape(-1), qh, sh, None)
    torch.cuda.synchronize()
    rng = np.random.default_rng(5)
    blk = np.sort(rng.choice(nblk, 4096, replace=False))
    blk[-1] = nblk - 1  # the last block of the tensor
    idx = torch.from_numpy(blk).cuda()

    def gather_blocks(t, width=128):
        return t.reshape(-1, width)[idx]

    xb = [bits(gather_blocks(x.reshape(-1))) for x in xs]
    ref = [oracle.quant_i8(b) for b in xb]
    for w in range(4):
        assert_same(gather_blocks(qs[w][0]), ref[w][0], f"source {w} payload")
        assert_same(qs[w][1][idx], ref[w][1], f"source {w} scales")
    qa_r, sa_r, _ = oracle.dequant_accum_i8([r[0] for r in ref], [r[1] for r in ref], materialize=False)
    assert_same(gather_blocks(qa), qa_r, "accumulated payload")
    assert_same(sa[idx], sa_r, "accumulated scales")
    assert_same(gather_blocks(out), oracle.dequant_i8(qa_r, sa_r), "materialized")
    qh_r, sh_r, _ = oracle.ring_hop_i8(ref[0][0], ref[0][1], xb[1])
    assert_same(gather_blocks(qh), qh_r, "hop payload")
    assert_same(sh[idx], sh_r, "hop scales")


# ------------------------------------------------------------------ edge cases
@pytest.mark.parametrize("nblk", [1, 2, 3, 5, 7, 8, 9, 15, 16, 17, 63, 64, 65, 1001, 4099])
def test_ragged_sizes_quant_dequant(nblk):
    rng = np.random.default_rng(nblk)
    xb = adversarial_blocks(rng, nblk).reshape(-1)
    n = xb.size
    x = from_bits_bf16(xb)
    gq, gs, go = Guarded(n), Guarded(4 * (n // 128)), Guarded(2 * n)
    q, s, out = gq.view(torch.int8), gs.view(torch.float32), go.view(torch.bfloat16)
    codec.quant_i8(x, q, s)
    codec.dequant_i8(q, s, out)
    q_ref, s_ref = oracle.quant_i8(xb)
    assert_same(q, q_ref, "payload")
    assert_same(s, s_ref, "scales")
    assert_same(out, oracle.dequant_i8(q_ref, s_ref), "materialized")
    assert gq.bands_intact() and gs.bands_intact() and go.bands_intact()


def test_near_half_quotients_take_exact_path():
    rng = np.random.default_rng(77)
    xb = near_half_blocks(rng, 64).reshape(-1)
    q, s = gpu_quant(from_bits_bf16(xb))
    q_ref, s_ref = oracle.quant_i8(xb)
    assert_same(q, q_ref, "payload")
    assert_same(s, s_ref, "scales")


def test_dequant_arbitrary_payloads():
    # every byte value (including -128, which quantization never writes) with scales
    # spanning zero, subnormal, normal and large binary32
    rng = np.random.default_rng(8)
    nblk = 512
    q = rng.integers(-128, 128, nblk * 128).astype(np.int8)
    q[:256] = np.arange(-128, 128)
    s = (rng.standard_normal(nblk) * 10.0 ** rng.uniform(-44, 36, nblk)).astype(np.float32)
    s[:4] = [0.0, np.float32(2.0 ** -149), np.float32(1.5e-39), np.float32(2.0e36)]
    s = np.abs(s)
    out = torch.empty(q.size, dtype=torch.bfloat16, device="cuda")
    codec.dequant_i8(torch.from_numpy(q).cuda(), torch.from_numpy(s).cuda(), out)
    assert_same(out, oracle.dequant_i8(q, s), "materialized")


@pytest.mark.parametrize("owner", [True, False])
@pytest.mark.parametrize("W", [1, 2, 3, 4, 5, 7, 8, 9, 16])
@pytest.mark.parametrize("nblk", [37, 8, 1])
def test_accumulate_any_width(W, owner, nblk):
    # with and without the owner output (separate kernels), whole and partial chunks
    rng = np.random.default_rng(100 + W + nblk)
    xs = [adversarial_blocks(rng, nblk, max_abs=1.0e37).reshape(-1) for _ in range(W)]  # sums stay finite
    ref = [oracle.quant_i8(x) for x in xs]
    qd = [torch.from_numpy(r[0]).cuda() for r in ref]
    sd = [torch.from_numpy(r[1]).cuda() for r in ref]
    n = nblk * 128
    gq, gs, go = Guarded(n), Guarded(4 * nblk), Guarded(2 * n)
    codec.dequant_accum_i8(qd, sd, gq.view(torch.int8), gs.view(torch.float32),
                           go.view(torch.bfloat16) if owner else None)
    qa, sa, oa = oracle.dequant_accum_i8([r[0] for r in ref], [r[1] for r in ref], materialize=True)
    assert np.all(np.isfinite(sa))
    assert_same(gq.view(torch.int8), qa, "payload")
    assert_same(gs.view(torch.float32), sa, "scales")
    if owner:
        assert_same(go.view(torch.bfloat16), oa, "materialized")
    else:
        assert (go.raw == Guarded.SENTINEL).all().item()  # no owner output: nothing written
    assert gq.bands_intact() and gs.bands_intact() and go.bands_intact()


def test_accumulate_repeated_source_and_tiny_sums():
    # the same payload passed twice (inputs may repeat), and FP32 sums in the binary32
    # subnormal range whose amax/127 is subnormal or underflows to zero
    nblk = 6
    q = np.zeros((nblk, 128), np.int8)
    s = np.zeros(nblk, np.float32)
    q[0, :3] = [1, -1, 0]
    s[0] = np.float32(2.0 ** -149)
    q[1, :3] = [95, -3, 7]
    s[1] = np.float32(2.0 ** -148)
    q[2, :3] = [-95, 3, 127]
    s[2] = np.float32(2.0 ** -140)
    q[3] = np.arange(-64, 64)
    s[3] = np.float32(1.0e-38)
    q[4] = 127
    s[4] = np.float32(3.0e30)
    q[5, 0] = -127
    s[5] = np.float32(1.0)
    q = q.reshape(-1)
    qd, sd = torch.from_numpy(q).cuda(), torch.from_numpy(s).cuda()
    for W in (3, 4):  # three sources, and four (the kernel without the owner output too)
        _, qo, so = codec.empty_wire_i8(q.size)
        out = torch.empty(q.size, dtype=torch.bfloat16, device="cuda")
        codec.dequant_accum_i8([qd] * W, [sd] * W, qo, so, out)
        qa, sa, oa = oracle.dequant_accum_i8([q] * W, [s] * W, materialize=True)
        assert_same(qo, qa, "payload")
        assert_same(so, sa, "scales")
        assert_same(out, oa, "materialized")
        _, qn, sn = codec.empty_wire_i8(q.size)
        codec.dequant_accum_i8([qd] * W, [sd] * W, qn, sn, None)
        assert_same(qn, qa, "payload without owner output")
        assert_same(sn, sa, "scales without owner output")


def test_bf16_pointers_aligned_to_16_but_not_32_bytes():
    # BF16 buffers need only 16-byte alignment; 32-byte-aligned ones take 256-bit
    # accesses, the others 16-byte ones: both must give the same bytes
    rng = np.random.default_rng(77)
    nblk = 45
    n = nblk * 128
    xs = [adversarial_blocks(rng, nblk, max_abs=1.0e37).reshape(-1) for _ in range(4)]
    for off in (0, 8):  # BF16 elements: 0 and 16 bytes past a 32-byte boundary
        def bf16_at(bits_):
            raw = torch.empty(n + 16, dtype=torch.bfloat16, device="cuda")
            t = raw[off:off + n]
            if bits_ is not None:
                t.copy_(from_bits_bf16(bits_))
            assert t.data_ptr() % 32 == 2 * off
            return t
        x = [bf16_at(b) for b in xs]
        qs, ss = [], []
        for w in range(4):
            _, q, s_ = codec.empty_wire_i8(n)
            codec.quant_i8(x[w], q, s_)
            qr, sr = oracle.quant_i8(xs[w])
            assert_same(q, qr, f"quant payload, offset {off}")
            assert_same(s_, sr, f"quant scales, offset {off}")
            qs.append(q)
            ss.append(s_)
        out = bf16_at(None)
        codec.dequant_i8(qs[0], ss[0], out)
        assert_same(out, oracle.dequant_i8(*oracle.quant_i8(xs[0])), f"materialize, offset {off}")
        ref = [oracle.quant_i8(b) for b in xs]
        _, qa, sa = codec.empty_wire_i8(n)
        codec.dequant_accum_i8(qs, ss, qa, sa, out)
        aq, as_, ao = oracle.dequant_accum_i8([r[0] for r in ref], [r[1] for r in ref], materialize=True)
        assert_same(qa, aq, f"accumulate payload, offset {off}")
        assert_same(out, ao, f"accumulate owner output, offset {off}")
        _, qh, sh = codec.empty_wire_i8(n)
        codec.ring_hop_i8(qs[0], ss[0], x[1], qh, sh, out)
        hq, hs, ho = oracle.ring_hop_i8(ref[0][0], ref[0][1], xs[1], materialize=True)
        assert_same(qh, hq, f"hop payload, offset {off}")
        assert_same(sh, hs, f"hop scales, offset {off}")
        assert_same(out, ho, f"hop owner output, offset {off}")


@pytest.mark.parametrize("owner", [True, False])
@pytest.mark.parametrize("nblk", [200, 45])
def test_ring_hop_edge_cases(nblk, owner):
    # whole and partial last chunks, with and without the owner output
    rng = np.random.default_rng(31)
    x_in = adversarial_blocks(rng, nblk, max_abs=1.0e38).reshape(-1)
    x_loc = adversarial_blocks(rng, nblk, max_abs=1.0e38).reshape(-1)
    x_loc[:128 * 9] = x_in[:128 * 9] ^ 0x8000  # blocks where the hop cancels to tiny sums
    q_in, s_in = oracle.quant_i8(x_in)
    n = x_in.size
    gq, gs, go = Guarded(n), Guarded(4 * nblk), Guarded(2 * n)
    codec.ring_hop_i8(torch.from_numpy(q_in).cuda(), torch.from_numpy(s_in).cuda(), from_bits_bf16(x_loc),
                      gq.view(torch.int8), gs.view(torch.float32), go.view(torch.bfloat16) if owner else None)
    qh, sh, oh = oracle.ring_hop_i8(q_in, s_in, x_loc, materialize=True)
    assert np.all(np.isfinite(sh))
    assert_same(gq.view(torch.int8), qh, "payload")
    assert_same(gs.view(torch.float32), sh, "scales")
    if owner:
        assert_same(go.view(torch.bfloat16), oh, "materialized")
    else:
        assert (go.raw == Guarded.SENTINEL).all().item()  # no owner output: nothing written
    assert gq.bands_intact() and gs.bands_intact() and go.bands_intact()


def test_empty_inputs_are_noops():
    e8 = torch.empty(0, dtype=torch.int8, device="cuda")
    ef = torch.empty(0, dtype=torch.float32, device="cuda")
    eb = torch.empty(0, dtype=torch.bfloat16, device="cuda")
    codec.quant_i8(eb, e8, ef)
    codec.dequant_i8(e8, ef, eb)
    codec.dequant_accum_i8([e8, e8], [ef, ef], e8, ef, eb)
    codec.ring_hop_i8(e8, ef, eb, e8, ef, eb)
    torch.cuda.synchronize()


def test_errors_surface_before_launch_on_gpu():
    x = torch.zeros(256, dtype=torch.bfloat16, device="cuda")
    _, q, s = codec.empty_wire_i8(256)
    with pytest.raises(BQError) as e:
        codec.quant_i8(x[1:129], q[:128], s[:1])  # x misaligned by 2 bytes
    assert e.value.status == 3
    with pytest.raises(BQError) as e:
        codec.quant_i8(x, x.view(torch.int8)[:256], s)  # payload inside x
    assert e.value.status == 4


def test_tiny_scale_blocks_across_the_exact_division_cutoff():
    # Blocks whose amax spans BF16 values from 2^-126 to 2^-90 (scales around 2^-100,
    # where a kernel's quotient remainders can reach the subnormal range), each with
    # random values below its amax, including the worst cases found by an exhaustive
    # sweep of the remainder-based quotient.
    rng = np.random.default_rng(2024)
    amax_codes = np.arange(0x0080, 0x12C0, 3, dtype=np.uint16)
    nblk = amax_codes.size
    x = np.zeros((nblk, 128), np.uint16)
    x[:, 0] = amax_codes
    for b, a in enumerate(amax_codes):
        x[b, 1:] = rng.integers(0, int(a) + 1, 127).astype(np.uint16) | (rng.integers(0, 2, 127) << 15).astype(np.uint16)
    x[0, :3] = [0x0438, 0x00EE, 0x00FA]
    x[1, :3] = [0x0437, 0x00C1, 0x00C5]
    xb = x.reshape(-1)
    q, s = gpu_quant(from_bits_bf16(xb))
    q_ref, s_ref = oracle.quant_i8(xb)
    assert_same(q, q_ref, "payload")
    assert_same(s, s_ref, "scales")
    # the same values as FP32 sums (one source, scale 1 pass-through of tiny values)
    _, qh, sh = codec.empty_wire_i8(xb.size)
    zero_q = torch.zeros(xb.size, dtype=torch.int8, device="cuda")
    zero_s = torch.zeros(xb.size // 128, dtype=torch.float32, device="cuda")
    codec.ring_hop_i8(zero_q, zero_s, from_bits_bf16(xb), qh, sh, None)
    qz, sz = oracle.quant_i8(np.zeros_like(xb))
    qh_r, sh_r, _ = oracle.ring_hop_i8(qz, sz, xb)
    assert_same(qh, qh_r, "hop payload")
    assert_same(sh, sh_r, "hop scales")


def _scales_at_4_mod_16(s: np.ndarray) -> torch.Tensor:
    buf = torch.zeros(s.size + 4, dtype=torch.float32, device="cuda")
    view = buf[1:1 + s.size]  # 4 bytes past a 16-byte boundary
    view.copy_(torch.from_numpy(s))
    assert view.data_ptr() % 16 == 4
    return view


def test_accumulate_with_scales_not_16_byte_aligned():
    # scale pointers only 4-byte aligned (allowed by the ABI) take the path that loads
    # from global memory directly; payloads still 16-byte aligned
    rng = np.random.default_rng(404)
    nblk, W = 1027, 4
    xs = [adversarial_blocks(rng, nblk, max_abs=1.0e37).reshape(-1) for _ in range(W)]
    ref = [oracle.quant_i8(x) for x in xs]
    qd, sd = [], []
    for q, s in ref:
        qd.append(torch.from_numpy(q).cuda())
        sd.append(_scales_at_4_mod_16(s))
    n = nblk * 128
    _, qo, so = codec.empty_wire_i8(n)
    out = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    codec.dequant_accum_i8(qd, sd, qo, so, out)
    qa, sa, oa = oracle.dequant_accum_i8([r[0] for r in ref], [r[1] for r in ref], materialize=True)
    assert_same(qo, qa, "payload")
    assert_same(so, sa, "scales")
    assert_same(out, oa, "materialized")


def test_ring_hop_with_scales_not_16_byte_aligned():
    # the hop stages its inputs through shared memory only when the incoming scales
    # are 16-byte aligned; 4-byte aligned scales take the direct-load path
    rng = np.random.default_rng(405)
    nblk = 1029
    x_in = adversarial_blocks(rng, nblk, max_abs=1.0e37).reshape(-1)
    x_loc = adversarial_blocks(rng, nblk, max_abs=1.0e37).reshape(-1)
    q_in, s_in = oracle.quant_i8(x_in)
    n = nblk * 128
    _, qo, so = codec.empty_wire_i8(n)
    out = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    codec.ring_hop_i8(torch.from_numpy(q_in).cuda(), _scales_at_4_mod_16(s_in), from_bits_bf16(x_loc), qo, so, out)
    qh, sh, oh = oracle.ring_hop_i8(q_in, s_in, x_loc, materialize=True)
    assert_same(qo, qh, "payload")
    assert_same(so, sh, "scales")
    assert_same(out, oh, "materialized")
