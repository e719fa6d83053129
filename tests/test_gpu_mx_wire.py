"""MXFP8 wire reductions (mx_a2a accumulate, mx_ring hop) vs the CPU oracle, bit for bit,
through the C ABI ("feat(pcie_dma): add INT8 and MXFP8 wire modes", Summary).

Expected values come only from the oracle run on the same input bits.
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
    gv, wv = g.view(np.uint8), w.view(np.uint8)
    if not np.array_equal(gv, wv):
        g2 = g.view(w.dtype)
        bad = np.nonzero(g2 != w)[0]
        raise AssertionError(f"{what}: {bad.size} mismatches, first at {bad[0]}: got {g2[bad[0]]} want {w[bad[0]]}")


def dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def random_wires(rng, W, nblk, e_lo=0, e_hi=240):
    """Flat MX wires with arbitrary finite codes and scale bytes in [e_lo, e_hi], plus
    groups that are all zero, all negative zero, and large-amax groups whose small
    elements scale into the binary32 subnormal range when requantized."""
    n = nblk * 128
    finite = np.array([c for c in range(256) if c & 0x7F != 0x7F], np.uint8)
    qs, ss = [], []
    for _ in range(W):
        q = rng.choice(finite, n).astype(np.uint8)
        s = rng.integers(e_lo, e_hi + 1, n // 32).astype(np.uint8)
        ng = n // 32
        q.reshape(-1, 32)[rng.integers(0, ng, max(1, ng // 16))] = 0x00
        q.reshape(-1, 32)[rng.integers(0, ng, max(1, ng // 16))] = 0x80
        big = rng.integers(0, ng, max(1, ng // 16))
        q.reshape(-1, 32)[big, 0] = 0x7E
        q.reshape(-1, 32)[big, 1:] = rng.choice(np.array([0x01, 0x81, 0x02, 0x00, 0x80], np.uint8), (big.size, 31))
        qs.append(q)
        ss.append(s)
    return qs, ss


# ------------------------------------------------------------------ workloads
def test_mx_a2a_bitexact():
    xs = [x.cuda() for x in inputs.a2a_3072(rows=1024)]
    q_out, s_out, owner, srcs = topology.mx_a2a(xs)
    refs = [oracle.quant_mx_flat(bits(x)) for x in xs]
    for (q, s), (qr, sr) in zip(srcs, refs):
        assert_same(q, qr, "source codes")
        assert_same(s, sr, "source scales")
    qa, sa, oa = oracle.dequant_accum_mx([r[0] for r in refs], [r[1] for r in refs], materialize=True)
    assert_same(q_out, qa, "accumulated codes")
    assert_same(s_out, sa, "accumulated scales")
    assert_same(owner, oa, "owner materialization")
    # without the fused BF16 output the wire is the same; the owner output equals a
    # separate materialization of that wire
    _, q2, s2 = codec.empty_wire_mx(q_out.numel())
    codec.dequant_accum_mx([q for q, _ in srcs], [s for _, s in srcs], q2, s2, None)
    assert torch.equal(q2, q_out) and torch.equal(s2, s_out)
    sep = torch.empty_like(owner)
    codec.dequant_mx_flat(q_out, s_out, sep)
    assert torch.equal(sep, owner)


def test_mx_ring_chain_bitexact():
    xs = [x.cuda() for x in inputs.ring_16384(rows=2048)]
    W = len(xs)
    outs, finals, owners = topology.mx_ring(xs)
    xb = [bits(x).reshape(W, -1) for x in xs]
    shard_rows = xs[0].shape[0] // W
    for c in range(W):
        chain = topology.ring_order(c, W)
        q, s = oracle.quant_mx_flat(xb[chain[0]][c])
        for rank in chain[1:-1]:
            q, s, _ = oracle.ring_hop_mx(q, s, xb[rank][c])
        q, s, o = oracle.ring_hop_mx(q, s, xb[chain[-1]][c], materialize=True)
        assert_same(finals[c][0], q, f"shard {c} final codes")
        assert_same(finals[c][1], s, f"shard {c} final scales")
        assert_same(owners[c], o, f"shard {c} owner")
    for o in outs[1:]:
        assert torch.equal(o, outs[0])
    for c in range(W):
        assert torch.equal(owners[c], outs[0][c * shard_rows:(c + 1) * shard_rows])


def test_mx_prefill_sampled_bitexact():
    # Full-size launch (4 x 65536 x 7168, the size the benchmark times); the oracle
    # recomputes 4096 sampled 128-value blocks from the same bits.
    torch.cuda.empty_cache()
    xs = inputs.prefill_65536()
    n = xs[0].numel()
    nblk = n // 128
    wires = []
    for x in xs:
        _, q, s = codec.empty_wire_mx(n)
        codec.quant_mx_flat(x.reshape(-1), q, s)
        wires.append((q, s))
    _, qa, sa = codec.empty_wire_mx(n)
    out = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    codec.dequant_accum_mx([q for q, _ in wires], [s for _, s in wires], qa, sa, out)
    _, qh, sh = codec.empty_wire_mx(n)
    codec.ring_hop_mx(wires[0][0], wires[0][1], xs[1].reshape(-1), qh, sh, None)
    torch.cuda.synchronize()
    rng = np.random.default_rng(6)
    blk = np.sort(rng.choice(nblk, 4096, replace=False))
    blk[-1] = nblk - 1
    idx = torch.from_numpy(blk).cuda()

    def gather(t, width):
        return t.reshape(-1, width)[idx]

    xb = [bits(gather(x.reshape(-1), 128)) for x in xs]
    ref = [oracle.quant_mx_flat(b) for b in xb]
    for w in range(4):
        assert_same(gather(wires[w][0], 128), ref[w][0], f"source {w} codes")
        assert_same(gather(wires[w][1], 4), ref[w][1], f"source {w} scales")
    qa_r, sa_r, oa_r = oracle.dequant_accum_mx([r[0] for r in ref], [r[1] for r in ref], materialize=True)
    assert_same(gather(qa, 128), qa_r, "accumulated codes")
    assert_same(gather(sa, 4), sa_r, "accumulated scales")
    assert_same(gather(out, 128), oa_r, "owner materialization")
    qh_r, sh_r, _ = oracle.ring_hop_mx(ref[0][0], ref[0][1], xb[1])
    assert_same(gather(qh, 128), qh_r, "hop codes")
    assert_same(gather(sh, 4), sh_r, "hop scales")


# ------------------------------------------------------------------ edge cases
@pytest.mark.parametrize("nblk", [1, 2, 3, 7, 8, 9, 17, 63, 65, 1029, 4099])
def test_mx_ragged_sizes(nblk):
    rng = np.random.default_rng(500 + nblk)
    W = 3
    qs, ss = random_wires(rng, W, nblk)
    n = nblk * 128
    gq, gs, go = Guarded(n), Guarded(n // 32), Guarded(2 * n)
    codec.dequant_accum_mx([dev(q) for q in qs], [dev(s) for s in ss], gq.view(torch.uint8), gs.view(torch.uint8),
                           go.view(torch.bfloat16))
    qa, sa, oa = oracle.dequant_accum_mx(qs, ss, materialize=True)
    assert_same(gq.view(torch.uint8), qa, "accumulated codes")
    assert_same(gs.view(torch.uint8), sa, "accumulated scales")
    assert_same(go.view(torch.bfloat16), oa, "materialized")
    assert gq.bands_intact() and gs.bands_intact() and go.bands_intact()
    x_loc = adversarial_blocks(rng, nblk, max_abs=1.0e37).reshape(-1)
    hq, hs, ho = Guarded(n), Guarded(n // 32), Guarded(2 * n)
    codec.ring_hop_mx(dev(qs[0]), dev(ss[0]), from_bits_bf16(x_loc), hq.view(torch.uint8), hs.view(torch.uint8),
                      ho.view(torch.bfloat16))
    qh, sh, oh = oracle.ring_hop_mx(qs[0], ss[0], x_loc, materialize=True)
    assert_same(hq.view(torch.uint8), qh, "hop codes")
    assert_same(hs.view(torch.uint8), sh, "hop scales")
    assert_same(ho.view(torch.bfloat16), oh, "hop materialized")
    assert hq.bands_intact() and hs.bands_intact() and ho.bands_intact()


@pytest.mark.parametrize("W", [1, 2, 3, 4, 5, 7, 8, 9, 16])
@pytest.mark.parametrize("owner", [True, False])
@pytest.mark.parametrize("nblk", [37, 8, 1])
def test_mx_accumulate_any_width(W, owner, nblk):
    # with and without the owner output, whole and partial chunks
    rng = np.random.default_rng(600 + W + nblk)
    qs, ss = random_wires(rng, W, nblk, e_lo=60, e_hi=200)
    n = nblk * 128
    _, qo, so = codec.empty_wire_mx(n)
    out = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    codec.dequant_accum_mx([dev(q) for q in qs], [dev(s) for s in ss], qo, so, out if owner else None)
    qa, sa, oa = oracle.dequant_accum_mx(qs, ss, materialize=True)
    assert_same(qo, qa, "codes")
    assert_same(so, sa, "scales")
    if owner:
        assert_same(out, oa, "materialized")


def test_mx_bf16_pointers_aligned_to_16_but_not_32_bytes():
    # the wide kernels take 256-bit BF16 accesses only at 32-byte-aligned pointers
    rng = np.random.default_rng(702)
    nblk, W = 45, 4
    qs, ss = random_wires(rng, W, nblk, e_lo=60, e_hi=200)
    n = nblk * 128
    x_loc = adversarial_blocks(rng, nblk, max_abs=1.0e37).reshape(-1)
    for off in (0, 8):  # BF16 elements: 0 and 16 bytes past a 32-byte boundary
        raw_out = torch.empty(n + 16, dtype=torch.bfloat16, device="cuda")
        out = raw_out[off:off + n]
        raw_x = torch.empty(n + 16, dtype=torch.bfloat16, device="cuda")
        x = raw_x[off:off + n]
        x.copy_(from_bits_bf16(x_loc))
        assert out.data_ptr() % 32 == 2 * off and x.data_ptr() % 32 == 2 * off
        _, qo, so = codec.empty_wire_mx(n)
        codec.dequant_accum_mx([dev(q) for q in qs], [dev(s) for s in ss], qo, so, out)
        qa, sa, oa = oracle.dequant_accum_mx(qs, ss, materialize=True)
        assert_same(qo, qa, f"accumulated codes, offset {off}")
        assert_same(out, oa, f"accumulate owner output, offset {off}")
        codec.ring_hop_mx(dev(qs[1]), dev(ss[1]), x, qo, so, out)
        qh, sh, oh = oracle.ring_hop_mx(qs[1], ss[1], x_loc, materialize=True)
        assert_same(qo, qh, f"hop codes, offset {off}")
        assert_same(so, sh, f"hop scales, offset {off}")
        assert_same(out, oh, f"hop owner output, offset {off}")


def test_mx_accumulate_tiny_and_cancelling_sums():
    # Two sources A and B:
    #   group 0  A: one element 448 * 2^13 (scale byte 140), B: elements m * 2^-136
    #            (scale byte 0); the sum requantizes with byte 140, which scales the
    #            small elements to m * 2^-149, binary32 subnormals, and rounds them to
    #            E4M3 zero with their sign
    #   group 1  negative zeros in both (-0 + -0 = -0)
    #   group 2  B = -A exactly (cancellation to +0, all-zero group -> byte 127)
    #   group 3  both at scale byte 0: sums down to 2^-135, requantized at byte 0
    n = 128
    qa = np.zeros(n, np.uint8)
    qb = np.zeros(n, np.uint8)
    sa = np.array([140, 9, 100, 0], np.uint8)
    sb = np.array([0, 17, 100, 0], np.uint8)
    qa[0] = 0x7E
    qb[1:32] = np.resize(np.array([0x01, 0x81, 0x05, 0x85, 0x07], np.uint8), 31)
    qa[32:64] = 0x80
    qb[32:64] = 0x80
    qa[64:96] = np.arange(0x40, 0x60)
    qb[64:96] = qa[64:96] ^ 0x80
    qa[96:128] = np.resize(np.array([0x01, 0x02, 0x83, 0x04], np.uint8), 32)
    qb[96:128] = np.resize(np.array([0x01, 0x81, 0x06], np.uint8), 32)
    for srcs, scs in (([qa, qb], [sa, sb]), ([qa, qa, qa], [sa, sa, sa]), ([qb], [sb]), ([qb, qa], [sb, sa])):
        _, qo, so = codec.empty_wire_mx(n)
        out = torch.empty(n, dtype=torch.bfloat16, device="cuda")
        codec.dequant_accum_mx([dev(a) for a in srcs], [dev(c) for c in scs], qo, so, out)
        qr, sr, orr = oracle.dequant_accum_mx(srcs, scs, materialize=True)
        assert_same(qo, qr, "codes")
        assert_same(so, sr, "scales")
        assert_same(out, orr, "materialized")
    qr, sr, _ = oracle.dequant_accum_mx([qa, qb], [sa, sb], materialize=False)
    assert sr[0] == 140 and np.all((qr[1:32] & 0x7F) == 0) and sr[2] == 127


def _scales_at_4_mod_16(s: np.ndarray) -> torch.Tensor:
    buf = torch.zeros(s.size + 16, dtype=torch.uint8, device="cuda")
    view = buf[4:4 + s.size]
    view.copy_(torch.from_numpy(s))
    assert view.data_ptr() % 16 == 4
    return view


def test_mx_reductions_with_scales_not_16_byte_aligned():
    rng = np.random.default_rng(700)
    nblk, W = 1031, 4
    qs, ss = random_wires(rng, W, nblk, e_lo=80, e_hi=180)
    n = nblk * 128
    _, qo, so = codec.empty_wire_mx(n)
    codec.dequant_accum_mx([dev(q) for q in qs], [_scales_at_4_mod_16(s) for s in ss], qo, so, None)
    qa, sa, _ = oracle.dequant_accum_mx(qs, ss, materialize=False)
    assert_same(qo, qa, "accumulated codes")
    assert_same(so, sa, "accumulated scales")
    x_loc = adversarial_blocks(rng, nblk, max_abs=1.0e37).reshape(-1)
    out = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    codec.ring_hop_mx(dev(qs[1]), _scales_at_4_mod_16(ss[1]), from_bits_bf16(x_loc), qo, so, out)
    qh, sh, oh = oracle.ring_hop_mx(qs[1], ss[1], x_loc, materialize=True)
    assert_same(qo, qh, "hop codes")
    assert_same(so, sh, "hop scales")
    assert_same(out, oh, "hop materialized")


def test_mx_hop_cancellation_and_negative_zero():
    rng = np.random.default_rng(701)
    nblk = 40
    x_in = adversarial_blocks(rng, nblk, max_abs=1.0e37).reshape(-1)
    q_in, s_in = oracle.quant_mx_flat(x_in)
    # the local shard cancels some incoming values exactly (-x), adds -0 to others
    x_loc = adversarial_blocks(rng, nblk, max_abs=1.0e37).reshape(-1)
    deq = oracle.dequant_mx_flat(q_in, s_in)
    x_loc[:1024] = deq[:1024] ^ 0x8000
    x_loc[1024:2048] = 0x8000
    n = x_in.size
    _, qo, so = codec.empty_wire_mx(n)
    out = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    codec.ring_hop_mx(dev(q_in), dev(s_in), from_bits_bf16(x_loc), qo, so, out)
    qh, sh, oh = oracle.ring_hop_mx(q_in, s_in, x_loc, materialize=True)
    assert_same(qo, qh, "codes")
    assert_same(so, sh, "scales")
    assert_same(out, oh, "materialized")


def test_mx_reductions_empty_and_errors():
    e8 = torch.empty(0, dtype=torch.uint8, device="cuda")
    codec.dequant_accum_mx([e8], [e8], e8, e8, None)
    codec.ring_hop_mx(e8, e8, torch.empty(0, dtype=torch.bfloat16, device="cuda"), e8, e8, None)
    n = 256
    _, q, s = codec.empty_wire_mx(n)
    _, q2, s2 = codec.empty_wire_mx(n)
    x = torch.zeros(n, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(BQError) as ei:  # output aliases an input
        codec.dequant_accum_mx([q], [s], q, s2)
    assert ei.value.status == 4
    with pytest.raises(BQError) as ei:
        codec.ring_hop_mx(q, s, x, q2, s)
    assert ei.value.status == 4
    big = torch.zeros(n + 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(BQError) as ei:  # payload not 16-byte aligned
        codec.dequant_accum_mx([big[1:1 + n]], [s], q2, s2)
    assert ei.value.status == 3
    with pytest.raises(BQError) as ei:  # W = 17
        codec.dequant_accum_mx([q] * 17, [s] * 17, q2, s2)
    assert ei.value.status == 2


def test_mx_reductions_graph_replay_is_bit_identical():
    xs = [x.cuda() for x in inputs.a2a_3072(rows=512)]
    n = xs[0].numel()
    wires = [codec.empty_wire_mx(n) for _ in range(6)]
    owner = torch.empty(n, dtype=torch.bfloat16, device="cuda")

    def step(stream=None):
        for w in range(4):
            codec.quant_mx_flat(xs[w].reshape(-1), wires[w][1], wires[w][2], stream)
        codec.dequant_accum_mx([wires[w][1] for w in range(4)], [wires[w][2] for w in range(4)], wires[4][1],
                               wires[4][2], owner, stream)
        codec.ring_hop_mx(wires[4][1], wires[4][2], xs[0].reshape(-1), wires[5][1], wires[5][2], None, stream)

    step()
    torch.cuda.synchronize()
    eager = [w[0].clone() for w in wires] + [owner.clone()]
    for w in wires:
        w[0].zero_()
    owner.zero_()
    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(st):
        with torch.cuda.graph(g, stream=st):
            step(st)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    for a, b in zip(eager, [w[0] for w in wires] + [owner]):
        assert torch.equal(a, b)


def test_mx_ring_chain_full_size_sampled():
    # the 16384-row ring chain (4 shards of 4096 rows, 1 quantize + 3 hops each) at full
    # size on the GPU; every element's chain is independent, so the oracle recomputes
    # the chain on 2048 sampled 128-value blocks of every shard
    xs = [x.cuda() for x in inputs.ring_16384()]
    W = len(xs)
    outs, finals, owners = topology.mx_ring(xs)
    torch.cuda.synchronize()
    nblk_shard = xs[0].numel() // W // 128
    rng = np.random.default_rng(61)
    for c in range(W):
        blk = np.sort(rng.choice(nblk_shard, 2048, replace=False))
        blk[-1] = nblk_shard - 1
        idx = torch.from_numpy(blk).cuda()
        shard = [x.reshape(W, -1)[c].reshape(-1, 128)[idx] for x in xs]
        chain = topology.ring_order(c, W)
        q, s = oracle.quant_mx_flat(bits(shard[chain[0]]))
        for rank in chain[1:]:
            q, s, _ = oracle.ring_hop_mx(q, s, bits(shard[rank]))
        assert_same(finals[c][0].reshape(-1, 128)[idx], q, f"shard {c} codes")
        assert_same(finals[c][1].reshape(-1, 4)[idx], s, f"shard {c} scales")
        assert_same(owners[c].reshape(-1, 128)[idx], oracle.dequant_mx_flat(q, s), f"shard {c} owner")
    for o in outs[1:]:
        assert torch.equal(o, outs[0])


def test_mx_modes_error_vs_unquantized_sum():
    # each MX requantization moves a value by at most half an E4M3 spacing at its
    # scaled magnitude, relative 2^-4 of the value for normal codes plus 2^-10 * 2^(e-127)
    # absolutely; the a2a owner output stays within the sum of those bounds of the exact
    # sum of the BF16 inputs (plus half a BF16 ulp of the output)
    xs = [x.cuda() for x in inputs.a2a_3072(rows=256)]
    q_out, s_out, owner, srcs = topology.mx_a2a(xs)
    exact = sum(x.double() for x in xs).reshape(-1, 32)
    def group_bound(s_bytes, vals):
        scale = torch.exp2(s_bytes.double() - 127)[:, None]
        return vals.abs() * 2.0 ** -4 + scale * 2.0 ** -10
    bound = sum(group_bound(s.reshape(-1), x.double().reshape(-1, 32)) for (_, s), x in zip(srcs, xs))
    # the requantization's term is relative to the binary32 sum, which exceeds the
    # owner output by at most 1 / (1 - 2^-4) and half a BF16 ulp: 1.1 covers both
    bound = bound + group_bound(s_out.reshape(-1), owner.double().reshape(-1, 32) * 1.1)
    bound = bound + owner.double().reshape(-1, 32).abs() * 2.0 ** -8 + 1e-30
    err = (owner.double().reshape(-1, 32) - exact).abs()
    assert bool((err <= bound * (1 + 2.0 ** -10)).all())
