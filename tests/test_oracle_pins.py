"""Pins of the CPU oracle to things other than itself (no GPU needed).

Each test checks the oracle against what the pull-request pages or the mathematics
fix: hand-derived closed forms (tests/golden), exhaustive sweeps, exact-rational
brute force, invariants the pages list (132-byte layout, zero blocks, the
half-quantization-step bound, amax mapping to +-127, canonical forwarding, staged ==
concatenated), and special cases that reduce to library routines.
"""
import os
import random
from fractions import Fraction as F

import numpy as np
import pytest
import torch

import oracle
from tests import exact

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf16_bits_of(values) -> np.ndarray:
    t = torch.tensor([float(v) for v in values], dtype=torch.float32).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


def _parse_i8_golden():
    cases, cur = [], None
    for line in open(os.path.join(GOLDEN, "i8_blocks.txt")):
        line = line.split("#", 1)[0].strip()
        if not line:
            continue
        key, _, val = line.partition(":")
        val = val.split()
        if key == "case":
            cur = {"name": val[0]}
            cases.append(cur)
        elif key in ("x", "scale", "q", "deq"):
            cur[key] = val
    return cases


# ------------------------------------------------------------------ layout
def test_wire_layout_132_bytes_per_block():
    # "add block-INT8 wire modes for AG, ring, and A2A", Summary: 128 payload bytes +
    # one FP32 scale = 132 bytes per block; "add INT8 and MXFP8 wire modes", Summary:
    # 132 vs 256 bytes per 128 values, a 48.4% reduction.
    for nblk in (0, 1, 7, 28672, 3670016 // 128):
        assert oracle.wire_bytes(128 * nblk) == 132 * nblk
    assert 1 - F(132, 256) == F(484375, 1000000)
    assert round(float(1 - F(132, 256)) * 100, 1) == 48.4
    # MX: 128 E4M3 bytes + 4 E8M0 bytes per 128 values is the same 132 bytes.
    x = np.zeros((1, 128), np.uint16)
    q, s = oracle.quant_mx(x)
    assert q.nbytes + s.nbytes == 132


# ------------------------------------------------------------------ golden (closed forms)
@pytest.mark.parametrize("case", _parse_i8_golden(), ids=lambda c: c["name"])
def test_i8_golden_blocks(case):
    xs = [float(v) for v in case["x"]]
    block = np.zeros(128, np.uint16)
    block[: len(xs)] = _bf16_bits_of(xs)
    # the listed inputs are exact BF16 numbers
    assert np.array_equal(_bits_to_f32(block[: len(xs)]), np.array(xs, np.float32))
    q, s = oracle.quant_i8(block)
    assert s[0] == np.float32(float(case["scale"][0]))
    assert not np.signbit(s[0])
    assert list(q[: len(xs)]) == [int(v) for v in case["q"]]
    assert np.all(q[len(xs):] == 0)
    if "deq" in case:
        out = oracle.dequant_i8(q, s)
        assert [int(h, 16) for h in case["deq"]] == list(out[: len(xs)].astype(int))


def test_mx_golden():
    for line in open(os.path.join(GOLDEN, "mx_scales.txt")):
        line = line.split("#", 1)[0].strip()
        if not line:
            continue
        if line.startswith("e8m0"):
            _, amax, byte = line.split()
            assert oracle.e8m0_scale(float(amax)) == int(byte), line
        elif line.startswith("e4m3"):
            _, y, code = line.split()
            assert oracle.e4m3_encode(float(y)) == int(code, 16), line
        elif line.startswith("group"):
            parts = [p.strip() for p in line[len("group"):].split("|")]
            xs = [float(v) for v in parts[0].split(":")[1].split()]
            e = int(parts[1].split(":")[1])
            codes = [int(c, 16) for c in parts[2].split(":")[1].split()]
            row = np.zeros((1, 128), np.uint16)
            row[0, : len(xs)] = _bf16_bits_of(xs)
            q, s = oracle.quant_mx(row)
            assert s[0, 0] == e
            assert list(q[0, : len(codes)]) == codes
            assert np.all(q[0, len(codes):32] == 0)
            assert list(s[0, 1:]) == [127, 127, 127]  # the other three groups are zero


# ------------------------------------------------------------------ zero blocks
def test_zero_blocks_i8_and_mx():
    # proofs list of the block-INT8 page: zero blocks -> scale 0, payload 0.
    x = np.zeros(128 * 5, np.uint16)
    x[128 * 2 + 7] = _bf16_bits_of([3.0])[0]
    q, s = oracle.quant_i8(x)
    assert list(s == 0) == [True, True, False, True, True]
    assert np.all(q[:256] == 0) and np.all(q[384:] == 0)
    out = oracle.dequant_i8(q, s)
    assert np.all(out[:256] == 0) and np.all(out[384:] == 0)
    # MX: zero group -> scale byte 127 and value bytes 0 (review rule of the MXFP8 page)
    qm, sm = oracle.quant_mx(np.zeros((2, 256), np.uint16))
    assert np.all(sm == 127) and np.all(qm == 0)
    assert np.all(oracle.dequant_mx(qm, sm) == 0)


# ------------------------------------------------------------------ amax -> +-127 (exhaustive)
def test_amax_maps_to_127_for_every_bf16_amax():
    # Every positive finite BF16 value a as the block's amax, with -a beside it.
    a = np.arange(1, 0x7F80, dtype=np.uint16)
    blocks = np.zeros((a.size, 128), np.uint16)
    blocks[:, 0] = a
    blocks[:, 1] = a | 0x8000
    blocks[:, 2] = a >> 1  # a smaller value in the same block (no constraint, exercised)
    q, s = oracle.quant_i8(blocks.reshape(-1))
    q = q.reshape(a.size, 128)
    assert np.all(q[:, 0] == 127)
    assert np.all(q[:, 1] == -127)
    assert np.all(np.abs(q) <= 127)
    # and the scale is the binary32 quotient amax/127 (library division, IEEE binary32)
    assert np.array_equal(s, (_bits_to_f32(a) / np.float32(127)).astype(np.float32))


# ------------------------------------------------------------------ half-step bound
def _random_blocks(rng, nblk):
    kinds = []
    out = np.zeros((nblk, 128), np.float32)
    for b in range(nblk):
        kind = b % 6
        if kind == 0:
            v = rng.standard_normal(128)
        elif kind == 1:
            v = rng.standard_normal(128) * 10.0 ** rng.uniform(-30, 30)
        elif kind == 2:  # one outlier
            v = rng.standard_normal(128)
            v[rng.integers(128)] *= 1000
        elif kind == 3:  # BF16 subnormal range
            v = rng.standard_normal(128) * 2.0 ** -128
        elif kind == 4:  # ties around integers of a power-of-two scale
            v = (rng.integers(-127, 128, 128) + 0.5) * 2.0 ** rng.integers(-20, 20)
            v[0] = 127 * 2.0 ** -3
        else:  # few distinct values
            v = rng.choice([0.0, 1.0, -1.0, 0.5, 3.0, -127.0], 128)
        out[b] = v
        kinds.append(kind)
    t = torch.from_numpy(out).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def test_half_step_error_bound():
    # proofs list of the block-INT8 page: |x - deq| <= scale / 2. On the binary32
    # dequantized value the exact bound is s * (1/2 + 2^-18) because fl(x/s) may be a
    # half-ulp (<= 2^-18 for |x/s| < 128) off x/s before rounding to an integer.
    rng = np.random.default_rng(7)
    x = _random_blocks(rng, 600)
    q, s = oracle.quant_i8(x.reshape(-1))
    xv = _bits_to_f32(x).astype(np.float64).reshape(-1, 128)
    deq = q.reshape(-1, 128).astype(np.float64) * s.astype(np.float64)[:, None]  # exact in float64
    err = np.abs(xv - deq)
    bound = s.astype(np.float64)[:, None] * (0.5 + 2.0 ** -18)
    assert np.all(err <= bound)
    # the bound is attained to within the slack somewhere (it is not vacuous)
    nz = s > 0
    assert np.max(err[nz] / s[nz, None]) > 0.49


# ------------------------------------------------------------------ brute force (exact rationals)
def _adversarial_blocks(rnd, nblk, max_abs=3.0e38):
    special = [0.0, -0.0, 1.0, -1.0, 0.5, 1.5, 2.5, 127.0, 126.5, 2.0 ** -133, 2.0 ** -126, 3.0e38, -3.0e38]
    blocks = []
    for b in range(nblk):
        base = 2.0 ** rnd.randint(-140, 120)
        vals = []
        for i in range(128):
            r = rnd.random()
            if r < 0.2:
                vals.append(rnd.choice(special) * (base if rnd.random() < 0.5 else 1.0))
            elif r < 0.5:
                vals.append((rnd.randint(-254, 254) / 2.0) * base)
            else:
                vals.append(rnd.gauss(0, 1) * base)
        blocks.append(vals)
    t = torch.tensor(blocks, dtype=torch.float32).clamp(-max_abs, max_abs).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def test_quant_dequant_i8_brute_force_exact():
    rnd = random.Random(11)
    x = _adversarial_blocks(rnd, 48)
    q, s = oracle.quant_i8(x.reshape(-1))
    out = oracle.dequant_i8(q, s)
    for b in range(x.shape[0]):
        vals = [exact.bits_to_value(int(v)) for v in x[b]]
        q_ref, s_ref = exact.quant_block_i8(vals)
        assert F(float(s[b])) == s_ref
        assert list(q[128 * b:128 * b + 128]) == q_ref
        for i in range(128):
            assert int(out[128 * b + i]) == exact.dequant_i8(q_ref[i], s_ref)


def test_accumulate_follows_source_order_exact():
    # "multi-source INT8 dequantization with FP32 accumulation": d_w = fl(q_w s_w) and
    # acc = ((d_0 + d_1) + d_2) + d_3 in binary32; sources chosen so that other orders
    # of the additions give other sums (absorption of small terms).
    rnd = random.Random(5)
    n = 128 * 6
    W = 4
    qs, ss = [], []
    for w in range(W):
        qs.append(np.array([rnd.randint(-127, 127) for _ in range(n)], np.int8))
        ss.append(np.array([np.float32(2.0 ** rnd.randint(-30, 30) * (1 + rnd.random())) for _ in range(n // 128)],
                           np.float32))
    # make block 0 order-sensitive: big, tiny, -big, tiny
    ss[0][0], ss[1][0], ss[2][0], ss[3][0] = np.float32(2.0 ** 20), np.float32(2.0 ** -10), np.float32(2.0 ** 20), np.float32(2.0 ** -10)
    qs[0][:128], qs[2][:128] = 100, -100
    q_out, s_out, out = oracle.dequant_accum_i8(qs, ss)
    for b in range(n // 128):
        acc = []
        for i in range(128):
            e = 128 * b + i
            a = exact.f32(int(qs[0][e]) * F(float(ss[0][b])))
            for w in range(1, W):
                a = exact.f32(a + exact.f32(int(qs[w][e]) * F(float(ss[w][b]))))
            acc.append(a)
        q_ref, s_ref = exact.quant_block_i8(acc)
        assert F(float(s_out[b])) == s_ref
        assert list(q_out[128 * b:128 * b + 128]) == q_ref
    # block 0: the sum in source order is 2 * tiny terms lost? check it is not the
    # reordered sum (d0 + d2) + (d1 + d3)
    e = 0
    d = [exact.f32(int(qs[w][e]) * F(float(ss[w][0]))) for w in range(W)]
    in_order = exact.f32(exact.f32(exact.f32(d[0] + d[1]) + d[2]) + d[3])
    regrouped = exact.f32(exact.f32(d[0] + d[2]) + exact.f32(d[1] + d[3]))
    assert in_order != regrouped
    # canonical forwarding: the owner output is the materialization of the payload
    assert np.array_equal(out, oracle.dequant_i8(q_out, s_out))


def test_ring_hop_exact():
    # "fused INT8 dequantize-add-requantize for each ring reduce-scatter hop"
    rnd = random.Random(3)
    x_in = _adversarial_blocks(rnd, 8).reshape(-1)
    x_loc = _adversarial_blocks(rnd, 8).reshape(-1)
    q_in, s_in = oracle.quant_i8(x_in)
    q_out, s_out, out = oracle.ring_hop_i8(q_in, s_in, x_loc, materialize=True)
    for b in range(8):
        v = []
        for i in range(128):
            e = 128 * b + i
            d = exact.f32(int(q_in[e]) * F(float(s_in[b])))
            v.append(exact.f32(d + exact.bits_to_value(int(x_loc[e]))))
        q_ref, s_ref = exact.quant_block_i8(v)
        assert F(float(s_out[b])) == s_ref
        assert list(q_out[128 * b:128 * b + 128]) == q_ref
    assert np.array_equal(out, oracle.dequant_i8(q_out, s_out))


def test_fp32_tiny_amax_scale_underflow():
    # Reading R2: an FP32 sum whose amax/127 underflows to 0 gives scale 0, payload 0;
    # one whose amax/127 is subnormal is quantized with the clamp engaged when the
    # rounded scale is far below amax/127.
    tiny = np.float32(2.0 ** -149)
    q0 = np.zeros(128, np.int8)
    q0[0] = 1
    q_out, s_out, _ = oracle.dequant_accum_i8([q0], [np.array([tiny], np.float32)], materialize=False)
    assert s_out[0] == 0 and np.all(q_out == 0)
    # amax = 190 * 2^-149 -> amax / 127 = 1.496 * 2^-149 -> scale 2^-149, quotient 190
    q1 = np.zeros(128, np.int8)
    q1[0], q1[1] = 95, -3
    q_out, s_out, _ = oracle.dequant_accum_i8([q1], [np.array([np.float32(2.0 ** -148)], np.float32)],
                                              materialize=False)
    assert s_out[0] == tiny
    assert q_out[0] == 127 and q_out[1] == -6
    # the same block negated clamps at -127 (the payload never holds -128)
    q_out, s_out, _ = oracle.dequant_accum_i8([-q1], [np.array([np.float32(2.0 ** -148)], np.float32)],
                                              materialize=False)
    assert q_out[0] == -127 and q_out[1] == 6


# ------------------------------------------------------------------ BF16 rounding vs library
def test_bf16_round_matches_torch_conversion():
    rng = np.random.default_rng(1)
    u = rng.integers(0, 2 ** 32, 20000, dtype=np.uint64).astype(np.uint32)
    # bias toward ties and subnormals and the overflow edge
    u[:2000] = (u[:2000] & 0xFFFF0000) | 0x8000
    u[2000:3000] = u[2000:3000] & 0x807FFFFF
    u[3000] = 0x7F7FFFFF
    u[3001] = 0x7F7F8000
    u[3002] = 0x7F7F7FFF
    f = u.view(np.float32)
    f = f[np.isfinite(f)]
    ref = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.bf16_round(float(v)) for v in f], np.uint16)
    assert np.array_equal(got, ref)


def test_dequant_i8_matches_library_double_rounding():
    # materialization: binary32 product (library multiply) then library BF16 rounding
    rng = np.random.default_rng(2)
    q = rng.integers(-128, 128, 128 * 512).astype(np.int8)
    s = (rng.standard_normal(512) * 10.0 ** rng.uniform(-40, 36, 512)).astype(np.float32)
    s[:3] = [0.0, np.float32(2.0 ** -149), np.float32(3.0e36)]
    out = oracle.dequant_i8(q, s)
    prod = torch.from_numpy(q.astype(np.float32)) * torch.from_numpy(np.repeat(s, 128))
    ref = prod.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(out, ref)


def test_double_rounding_differs_from_single_rounding_somewhere():
    # The definition rounds q*s to binary32 first. Near a BF16 midpoint m, a product
    # q*s slightly off m can round to m in binary32 and then to the even BF16 neighbour,
    # where rounding q*s once would pick the other neighbour. Search the binary32 scales
    # next to m/q for such cases and check that the oracle rounds twice.
    found = 0
    for m in (1 + F(1, 256), 1 + F(3, 256), F(3, 2) + F(1, 128), 100 + F(1, 4)):
        for qv in range(3, 128, 2):
            centre = np.float32(float(m / qv))
            for k in range(-3, 4):
                s = np.nextafter(centre, np.float32(np.inf) if k > 0 else np.float32(0), dtype=np.float32)
                for _ in range(abs(k) - 1):
                    s = np.nextafter(s, np.float32(np.inf) if k > 0 else np.float32(0), dtype=np.float32)
                if k == 0:
                    s = centre
                exact_prod = qv * F(float(s))
                once = exact.bf16_bits(exact.bf16(exact_prod))
                twice = exact.bf16_bits(exact.bf16(exact.f32(exact_prod)))
                if once != twice:
                    qq = np.zeros(128, np.int8)
                    qq[0] = qv
                    assert int(oracle.dequant_i8(qq, np.array([s], np.float32))[0]) == twice
                    found += 1
    assert found >= 3


# ------------------------------------------------------------------ E8M0 (exhaustive)
def test_e8m0_scale_exhaustive_over_bf16_amax():
    # review rule of the MXFP8 page; checked for every positive finite BF16 amax against
    # a closed form from the library's frexp: v = m * 2^k with m in [0.5, 1); the
    # smallest power of two >= v is 2^(k-1) when m == 0.5, else 2^k.
    a_bits = np.arange(1, 0x7F80, dtype=np.uint16)
    a = _bits_to_f32(a_bits)
    v = (a / np.float32(448.0)).astype(np.float32)
    m, k = np.frexp(v.astype(np.float64))
    expect = np.where(m == 0.5, k - 1, k) + 127
    expect = np.clip(expect, 0, 254)
    ngroups = ((a.size + 3) // 4) * 4
    groups = np.zeros((ngroups, 32), np.uint16)
    groups[: a.size, 0] = a_bits
    groups[: a.size, 5] = a_bits | 0x8000
    q, s = oracle.quant_mx(groups.reshape(-1, 128))
    got = s.reshape(-1)
    assert np.all(got[a.size:] == 127)
    got = got[: a.size]
    assert np.array_equal(got, expect.astype(np.uint8))
    # the largest magnitude lands in (224, 448] unless the scale byte bottoms out at 0,
    # so saturation never engages for finite BF16 input
    y = a.astype(np.float64) * np.exp2(127.0 - got.astype(np.float64))
    assert np.all(y <= 448.0)
    assert np.all((y > 224.0) | (got == 0))
    assert got.max() <= 247


def test_e8m0_brute_force_exact_subnormal_range():
    # exact: v = fl(amax / 448) then the smallest 2^(b-127) >= v, by direct comparison
    for a_bits in list(range(1, 0x200)) + list(range(0x0300, 0x0400)):
        a = exact.bits_to_value(a_bits)
        v = exact.f32(a / 448)
        assert oracle.e8m0_scale(float(a)) == exact.e8m0_up(v), hex(a_bits)


# ------------------------------------------------------------------ E4M3 (exhaustive)
def test_e4m3_encode_exhaustive_vs_nearest_search():
    # Every BF16 value with |y| < 2^10 (this covers every E4M3 tie point, the
    # subnormal range, and the saturation region), against a nearest-value search over
    # the 126 non-negative finite E4M3 values written out from the format definition.
    codes = []
    vals = []
    for code, v in exact.e4m3_values():
        codes.append(code)
        vals.append(float(v))
    vals = np.array(vals)
    bits = np.arange(0, 0x4480, dtype=np.uint16)  # 0 .. 2^10 (exclusive-ish)
    ys = _bits_to_f32(bits).astype(np.float64)
    # nearest search: distances are exact here except when one candidate is far away
    d = np.abs(vals[None, :] - ys[:, None])
    best = d.min(axis=1)
    cand = d == best[:, None]
    even = cand & (np.array(codes)[None, :] % 2 == 0)
    pick = np.where(even.any(axis=1), np.argmax(even, axis=1), np.argmax(cand, axis=1))
    expect = np.array(codes)[pick]
    got = np.array([oracle.e4m3_encode(y) for y in ys])
    got_neg = np.array([oracle.e4m3_encode(-y) for y in ys])
    assert np.array_equal(got, expect)
    assert np.array_equal(got_neg, expect | 0x80)


def test_e4m3_encode_matches_torch_float8_e4m3fn():
    # PyTorch's float8_e4m3fn is an independent implementation of OCP E4M3 (the format
    # "standard MXFP8" names): its largest finite value is the 448 the scale rules
    # divide by, and its round-to-nearest-even conversion keeps the sign of zero. Every
    # BF16 value with |y| <= 464 (beyond 464 PyTorch's conversion gives NaN where a
    # saturating one gives 448; no scaled MX value gets there), both signs, subnormals
    # and zeros included, encodes to the same byte.
    f8 = getattr(torch, "float8_e4m3fn", None)
    if f8 is None:
        pytest.skip("this torch has no float8_e4m3fn")
    assert float(torch.finfo(f8).max) == 448.0
    bits = np.arange(0, 0x43E9, dtype=np.uint16)  # 0 .. 464 in BF16
    ys = _bits_to_f32(bits)
    for sign in (1.0, -1.0):
        v = (ys * np.float32(sign)).astype(np.float32)
        want = torch.from_numpy(v).to(f8).view(torch.uint8).numpy()
        got = np.array([oracle.e4m3_encode(float(y)) for y in v], np.uint8)
        bad = np.flatnonzero(got != want)
        assert bad.size == 0, (sign, [(float(v[i]), int(got[i]), int(want[i])) for i in bad[:5]])
    assert oracle.e4m3_encode(-0.0) == 0x80 and oracle.e4m3_encode(0.0) == 0x00


def test_e4m3_decode_exhaustive():
    for code, v in exact.e4m3_values():
        assert F(oracle.e4m3_decode(code)) == v
        assert F(oracle.e4m3_decode(code | 0x80)) == -v
    assert np.isnan(oracle.e4m3_decode(0x7F)) and np.isnan(oracle.e4m3_decode(0xFF))


def test_mx_quant_dequant_brute_force_exact():
    rnd = random.Random(4)
    x = _adversarial_blocks(rnd, 16).reshape(8, 256)
    q, s = oracle.quant_mx(x)
    out = oracle.dequant_mx(q, s)
    for r in range(8):
        for g in range(8):
            vals = [exact.bits_to_value(int(b)) for b in x[r, 32 * g:32 * g + 32]]
            amax = max(abs(v) for v in vals)
            e = 127 if amax == 0 else exact.e8m0_up(exact.f32(amax / 448))
            assert s[r, g] == e
            for i, v in enumerate(vals):
                negative_input = bool(x[r, 32 * g + i] & 0x8000)
                c = exact.e4m3_nearest(v * F(2) ** (127 - e))
                if v == 0 and negative_input:
                    c = 0x80  # -0 keeps its sign (reading R5)
                assert q[r, 32 * g + i] == c
                dv = dict(exact.e4m3_values())[c & 0x7F] * F(2) ** (e - 127)
                want = exact.bf16_bits_signed(-dv if c & 0x80 else dv, bool(c & 0x80))
                assert int(out[r, 32 * g + i]) == want


def test_mx_dequant_of_e4m3_relative_error_bound():
    # |x - deq| <= half an E4M3 spacing at y, times the scale (relative 2^-4 for normal y)
    rng = np.random.default_rng(3)
    xf = (rng.standard_normal((64, 512)) * 10.0 ** rng.uniform(-5, 5, (64, 1))).astype(np.float32)
    x = torch.from_numpy(xf).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    q, s = oracle.quant_mx(x)
    out = oracle.dequant_mx(q, s)
    xv = _bits_to_f32(x).astype(np.float64)
    dv = _bits_to_f32(out).astype(np.float64)
    scale = np.repeat(np.exp2(s.astype(np.float64) - 127), 32, axis=1)
    y = np.abs(xv) / scale
    spacing = np.where(y < 2.0 ** -6, 2.0 ** -9, np.exp2(np.floor(np.log2(np.maximum(y, 2.0 ** -6))) - 3))
    bf16_half_ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(dv), 2.0 ** -126))) - 8)
    assert np.all(np.abs(xv - dv) <= spacing / 2 * scale + bf16_half_ulp)


# ------------------------------------------------------------------ MX wire reductions
def _mx_sources(rnd, W, ngroups, e_lo=100, e_hi=150):
    """Random flat MX wires: finite codes (no 0x7F/0xFF), scale bytes in [e_lo, e_hi]."""
    qs, ss = [], []
    finite = [c for c in range(256) if c & 0x7F != 0x7F]
    for _ in range(W):
        qs.append(np.array([rnd.choice(finite) for _ in range(32 * ngroups)], np.uint8))
        ss.append(np.array([rnd.randint(e_lo, e_hi) for _ in range(ngroups)], np.uint8))
    return qs, ss


def test_mx_accumulate_follows_source_order_exact():
    # mx_a2a (reading R11): d_w = decode(q_w) 2^(e_w-127) exactly, acc = ((d_0 + d_1) +
    # d_2) + d_3 in binary32, requantized per group from the binary32 amax. Checked
    # against exact rationals with the sign of zero tracked.
    rnd = random.Random(11)
    W, ng = 4, 24
    qs, ss = _mx_sources(rnd, W, ng)
    # group 0: big, tiny, -big, tiny (absorption makes the order visible)
    ss[0][0], ss[1][0], ss[2][0], ss[3][0] = 150, 100, 150, 100
    qs[0][:32] = 0x70  # 256
    qs[2][:32] = 0xF0  # -256
    qs[1][:32] = 0x01
    qs[3][:32] = 0x01
    # group 1: every source -0 except a +0 in element 0 (IEEE: -0 + -0 = -0, -0 + +0 = +0)
    for w in range(W):
        qs[w][32:64] = 0x80
    qs[2][32] = 0x00
    # group 2: all zero codes in every source (amax 0 -> byte 127)
    for w in range(W):
        qs[w][64:96] = 0x00
    # group 3: scale byte 0 and small codes: decoded values down to 2^-136, below the
    # BF16 subnormal range but exact in binary32
    for w in range(W):
        ss[w][3] = 0
        qs[w][96:128] = [rnd.choice([0x01, 0x02, 0x03, 0x05, 0x09, 0x81, 0x83, 0x8A]) for _ in range(32)]
    q_out, s_out, out = oracle.dequant_accum_mx(qs, ss)
    for g in range(ng):
        acc = []
        for i in range(32):
            e = 32 * g + i
            a = exact.mx_element(int(qs[0][e]), int(ss[0][g]))
            for w in range(1, W):
                a = exact.f32_add_signed(a, exact.mx_element(int(qs[w][e]), int(ss[w][g])))
            acc.append(a)
        codes, eg = exact.quant_group_mx(acc)
        assert s_out[g] == eg, g
        assert list(q_out[32 * g:32 * g + 32]) == codes, g
        assert [int(b) for b in out[32 * g:32 * g + 32]] == [exact.dequant_mx(c, eg) for c in codes]
    assert s_out[2] == 127 and np.all(q_out[64:96] == 0)
    assert q_out[32] == 0x00 and np.all(q_out[33:64] == 0x80)
    # source order matters for group 0
    d = [exact.mx_element(int(qs[w][0]), int(ss[w][0]))[0] for w in range(W)]
    in_order = exact.f32(exact.f32(exact.f32(d[0] + d[1]) + d[2]) + d[3])
    regrouped = exact.f32(exact.f32(d[0] + d[2]) + exact.f32(d[1] + d[3]))
    assert in_order != regrouped
    # canonical forwarding: the owner output is the materialization of the payload
    assert np.array_equal(out, oracle.dequant_mx_flat(q_out, s_out))


def test_mx_ring_hop_exact():
    # mx_ring (reading R12): v = fl(decode(q_in) 2^(e_in-127) + x_local), requantized
    rnd = random.Random(12)
    x_in = _adversarial_blocks(rnd, 6).reshape(-1)
    x_loc = _adversarial_blocks(rnd, 6).reshape(-1)
    x_loc[:64] = x_in[:64] ^ 0x8000  # cancellations to exact zeros and tiny sums
    q_in, s_in = oracle.quant_mx_flat(x_in)
    q_out, s_out, out = oracle.ring_hop_mx(q_in, s_in, x_loc, materialize=True)
    for g in range(x_in.size // 32):
        v = []
        for i in range(32):
            e = 32 * g + i
            xl = (exact.bits_to_value(int(x_loc[e])), int(x_loc[e]) == 0x8000)
            v.append(exact.f32_add_signed(exact.mx_element(int(q_in[e]), int(s_in[g])), xl))
        codes, eg = exact.quant_group_mx(v)
        assert s_out[g] == eg, g
        assert list(q_out[32 * g:32 * g + 32]) == codes, g
    assert np.array_equal(out, oracle.dequant_mx_flat(q_out, s_out))


def test_mx_single_source_accumulate_preserves_quantized_wires():
    # For a wire quantized from BF16, each group's largest |x 2^(127-e)| exceeds 224,
    # so its largest code is in [224, 448]. Requantizing the exact decode keeps the
    # scale byte and every code when that code is above 224, and otherwise (largest
    # code exactly 224) lowers the byte by one and doubles every code exactly. Either
    # way the one-source reduction preserves every value, and the sign of zero.
    rnd = random.Random(13)
    x = _adversarial_blocks(rnd, 16).reshape(-1)
    q, s = oracle.quant_mx_flat(x)
    q1, s1, out1 = oracle.dequant_accum_mx([q], [s])
    assert np.array_equal(out1, oracle.dequant_mx_flat(q, s))
    cmax = (q.reshape(-1, 32) & 0x7F).max(axis=1)
    same = cmax > 0x76  # largest magnitude above 224
    assert np.array_equal(s1[same], s[same])
    assert np.array_equal(q1.reshape(-1, 32)[same], q.reshape(-1, 32)[same])
    moved = ~same & (s > 0) & (cmax > 0)
    assert moved.any() and np.all(cmax[moved] == 0x76) and np.array_equal(s1[moved], s[moved] - 1)
    # a hop onto +0 is the same requantization, except -0 + +0 = +0
    zeros = np.zeros(x.size, np.uint16)
    q2, s2, out2 = oracle.ring_hop_mx(q, s, zeros, materialize=True)
    assert np.array_equal(s2, s1)
    assert np.array_equal(q2, np.where(q1 == 0x80, 0, q1).astype(np.uint8))
    assert np.array_equal(out2, np.where(out1 == 0x8000, 0, out1).astype(np.uint16))


def test_e8m0_scale_over_fp32_amax_closed_form():
    # The MX reductions take the scale of binary32 sums, so the scale rule is pinned
    # over binary32 amax too: a stride through every positive finite binary32 pattern
    # plus the powers of two and their neighbours, against the frexp closed form.
    bits = np.concatenate([np.arange(1, 0x7F800000, 4099, dtype=np.uint32),
                           np.array([(k << 23) + d for k in range(1, 255) for d in (-1, 0, 1)], np.uint32),
                           np.arange(1, 64, dtype=np.uint32)])
    a = bits.view(np.float32)
    v = (a / np.float32(448.0)).astype(np.float32)
    m, k = np.frexp(v.astype(np.float64))
    expect = np.clip(np.where(v == 0, -127, np.where(m == 0.5, k - 1, k)) + 127, 0, 254)
    got = np.array([oracle.e8m0_scale(float(t)) for t in a], np.int64)
    assert np.array_equal(got, expect)


def test_e4m3_encode_of_fp32_values_at_and_around_every_tie():
    # binary32 inputs carry more bits than BF16: every midpoint between consecutive
    # E4M3 values, its binary32 neighbours, and random binary32 values, against the
    # nearest-value search (both signs).
    vals = [v for _, v in exact.e4m3_values()]
    pts = []
    for lo, hi in zip(vals, vals[1:]):
        mid = np.float32(float((lo + hi) / 2))
        pts += [mid, np.nextafter(mid, np.float32(0)), np.nextafter(mid, np.float32(1e9))]
    rng = np.random.default_rng(14)
    pts += list((rng.random(3000) * 470).astype(np.float32)) + list(np.float32(2.0) ** rng.uniform(-16, -8, 500).astype(np.float32))
    for y in pts:
        want = exact.e4m3_nearest(F(float(y)))
        assert oracle.e4m3_encode(float(y)) == want, float(y)
        assert oracle.e4m3_encode(-float(y)) == (want | 0x80), float(y)


# ------------------------------------------------------------------ legacy E4M3 codec
def _parse_e4m3_golden():
    cases, cur = [], None
    for line in open(os.path.join(GOLDEN, "e4m3_blocks.txt")):
        line = line.split("#", 1)[0].strip()
        if not line:
            continue
        key, _, val = line.partition(":")
        val = val.split()
        if key == "case":
            cur = {"name": val[0]}
            cases.append(cur)
        else:
            cur[key] = val
    return cases


@pytest.mark.parametrize("case", _parse_e4m3_golden(), ids=lambda c: c["name"])
def test_e4m3_golden_blocks(case):
    xs = [float(v) for v in case["x"]]
    block = np.zeros(128, np.uint16)
    block[: len(xs)] = _bf16_bits_of(xs)
    assert np.array_equal(_bits_to_f32(block[: len(xs)]), np.array(xs, np.float32))
    q, s = oracle.quant_e4m3(block)
    assert int(s.view(np.uint32)[0]) == int(case["scale_bits"][0], 16)
    assert [int(v) for v in q[: len(xs)]] == [int(c, 16) for c in case["codes"]]
    assert np.all(q[len(xs):] == 0)
    out = oracle.dequant_e4m3(q, s)
    assert [int(h, 16) for h in case["deq"]] == list(out[: len(xs)].astype(int))


def test_e4m3_amax_maps_to_448_for_every_bf16_amax():
    # Reading R14 with a BF16 amax a: s = fl(a / 448) (checked against numpy's binary32
    # division) and the element holding the amax encodes to +-448 (0x7e / 0xfe) for
    # every positive finite BF16 amax: fl(a / s) lies within 0.34% of 448 even where s
    # is a binary32 subnormal, and 448 is the nearest (or saturated) E4M3 value.
    a_bits = np.arange(1, 0x7F80, dtype=np.uint16)
    blocks = np.zeros((a_bits.size, 128), np.uint16)
    blocks[:, 0] = a_bits
    blocks[:, 77] = a_bits | 0x8000
    blocks[:, 5] = 0x8000
    q, s = oracle.quant_e4m3(blocks.reshape(-1))
    q = q.reshape(-1, 128)
    a = _bits_to_f32(a_bits)
    assert np.array_equal(s, (a / np.float32(448.0)).astype(np.float32))
    assert np.all(q[:, 0] == 0x7E) and np.all(q[:, 77] == 0xFE)
    assert np.all(q[:, 5] == 0x80)  # -0 in a non-zero block keeps its sign
    assert np.all(q[:, [1, 2, 3, 4, 6, 100]] == 0)


def test_e4m3_codec_brute_force_exact():
    rnd = random.Random(21)
    x = _adversarial_blocks(rnd, 16).reshape(-1)
    q, s = oracle.quant_e4m3(x)
    out = oracle.dequant_e4m3(q, s)
    for b in range(16):
        vals = [(exact.bits_to_value(int(v)), int(v) == 0x8000) for v in x[128 * b:128 * b + 128]]
        codes, sc = exact.quant_block_e4m3(vals)
        assert F(float(s[b])) == sc, b
        assert [int(c) for c in q[128 * b:128 * b + 128]] == codes, b
        assert [int(o) for o in out[128 * b:128 * b + 128]] == [exact.dequant_e4m3(c, sc) for c in codes], b


def test_e4m3_dequant_rounds_twice():
    # As for block INT8 (reading R3 applied by R14): decode(code) * s is rounded to
    # binary32, then to BF16. Search binary32 scales next to m / d for BF16 midpoints m
    # and E4M3 values d with more than one significant bit, where the two roundings
    # differ from one rounding of the exact product, and check the oracle rounds twice.
    found = 0
    vals = dict(exact.e4m3_values())
    for m in (1 + F(1, 256), 1 + F(3, 256), F(3, 2) + F(1, 128), 100 + F(1, 4)):
        for code in (0x39, 0x3B, 0x3D, 0x3F, 0x43, 0x47, 0x4D, 0x55):
            d = vals[code]
            centre = np.float32(float(m / d))
            cands = [centre]
            lo = hi = centre
            for _ in range(3):
                lo = np.nextafter(lo, np.float32(0), dtype=np.float32)
                hi = np.nextafter(hi, np.float32(np.inf), dtype=np.float32)
                cands += [lo, hi]
            for sc in cands:
                exact_prod = d * F(float(sc))
                once = exact.bf16_bits(exact.bf16(exact_prod))
                twice = exact.bf16_bits(exact.bf16(exact.f32(exact_prod)))
                if once != twice:
                    qq = np.zeros(128, np.uint8)
                    qq[0] = code
                    assert int(oracle.dequant_e4m3(qq, np.array([sc], np.float32))[0]) == twice
                    found += 1
    assert found >= 3


# ------------------------------------------------------------------ BF16 reduce + quantize
def test_reduce_quant_follows_rank_order_then_bf16_exact():
    # Reading R13: binary32 sum in rank order, one rounding to BF16, then the codec.
    rnd = random.Random(22)
    W = 4
    xs = [_adversarial_blocks(rnd, 6, max_abs=1.0e37).reshape(-1) for _ in range(W)]  # sums stay finite
    # block 0: big, tiny, -big, tiny (the order is visible); block 1: negative zeros
    xs[0][:128], xs[2][:128] = 0x4B80, 0xCB80  # +-2^24
    xs[1][:128], xs[3][:128] = 0x3F80, 0x3F80  # 1
    for w in range(W):
        xs[w][128:256] = 0x8000
    xs[1][130] = 0x0000
    qi, si, oi = oracle.reduce_quant_i8(xs, materialize=True)
    qe, se, oe = oracle.reduce_quant_e4m3(xs, materialize=True)
    for b in range(6):
        y = []
        for i in range(128):
            e = 128 * b + i
            a = (exact.bits_to_value(int(xs[0][e])), int(xs[0][e]) == 0x8000)
            for w in range(1, W):
                a = exact.f32_add_signed(a, (exact.bits_to_value(int(xs[w][e])), int(xs[w][e]) == 0x8000))
            y.append((exact.bf16(a[0]), a[1]))
        q_ref, s_ref = exact.quant_block_i8([v for v, _ in y])
        assert F(float(si[b])) == s_ref and list(qi[128 * b:128 * b + 128]) == q_ref, b
        c_ref, se_ref = exact.quant_block_e4m3(y)
        assert F(float(se[b])) == se_ref and [int(c) for c in qe[128 * b:128 * b + 128]] == c_ref, b
    # the order matters in block 0: ((2^24 + 1) - 2^24) + 1 = 1 in binary32 (2^24 + 1
    # rounds to 2^24), while (2^24 - 2^24) + (1 + 1) = 2
    d = [exact.bits_to_value(int(xs[w][0])) for w in range(W)]
    in_order = exact.f32(exact.f32(exact.f32(d[0] + d[1]) + d[2]) + d[3])
    regrouped = exact.f32(exact.f32(d[0] + d[2]) + exact.f32(d[1] + d[3]))
    assert in_order != regrouped
    # canonical forwarding
    assert np.array_equal(oi, oracle.dequant_i8(qi, si))
    assert np.array_equal(oe, oracle.dequant_e4m3(qe, se))


def test_reduce_quant_of_one_source_is_quantize():
    rnd = random.Random(23)
    x = _adversarial_blocks(rnd, 12).reshape(-1)
    qi, si, _ = oracle.reduce_quant_i8([x])
    q0, s0 = oracle.quant_i8(x)
    assert np.array_equal(qi, q0) and np.array_equal(si, s0)
    qe, se, _ = oracle.reduce_quant_e4m3([x])
    q1, s1 = oracle.quant_e4m3(x)
    assert np.array_equal(qe, q1) and np.array_equal(se, s1)


# ------------------------------------------------------------------ FP16 slices for MX
def test_f16_widening_exhaustive_vs_numpy():
    bits = np.arange(0, 0x10000, dtype=np.uint32)
    finite = ((bits >> 10) & 0x1F) != 0x1F
    bits = bits[finite].astype(np.uint16)
    want = bits.view(np.float16).astype(np.float32)
    got = np.array([oracle.f16_to_float(int(b)) for b in bits], np.float32)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def test_mx_f16_scale_exhaustive_over_fp16_amax():
    # every positive finite FP16 amax against the frexp closed form of fl(a / 448)
    a_bits = np.arange(1, 0x7C00, dtype=np.uint16)
    a = a_bits.view(np.float16).astype(np.float32)
    v = (a / np.float32(448.0)).astype(np.float32)
    m, k = np.frexp(v.astype(np.float64))
    expect = np.clip(np.where(m == 0.5, k - 1, k) + 127, 0, 254)
    ng = ((a_bits.size + 3) // 4) * 4
    groups = np.zeros((ng, 32), np.uint16)
    groups[: a_bits.size, 0] = a_bits
    groups[: a_bits.size, 9] = a_bits | 0x8000
    q, s = oracle.quant_mx(groups.reshape(-1, 128), fmt="f16")
    got = s.reshape(-1)[: a_bits.size]
    assert np.array_equal(got, expect.astype(np.uint8))
    codes = q.reshape(-1, 32)[: a_bits.size]
    y = a.astype(np.float64) * np.exp2(127.0 - got.astype(np.float64))
    assert np.all(y <= 448.0) and np.all(y > 224.0)  # FP16's range never reaches byte 0
    assert np.all((codes[:, 9] & 0x80) == 0x80)


def test_mx_f16_brute_force_exact():
    rng = np.random.default_rng(24)
    vals = (rng.standard_normal((8, 128)) * 10.0 ** rng.uniform(-6, 4, (8, 1))).astype(np.float16)
    vals[0, :8] = np.array([65504, -65504, 6e-8, -6e-8, 0.0, -0.0, 1.0, 0.5], np.float16)
    vals[1, :32] = np.float16(2.0 ** -24) * np.arange(32)
    x = vals.view(np.uint16)
    q, s = oracle.quant_mx(x, fmt="f16")
    for r in range(8):
        for g in range(4):
            vs = [exact.f16_value(int(b)) for b in x[r, 32 * g:32 * g + 32]]
            amax = max(abs(v) for v in vs)
            e = 127 if amax == 0 else exact.e8m0_up(exact.f32(amax / 448))
            assert s[r, g] == e
            for i, v in enumerate(vs):
                c = exact.e4m3_nearest(v * F(2) ** (127 - e))
                if v == 0 and x[r, 32 * g + i] & 0x8000:
                    c = 0x80
                assert q[r, 32 * g + i] == c


def test_mx_f16_staged_slices_equal_concatenated():
    rng = np.random.default_rng(25)
    slices = [(rng.standard_normal((16, 256)) * 30).astype(np.float16).view(np.uint16) for _ in range(3)]
    q_buf = np.zeros((16, 768), np.uint8)
    s_buf = np.zeros((16, 24), np.uint8)
    for i, sl in enumerate(slices):
        oracle.quant_mx_into(sl, q_buf, s_buf, 256 * i, fmt="f16")
    q, s = oracle.quant_mx(np.concatenate(slices, axis=1), fmt="f16")
    assert np.array_equal(q_buf, q) and np.array_equal(s_buf, s)


# ------------------------------------------------------------------ tiled scale layout
# The staged-input page ("[II] Support staged MXFP8 linear inputs", Behavior) has
# empty_input allocate "MXFP8 values and scale layouts" for its GEMM but prints no
# layout. The oracle's tiled layout is pinned to an independent statement of the
# layout that Blackwell block-scaled GEMMs read: PyTorch's own test helpers
# `to_blocked` (tile rearrangement by reshapes, citing cuBLAS's "1D block scaling
# factors layout") and `from_blocked` (the per-element offset formula of the same
# cuBLAS section, written as loops). They live in a torch test module whose import
# needs test-only packages, so the two functions are parsed out of the installed file
# and executed on their own; nothing of them is copied here.
def _torch_block_layout():
    import ast
    path = os.path.join(os.path.dirname(torch.__file__), "testing", "_internal", "common_quantized.py")
    if not os.path.exists(path):
        pytest.skip("this torch build does not ship common_quantized.py")
    tree = ast.parse(open(path).read(), path)
    want = {"ceil_div", "to_blocked", "from_blocked"}
    funcs = [n for n in tree.body if isinstance(n, ast.FunctionDef) and n.name in want]
    if {f.name for f in funcs} != want:
        pytest.skip("torch's common_quantized.py has no to_blocked/from_blocked")
    ns = {"torch": torch, "Tensor": torch.Tensor}
    exec(compile(ast.Module(body=funcs, type_ignores=[]), path, "exec"), ns)
    return ns["to_blocked"], ns["from_blocked"]


def _torch_to_mxfp():
    import ast
    path = os.path.join(os.path.dirname(torch.__file__), "testing", "_internal", "common_quantized.py")
    if not os.path.exists(path) or not hasattr(torch, "float8_e8m0fnu"):
        pytest.skip("this torch build has no MX reference")
    tree = ast.parse(open(path).read(), path)
    funcs = [n for n in tree.body if isinstance(n, ast.FunctionDef) and n.name == "to_mxfp"]
    if not funcs:
        pytest.skip("torch's common_quantized.py has no to_mxfp")
    ns = {"torch": torch}
    exec(compile(ast.Module(body=funcs, type_ignores=[]), path, "exec"), ns)
    return ns["to_mxfp"]


def test_mx_quant_equals_torch_to_mxfp():
    # PyTorch's MXFP8 reference for its block-scaled GEMM tests (to_mxfp, "RCEIL") states
    # the same rule independently: E8M0 = ceil(log2(fl(amax/448))) + 127, elements
    # x * 2^(127 - E8M0) saturated to +-448 and cast to E4M3 with ties to even. Its
    # readings differ only where this test does not go: an all-zero group gets E8M0 0
    # there (127 by the pages' rule), and groups with amax/448 below 2^-127 are clamped.
    # Magnitudes per group span 2^-100 .. 2^100; a BF16 amax is never close enough above
    # a power of two for its float32 log2 to round to the power itself.
    to_mxfp = _torch_to_mxfp()
    rng = np.random.default_rng(61)
    rows, cols = 96, 2048
    mag = np.exp2(rng.integers(-100, 101, size=(rows, cols // 32))).repeat(32, axis=1)
    v = rng.standard_normal((rows, cols)) * mag
    v[0, :32] = 448.0 * np.exp2(np.arange(32) % 5 - 2)  # amax exactly 448 * 2^k
    v[1, :32] = np.where(np.arange(32) == 7, 1.0e4, rng.standard_normal(32))  # one outlier
    xt = torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16)
    xb = xt.view(torch.int16).numpy().view(np.uint16)
    scale_t, data_t = to_mxfp(xt, 32, "mxfp8")
    q, sc = oracle.quant_mx(xb)
    assert np.array_equal(sc, scale_t.view(torch.uint8).numpy())
    assert np.array_equal(q, data_t.view(torch.uint8).numpy())


@pytest.mark.parametrize("rows,g", [(128, 4), (128, 224), (200, 8), (200, 224), (4096, 4), (4096, 224),
                                    (4096, 1344), (257, 1344)])
def test_mx_tiled_scale_layout_equals_torch_to_blocked(rows, g):
    to_blocked, _ = _torch_block_layout()
    rng = np.random.default_rng(rows * 7919 + g)
    s = rng.integers(0, 256, size=(rows, g), dtype=np.uint8)
    want = to_blocked(torch.from_numpy(s)).numpy()
    got = oracle.mx_scales_to_tiled(s, fill=0)  # to_blocked pads with zeros
    assert got.shape == want.shape
    assert np.array_equal(got, want)


def test_mx_tiled_scale_layout_inverts_torch_from_blocked():
    _, from_blocked = _torch_block_layout()
    rng = np.random.default_rng(31)
    for rows, g in [(200, 8), (256, 12)]:
        s = rng.integers(0, 256, size=(rows, g), dtype=np.uint8)
        tiled = torch.from_numpy(oracle.mx_scales_to_tiled(s))
        shape_only = torch.empty((rows, 32 * g), dtype=torch.uint8)
        back = from_blocked(shape_only, tiled, 32).numpy()
        assert np.array_equal(back, s)


def test_mx_tiled_scale_positions_of_staged_slices():
    # The staged workload: six 4096 x 7168 slices at scale-column offsets 224 i of one
    # 4096 x 1344 scale matrix. Every (row, column) of every slice must land where
    # to_blocked puts it; the element's index is carried through the oracle's layout
    # in three byte planes and compared with to_blocked of the index matrix.
    to_blocked, _ = _torch_block_layout()
    rows, g_total, g_slice = 4096, 1344, 224
    idx = np.arange(rows * g_total, dtype=np.int64).reshape(rows, g_total)
    want = to_blocked(torch.from_numpy(idx.astype(np.int32))).numpy().astype(np.int64)
    got = np.zeros(want.shape, np.int64)
    for b in range(3):
        plane = ((idx >> (8 * b)) & 0xFF).astype(np.uint8)
        got |= oracle.mx_scales_to_tiled(plane).astype(np.int64) << (8 * b)
    assert np.array_equal(got, want)
    # and the oracle's per-element offset agrees for sampled elements of each slice
    rng = np.random.default_rng(32)
    where = np.empty(want.size, np.int64)
    where[want] = np.arange(want.size)
    for i in range(6):
        for r, c in zip(rng.integers(0, rows, 64), rng.integers(g_slice * i, g_slice * (i + 1), 64)):
            assert oracle.mx_tiled_scale_offset(int(r), int(c), g_total) == where[r * g_total + c]


# ------------------------------------------------------------------ staged == concatenated
def test_staged_slices_equal_concatenated():
    # "[II] Support staged MXFP8 linear inputs": quantizing 128-column-aligned slices
    # into column offsets of one buffer gives bitwise the result of quantizing the
    # concatenation (Validation: staged and concatenated outputs are bitwise equal).
    rng = np.random.default_rng(12)
    rows, widths = 24, [128, 256, 384, 128]
    slices = []
    for w in widths:
        xf = (rng.standard_normal((rows, w)) * 0.02).astype(np.float32)
        xf[rng.random(xf.shape) < 0.01] *= 100
        slices.append(torch.from_numpy(xf).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16))
    cat = np.concatenate(slices, axis=1)
    q_ref, s_ref = oracle.quant_mx(cat)
    C = cat.shape[1]
    q_buf = np.full((rows, C), 0xAA, np.uint8)
    s_buf = np.full((rows, C // 32), 0xAA, np.uint8)
    col = 0
    for sl in slices:
        oracle.quant_mx_into(sl, q_buf, s_buf, col)
        col += sl.shape[1]
    assert np.array_equal(q_buf, q_ref)
    assert np.array_equal(s_buf, s_ref)
    with pytest.raises(ValueError):
        oracle.quant_mx_into(slices[0], q_buf, s_buf, 64)


# ------------------------------------------------------------------ canonical forwarding
def test_ring_chain_owner_and_replicas_identical():
    # "Owners materialize their shard from the same final wire payload forwarded to
    # peers": every simulated rank materializes the final payload identically, and the
    # owner's fused output equals the materialization of that payload.
    rng = np.random.default_rng(21)
    W, n = 4, 128 * 16
    xs = [torch.from_numpy(rng.standard_normal(n).astype(np.float32)).to(torch.bfloat16)
          .view(torch.int16).numpy().view(np.uint16) for _ in range(W)]
    q, s = oracle.quant_i8(xs[1])
    for w in (2, 3):
        q, s, _ = oracle.ring_hop_i8(q, s, xs[w])
    q, s, owner = oracle.ring_hop_i8(q, s, xs[0], materialize=True)
    replicas = [oracle.dequant_i8(q, s) for _ in range(W)]
    for r in replicas:
        assert np.array_equal(r, owner)
    # error against the exact BF16 sum stays within the chained half-step bounds
    total = sum(_bits_to_f32(x).astype(np.float64) for x in xs)
    err = np.abs(_bits_to_f32(owner).astype(np.float64) - total)
    assert err.max() < 0.25
