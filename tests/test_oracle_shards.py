"""The shard runner the full-size parity test and the CPU baseline use: oracle calls on
contiguous row ranges, run in host threads, give exactly the bytes of one call on the
whole input (every block and MX group depends on its own values only), and the ranges
cover every row once."""
import numpy as np
import pytest
import torch

import oracle
from block_quantized_wire_gb300.inputs import bf16_bits
from oracle import shards

H = 7168


@pytest.mark.parametrize("rows,parts", [(0, 4), (1, 4), (7, 3), (16, 16), (100, 7), (5, 1)])
def test_row_ranges_cover_every_row_once(rows, parts):
    rr = shards.row_ranges(rows, parts)
    assert len(rr) == min(rows, max(1, parts))
    seen = []
    for lo, hi in rr:
        assert hi > lo
        seen.extend(range(lo, hi))
    assert seen == list(range(rows))
    if rr:
        sizes = [hi - lo for lo, hi in rr]
        assert max(sizes) - min(sizes) <= 1


def test_run_returns_in_order_and_raises():
    assert shards.run(lambda lo, hi: (lo, hi), 10, 4) == shards.row_ranges(10, 4)
    assert shards.run(lambda lo, hi: (lo, hi), 50, 3, parts=9) == shards.row_ranges(50, 9)
    with pytest.raises(ZeroDivisionError):
        shards.run(lambda lo, hi: 1 // (lo - 3) if lo == 3 else 0, 12, 4)


def _bits(rows, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(rows, H, generator=g) * torch.exp(torch.randn(rows, 1, generator=g))
    x[rows // 2] = 0.0
    return bf16_bits(x.to(torch.bfloat16)).reshape(rows, H)


def _sharded(fn, arrays, rows, parts):
    outs = shards.run(lambda lo, hi: fn(*[a[lo:hi] for a in arrays]), rows, parts)
    return [np.concatenate([o[k].reshape(hi - lo, -1) for o, (lo, hi) in zip(outs, shards.row_ranges(rows, parts))])
            for k in range(len(outs[0]))]


def test_sharded_int8_calls_equal_one_call():
    rows = 13
    xs = [_bits(rows, 70 + w) for w in range(3)]
    whole_q = [oracle.quant_i8(x.reshape(-1)) for x in xs]
    for parts in (2, 5):
        for x, (q, s) in zip(xs, whole_q):
            sq, ss = _sharded(lambda a: oracle.quant_i8(a.reshape(-1)), [x], rows, parts)
            assert np.array_equal(sq.reshape(-1), q) and np.array_equal(ss.reshape(-1), s)
    qs = [q.reshape(rows, H) for q, _ in whole_q]
    ss_ = [s.reshape(rows, H // 128) for _, s in whole_q]
    qa, sa, oa = oracle.dequant_accum_i8([q for q, _ in whole_q], [s for _, s in whole_q])
    got = _sharded(lambda *a: oracle.dequant_accum_i8([v.reshape(-1) for v in a[:3]], [v.reshape(-1) for v in a[3:]]),
                   qs + ss_, rows, 4)
    for g, w in zip(got, (qa, sa, oa)):
        assert np.array_equal(g.reshape(-1), w)
    hq, hs, ho = oracle.ring_hop_i8(whole_q[0][0], whole_q[0][1], xs[1].reshape(-1), materialize=True)
    got = _sharded(lambda q, s, x: oracle.ring_hop_i8(q.reshape(-1), s.reshape(-1), x.reshape(-1), materialize=True),
                   [qs[0], ss_[0], xs[1]], rows, 3)
    for g, w in zip(got, (hq, hs, ho)):
        assert np.array_equal(g.reshape(-1), w)


def test_sharded_mx_calls_equal_one_call():
    rows = 11
    x = _bits(rows, 80)
    q, s = oracle.quant_mx(x)
    gq, gs = _sharded(lambda a: oracle.quant_mx(a), [x], rows, 4)
    assert np.array_equal(gq, q) and np.array_equal(gs, s)
    (out,) = _sharded(lambda a, b: (oracle.dequant_mx(a, b),), [q, s], rows, 3)
    assert np.array_equal(out, oracle.dequant_mx(q, s))
