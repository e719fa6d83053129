"""The debug build stays inside its buffers and changes no result.

libbq_debug.so is the same sources compiled with BQ_DEBUG=1. There, every kernel lists
the byte ranges of the buffers its arguments describe (inputs read-only, outputs
writable). Every global load, store and bulk copy is then checked against them; an access
outside them is not performed and is counted. This module reruns parity tests through
that build, covering every kernel family, ragged sizes, every source count, strided and
staged MX, 4-byte-aligned scales, and sizes where every warp walks several chunks. The results must stay bit-exact and the count of
declined accesses must stay 0. A self-test shows that an access outside the listed
ranges is declined and counted, without it touching memory.
"""
import pytest
import torch

import oracle
from block_quantized_wire_gb300 import _lib, build, codec
from block_quantized_wire_gb300._lib import BQError
from tests import test_gpu_i8 as t8
from tests import test_gpu_mx as tx
from tests import test_gpu_mx_wire as tw
from tests import test_gpu_next_rows as tn
from tests import test_gpu_multipass as tm
from tests import test_gpu_properties as tp

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dbg(bq_lib):
    return build.build_debug_library()


def test_declined_access_is_counted_not_performed(dbg):
    buf = torch.zeros(1024, dtype=torch.uint8, device="cuda")
    buf[:16] = 9
    buf[512:528] = 7
    with _lib.use_library(dbg):
        assert codec.debug_build()
        codec.take_index_errors()
        codec.selftest_index_check(buf)
        torch.cuda.synchronize()
        assert codec.take_index_errors() == 1
        assert codec.take_index_errors() == 0
    # the load at byte 512 lay outside the listed 256 bytes: it was declined and yielded
    # zeros, which the store inside the listed range then wrote
    assert bool((buf[:16] == 0).all()) and bool((buf[512:528] == 7).all())
    # the default build has no checks: it refuses the self-test before any launch
    assert not codec.debug_build()
    with pytest.raises(BQError) as e:
        codec.selftest_index_check(buf)
    assert e.value.status == 6
    assert codec.take_index_errors() == 0


def _no_declined_access():
    torch.cuda.synchronize()
    return codec.take_index_errors() == 0


def test_int8_kernels_stay_in_bounds(dbg):
    with _lib.use_library(dbg):
        codec.take_index_errors()
        for nblk in (1, 7, 9, 65, 1001):
            t8.test_ragged_sizes_quant_dequant(nblk)
        for W in (1, 2, 3, 4, 5, 16):
            for owner in (True, False):
                for nblk in (37, 8, 1):
                    t8.test_accumulate_any_width(W, owner, nblk)
        for nblk in (200, 45):
            for owner in (True, False):
                t8.test_ring_hop_edge_cases(nblk, owner)
        t8.test_accumulate_with_scales_not_16_byte_aligned()
        t8.test_ring_hop_with_scales_not_16_byte_aligned()
        t8.test_bf16_pointers_aligned_to_16_but_not_32_bytes()
        t8.test_tiny_scale_blocks_across_the_exact_division_cutoff()
        t8.test_a2a_3072_bitexact()
        assert _no_declined_access()


def test_mx_kernels_stay_in_bounds(dbg):
    with _lib.use_library(dbg):
        codec.take_index_errors()
        tx.test_mixed_3072_mx_bitexact()
        tx.test_strided_shapes(17, 384, 24, 48, 12)
        tx.test_strided_shapes(64, 128, 128, 0, 60)
        tx.test_staged_slices_4096_bitexact_and_equal_to_concatenated()
        tx.test_slices_in_one_call_ragged_widths(torch.bfloat16)
        tx.test_slices_in_one_call_sixteen_narrow_slices_and_an_empty_one()
        tn.test_mx_f16_every_value_and_ragged_rows()
        tn.test_mx_tiled_scales_staged_slices(torch.float16)
        for nblk in (1, 9, 65, 1029):
            tw.test_mx_ragged_sizes(nblk)
        for W in (1, 4, 5, 16):
            for owner in (True, False):
                tw.test_mx_accumulate_any_width(W, owner, 37)
        tw.test_mx_reductions_with_scales_not_16_byte_aligned()
        tw.test_mx_bf16_pointers_aligned_to_16_but_not_32_bytes()
        tw.test_mx_ring_chain_bitexact()
        assert _no_declined_access()


def test_allgather_and_e4m3_kernels_stay_in_bounds(dbg):
    with _lib.use_library(dbg):
        codec.take_index_errors()
        for name in list(tn.CODECS):
            for nblk in (1, 9, 65, 1027):
                tn.test_reduce_quant_ragged(name, nblk)
            for W in (1, 5, 16):
                tn.test_reduce_quant_any_width(name, W)
        for nblk in (1, 17, 1001):
            tn.test_e4m3_ragged_and_adversarial(nblk)
        tn.test_e4m3_input_aligned_to_16_but_not_32_bytes()
        tn.test_e4m3_scales_across_the_exact_division_cutoff()
        tp.test_fused_owner_output_equals_separate_materialization()
        assert _no_declined_access()


def test_multipass_kernels_stay_in_bounds(dbg):
    # every warp several chunks deep: the async copy stages refilled, the grid-stride
    # loops of the one-CTA-per-SM launches past their first pass, then a ragged tail
    nblk = tm.multipass_nblk()
    xs = [tm.source_bits(900 + i, nblk) for i in range(4)]
    sources = (nblk, xs, [oracle.quant_i8(x) for x in xs])
    with _lib.use_library(dbg):
        codec.take_index_errors()
        tm.test_quant_dequant_multipass(sources)
        tm.test_ring_hop_multipass(sources, True)
        for W in (1, 4):
            tm.test_accumulate_multipass(sources, W, False)
        for name in ("i8", "e4m3"):
            tm.test_reduce_quant_multipass(sources, name, 4, False)
        tm.test_e4m3_quant_dequant_multipass(sources)
        tm.test_mx_accumulate_multipass(4)
        assert _no_declined_access()
