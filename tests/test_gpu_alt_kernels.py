"""The compile-time alternatives of the measured default kernels stay bit-exact.

The defaults were chosen by measurement: 16 values per lane for the INT8 quantize,
accumulate and ring hop and the MX wire reductions, 256-bit BF16 accesses, and direct
loads in the hops. The alternatives (8 values per lane; bulk-copy-staged hops with
their bounded mbarrier waits; 16-byte accesses only) remain in the sources as the
baseline of those measurements. This module builds them into libbq_alt.so and reruns
the parity tests that reach them through it.

libbq_direct.so holds the other measured alternatives: direct loads instead of the
per-lane async copies in the accumulates and the fused reduce, and 256-thread CTAs
instead of one CTA per SM. The multipass and small-size parity tests rerun through it.
"""
import pytest

import oracle
from block_quantized_wire_gb300 import _lib, build
from tests import test_gpu_i8 as t8
from tests import test_gpu_multipass as tmp
from tests import test_gpu_mx_wire as tm
from tests import test_gpu_next_rows as tn
from tests import test_gpu_properties as tp

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def alt(bq_lib):
    return build.build_alt_library()


def test_alt_int8_kernels(alt):
    with _lib.use_library(alt):
        for nblk in (1, 7, 9, 1001):
            t8.test_ragged_sizes_quant_dequant(nblk)
        for W in (1, 2, 3, 4, 5, 9):
            for owner in (True, False):
                for nblk in (37, 8, 1):
                    t8.test_accumulate_any_width(W, owner, nblk)
        t8.test_accumulate_repeated_source_and_tiny_sums()
        t8.test_near_half_quotients_take_exact_path()
        t8.test_tiny_scale_blocks_across_the_exact_division_cutoff()
        for nblk in (200, 45):
            for owner in (True, False):
                t8.test_ring_hop_edge_cases(nblk, owner)
        t8.test_accumulate_with_scales_not_16_byte_aligned()
        t8.test_ring_hop_with_scales_not_16_byte_aligned()
        t8.test_bf16_pointers_aligned_to_16_but_not_32_bytes()
        t8.test_a2a_3072_bitexact()
        t8.test_ring_16384_chain_bitexact()


def test_alt_mx_wire_kernels(alt):
    with _lib.use_library(alt):
        for W in (1, 4, 5):
            for owner in (True, False):
                for nblk in (37, 8, 1):
                    tm.test_mx_accumulate_any_width(W, owner, nblk)
        tm.test_mx_accumulate_tiny_and_cancelling_sums()
        tm.test_mx_reductions_with_scales_not_16_byte_aligned()
        tm.test_mx_hop_cancellation_and_negative_zero()
        tm.test_mx_bf16_pointers_aligned_to_16_but_not_32_bytes()
        tm.test_mx_a2a_bitexact()
        tm.test_mx_ring_chain_bitexact()


def test_alt_staged_hops_leave_no_abandoned_wait(alt):
    with _lib.use_library(alt):
        tp.test_bounded_waits_do_not_run_out_and_can_be_observed()
        tp.test_fused_owner_output_equals_separate_materialization()


@pytest.fixture(scope="module")
def direct(bq_lib):
    return build.build_direct_library()


def test_direct_loads_and_small_ctas(direct):
    nblk = tmp.multipass_nblk()
    xs = [tmp.source_bits(900 + i, nblk) for i in range(4)]
    sources = (nblk, xs, [oracle.quant_i8(x) for x in xs])
    with _lib.use_library(direct):
        tmp.test_quant_dequant_multipass(sources)
        for owner in (False, True):
            tmp.test_ring_hop_multipass(sources, owner)
        for W in (1, 4):
            tmp.test_accumulate_multipass(sources, W, False)
        for name in ("i8", "e4m3"):
            tmp.test_reduce_quant_multipass(sources, name, 4, False)
        tmp.test_e4m3_quant_dequant_multipass(sources)
        tmp.test_mx_accumulate_multipass(4)
        for W in (1, 2, 3, 4):
            for nblk_small in (37, 8, 1):
                t8.test_accumulate_any_width(W, False, nblk_small)
                tm.test_mx_accumulate_any_width(W, False, nblk_small)
        for name in list(tn.CODECS):
            for nblk_small in (1, 9, 65):
                tn.test_reduce_quant_ragged(name, nblk_small)
