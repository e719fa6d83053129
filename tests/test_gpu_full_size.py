"""Whole-tensor parity at full size, in the launch configuration the benchmark times.

The benchmark's own step (four 65536x7168 BF16 buffers through quant_i8 x4,
dequant_accum_i8 (W=4), dequant_i8 and ring_hop_i8; six 4096x7168 slices staged by
quant_mx into one 4096x43008 buffer, then dequant_mx) runs once on the GPU. Then the
oracle recomputes every output byte from the same BF16 input bits. It runs on row
ranges in host threads (blocks are independent, so the bytes are those of one call),
and the oracle chains its own results: it never sees a value the GPU produced. Every
payload byte, scale word and BF16 output is compared. Each range copies only its own
rows from the device, which bounds host memory.
"""
import pytest
import torch

import bench
from oracle import shards
from tests.step_check import compare_step

pytestmark = pytest.mark.gpu

ROWS, SLICE_ROWS = 65536, 4096  # the benchmark's buffers and slices


@pytest.fixture(scope="module", autouse=True)
def _lib(bq_lib):
    return bq_lib


def test_prefill_step_whole_tensors_bitexact():
    torch.cuda.empty_cache()
    pipe = bench.Pipeline(ROWS, SLICE_ROWS, torch.device("cuda"))
    pipe.run()
    torch.cuda.synchronize()
    # 1024-row ranges: about 0.2 GB of host memory per thread at a time
    errs = compare_step(pipe, shards.host_cores())
    assert not errs, "\n".join(errs[:20])
