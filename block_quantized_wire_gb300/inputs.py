"""Seeded synthetic inputs for the codec workloads.

This module only draws random BF16 tensors with the shapes, value distributions and
structure of the workloads the codec is measured on. It holds none of the codec's
arithmetic, and it is the one module that both the CUDA path's tests/benchmark and
the CPU oracle's callers use.

Recipe (fixed seeds; every tensor is drawn in FP32, given its structure in FP32, then
rounded once to BF16):

* ``roundtrip_512``   512 x 7168, N(0,1), seed 1001. Of its 28,672 128-value blocks
  (a random permutation), the first 573 (2%) are set to zero and the next 287 (1%)
  get one element, at a random position, multiplied by 100.
* ``mixed_3072``      3072 x 7168, N(0,1), seed 2001. Every row is multiplied by a
  lognormal(0,1) factor, then each element independently with probability 0.005 is
  multiplied by 1000, then 31 random rows (1%) are set to zero.
* ``a2a_3072``        W = 4 sources of 3072 x 7168, N(0,1), seeds 3001..3004.
* ``ring_16384``      W = 4 buffers of 16384 x 7168, N(0,1), seeds 4001..4004.
* ``prefill_65536``   W = 4 buffers of 65536 x 7168, 0.02 * N(0,1), seeds 5001..5004;
  each element independently with probability 0.001 is multiplied by 100.
* ``mx_slices_4096``  six slices of 4096 x 7168, 0.02 * N(0,1) with the same 0.1% x100
  outliers, seeds 5101..5106, quantized into one 4096 x 43008 MXFP8 buffer.

The hidden width 7168 and the row counts 512 and 3072 are the projection geometry
and the validation row counts of the pages ("[II] Support staged MXFP8 linear
inputs", Validation; "feat(pcie_dma): add block-INT8 wire modes for AG, ring, and
A2A", Evidence and validation status). The pages' activations come from serving
real models whose weights are not available, so these draws stand in for them.

``device`` selects the generator: a CPU generator gives the same bits on every run of
one machine; a CUDA generator (used for the largest workload, where CPU drawing is
slow) gives the same bits on every run of one GPU type. Either way, the tests and the
oracle consume the very bits that the CUDA path consumes.
"""
from __future__ import annotations

import torch

HIDDEN = 7168
W_SOURCES = 4

WORKLOADS = ("roundtrip_512", "mixed_3072", "a2a_3072", "ring_16384", "prefill_65536", "mx_slices_4096")


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def randn_bf16(shape, seed: int, std: float = 1.0, device="cpu") -> torch.Tensor:
    """std * N(0,1) drawn in FP32 and rounded once to BF16."""
    g = _gen(seed, device)
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(torch.bfloat16)


def _with_outliers(x: torch.Tensor, g: torch.Generator, p: float, factor: float) -> torch.Tensor:
    mask = torch.rand(x.shape, generator=g, device=x.device) < p
    return torch.where(mask, x * factor, x)


def roundtrip_512(device="cpu", rows: int = 512, cols: int = HIDDEN, seed: int = 1001) -> torch.Tensor:
    g = _gen(seed, device)
    x = torch.randn((rows, cols), generator=g, device=device, dtype=torch.float32)
    blocks = x.view(-1, 128)
    nb = blocks.shape[0]
    perm = torch.randperm(nb, generator=g, device=device)
    n_zero = int(round(nb * 0.02))
    n_out = int(round(nb * 0.01))
    blocks[perm[:n_zero]] = 0.0
    rows_out = perm[n_zero:n_zero + n_out]
    pos = torch.randint(0, 128, (n_out,), generator=g, device=device)
    blocks[rows_out, pos] *= 100.0
    return x.to(torch.bfloat16)


def mixed_3072(device="cpu", rows: int = 3072, cols: int = HIDDEN, seed: int = 2001) -> torch.Tensor:
    g = _gen(seed, device)
    x = torch.randn((rows, cols), generator=g, device=device, dtype=torch.float32)
    row_scale = torch.exp(torch.randn((rows, 1), generator=g, device=device, dtype=torch.float32))
    x = x * row_scale
    x = _with_outliers(x, g, 0.005, 1000.0)
    zero_rows = torch.randperm(rows, generator=g, device=device)[: max(1, int(round(rows * 0.01)))]
    x[zero_rows] = 0.0
    return x.to(torch.bfloat16)


def a2a_3072(device="cpu", rows: int = 3072, cols: int = HIDDEN, W: int = W_SOURCES, seed0: int = 3001):
    return [randn_bf16((rows, cols), seed0 + w, device=device) for w in range(W)]


def ring_16384(device="cpu", rows: int = 16384, cols: int = HIDDEN, W: int = W_SOURCES, seed0: int = 4001):
    return [randn_bf16((rows, cols), seed0 + w, device=device) for w in range(W)]


def prefill_buffer(w: int, device="cuda", rows: int = 65536, cols: int = HIDDEN, seed0: int = 5001):
    g = _gen(seed0 + w, device)
    x = torch.randn((rows, cols), generator=g, device=device, dtype=torch.float32).mul_(0.02)
    mask = torch.rand((rows, cols), generator=g, device=device) < 0.001
    x[mask] *= 100.0
    del mask
    return x.to(torch.bfloat16)


def prefill_65536(device="cuda", rows: int = 65536, cols: int = HIDDEN, W: int = W_SOURCES, seed0: int = 5001):
    return [prefill_buffer(w, device, rows, cols, seed0) for w in range(W)]


def mx_slices_4096(device="cuda", rows: int = 4096, cols: int = HIDDEN, n_slices: int = 6, seed0: int = 5101,
                   dtype: torch.dtype = torch.bfloat16):
    """The staged MX slices; dtype torch.float16 gives the FP16 slices the staged-input
    page also accepts (the same FP32 draws, rounded once to FP16; they stay far inside
    the FP16 range)."""
    out = []
    for i in range(n_slices):
        g = _gen(seed0 + i, device)
        x = torch.randn((rows, cols), generator=g, device=device, dtype=torch.float32).mul_(0.02)
        x = _with_outliers(x, g, 0.001, 100.0)
        out.append(x.to(dtype))
    return out


def bf16_bits(t: torch.Tensor):
    """The uint16 bit patterns of a BF16 tensor, as a host numpy array."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view("uint16")
