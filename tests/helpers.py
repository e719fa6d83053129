"""Small helpers shared by the tests: bit views between torch and numpy, guarded
allocations, and adversarial BF16 blocks. No codec arithmetic lives here."""
from __future__ import annotations

import numpy as np
import torch


def bits(t: torch.Tensor) -> np.ndarray:
    """Raw bit patterns of a tensor as a host numpy array (BF16 -> uint16, int8, float32, uint8)."""
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def from_bits_bf16(b: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).to(device)


def bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32)


def bf16_of(values, device="cpu") -> torch.Tensor:
    return torch.as_tensor(np.asarray(values, np.float32)).to(torch.bfloat16).to(device)


class Guarded:
    """A device buffer with sentinel bands on both sides of the usable region."""

    BAND = 4096
    SENTINEL = 0xA5

    def __init__(self, nbytes: int, device="cuda"):
        self.raw = torch.full((nbytes + 2 * self.BAND,), self.SENTINEL, dtype=torch.uint8, device=device)
        self.nbytes = nbytes

    def view(self, dtype: torch.dtype, shape=None) -> torch.Tensor:
        t = self.raw[self.BAND:self.BAND + self.nbytes].view(dtype)
        return t.view(shape) if shape is not None else t

    def bands_intact(self) -> bool:
        lo = self.raw[: self.BAND]
        hi = self.raw[self.BAND + self.nbytes:]
        return bool((lo == self.SENTINEL).all().item() and (hi == self.SENTINEL).all().item())


def adversarial_blocks(rng: np.random.Generator, nblk: int, max_abs: float = 3.3e38) -> np.ndarray:
    """BF16 bit patterns [nblk, 128]: normal, wide-range, outlier, subnormal, tie-heavy,
    near-maximum, negative-zero and all-zero blocks; magnitudes clipped to max_abs so
    that callers summing several of them can keep FP32 sums finite."""
    out = np.zeros((nblk, 128), np.float32)
    for b in range(nblk):
        kind = b % 9
        if kind == 0:
            v = rng.standard_normal(128)
        elif kind == 1:
            v = rng.standard_normal(128) * 10.0 ** rng.uniform(-35, 35)
        elif kind == 2:
            v = rng.standard_normal(128)
            v[rng.integers(128)] *= 1e4
        elif kind == 3:
            v = rng.standard_normal(128) * 2.0 ** rng.integers(-133, -120)
        elif kind == 4:
            p = 2.0 ** rng.integers(-30, 30)
            v = (rng.integers(-127, 127, 128) + 0.5) * p
            v[0] = 127 * p
        elif kind == 5:
            v = rng.choice([3.3e38, -3.3e38, 1.0e38, 2.0 ** -133, 0.0], 128)
        elif kind == 6:
            v = np.full(128, -0.0)
        elif kind == 7:
            v = np.zeros(128)
        else:
            v = rng.choice([0.0, 1.0, -1.0, 0.5, -0.5, 1.5, 127.0], 128) * 2.0 ** rng.integers(-10, 10)
        out[b] = np.clip(v, -max_abs, max_abs)
    t = torch.from_numpy(out).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def near_half_blocks(rng: np.random.Generator, nblk: int) -> np.ndarray:
    """Blocks whose quotients x / fl(amax/127) lie within 2^-13 of a half-integer but are
    not exact ties: they exercise the exact-division path of a reciprocal-based kernel."""
    blocks = np.zeros((nblk, 128), np.uint16)
    all_pos = np.arange(1, 0x7F80, dtype=np.uint32)
    vals = (all_pos << 16).view(np.float32).astype(np.float64)
    for b in range(nblk):
        while True:
            amax_bits = np.uint16(rng.integers(0x3C00, 0x4400))
            amax = float((np.uint32(amax_bits) << 16).view(np.float32))
            s = float(np.float32(np.float32(amax) / np.float32(127)))
            r = vals / s
            f = np.abs(r - np.floor(r) - 0.5)
            sel = np.nonzero((vals < amax) & (f < 2.0 ** -13) & (f > 0))[0]
            if sel.size >= 1:
                break
        pick = rng.choice(sel, size=127, replace=True)
        row = (all_pos[pick]).astype(np.uint16)
        signs = rng.integers(0, 2, 127).astype(np.uint16) << 15
        blocks[b, 0] = amax_bits
        blocks[b, 1:] = row | signs
    return blocks
