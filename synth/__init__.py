"""Seeded synthetic inputs shared by the oracle side and the CUDA side.

This module holds only random-number generation: no operation of the
streaming path (scale, row shift, polynomial, cluster hand-off) is computed
here, so that the oracle and the CUDA path can both be fed the same bytes
without sharing any of the method's arithmetic.

Generator (counter based, so any element can be regenerated on its own):

    z_i = splitmix64(seed XOR i)
    k_i = z_i >> 40                      (a 24-bit integer, 0 <= k_i < 2**24)
    x_i = (k_i - 2**23) * 2**-23         (uniform on the grid [-1, 1), float32)
    c_i = (k_i - 2**23) * 2**-24         (uniform on the grid [-0.5, 0.5))

splitmix64 is the output function of Steele, Lea and Flood's SplittableRandom
("Fast splittable pseudorandom number generators", OOPSLA 2014) with the
mixing constants of Stafford's "Mix13" variant, as used by Vigna's public
splitmix64 generator:

    z += 0x9E3779B97F4A7C15
    z  = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9
    z  = (z ^ (z >> 27)) * 0x94D049BB133111EB
    z  =  z ^ (z >> 31)

Every value on the grid is an exact float32 (a 24-bit integer times a power of
two), with no subnormals, so the host (numpy) and device (torch) versions give
identical bits.
"""

from __future__ import annotations

import numpy as np

__all__ = [
    "SEED_ROLL_SMALL",
    "SEED_SCALE",
    "SEED_POLY",
    "SEED_ROLL",
    "SEED_EXCHANGE",
    "coeff_seed",
    "splitmix64_np",
    "uniform_pm1_np",
    "coeffs_np",
    "arange_matrix_np",
    "uniform_pm1_torch",
]

# One seed per workload; the polynomial coefficients get their own seed per degree.
SEED_ROLL_SMALL = 0xA5A50000 + 1
SEED_SCALE = 0xA5A50000 + 2
SEED_POLY = 0xA5A50000 + 3
SEED_ROLL = 0xA5A50000 + 4
SEED_EXCHANGE = 0xA5A50000 + 5


def coeff_seed(degree: int) -> int:
    return 0xC0EF0000 + int(degree)


_C0 = 0x9E3779B97F4A7C15
_C1 = 0xBF58476D1CE4E5B9
_C2 = 0x94D049BB133111EB
_MASK64 = (1 << 64) - 1


def splitmix64_np(x: np.ndarray) -> np.ndarray:
    """splitmix64 output function on a uint64 array (wrapping arithmetic)."""
    z = np.asarray(x, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = z + np.uint64(_C0)
        z = (z ^ (z >> np.uint64(30))) * np.uint64(_C1)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(_C2)
        z = z ^ (z >> np.uint64(31))
    return z


def _grid24_np(seed: int, start: int, count: int) -> np.ndarray:
    idx = np.arange(start, start + count, dtype=np.uint64)
    z = splitmix64_np(idx ^ np.uint64(seed & _MASK64))
    return (z >> np.uint64(40)).astype(np.int64)


def uniform_pm1_np(seed: int, count: int, start: int = 0) -> np.ndarray:
    """float32 values x_i, i in [start, start+count), on the grid of [-1, 1)."""
    k = _grid24_np(seed, start, count)
    return ((k - (1 << 23)).astype(np.float32) * np.float32(2.0**-23)).astype(np.float32)


def coeffs_np(degree: int) -> np.ndarray:
    """degree+1 float32 polynomial coefficients on the grid of [-0.5, 0.5)."""
    k = _grid24_np(coeff_seed(degree), 0, int(degree) + 1)
    return ((k - (1 << 23)).astype(np.float32) * np.float32(2.0**-24)).astype(np.float32)


def arange_matrix_np(rows: int = 64, cols: int = 4) -> np.ndarray:
    """The worked example's input: arange(rows*cols) as a rows x cols float32 matrix."""
    return np.arange(rows * cols, dtype=np.float32).reshape(rows, cols)


def _signed64(v: int) -> int:
    v &= _MASK64
    return v - (1 << 64) if v >= (1 << 63) else v


def uniform_pm1_torch(seed: int, count: int, device, out=None, chunk: int = 1 << 26):
    """Same values as :func:`uniform_pm1_np`, generated with torch int64 ops.

    torch has no unsigned 64-bit arithmetic, so the uint64 bits are carried in
    int64 tensors: addition and multiplication wrap modulo 2**64 either way,
    and a logical right shift is an arithmetic shift followed by a mask.
    Generated in chunks so that a multi-GiB buffer needs only a few hundred MiB
    of temporaries.
    """
    import torch

    if out is None:
        out = torch.empty(count, dtype=torch.float32, device=device)
    c0, c1, c2 = _signed64(_C0), _signed64(_C1), _signed64(_C2)
    s = _signed64(seed)

    def srl(z, k):
        return (z >> k) & ((1 << (64 - k)) - 1)

    for lo in range(0, count, chunk):
        hi = min(count, lo + chunk)
        z = torch.arange(lo, hi, dtype=torch.int64, device=out.device) ^ s
        z = z + c0
        z = (z ^ srl(z, 30)) * c1
        z = (z ^ srl(z, 27)) * c2
        z = z ^ srl(z, 31)
        k = srl(z, 40)
        out[lo:hi] = (k - (1 << 23)).to(torch.float32) * (2.0**-23)
    return out
