"""Seeded synthetic inputs shared by the oracle harness and the GPU path.

This module holds no arithmetic of the join-agg method: it only turns a
(seed, element index) pair into a number.  Both sides of every parity test
read the exact same bits from here, so a difference between them can only
come from the method.

Generator: a counter-based SplitMix64 (Steele, Lea and Flood, "Fast
splittable pseudorandom number generators", OOPSLA 2014).  Element ``n`` of
stream ``seed`` is ``mix64(mix64(seed) + (n + 1) * GAMMA)``, so any element
can be drawn on its own and the streams of different seeds do not overlap in
practice.

* uniform(a, b):  a + (b - a) * u,  u = (z >> 11) * 2**-53 in [0, 1)
* normal(mu, sd): Box-Muller on the pair (u_{2n}, u_{2n+1}):
  mu + sd * sqrt(-2 ln(1 - u1)) * cos(2 pi u2)
* intgrid(lo, hi): lo + floor(u * (hi - lo + 1)), integers in [lo, hi]

Values are produced in float64, rounded to float32 with round-to-nearest-even
and, for bf16 tensors, rounded once more from float32 to bf16 with
round-to-nearest-even.  ``to_f64`` returns the exact value of the stored
bits, which is what the oracle consumes.
"""
from __future__ import annotations

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

_CHUNK = 1 << 22


def _mix64(z: np.ndarray) -> np.ndarray:
    z = z.copy()
    z ^= z >> np.uint64(30)
    z *= _M1
    z ^= z >> np.uint64(27)
    z *= _M2
    z ^= z >> np.uint64(31)
    return z


def raw_u64(seed: int, start: int, count: int) -> np.ndarray:
    """SplitMix64 outputs for element indices [start, start + count)."""
    with np.errstate(over="ignore"):
        base = _mix64(np.array([seed & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64))[0]
        idx = np.arange(start + 1, start + count + 1, dtype=np.uint64)
        return _mix64(base + idx * GAMMA)


def unit_f64(seed: int, start: int, count: int) -> np.ndarray:
    """Uniform doubles in [0, 1) with 53 random bits."""
    return (raw_u64(seed, start, count) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def _fill(n: int, fn) -> np.ndarray:
    out = np.empty(n, dtype=np.float64)
    for s in range(0, n, _CHUNK):
        c = min(_CHUNK, n - s)
        out[s:s + c] = fn(s, c)
    return out


def uniform_f64(seed: int, n: int, lo: float, hi: float) -> np.ndarray:
    return _fill(n, lambda s, c: lo + (hi - lo) * unit_f64(seed, s, c))


def normal_f64(seed: int, n: int, mu: float, sd: float) -> np.ndarray:
    def gen(s, c):
        u = unit_f64(seed, 2 * s, 2 * c)
        u1, u2 = u[0::2], u[1::2]
        return mu + sd * np.sqrt(-2.0 * np.log1p(-u1)) * np.cos(2.0 * np.pi * u2)
    return _fill(n, gen)


def intgrid_f64(seed: int, n: int, lo: int, hi: int) -> np.ndarray:
    span = hi - lo + 1
    return _fill(n, lambda s, c: lo + np.floor(unit_f64(seed, s, c) * span))


# ---------------------------------------------------------------- rounding

def f64_to_f32(x: np.ndarray) -> np.ndarray:
    """Round to float32, nearest-even (numpy's cast rounds that way)."""
    return np.asarray(x, dtype=np.float64).astype(np.float32)


def f32_to_bf16_bits(x32: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round-to-nearest-even.

    Inputs are finite by construction (no NaN handling needed here).
    """
    b = np.ascontiguousarray(x32, dtype=np.float32).view(np.uint32)
    lsb = (b >> np.uint32(16)) & np.uint32(1)
    r = (b + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


class Tensor:
    """A generated tensor: its storage bits and their exact float64 value.

    ``dtype`` is "f32" or "bf16".  ``host`` holds the storage (float32 array
    or uint16 bf16 bit patterns), row-major with ``shape``.
    """

    def __init__(self, host: np.ndarray, dtype: str, shape):
        self.host = host
        self.dtype = dtype
        self.shape = tuple(int(s) for s in shape)

    def to_f64(self) -> np.ndarray:
        if self.dtype == "bf16":
            return bf16_bits_to_f32(self.host).astype(np.float64).reshape(self.shape)
        return self.host.astype(np.float64).reshape(self.shape)

    def to_f32(self) -> np.ndarray:
        if self.dtype == "bf16":
            return bf16_bits_to_f32(self.host).reshape(self.shape)
        return self.host.reshape(self.shape)

    @property
    def nbytes(self) -> int:
        return self.host.nbytes


def make(dtype: str, shape, dist: str, seed: int, a: float = 0.0, b: float = 1.0) -> Tensor:
    """Draw a tensor.

    dist: "uniform" (range [a, b)), "normal" (mean a, std b) or "int"
    (integers in [a, b]).
    """
    shape = tuple(int(s) for s in shape)
    n = int(np.prod(shape)) if shape else 1
    if dist == "uniform":
        v = uniform_f64(seed, n, a, b)
    elif dist == "normal":
        v = normal_f64(seed, n, a, b)
    elif dist == "int":
        v = intgrid_f64(seed, n, int(a), int(b))
    else:
        raise ValueError(f"unknown distribution {dist!r}")
    v32 = f64_to_f32(v)
    if dtype == "f32":
        return Tensor(v32, "f32", shape)
    if dtype == "bf16":
        return Tensor(f32_to_bf16_bits(v32), "bf16", shape)
    raise ValueError(f"unknown dtype {dtype!r}")


def subset_rows(seed: int, n_total: int, n_pick: int) -> np.ndarray:
    """A seeded sorted choice of n_pick distinct indices out of n_total."""
    keys = raw_u64(seed, 0, n_total)
    return np.sort(np.argsort(keys, kind="stable")[:n_pick])


# ------------------------------------------------------------ torch variant

def _torch_mix64(z):
    import torch
    m1 = 0xBF58476D1CE4E5B9 - (1 << 64)
    m2 = 0x94D049BB133111EB - (1 << 64)

    def lsr(x, k):
        return (x >> k) & ((1 << (64 - k)) - 1)

    z = z ^ lsr(z, 30)
    z = z * m1
    z = z ^ lsr(z, 27)
    z = z * m2
    return z ^ lsr(z, 31)


def _signed(v: int) -> int:
    v &= (1 << 64) - 1
    return v - (1 << 64) if v >= (1 << 63) else v


def _py_mix64(z: int) -> int:
    mask = (1 << 64) - 1
    z &= mask
    z ^= z >> 30
    z = (z * 0xBF58476D1CE4E5B9) & mask
    z ^= z >> 27
    z = (z * 0x94D049BB133111EB) & mask
    return z ^ (z >> 31)


def make_torch(dtype: str, shape, dist: str, seed: int, a: float = 0.0, b: float = 1.0, device="cuda"):
    """Same stream as ``make`` computed with torch on ``device`` (fast for
    large tensors).  Uniform and integer draws are bit-identical to
    ``make``; normals agree except where the last ulp of the fp64 log / cos
    differs between libraries.  Returns a torch tensor of the dtype."""
    import torch
    shape = tuple(int(s) for s in shape)
    n = 1
    for s in shape:
        n *= s
    base = _signed(_py_mix64(seed))
    gamma = _signed(0x9E3779B97F4A7C15)
    out = torch.empty(n, dtype=torch.float64 if dtype == "f64" else torch.float32, device=device)
    chunk = 1 << 24
    per = 2 if dist == "normal" else 1
    for s0 in range(0, n, chunk):
        c = min(chunk, n - s0)
        idx = torch.arange(per * s0 + 1, per * (s0 + c) + 1, dtype=torch.int64, device=device)
        z = _torch_mix64(base + idx * gamma)
        u = ((z >> 11) & ((1 << 53) - 1)).to(torch.float64) * (2.0 ** -53)
        if dist == "uniform":
            v = a + (b - a) * u
        elif dist == "int":
            v = a + torch.floor(u * (int(b) - int(a) + 1))
        elif dist == "normal":
            u1, u2 = u[0::2], u[1::2]
            v = a + b * torch.sqrt(-2.0 * torch.log1p(-u1)) * torch.cos(2.0 * torch.pi * u2)
        else:
            raise ValueError(dist)
        out[s0:s0 + c] = v.to(torch.float32)
    if dtype == "bf16":
        return out.to(torch.bfloat16).reshape(shape)
    return out.reshape(shape)
