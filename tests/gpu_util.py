"""Helpers of the GPU parity tests: upload seeded inputs, read relations back,
compare against the oracle."""
from __future__ import annotations

import numpy as np
import torch

import synth
from tensor_relational_einsum_gb300 import _abi
from tensor_relational_einsum_gb300.relation import Relation, exchange, joinagg  # noqa: F401

FP32_TOL = 1e-5
BF16_TOL = 2e-2


def to_device(t: synth.Tensor) -> torch.Tensor:
    if t.dtype == "bf16":
        return torch.from_numpy(t.host.view(np.int16).copy()).view(torch.bfloat16).reshape(t.shape).cuda()
    return torch.from_numpy(t.host.copy()).reshape(t.shape).cuda()


def rel(t: synth.Tensor, parts) -> Relation:
    return Relation.from_dense(to_device(t), parts, dtype=t.dtype)


def dense64(r: Relation) -> np.ndarray:
    return r.to_dense().float().cpu().numpy().astype(np.float64)


def arena_bits(r: Relation) -> np.ndarray:
    a = r.arena().cpu()
    return a.view(torch.int16).numpy().view(np.uint16) if r.dtype == "bf16" else a.view(torch.int32).numpy()


def bounds_of(dims, parts):
    return [synth_bounds(n, p) for n, p in zip(dims, parts)]


def synth_bounds(n, p):
    return [(i * n) // p for i in range(p + 1)] if isinstance(p, int) else list(p)


def rel_frob(got: np.ndarray, want: np.ndarray) -> float:
    """Relative Frobenius error over the cells present in ``want`` (NaN in
    ``want`` marks an absent cell)."""
    m = ~np.isnan(want)
    num = np.linalg.norm((got - want)[m])
    den = np.linalg.norm(want[m])
    return float(num / den) if den > 0 else float(num)


def max_block_rel_frob(got, want, bounds) -> float:
    """Max over output blocks of the relative Frobenius error."""
    import itertools
    worst = 0.0
    for combo in itertools.product(*[range(len(b) - 1) for b in bounds]):
        sl = tuple(slice(b[i], b[i + 1]) for b, i in zip(bounds, combo))
        worst = max(worst, rel_frob(got[sl], want[sl]))
    return worst


def last():
    return _abi.last_plan()
