"""Block-level join-agg: Definition 3.7 executed over sub-tensor relations.

TEST INFRASTRUCTURE (see the package docstring).

For each function specification F (a tuple of input blocks, from
``oracle.worklist``): project every input onto F's input types, run the
concrete operator f[F] on the projections (the cell-level join-agg of the
same spec, restricted to the blocks), then combine the outputs that share
an output type with the aggregation op and recompose the aggregated blocks
into the output ("Every Kernel Is a Join", Definition 3.7 steps 1-3).

Because the aggregation op is associative and commutative, the result must
not depend on the block decomposition; the tests use this as an invariant.
"""
from __future__ import annotations

import numpy as np

from . import joinagg, letter_extents, parse
from .worklist import letters_in_order, worklist


def _combine(agg: str, a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """a (+) b cell by cell, where an absent (NaN) cell is no tuple at all."""
    if agg == "sum":
        both = a + b
    elif agg == "max":
        both = np.fmax(a, b)
    else:
        raise ValueError("a group with several tuples needs a SUM or MAX aggregation")
    return np.where(np.isnan(a), b, np.where(np.isnan(b), a, both))


def joinagg_blocked(spec: str, arrays, bounds: dict, map: str = "product", agg: str = "sum", scale: float = 1.0,
                    eps: float = 0.0, pred: str | None = None, tier: str = "idx") -> np.ndarray:
    ins, out = parse(spec)
    arrays = [np.asarray(a, dtype=np.float64) for a in arrays]
    ext = letter_extents(spec, [a.shape for a in arrays])
    letters = letters_in_order(spec)
    for l in letters:
        if bounds[l][0] != 0 or bounds[l][-1] != ext[l]:
            raise ValueError(f"bounds of {l!r} do not span its extent")
    nblk = {l: len(bounds[l]) - 1 for l in letters}
    wl = worklist(spec, bounds, pred)
    res = np.full(tuple(ext[l] for l in out), np.nan)

    def decode(term, bid):
        iv = {}
        for l in reversed(term):
            iv[l] = bid % nblk[l]
            bid //= nblk[l]
        return iv

    for g, ob in enumerate(wl["groups"]):
        acc = None
        for tup in wl["tuples"][wl["grp_ptr"][g]:wl["grp_ptr"][g + 1]]:
            iv = {}
            for term, bid in zip(ins, tup):
                iv.update(decode(term, bid))
            proj = []
            for term, a in zip(ins, arrays):
                sl = tuple(slice(bounds[l][iv[l]], bounds[l][iv[l] + 1]) for l in term)
                proj.append(a[sl])
            lo = {l: bounds[l][iv[l]] for l in iv}
            part = joinagg(spec, proj, map=map, agg=agg, scale=scale, eps=eps, pred=pred, tier=tier, lo=lo)
            acc = part if acc is None else _combine(agg, acc, part)
        oiv = decode(out, ob)
        osl = tuple(slice(bounds[l][oiv[l]], bounds[l][oiv[l] + 1]) for l in out)
        res[osl] = acc
    return res


def joinagg_partials(spec: str, arrays, bounds: dict, map: str = "product", tier: str = "idx") -> np.ndarray:
    """Definition 3.7 without its aggregation step: every output block keeps
    one unaggregated copy per function specification of its group, copy q
    holding the q-th in canonical order (the contracted letters' block ids,
    outer first).  Returns [m, *output extents], m the common group size --
    the m partial copies that an exchange with aggregation later combines
    ("Every Kernel Is a Join", Section 5.3 and Example 5.4, where the copies
    of C1 are X and Y)."""
    ins, out = parse(spec)
    arrays = [np.asarray(a, dtype=np.float64) for a in arrays]
    ext = letter_extents(spec, [a.shape for a in arrays])
    letters = letters_in_order(spec)
    nblk = {l: len(bounds[l]) - 1 for l in letters}
    wl = worklist(spec, bounds)
    sizes = {wl["grp_ptr"][g + 1] - wl["grp_ptr"][g] for g in range(len(wl["groups"]))}
    if len(sizes) != 1:
        raise ValueError("partials need the same number of function specifications in every group")
    m = sizes.pop()
    res = np.full((m,) + tuple(ext[l] for l in out), np.nan)

    def decode(term, bid):
        iv = {}
        for l in reversed(term):
            iv[l] = bid % nblk[l]
            bid //= nblk[l]
        return iv

    for g, ob in enumerate(wl["groups"]):
        oiv = decode(out, ob)
        osl = tuple(slice(bounds[l][oiv[l]], bounds[l][oiv[l] + 1]) for l in out)
        for q, tup in enumerate(wl["tuples"][wl["grp_ptr"][g]:wl["grp_ptr"][g + 1]]):
            iv = {}
            for term, bid in zip(ins, tup):
                iv.update(decode(term, bid))
            proj = [a[tuple(slice(bounds[l][iv[l]], bounds[l][iv[l] + 1]) for l in term)]
                    for term, a in zip(ins, arrays)]
            lo = {l: bounds[l][iv[l]] for l in iv}
            res[(q,) + osl] = joinagg(spec, proj, map=map, agg="sum", tier=tier, lo=lo)
    return res


def aggregate_copies(parts: np.ndarray, agg: str) -> np.ndarray:
    """x[...] = parts[0, ...] (+) parts[1, ...] (+) ... in copy order, (+) the
    SUM or MAX of the producer's aggregation: the "X1 + Y1" of the exchange
    with aggregation ("Every Kernel Is a Join", Example 5.4).  fp64."""
    parts = np.asarray(parts, dtype=np.float64)
    acc = parts[0].copy()
    for q in range(1, parts.shape[0]):
        acc = _combine(agg, acc, parts[q])
    return acc
