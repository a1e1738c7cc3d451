"""Block-level join enumeration: the function specifications of a join-agg
spec and their aggregation groups.

TEST INFRASTRUCTURE (see the package docstring).

"Every Kernel Is a Join", Section 3.3: once every index letter is split into
intervals, the join-agg spec holds exactly one function specification per
combination of intervals (prod_s intervals[s] of them).  Definition 3.7 step
(2) groups the specifications whose output type is the same; Definition 3.6
requires the distinct output types to tile the output.

Canonical order (the pages fix none; this order is what the bit-exact work
list comparison uses):
  * groups in increasing output block id, the id being row-major over the
    output block grid with letters in output-term order (this is the
    lexicographic order of the output block keys);
  * inside a group, tuples in lexicographic order of the interval indices
    of the contracted letters, taken in order of first appearance in the
    spec string;
  * a tuple lists one block id per input, each id row-major over that
    input's block grid in its term's letter order.

A cell predicate ``pred="ts"`` (keep t <= s) drops every tuple whose blocks
hold no cell pair with t <= s, i.e. keeps a tuple iff lo_t <= hi_s - 1.
"""
from __future__ import annotations

import itertools

from . import parse


def letters_in_order(spec: str):
    seen = []
    for ch in spec:
        if "a" <= ch <= "z" and ch not in seen:
            seen.append(ch)
    return seen


def block_id(term: str, iv: dict, nblk: dict) -> int:
    bid = 0
    for l in term:
        bid = bid * nblk[l] + iv[l]
    return bid


def worklist(spec: str, bounds: dict, pred: str | None = None):
    """Enumerate the join of a spec under per-letter interval bounds.

    bounds: letter -> list of boundaries [b_0 = 0, ..., b_k = extent].
    Returns a dict with
      groups:  list of output block ids, in canonical order
      grp_ptr: CSR offsets into ``tuples`` (len(groups) + 1)
      tuples:  list of tuples of input block ids (one per input)
      join_volume: sum over tuples of the cells of its input blocks
                   ("Every Kernel Is a Join", Section 4.3, sub-cost (2))
      agg_volume:  sum over groups of (m - 1) * cells of the output block
                   (Section 4.3, sub-cost (3))
    """
    ins, out = parse(spec)
    letters = letters_in_order(spec)
    contracted = [l for l in letters if l not in out]
    nblk = {l: len(bounds[l]) - 1 for l in letters}
    size = {l: [bounds[l][i + 1] - bounds[l][i] for i in range(nblk[l])] for l in letters}

    def keep(iv):
        if not pred:
            return True
        a, b = pred[0], pred[1]
        lo_a = bounds[a][iv[a]]
        hi_b = bounds[b][iv[b] + 1]
        return lo_a <= hi_b - 1

    groups = {}
    for combo in itertools.product(*[range(nblk[l]) for l in letters]):
        iv = dict(zip(letters, combo))
        if not keep(iv):
            continue
        ob = block_id(out, iv, nblk)
        ckey = tuple(iv[l] for l in contracted)
        tup = tuple(block_id(t, iv, nblk) for t in ins)
        jv = 0
        for t in ins:
            c = 1
            for l in t:
                c *= size[l][iv[l]]
            jv += c
        ocells = 1
        for l in out:
            ocells *= size[l][iv[l]]
        groups.setdefault(ob, []).append((ckey, tup, jv, ocells))
    order = sorted(groups)
    grp_ptr = [0]
    tuples = []
    join_volume = 0
    agg_volume = 0
    for ob in order:
        members = sorted(groups[ob], key=lambda m: m[0])
        for _, tup, jv, _ in members:
            tuples.append(tup)
            join_volume += jv
        agg_volume += (len(members) - 1) * members[0][3]
        grp_ptr.append(len(tuples))
    return {"groups": order, "grp_ptr": grp_ptr, "tuples": tuples,
            "join_volume": join_volume, "agg_volume": agg_volume}


def overlay(bounds_a, bounds_b):
    """Per-dimension union of the split points of two tilings
    ("Every Kernel Is a Join", Section 5.3); the grid cells are the atoms."""
    return [sorted(set(a) | set(b)) for a, b in zip(bounds_a, bounds_b)]


def atoms(bounds_a, bounds_b):
    """List of atoms as tuples of per-dimension (lo, hi) intervals, row-major."""
    ov = overlay(bounds_a, bounds_b)
    per_dim = [[(p[i], p[i + 1]) for i in range(len(p) - 1)] for p in ov]
    return list(itertools.product(*per_dim))
