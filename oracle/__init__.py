"""fp64 CPU oracle for the tensor-relational join-agg hot path.

TEST INFRASTRUCTURE.  Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  It shares no
code with the CUDA path (``tensor_relational_einsum_gb300``) and never
imports it.

Layers
------
* ``joinagg``    -- one join-agg in the degenerate relational form (every key
  one cell), computed by the C tiers in ``orc.c``: "lit" (hash join +
  hash group-by) or "idx" (index nested loop over dense keys).
* ``exchange``   -- re-blocking of a block arena by definition.
* ``worklist``   -- the block-level join: function specifications (tuples of
  input blocks) grouped by output block (``oracle.worklist``).
* ``blocked``    -- the block-level implementation of Definition 3.7
  (join per tuple, aggregate per output block, recompose).
* ``chains``     -- compositions used by the workloads (attention, SwiGLU
  FFN, RMSNorm, RoPE, a LLaMA-style block).

Cell values are float64; NaN marks an ABSENT cell (no tuple).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "liborc.so")
_lock = threading.Lock()
_lib = None

MAPS = {"product": 0, "identity": 1, "silu_mul": 2, "add": 3, "exp_sub": 4, "div": 5,
        "square": 6, "rms_apply": 7}
AGGS = {"none": 0, "sum": 1, "max": 2}


def build(force: bool = False) -> str:
    """Compile orc.c into liborc.so with gcc (plain C11, no CUDA)."""
    src = os.path.join(_HERE, "orc.c")
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(src):
        tmp = _SO + ".tmp.%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=gnu11", "-shared", "-fPIC", "-pthread", src,
                               "-o", tmp, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            P = ctypes.POINTER
            L.orc_last_error.restype = ctypes.c_char_p
            L.orc_joinagg_lit.argtypes = [ctypes.c_char_p, P(ctypes.c_int64), P(ctypes.c_void_p), ctypes.c_int,
                                          ctypes.c_int, ctypes.c_double, ctypes.c_double, ctypes.c_char_p,
                                          P(ctypes.c_int64), ctypes.c_void_p, P(ctypes.c_int64)]
            L.orc_joinagg_idx.argtypes = [ctypes.c_char_p, P(ctypes.c_int64), P(ctypes.c_void_p), ctypes.c_int,
                                          ctypes.c_int, ctypes.c_double, ctypes.c_double, ctypes.c_char_p,
                                          P(ctypes.c_int64), ctypes.c_void_p, ctypes.c_int]
            L.orc_exchange.argtypes = [ctypes.c_int, P(ctypes.c_int64), ctypes.c_int, P(ctypes.c_int32),
                                       P(ctypes.c_int64), P(ctypes.c_int32), P(ctypes.c_int64), ctypes.c_void_p,
                                       ctypes.c_void_p, ctypes.c_int]
            L.orc_exchange_perm.argtypes = [ctypes.c_int, P(ctypes.c_int64), P(ctypes.c_int32), P(ctypes.c_int64),
                                            P(ctypes.c_int32), P(ctypes.c_int64), P(ctypes.c_int64), ctypes.c_int]
            L.orc_threads.restype = ctypes.c_int
            _lib = L
    return _lib


class OracleError(RuntimeError):
    pass


def _check(rc):
    if rc != 0:
        raise OracleError(lib().orc_last_error().decode())


def parse(spec: str):
    """Split "ij,jk->ik" into (["ij", "jk"], "ik")."""
    lhs, out = spec.split("->")
    return lhs.split(","), out


def letter_extents(spec: str, shapes):
    ins, _ = parse(spec)
    ext = {}
    for term, shp in zip(ins, shapes):
        if len(term) != len(shp):
            raise OracleError(f"input {term!r} has rank {len(term)} but shape {tuple(shp)}")
        for l, e in zip(term, shp):
            if ext.setdefault(l, int(e)) != int(e):
                raise OracleError(f"letter {l!r} has two extents")
    return ext


def joinagg(spec: str, arrays, map: str = "product", agg: str = "sum", scale: float = 1.0, eps: float = 0.0,
            pred: str | None = None, tier: str = "idx", nthreads: int = 0, lo: dict | None = None,
            return_joined: bool = False):
    """One join-agg ("Every Kernel Is a Join", Definition 3.7) in the
    degenerate form: join cells on shared letters, map, group by the output
    letters, aggregate; output cells with no joined tuple are NaN (absent).

    ``pred="ts"`` keeps only joined tuples with t <= s (a cell predicate on
    global letter values; ``lo`` gives each letter's global offset when the
    arrays are projections).
    """
    ins, out = parse(spec)
    if len(ins) != len(arrays):
        raise OracleError("number of arrays does not match the spec")
    arrs = [np.ascontiguousarray(a, dtype=np.float64) for a in arrays]
    ext = letter_extents(spec, [a.shape for a in arrs])
    shapes = np.array([e for a in arrs for e in a.shape] or [0], dtype=np.int64)
    out_shape = tuple(ext[l] for l in out)
    res = np.empty(out_shape, dtype=np.float64)
    ptrs = (ctypes.c_void_p * len(arrs))(*[a.ctypes.data for a in arrs])
    los = np.zeros(26, dtype=np.int64)
    for l, v in (lo or {}).items():
        los[ord(l) - 97] = int(v)
    P64 = ctypes.POINTER(ctypes.c_int64)
    pred_b = pred.encode() if pred else None
    L = lib()
    if tier == "lit":
        nj = ctypes.c_int64(0)
        _check(L.orc_joinagg_lit(spec.encode(), shapes.ctypes.data_as(P64), ptrs, MAPS[map], AGGS[agg], scale, eps,
                                 pred_b, los.ctypes.data_as(P64), res.ctypes.data, ctypes.byref(nj)))
        if return_joined:
            return res, nj.value
    elif tier == "idx":
        _check(L.orc_joinagg_idx(spec.encode(), shapes.ctypes.data_as(P64), ptrs, MAPS[map], AGGS[agg], scale, eps,
                                 pred_b, los.ctypes.data_as(P64), res.ctypes.data, int(nthreads)))
    else:
        raise OracleError(f"unknown tier {tier!r}")
    return res


def near_equal_bounds(n: int, k: int):
    """Block boundaries b_i = floor(i * n / k), i = 0..k (near-equal intervals,
    "Every Kernel Is a Join", Section 4.3)."""
    return [(i * n) // k for i in range(k + 1)]


def _flat_bounds(bounds):
    nb = np.array([len(b) - 1 for b in bounds], dtype=np.int32)
    flat = np.array([int(x) for b in bounds for x in b], dtype=np.int64)
    return nb, flat


def exchange(arena: np.ndarray, dims, src_bounds, dst_bounds, nthreads: int = 0) -> np.ndarray:
    """Re-block ``arena`` (blocks of the source tiling, each row-major, in
    row-major block-id order) into the arena of the destination tiling.
    Every element keeps its global coordinates ("Every Kernel Is a Join",
    Section 5.3).  Works on raw element bytes, so the result is bit-exact."""
    dims = np.array([int(d) for d in dims], dtype=np.int64)
    a = np.ascontiguousarray(arena)
    out = np.empty_like(a)
    snb, sb = _flat_bounds(src_bounds)
    dnb, db = _flat_bounds(dst_bounds)
    P64 = ctypes.POINTER(ctypes.c_int64)
    P32 = ctypes.POINTER(ctypes.c_int32)
    _check(lib().orc_exchange(len(dims), dims.ctypes.data_as(P64), a.itemsize, snb.ctypes.data_as(P32),
                              sb.ctypes.data_as(P64), dnb.ctypes.data_as(P32), db.ctypes.data_as(P64),
                              a.ctypes.data, out.ctypes.data, int(nthreads)))
    return out


def exchange_perm(dims, src_bounds, dst_bounds, nthreads: int = 0) -> np.ndarray:
    """perm[i] = source-arena position of destination-arena element i."""
    dims = np.array([int(d) for d in dims], dtype=np.int64)
    perm = np.empty(int(np.prod(dims)), dtype=np.int64)
    snb, sb = _flat_bounds(src_bounds)
    dnb, db = _flat_bounds(dst_bounds)
    P64 = ctypes.POINTER(ctypes.c_int64)
    P32 = ctypes.POINTER(ctypes.c_int32)
    _check(lib().orc_exchange_perm(len(dims), dims.ctypes.data_as(P64), snb.ctypes.data_as(P32),
                                   sb.ctypes.data_as(P64), dnb.ctypes.data_as(P32), db.ctypes.data_as(P64),
                                   perm.ctypes.data_as(P64), int(nthreads)))
    return perm


def threads() -> int:
    return int(lib().orc_threads())


from . import worklist, blocked, chains  # noqa: E402,F401
