"""GB300 (sm_103a) join-agg hot path of Einsummable.

Tensor relations, join-agg specs and the exchange ("Every Kernel Is a Join:
Automatic Multi-GPU Parallelism for AI Computations in Einsummable"),
executed on one GPU by libea.so (C ABI in include/ea.h):

* ``Relation``  -- a CUDA tensor stored as blocks of a tiling;
* ``joinagg``   -- one join-agg: join on shared letters, per-tuple kernel,
                   SUM/MAX aggregation fused into the kernel;
* ``exchange``  -- re-block a relation from one tiling to another.

The Python layer only marshals arguments.  Importing this package loads
libea.so lazily; calls raise if it is missing (no CPU fallback).
"""
from ._abi import EaError, lib  # noqa: F401

__all__ = ["Relation", "joinagg", "exchange", "check", "EaError", "lib", "plan_cache_clear"]


def __getattr__(name):
    if name in ("Relation", "joinagg", "exchange", "check", "plan_cache_clear", "output_layout"):
        from . import relation
        return getattr(relation, name)
    raise AttributeError(name)
