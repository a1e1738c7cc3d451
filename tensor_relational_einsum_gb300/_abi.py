"""ctypes binding of libea.so (the C ABI declared in include/ea.h).

Argument marshalling only: every step of a join-agg or an exchange runs in
libea.so's planner and CUDA kernels.  PyTorch provides device memory and
the current CUDA stream.  There is no CPU fallback: if libea.so is missing
or the GPU is absent, the calls raise.
"""
from __future__ import annotations

import ctypes
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
# EA_BOUNDS_CHECK=1 loads the bounds-checking build (EA_DEBUG_BOUNDS).
LIB_PATH = os.path.join(PKG, "libea_bounds.so" if os.environ.get("EA_BOUNDS_CHECK", "") == "1" else "libea.so")

F32, BF16 = 0, 1
DTYPES = {"f32": F32, "bf16": BF16}
AGGS = {"none": 0, "sum": 1, "max": 2, "max_sumexp": 3}
MAPS = {"product": 0, "identity": 1, "silu_mul": 2, "add": 3, "exp_sub": 4, "div": 5, "square": 6,
        "rms_apply": 7, "exp_sub_div": 8, "rope": 9}
STATUS = {0: "EA_OK", 1: "EA_ERR_SPEC", 2: "EA_ERR_SHAPE", 3: "EA_ERR_PARTITION", 4: "EA_ERR_DTYPE",
          5: "EA_ERR_ALLOC", 6: "EA_ERR_CUDA", 7: "EA_ERR_ARG", 8: "EA_ERR_UNSUPPORTED", 9: "EA_ERR_DEVICE",
          10: "EA_ERR_BOUNDS"}


class EaError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{STATUS.get(code, code)}: {msg}")
        self.code = code


class DimPart(ctypes.Structure):
    _fields_ = [("nblocks", ctypes.c_int32), ("reserved", ctypes.c_int32), ("bounds", ctypes.POINTER(ctypes.c_int64))]


class IndexPart(ctypes.Structure):
    _fields_ = [("index", ctypes.c_char), ("reserved", ctypes.c_char * 3), ("nblocks", ctypes.c_int32),
                ("bounds", ctypes.POINTER(ctypes.c_int64))]


class Opts(ctypes.Structure):
    _fields_ = [("out_dtype", ctypes.c_int32), ("scale", ctypes.c_float), ("eps", ctypes.c_float),
                ("pred_lo", ctypes.c_char), ("pred_hi", ctypes.c_char), ("rope_pos", ctypes.c_char),
                ("epi_pair", ctypes.c_char), ("rope_table", ctypes.c_void_p), ("rope_npos", ctypes.c_int64),
                ("out2", ctypes.c_void_p), ("epi_in", ctypes.c_void_p), ("epi_map", ctypes.c_int32),
                ("rope_dim", ctypes.c_int32), ("row_rms", ctypes.c_void_p), ("partials", ctypes.c_int32),
                ("rope_layout", ctypes.c_int32), ("simt_bf16", ctypes.c_int32)]


class AttnOpts(ctypes.Structure):
    _fields_ = [("scale", ctypes.c_float), ("causal", ctypes.c_int32), ("n_seq_ends", ctypes.c_int32),
                ("reserved0", ctypes.c_int32), ("seq_ends", ctypes.c_void_p), ("m_out", ctypes.c_void_p),
                ("l_out", ctypes.c_void_p), ("reserved", ctypes.c_int64 * 4)]


_lib = None
_lock = threading.Lock()

P64 = ctypes.POINTER(ctypes.c_int64)
P32 = ctypes.POINTER(ctypes.c_int32)
VP = ctypes.c_void_p
ALLOC_FN = ctypes.CFUNCTYPE(ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p)
FREE_FN = ctypes.CFUNCTYPE(None, ctypes.c_void_p, ctypes.c_void_p)


def lib():
    """Load libea.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with tensor_relational_einsum_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        L.ea_abi_version.restype = ctypes.c_int
        L.ea_debug_bounds.restype = ctypes.c_int
        L.ea_last_error.restype = ctypes.c_char_p
        L.ea_check.argtypes = [VP]
        L.ea_plan_cache_clear.argtypes = []
        L.ea_relation_create.argtypes = [ctypes.c_int, ctypes.c_int, P64, ctypes.POINTER(DimPart), VP,
                                         ctypes.POINTER(VP)]
        L.ea_relation_destroy.argtypes = [VP]
        L.ea_relation_info.argtypes = [VP, P32, P32, P64, P64]
        L.ea_relation_block.argtypes = [VP, ctypes.c_int64, ctypes.POINTER(VP), P64, P64]
        L.ea_relation_data.argtypes = [VP, ctypes.POINTER(VP), ctypes.POINTER(ctypes.c_size_t)]
        L.ea_relation_bounds.argtypes = [VP, ctypes.c_int, P32, P64]
        L.ea_joinagg_run.argtypes = [ctypes.c_char_p, ctypes.POINTER(VP), ctypes.c_int, ctypes.POINTER(IndexPart),
                                     ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.POINTER(Opts), VP,
                                     ctypes.POINTER(VP)]
        L.ea_exchange.argtypes = [VP, ctypes.POINTER(DimPart), VP, ctypes.POINTER(VP)]
        L.ea_plan_worklist.argtypes = [ctypes.c_char_p, P64, ctypes.POINTER(IndexPart), ctypes.c_int, ctypes.c_char,
                                       ctypes.c_char, ctypes.c_int64, ctypes.c_int64, P64, P64, P64, P64, P64, P64,
                                       P64]
        L.ea_exchange_permutation.argtypes = [ctypes.c_int, P64, ctypes.POINTER(DimPart), ctypes.POINTER(DimPart), P64]
        L.ea_overlay_atoms.argtypes = [ctypes.c_int, P64, ctypes.POINTER(DimPart), ctypes.POINTER(DimPart), P64]
        L.ea_last_plan.argtypes = [P32, P32, P64, P64, P64]
        L.ea_last_plan_cluster.argtypes = [P32]
        L.ea_exchange_noalloc.argtypes = [VP, VP, VP]
        L.ea_exchange_agg.argtypes = [VP, ctypes.c_int, ctypes.POINTER(DimPart), VP, ctypes.POINTER(VP)]
        L.ea_set_allocator.argtypes = [ALLOC_FN, FREE_FN, VP]
        L.ea_relation_copy_host.argtypes = [VP, VP, ctypes.c_int, VP]
        L.ea_selftest_wait_timeout.argtypes = [ctypes.c_int64, VP]
        L.ea_plan_check_exchange.argtypes = [P64, ctypes.c_int64, P64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64]
        L.ea_attention_run.argtypes = [ctypes.c_char_p, VP, VP, VP, ctypes.POINTER(AttnOpts), VP, ctypes.POINTER(VP)]
        for name in ("ea_check", "ea_plan_cache_clear", "ea_relation_create", "ea_relation_destroy",
                     "ea_relation_info", "ea_relation_block", "ea_relation_data", "ea_relation_bounds",
                     "ea_joinagg_run", "ea_exchange", "ea_plan_worklist", "ea_exchange_permutation",
                     "ea_overlay_atoms", "ea_last_plan", "ea_last_plan_cluster", "ea_exchange_noalloc", "ea_attention_run", "ea_exchange_agg",
                     "ea_set_allocator", "ea_relation_copy_host", "ea_selftest_wait_timeout", "ea_plan_check_exchange"):
            getattr(L, name).restype = ctypes.c_int
        if L.ea_abi_version() != 5:
            raise ImportError("libea.so ABI version mismatch")
        _lib = L
        return _lib


def check_status(rc: int):
    if rc != 0:
        raise EaError(rc, lib().ea_last_error().decode(errors="replace"))


# ------------------------------------------------------------- marshalling

def i64(values):
    arr = (ctypes.c_int64 * max(1, len(values)))(*[int(v) for v in values])
    return arr


def near_equal(n: int, k: int):
    return [(i * n) // k for i in range(k + 1)]


def dim_parts(dims, parts):
    """parts: per dimension an int (near-equal block count) or a bounds list.

    Returns (ctypes array of DimPart, keepalive list, bounds as lists)."""
    keep = []
    arr = (DimPart * len(dims))()
    bounds = []
    for d, (n, p) in enumerate(zip(dims, parts)):
        if isinstance(p, int):
            b = near_equal(n, p) if n > 0 else [0, 0]
        else:
            b = [int(x) for x in p]
        bounds.append(b)
        cb = i64(b)
        keep.append(cb)
        arr[d].nblocks = len(b) - 1
        arr[d].bounds = ctypes.cast(cb, P64)
    return arr, keep, bounds


def index_parts(parts: dict | None):
    parts = parts or {}
    keep = []
    arr = (IndexPart * max(1, len(parts)))()
    for i, (letter, p) in enumerate(parts.items()):
        arr[i].index = letter.encode()
        if isinstance(p, int):
            arr[i].nblocks = p
            arr[i].bounds = None
        else:
            cb = i64(p)
            keep.append(cb)
            arr[i].nblocks = len(p) - 1
            arr[i].bounds = ctypes.cast(cb, P64)
    return arr, len(parts), keep


KERNEL_CLASS = {0: "exchange", 1: "elementwise", 2: "rowreduce", 3: "contract_simt", 4: "contract_tc", 5: "attention", 6: "exchange_agg"}


def last_plan():
    """What the last join-agg / exchange call of this thread launched."""
    k, n = ctypes.c_int32(), ctypes.c_int32()
    t, g, u = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
    check_status(lib().ea_last_plan(ctypes.byref(k), ctypes.byref(n), ctypes.byref(t), ctypes.byref(g),
                                    ctypes.byref(u)))
    c = ctypes.c_int32()
    check_status(lib().ea_last_plan_cluster(ctypes.byref(c)))
    return {"kernel": KERNEL_CLASS.get(k.value, None), "launches": n.value, "tiles": t.value, "groups": g.value,
            "tuples": u.value, "cta_pair": c.value == 2}
