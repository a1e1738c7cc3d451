"""Tensor relations on the GPU and the two hot-path calls on them.

A ``Relation`` is a tensor stored as its blocks ("Every Kernel Is a Join",
Section 1: a set of (sub-tensor key, sub-tensor) pairs; Definitions 3.1 and
3.2: the keys are tensor types that tile the tensor).  Its arena is a torch
CUDA tensor; libea.so holds the handle.  ``joinagg`` and ``exchange`` call
the C ABI on the current torch stream.
"""
from __future__ import annotations

import ctypes

import torch

from . import _abi
from ._abi import AGGS, DTYPES, MAPS, check_status, lib

_TORCH = {"f32": torch.float32, "bf16": torch.bfloat16}
_NAMES = {0: "f32", 1: "bf16"}


def _stream_ptr(stream=None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


class Relation:
    """A tensor of ``dims`` tiled per dimension by ``parts`` (an int = that
    many near-equal blocks, or an explicit bounds list).

    ``storage``: an existing CUDA tensor holding the arena (borrowed, must
    have at least prod(dims) elements of the dtype); default: a new one."""

    def __init__(self, dtype: str, dims, parts, storage: torch.Tensor | None = None, device=None):
        self.dtype = dtype
        self.dims = tuple(int(d) for d in dims)
        n = 1
        for d in self.dims:
            n *= d
        if storage is None:
            storage = torch.empty(max(n, 1), dtype=_TORCH[dtype], device=device or "cuda")
        else:
            if storage.dtype != _TORCH[dtype] or storage.numel() < n or not storage.is_cuda:
                raise ValueError("storage must be a CUDA tensor of the relation's dtype with enough elements")
            if not storage.is_contiguous():
                raise ValueError("storage must be contiguous")
        self.storage = storage
        arr, keep, bounds = _abi.dim_parts(self.dims, parts)
        self.bounds = bounds
        h = ctypes.c_void_p()
        check_status(lib().ea_relation_create(DTYPES[dtype], len(self.dims), _abi.i64(self.dims), arr,
                                              ctypes.c_void_p(storage.data_ptr()), ctypes.byref(h)))
        self.handle = h

    # -- lifetime
    def __del__(self):
        h = getattr(self, "handle", None)
        if h is not None and h.value and _abi._lib is not None:
            _abi._lib.ea_relation_destroy(h)
            self.handle = None

    # -- queries
    @property
    def nblocks(self) -> int:
        n = ctypes.c_int64()
        check_status(lib().ea_relation_info(self.handle, None, None, None, ctypes.byref(n)))
        return n.value

    @property
    def parts(self):
        return [list(b) for b in self.bounds]

    def block(self, i: int):
        """(device pointer, lo, hi) of block i."""
        p = ctypes.c_void_p()
        lo = (ctypes.c_int64 * 8)()
        hi = (ctypes.c_int64 * 8)()
        check_status(lib().ea_relation_block(self.handle, i, ctypes.byref(p), lo, hi))
        r = len(self.dims)
        return p.value, tuple(lo[:r]), tuple(hi[:r])

    def arena(self) -> torch.Tensor:
        n = 1
        for d in self.dims:
            n *= d
        return self.storage[:n]

    # -- conversion (all on the GPU, through the exchange kernel)
    @classmethod
    def from_dense(cls, t: torch.Tensor, parts, dtype: str | None = None) -> "Relation":
        """Relation with tiling ``parts`` holding the row-major tensor ``t``."""
        dtype = dtype or {torch.float32: "f32", torch.bfloat16: "bf16"}[t.dtype]
        t = t.contiguous()
        whole = cls(dtype, t.shape, [1] * t.dim(), storage=t.reshape(-1))
        if all((isinstance(p, int) and p == 1) or (not isinstance(p, int) and len(p) == 2) for p in parts):
            out = cls(dtype, t.shape, parts)
            out.storage.copy_(t.reshape(-1)) if t.numel() else None
            return out
        return exchange(whole, parts)

    def load(self, t: torch.Tensor, stream=None) -> "Relation":
        """Fill this relation with the row-major tensor ``t`` (same extents
        and dtype) through the exchange kernel."""
        t = t.contiguous()
        if tuple(t.shape) != self.dims or t.dtype != _TORCH[self.dtype]:
            raise ValueError("load: tensor shape or dtype differs from the relation")
        if all(len(b) == 2 for b in self.bounds):
            self.arena().copy_(t.reshape(-1))
            return self
        whole = Relation(self.dtype, self.dims, [1] * len(self.dims), storage=t.reshape(-1))
        exchange(whole, None, out=self, stream=stream)
        return self

    def copy_host(self, host: torch.Tensor, to_device: bool = True, stream=None) -> torch.Tensor:
        """Load this relation from (``to_device``) or offload it to the dense
        row-major CPU tensor ``host`` with strided copies straight between
        host memory and the blocks (no device-side re-blocking).  Pinned host
        memory makes the copies asynchronous on ``stream``."""
        n = 1
        for d in self.dims:
            n *= d
        if host.device.type != "cpu" or not host.is_contiguous() or host.dtype != _TORCH[self.dtype] or \
                host.numel() != n:
            raise ValueError("host must be a contiguous CPU tensor of the relation's dtype and size")
        check_status(lib().ea_relation_copy_host(self.handle, ctypes.c_void_p(host.data_ptr()), 1 if to_device else 0,
                                                 ctypes.c_void_p(_stream_ptr(stream))))
        return host

    def to_dense(self) -> torch.Tensor:
        """The tensor, row-major, as a new CUDA tensor."""
        if all(len(b) == 2 for b in self.bounds):
            return self.arena().clone().reshape(self.dims)
        whole = exchange(self, [1] * len(self.dims))
        return whole.arena().reshape(self.dims)


def exchange(rel: Relation, parts, out: Relation | None = None, stream=None) -> Relation:
    """Re-block ``rel`` into the tiling ``parts`` ("Every Kernel Is a Join",
    Section 5.3).  Bit-exact."""
    if out is None:
        out = Relation(rel.dtype, rel.dims, parts, device=rel.storage.device)
        arr = None
    else:
        arr = None
    h = ctypes.c_void_p(out.handle.value)
    check_status(lib().ea_exchange(rel.handle, arr, ctypes.c_void_p(_stream_ptr(stream)), ctypes.byref(h)))
    return out


def exchange_agg(rel: Relation, agg: str, parts=None, out: Relation | None = None, stream=None) -> Relation:
    """Aggregate the m copies along ``rel``'s leading (copy) dimension with
    ``agg`` ("sum" or "max", in copy order) and re-block the result into the
    tiling ``parts`` of the remaining dimensions: the exchange with
    aggregation of "Every Kernel Is a Join", Section 5.3 / Example 5.4."""
    if out is None:
        out = Relation(rel.dtype, rel.dims[1:], parts, device=rel.storage.device)
    h = ctypes.c_void_p(out.handle.value)
    check_status(lib().ea_exchange_agg(rel.handle, AGGS[agg], None, ctypes.c_void_p(_stream_ptr(stream)),
                                       ctypes.byref(h)))
    return out


def copy_count(spec: str, inputs) -> int:
    """Function specifications per output block of a contraction: the
    product of the block counts of its aggregated letters."""
    terms, outl = _parse(spec)
    nb = {}
    for term, r in zip(terms, inputs):
        for l, b in zip(term, r.bounds):
            nb.setdefault(l, len(b) - 1)
    m = 1
    for l, n in nb.items():
        if l not in outl:
            m *= n
    return m


def _parse(spec: str):
    lhs, out = spec.split("->")
    return lhs.split(","), out


def output_layout(spec: str, inputs):
    """Extents and tilings of the output letters, taken from the inputs."""
    terms, out = _parse(spec)
    ext, bnd = {}, {}
    for term, r in zip(terms, inputs):
        for l, n, b in zip(term, r.dims, r.bounds):
            ext.setdefault(l, n)
            bnd.setdefault(l, b)
    return [ext[l] for l in out], [bnd[l] for l in out]


def joinagg(spec: str, inputs, agg: str = "sum", map: str = "product", out: Relation | None = None,
            out_dtype: str | None = None, scale: float = 1.0, eps: float = 0.0, pred: str | None = None,
            parts: dict | None = None, rope_table: torch.Tensor | None = None, rope_pos: str | None = None,
            out2: Relation | None = None, epi_map: str | None = None, epi_in: Relation | None = None,
            epi_pair: str | None = None, rope_dim: int = 0, row_rms: Relation | None = None,
            partials: bool = False, rope_layout: int = 0, simt_bf16: bool = False, stream=None) -> Relation:
    """Run one join-agg ("Every Kernel Is a Join", Definition 3.7) with
    libea.so.  ``pred="ts"`` keeps joined tuples with t <= s.  With
    ``agg="max_sumexp"`` the output receives the MAX and ``out2`` the SUM
    of exp(value - max).  A contraction may fuse an elementwise join into
    its epilogue: ``epi_map="add", epi_in=R`` stores value + R;
    ``epi_map="rope"`` rotates the output's column pairs (``rope_table``,
    ``rope_pos`` the row letter, pairs of period ``rope_dim``; a table
    [pairs, positions, 2] with ``rope_layout=1``);
    ``row_rms=ms`` multiplies every row r by rsqrt(ms[r] + eps) first;
    ``epi_map="silu_mul", epi_pair="c"`` plans letter c (extent 2, second
    input only) as the innermost output letter and stores SiLU(c=0) * (c=1).
    ``partials=True`` runs a contraction without its aggregation: the output
    gains a leading copy dimension of m unit blocks, copy q holding each
    block's q-th function specification alone (``exchange_agg`` sums them).
    A bf16 contraction the tensor-core kernel cannot tile raises unless
    ``simt_bf16=True`` lets it run on the (much slower) SIMT kernel."""
    if out is None:
        dims, bounds = output_layout(spec, inputs)
        if partials:
            m = copy_count(spec, inputs)
            dims, bounds = [m] + list(dims), [list(range(m + 1))] + list(bounds)
        out = Relation(out_dtype or inputs[0].dtype, dims, bounds, device=inputs[0].storage.device)
    handles = (ctypes.c_void_p * len(inputs))(*[r.handle.value for r in inputs])
    ip, n_parts, keep = _abi.index_parts(parts)
    o = _abi.Opts()
    o.out_dtype = 0
    o.scale = scale
    o.eps = eps
    if pred:
        o.pred_lo, o.pred_hi = pred[0].encode(), pred[1].encode()
    if rope_table is not None:
        o.rope_table = rope_table.data_ptr()
        o.rope_npos = rope_table.shape[1] if rope_layout == 1 else rope_table.shape[0]
        o.rope_pos = rope_pos.encode()
        o.rope_dim = rope_dim
        o.rope_layout = rope_layout
    if out2 is not None:
        o.out2 = out2.handle.value
    if row_rms is not None:
        o.row_rms = row_rms.handle.value
    o.partials = 1 if partials else 0
    o.simt_bf16 = 1 if simt_bf16 else 0
    if epi_map is not None:
        o.epi_map = MAPS[epi_map]
        if epi_in is not None:
            o.epi_in = epi_in.handle.value
        if epi_pair:
            o.epi_pair = epi_pair.encode()
    h = ctypes.c_void_p(out.handle.value)
    check_status(lib().ea_joinagg_run(spec.encode(), handles, len(inputs), ip, n_parts, AGGS[agg], MAPS[map],
                                      ctypes.byref(o), ctypes.c_void_p(_stream_ptr(stream)), ctypes.byref(h)))
    return out


def attention(spec: str, q: Relation, k: Relation, v: Relation, scale: float = 0.0, causal: bool = False,
              seq_ends=None, out: Relation | None = None, m_out: Relation | None = None,
              l_out: Relation | None = None, stream=None) -> Relation:
    """Flash attention as one join-agg ("Every Kernel Is a Join", Example
    3.10) with libea.so: ``spec`` such as "bshd,bthd,bthd->bshd"; a shared
    letter with g times more values in Q than in K groups query heads;
    ``seq_ends`` lists the end positions of packed sequences; ``scale`` 0
    means 1/sqrt(head dim).  Optional ``m_out``/``l_out`` (f32 over Q's
    letters without the head dim) receive the row max and row sum of exp."""
    if out is None:
        out = Relation("bf16", q.dims, q.bounds, device=q.storage.device)
    o = _abi.AttnOpts()
    o.scale = scale
    o.causal = 1 if causal else 0
    keep = None
    if seq_ends is not None:
        keep = _abi.i64(list(seq_ends))
        o.n_seq_ends = len(seq_ends)
        o.seq_ends = ctypes.cast(keep, ctypes.c_void_p)
    if m_out is not None:
        o.m_out = m_out.handle.value
    if l_out is not None:
        o.l_out = l_out.handle.value
    h = ctypes.c_void_p(out.handle.value)
    check_status(lib().ea_attention_run(spec.encode(), q.handle, k.handle, v.handle, ctypes.byref(o),
                                        ctypes.c_void_p(_stream_ptr(stream)), ctypes.byref(h)))
    del keep
    return out


# Callbacks handed to ea_set_allocator stay referenced for the life of the
# process: memory taken through them is released through them, possibly
# after the allocator has been switched back.
_allocators = []


def use_torch_allocator(enable: bool = True):
    """Route the library's own device memory (arenas of relations it creates
    with no storage given, device copies of cached plans) through torch's
    caching allocator on the current stream; ``enable=False`` goes back to
    cudaMalloc.  Relations built from Python always borrow torch storage."""
    if not enable:
        check_status(lib().ea_set_allocator(_abi.ALLOC_FN(), _abi.FREE_FN(), None))
        return

    def _alloc(n, ctx):
        try:
            return torch.cuda.caching_allocator_alloc(max(int(n), 1))
        except Exception:  # out of memory: the library reports EA_ERR_ALLOC
            return None

    def _free(p, ctx):
        torch.cuda.caching_allocator_delete(p)

    pair = (_abi.ALLOC_FN(_alloc), _abi.FREE_FN(_free))
    _allocators.append(pair)
    check_status(lib().ea_set_allocator(pair[0], pair[1], None))


def check(stream=None):
    """Synchronise the stream and raise on an asynchronous CUDA error or a
    raised device error flag."""
    check_status(lib().ea_check(ctypes.c_void_p(_stream_ptr(stream))))


def plan_cache_clear():
    check_status(lib().ea_plan_cache_clear())
