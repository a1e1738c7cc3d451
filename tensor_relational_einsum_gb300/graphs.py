"""Workloads of the hot path as graphs of join-aggs and exchanges.

Each class allocates its relations once and ``run()`` enqueues the calls on
the current stream -- the single-GPU counterpart of compiling a plan into
one CUDA graph of kernel invocations ("Every Kernel Is a Join", Section 6).
All arithmetic runs in libea.so.

* ``AttentionChain``  scores -> MAX -> SUM of exp -> normalise -> values
                      (softmax over t as MAX then SUM aggregations with an
                      exp map, Section 1's "softmax as join + aggregation").
* ``FusedAttention``  the same attention as one join-agg (Example 3.10):
                      the key tiles of a query tile aggregated with the
                      merge of (max, sum of exp, weighted sum) triples in one
                      tcgen05 kernel.
* ``SwigluFFN``       gate/up contractions (SUM over model-dim blocks),
                      SiLU(gate) * up elementwise join, down contraction.
* ``MatrixChain``     the pages' matrix-chain workloads (chains A-E): a
                      fixed parenthesization, every multiply one contraction
                      join-agg over near-equal blocks.
* ``LlamaBlock``      pre-norm block: RMSNorm, Q,K contraction with RoPE in its
                      epilogue and V contraction (or fused QKV then RoPE),
                      causal attention (fused, or the chain), O projection
                      reading the attention output in place (+ residual in
                      its epilogue), RMSNorm, SwiGLU FFN (SiLU * up and the
                      second residual in the contraction epilogues); or the
                      same with every join unfused and an exchange of the
                      attention output into the O projection's tiling.
"""
from __future__ import annotations

import math

import numpy as np
import torch

from . import _abi
from .relation import Relation, attention, exchange, joinagg


class Recorder:
    """Brackets every call with CUDA events on the current stream and notes
    which kernel class it launched (for per-kernel timing and launch
    counts)."""

    def __init__(self):
        self.calls = []  # (name, kernel class, launches, start event, end event)

    def call(self, name, fn):
        s = torch.cuda.Event(enable_timing=True)
        e = torch.cuda.Event(enable_timing=True)
        s.record()
        fn()
        e.record()
        lp = _abi.last_plan()
        self.calls.append((name, lp["kernel"], lp["launches"], s, e))

    def summary(self):
        """name -> (kernel class, launches per call, list of ms)."""
        out = {}
        for name, k, n, s, e in self.calls:
            ent = out.setdefault(name, [k, n, []])
            ent[2].append(s.elapsed_time(e))
        return out


def _direct(name, fn):
    fn()


def capture(fn, warmup: int = 2) -> "torch.cuda.CUDAGraph":
    """Record ``fn``'s libea launches into one CUDA graph ("Every Kernel Is a
    Join", Section 6: every plan is compiled to a CUDA graph and executed
    directly).  ``fn`` runs ``warmup`` times first on a side stream, which
    builds, uploads and caches every plan, so the capture itself makes no
    allocation or synchronisation; ``graph.replay()`` then launches the same
    kernels with the same arguments on the current stream."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(warmup):
            fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, capture_error_mode="thread_local"):
        fn()
    return g


def view(parent: Relation, offset_elems: int, dims, parts) -> Relation:
    """A relation over a contiguous piece of ``parent``'s arena (zero-copy)."""
    n = int(np.prod(dims))
    return Relation(parent.dtype, dims, parts, storage=parent.storage[offset_elems:offset_elems + n])


def rope_table(n_pos: int, d_head: int, theta: float, device="cuda") -> torch.Tensor:
    """fp32 [n_pos, d_head/2, 2] = (cos, sin) of pos * theta^(-2i/d_head),
    angles evaluated in float64 on the host."""
    i = np.arange(d_head // 2, dtype=np.float64)
    inv = np.power(theta, -2.0 * i / d_head)
    ang = np.arange(n_pos, dtype=np.float64)[:, None] * inv[None, :]
    tab = np.stack([np.cos(ang), np.sin(ang)], axis=-1).astype(np.float32)
    return torch.from_numpy(tab).to(device)


class AttentionChain:
    """Q, K, V relations [b, h, s|t, d] (bf16) tiled on b and h; t (and the
    scores' t) in ``t_blocks`` blocks; optional causal predicate t <= s and
    score scale."""

    def __init__(self, Q: Relation, K: Relation, V: Relation, scale: float = 1.0, causal: bool = False,
                 qspec: str = "bhsd", kspec: str = "bhtd", vspec: str = "bhtd", ospec: str = "bhsd",
                 fused_stats: bool = True):
        self.Q, self.K, self.V = Q, K, V
        self.fused_stats = fused_stats
        self.scale, self.pred = scale, ("ts" if causal else None)
        self.s_spec = f"{qspec},{kspec}->bhst"
        self.o_spec = f"bhst,{vspec}->{ospec}"
        ext, bnd = {}, {}
        for spec, r in ((qspec, Q), (kspec, K), (vspec, V)):
            for l, n, b in zip(spec, r.dims, r.bounds):
                ext[l], bnd[l] = n, b
        dev = Q.storage.device
        self.S = Relation("f32", [ext[l] for l in "bhst"], [bnd[l] for l in "bhst"], device=dev)
        self.m = Relation("f32", [ext[l] for l in "bhs"], [bnd[l] for l in "bhs"], device=dev)
        self.l = Relation("f32", [ext[l] for l in "bhs"], [bnd[l] for l in "bhs"], device=dev)
        self.P = Relation("bf16", [ext[l] for l in "bhst"], [bnd[l] for l in "bhst"], device=dev)
        self.O = Relation("bf16", [ext[l] for l in ospec], [bnd[l] for l in ospec], device=dev)
        self.ext = ext

    def run(self, rec: Recorder | None = None):
        c = rec.call if rec is not None else _direct
        c("attn.scores", lambda: joinagg(self.s_spec, [self.Q, self.K], "sum", "product", out=self.S,
                                         scale=self.scale, pred=self.pred))
        if self.fused_stats:
            # MAX and SUM of exp in one pass over the scores
            c("attn.stats", lambda: joinagg("bhst->bhs", [self.S], "max_sumexp", "identity", out=self.m,
                                            out2=self.l, pred=self.pred))
        else:
            c("attn.max", lambda: joinagg("bhst->bhs", [self.S], "max", "identity", out=self.m, pred=self.pred))
            c("attn.sumexp", lambda: joinagg("bhst,bhs->bhs", [self.S, self.m], "sum", "exp_sub", out=self.l,
                                             pred=self.pred))
        c("attn.normalise", lambda: joinagg("bhst,bhs,bhs->bhst", [self.S, self.m, self.l], "none", "exp_sub_div",
                                            out=self.P, pred=self.pred))
        c("attn.values", lambda: joinagg(self.o_spec, [self.P, self.V], "sum", "product", out=self.O,
                                         pred=self.pred))
        return self.O

    def flops(self) -> float:
        e = self.ext
        full = 2.0 * e["b"] * e["h"] * e["s"] * e["t"] * e["d"] * 2
        return full


class FusedAttention:
    """Q [.., s, .., d], K and V [.., t, .., d] (bf16) as one attention
    join-agg; ``spec`` names the roles ("bshd,bthd,bthd->bshd")."""

    def __init__(self, Q: Relation, K: Relation, V: Relation, spec: str, scale: float = 0.0, causal: bool = False):
        self.Q, self.K, self.V, self.spec = Q, K, V, spec
        self.scale, self.causal = scale, causal
        self.O = Relation("bf16", Q.dims, Q.bounds, device=Q.storage.device)

    def run(self, rec: Recorder | None = None):
        c = rec.call if rec is not None else _direct
        c("attn.fused", lambda: attention(self.spec, self.Q, self.K, self.V, scale=self.scale, causal=self.causal,
                                          out=self.O))
        return self.O


class SwigluFFN:
    """x [T, D] tiled (t_blocks, 4); w_gate, w_up [D, F] and w_down [F, D];
    contracted dims in ``k_blocks`` blocks (partial products SUM-aggregate).

    fused: gate and up are one weight relation [D, F, 2] (c innermost), and
    the elementwise join H = SiLU(G) * U runs in the contraction's epilogue
    over the c pairs, so G and U are never written; the down projection can
    fuse a residual join (Y = H w_down + residual).  Unfused: the three
    join-aggs of the chain, with G and U as halves of one [2, T, F] output."""

    def __init__(self, x: Relation, w_gate: torch.Tensor, w_up: torch.Tensor, w_down: torch.Tensor,
                 k_blocks: int = 4, out: Relation | None = None, fused: bool = True,
                 residual: Relation | None = None, gain: Relation | None = None,
                 row_rms: Relation | None = None, eps: float = 0.0):
        T, D = x.dims
        F = w_gate.shape[1]
        tb = x.bounds[0]
        dev = x.storage.device
        self.x = x
        self.fused = fused
        self.residual = residual
        self.row_rms, self.eps = row_rms, eps
        if fused:
            self.wgu = Relation.from_dense(torch.stack([w_gate, w_up], dim=2).contiguous(), [x.bounds[1], k_blocks, 1])
            if gain is not None:  # an RMSNorm gain over the contracted letter, folded into the weight once
                self.wgu = joinagg("dfc,d->dfc", [self.wgu, gain], "none", "product")
            self.G = self.U = None
        else:
            # gate and up share their join: one relation [D, 2, F] (c = 0 gate, 1 up)
            gu = torch.stack([w_gate, w_up], dim=1).contiguous()
            self.wgu = Relation.from_dense(gu, [x.bounds[1], 2, k_blocks])
            self.gu = Relation("bf16", (2, T, F), [2, tb, k_blocks], device=dev)
            half = T * F
            self.G = view(self.gu, 0, (T, F), [tb, k_blocks])
            self.U = view(self.gu, half, (T, F), [tb, k_blocks])
        self.wd = Relation.from_dense(w_down.contiguous(), [k_blocks, x.bounds[1]])
        self.H = Relation("bf16", (T, F), [tb, k_blocks], device=dev)
        self.Y = out if out is not None else Relation("bf16", (T, D), [tb, x.bounds[1]], device=dev)
        self.T, self.D, self.F = T, D, F

    def run(self, x: Relation | None = None, rec: Recorder | None = None, out: Relation | None = None):
        x = x or self.x
        Y = out or self.Y
        c = rec.call if rec is not None else _direct
        if self.fused:
            c("ffn.gate_up", lambda: joinagg("td,dfc->tf", [x, self.wgu], "sum", "product", out=self.H,
                                             epi_map="silu_mul", epi_pair="c", row_rms=self.row_rms, eps=self.eps))
        else:
            c("ffn.gate_up", lambda: joinagg("td,dcf->ctf", [x, self.wgu], "sum", "product", out=self.gu))
            c("ffn.silu_mul", lambda: joinagg("tf,tf->tf", [self.G, self.U], "none", "silu_mul", out=self.H))
        if self.residual is not None:
            c("ffn.down", lambda: joinagg("tf,fd->td", [self.H, self.wd], "sum", "product", out=Y,
                                          epi_map="add", epi_in=self.residual))
        else:
            c("ffn.down", lambda: joinagg("tf,fd->td", [self.H, self.wd], "sum", "product", out=Y))
        return Y

    def flops(self) -> float:
        return 2.0 * self.T * self.D * self.F * 3


# The matrix chains of the evaluation ("Every Kernel Is a Join", Section 7):
# dimensions d0..dn (matrix i is d[i-1] x d[i]) and the fixed parenthesization.
def _alt(ends, a, b, n):
    return [ends] + [a if i % 2 == 0 else b for i in range(n - 1)] + [ends]


def _necked(ends, neck, inner, n):
    return [ends, neck] + [inner] * (n - 3) + [neck, ends]


def _right_nested(lo, hi):
    node = (hi - 1, hi)
    for i in range(hi - 2, lo - 1, -1):
        node = (i, node)
    return node


CHAINS = {
    "A": (_alt(10240, 16384, 6144, 9), (((1, 2), ((3, 4), ((5, 6), (7, 8)))), 9)),
    "B": (_alt(9216, 20480, 5120, 5), ((1, 2), ((3, 4), 5))),
    "C": ([10240, 12288, 32768, 2048], (1, (2, 3))),
    "D": (_necked(24576, 1536, 20480, 9), ((1, _right_nested(2, 8)), 9)),
    "E": (_necked(49152, 1024, 20480, 13), ((1, _right_nested(2, 12)), 13)),
}


def chain_blocks(d: int, block: int = 4096) -> int:
    """Near-equal blocks of about ``block`` along a chain dimension."""
    return max(1, round(d / block))


class MatrixChain:
    """A chain of bf16 matrices multiplied in a fixed parenthesization, every
    multiply the contraction join-agg "ij,jk->ik" (SUM over the contracted
    dimension's blocks fused in the accumulator); every dimension tiled into
    near-equal blocks of about 4096.  ``mats``: torch tensors M1..Mn."""

    def __init__(self, mats, paren, block: int = 4096):
        self.paren = paren
        self.rels = [Relation.from_dense(m.contiguous(), [chain_blocks(m.shape[0], block),
                                                          chain_blocks(m.shape[1], block)]) for m in mats]
        self.steps = []          # (left, right, out) in evaluation order
        self.flop = 0.0
        self.out = self._plan(paren)

    def _plan(self, node):
        if isinstance(node, int):
            return self.rels[node - 1]
        left, right = self._plan(node[0]), self._plan(node[1])
        out = Relation("bf16", (left.dims[0], right.dims[1]), [left.bounds[0], right.bounds[1]],
                       device=left.storage.device)
        self.steps.append((left, right, out))
        self.flop += 2.0 * left.dims[0] * left.dims[1] * right.dims[1]
        return out

    def run(self, rec: Recorder | None = None):
        c = rec.call if rec is not None else _direct
        for i, (l, r, o) in enumerate(self.steps):
            c(f"chain.{i}", lambda l=l, r=r, o=o: joinagg("ij,jk->ik", [l, r], "sum", "product", out=o))
        return self.out


class LlamaBlock:
    """Pre-norm LLaMA-style block over x [b * s, D] (bf16), tokens tiled one
    sequence per block and the model dimension in ``d_blocks`` blocks."""

    def __init__(self, b: int, s: int, D: int, n_heads: int, F: int, W: dict, eps: float = 1e-6,
                 theta: float = 10000.0, d_blocks: int = 4, s_blocks: int = 4, device="cuda",
                 fused_attention: bool = True, fused_epilogues: bool = True):
        self.b, self.s, self.D, self.H, self.F = b, s, D, n_heads, F
        self.dh = D // n_heads
        T = b * s
        self.T = T
        self.eps = eps
        dev = device
        db, sb = d_blocks, s_blocks
        tb = b  # one block of tokens per sequence
        self.x = Relation("bf16", (T, D), [tb, db], device=dev)
        self.g1 = Relation.from_dense(W["g1"].contiguous(), [db])
        self.g2 = Relation.from_dense(W["g2"].contiguous(), [db])
        if fused_epilogues:
            # Q and K in one contraction with RoPE in its epilogue, V in another;
            # RMSNorm's gain folded into the weights, its row scale in the epilogues
            wqk = Relation.from_dense(torch.stack([W["wq"], W["wk"]], dim=1).contiguous(), [db, 2, 1])
            self.wqk = joinagg("dce,d->dce", [wqk, self.g1], "none", "product")
            self.wv = joinagg("de,d->de", [Relation.from_dense(W["wv"].contiguous(), [db, 1]), self.g1], "none",
                              "product")
        else:
            wqkv = torch.stack([W["wq"], W["wk"], W["wv"]], dim=1).contiguous()     # [D, 3, D]
            self.wqkv = Relation.from_dense(wqkv, [db, 3, 1])
        # the O projection contracts the whole model dim (one block) when it
        # reads the attention output in place (fused path), else db blocks
        self.wo = Relation.from_dense(W["wo"].contiguous(), [1 if fused_epilogues else db, db])
        self.ms1 = Relation("f32", (T,), [tb], device=dev)
        self.n1 = None if fused_epilogues else Relation("bf16", (T, D), [tb, db], device=dev)
        self.qkv = Relation("bf16", (3, T, D), [3, tb, 1], device=dev)
        hd = (b, s, n_heads, self.dh)
        attn_parts = [b, sb, 1, 1]
        self.q = view(self.qkv, 0, hd, attn_parts)
        self.k = view(self.qkv, T * D, hd, attn_parts)
        self.v = view(self.qkv, 2 * T * D, hd, attn_parts)
        self.qk_out = view(self.qkv, 0, (2, T, D), [2, tb, 1])
        self.v_out = view(self.qkv, 2 * T * D, (T, D), [tb, 1])
        if fused_epilogues:
            self.qr, self.kr = self.q, self.k      # rotated in place by the epilogue
        else:
            self.qr = Relation("bf16", hd, attn_parts, device=dev)
            self.kr = Relation("bf16", hd, attn_parts, device=dev)
        self.table = rope_table(s, self.dh, theta, device=dev)
        self.table_pm = self.table.transpose(0, 1).contiguous()  # [pairs, positions, 2] for the epilogue
        self.fused_epilogues = fused_epilogues
        self.fused_attention = fused_attention
        if fused_attention:
            self.attn = FusedAttention(self.qr, self.kr, self.v, "bshd,bthd,bthd->bshd", scale=1.0 / math.sqrt(self.dh),
                                       causal=True)
        else:
            self.attn = AttentionChain(self.qr, self.kr, self.v, scale=1.0 / math.sqrt(self.dh), causal=True,
                                       qspec="bshd", kspec="bthd", vspec="bthd", ospec="bshd")
        # the attention output, seen as [T, D] in blocks of s / s_blocks tokens x all heads ...
        self.o_tok = view(self.attn.O, 0, (T, D), [b * sb, 1])
        # ... re-blocked by the exchange into the O projection's contraction
        # tiling (unfused path); with the model dim in one block the same
        # arena is already a [T, D] relation in blocks of one sequence (the
        # rows of all heads of a token are contiguous), which the fused path's
        # O projection reads in place
        self.o_ex = None if fused_epilogues else Relation("bf16", (T, D), [tb, db], device=dev)
        self.o_rows = view(self.attn.O, 0, (T, D), [tb, 1])
        self.a = None if fused_epilogues else Relation("bf16", (T, D), [tb, db], device=dev)
        self.h = Relation("bf16", (T, D), [tb, db], device=dev)
        self.ms2 = Relation("f32", (T,), [tb], device=dev)
        self.n2 = None if fused_epilogues else Relation("bf16", (T, D), [tb, db], device=dev)
        self.y = Relation("bf16", (T, D), [tb, db], device=dev)
        if fused_epilogues:
            # residual joins in the O-projection and down-projection epilogues
            self.ffn = SwigluFFN(self.h, W["w_gate"], W["w_up"], W["w_down"], k_blocks=db, out=self.y, fused=True,
                                 residual=self.h, gain=self.g2, row_rms=self.ms2, eps=eps)
        else:
            self.ffn = SwigluFFN(self.n2, W["w_gate"], W["w_up"], W["w_down"], k_blocks=db, out=None, fused=False)
        self.ffn_out = self.ffn.Y

    def rmsnorm(self, x, ms, g, out, c, tag):
        c(tag + ".sumsq", lambda: joinagg("td->t", [x], "sum", "square", out=ms, scale=1.0 / self.D))
        c(tag + ".apply", lambda: joinagg("td,t,d->td", [x, ms, g], "none", "rms_apply", out=out, eps=self.eps))

    def run(self, rec: Recorder | None = None, x: Relation | None = None, y: Relation | None = None):
        """One block forward on ``x`` (default: the block's own input
        relation) into ``y`` (default: its own output); both tiled like the
        block's, e.g. double buffers a pipelined caller fills and drains."""
        c = rec.call if rec is not None else _direct
        x = x or self.x
        y = y or self.y
        if self.fused_epilogues:
            c("norm1.sumsq", lambda: joinagg("td->t", [x], "sum", "square", out=self.ms1, scale=1.0 / self.D))
            c("qkv", lambda: joinagg("td,dce->cte", [x, self.wqk], "sum", "product", out=self.qk_out,
                                     epi_map="rope", rope_table=self.table_pm, rope_layout=1, rope_pos="t",
                                     rope_dim=self.dh, row_rms=self.ms1, eps=self.eps))
            c("qkv.v", lambda: joinagg("td,de->te", [x, self.wv], "sum", "product", out=self.v_out,
                                       row_rms=self.ms1, eps=self.eps))
        else:
            self.rmsnorm(x, self.ms1, self.g1, self.n1, c, "norm1")
            c("qkv", lambda: joinagg("td,dce->cte", [self.n1, self.wqkv], "sum", "product", out=self.qkv))
            c("rope.q", lambda: joinagg("bshd->bshd", [self.q], "none", "rope", out=self.qr, rope_table=self.table,
                                        rope_pos="s"))
            c("rope.k", lambda: joinagg("bshd->bshd", [self.k], "none", "rope", out=self.kr, rope_table=self.table,
                                        rope_pos="s"))
        self.attn.run(rec)
        if self.fused_epilogues:
            c("o_proj", lambda: joinagg("te,ed->td", [self.o_rows, self.wo], "sum", "product", out=self.h,
                                        epi_map="add", epi_in=x))
        else:
            c("exchange.attn_out", lambda: exchange(self.o_tok, None, out=self.o_ex))
            c("o_proj", lambda: joinagg("te,ed->td", [self.o_ex, self.wo], "sum", "product", out=self.a))
            c("residual1", lambda: joinagg("td,td->td", [x, self.a], "none", "add", out=self.h))
        if self.fused_epilogues:
            c("norm2.sumsq", lambda: joinagg("td->t", [self.h], "sum", "square", out=self.ms2, scale=1.0 / self.D))
            self.ffn.run(self.h, rec, out=y)
        else:
            self.rmsnorm(self.h, self.ms2, self.g2, self.n2, c, "norm2")
            self.ffn.run(self.n2, rec)
        if not self.fused_epilogues:
            c("residual2", lambda: joinagg("td,td->td", [self.h, self.ffn_out], "none", "add", out=y))
        return y

    def call_bytes(self) -> dict:
        """Algorithmic bytes of each call: every input relation read once,
        every output relation written once (written score blocks only)."""
        T, D, F = self.T, self.D, self.F
        x = T * D * 2
        nb = len(self.qr.bounds[1]) - 1                # s (and t) blocks
        sb = self.s // nb
        kept = nb * (nb + 1) // 2                     # (s, t) blocks the causal filter keeps
        S = self.b * self.H * kept * sb * sb * 4
        P = S // 2
        ml = self.b * self.H * self.s * 4
        fe = self.fused_epilogues
        return {"norm1.sumsq": x + T * 4, "norm1.apply": 2 * x + T * 4 + D * 2,
                "qkv": (3 * x + 2 * D * D * 2) if fe else (4 * x + 3 * D * D * 2), "qkv.v": 2 * x + D * D * 2,
                "rope.q": 2 * x, "rope.k": 2 * x, "attn.scores": 2 * x + S, "attn.stats": S + 2 * ml,
                "attn.normalise": S + 2 * ml + P, "attn.values": P + 2 * x, "attn.fused": 4 * x,
                "exchange.attn_out": 2 * x,
                "o_proj": (3 if fe else 2) * x + D * D * 2, "residual1": 3 * x, "norm2.sumsq": x + T * 4,
                "norm2.apply": 2 * x + T * 4 + D * 2,
                "ffn.gate_up": x + 2 * D * F * 2 + (1 if fe else 2) * T * F * 2,
                "ffn.silu_mul": 3 * T * F * 2, "ffn.down": T * F * 2 + F * D * 2 + (2 if fe else 1) * x,
                "residual2": 3 * x}

    def call_flops(self) -> dict:
        """Algorithmic FLOPs of each contraction call."""
        T, D, F = self.T, self.D, self.F
        causal_pairs = self.b * self.H * self.s * (self.s + 1) / 2
        qkv = 2.0 * T * D * (2 if self.fused_epilogues else 3) * D
        return {"qkv": qkv, "qkv.v": 2.0 * T * D * D, "o_proj": 2.0 * T * D * D, "ffn.gate_up": 2.0 * T * D * 2 * F,
                "ffn.down": 2.0 * T * F * D, "attn.scores": 2.0 * causal_pairs * self.dh,
                "attn.values": 2.0 * causal_pairs * self.dh, "attn.fused": 4.0 * causal_pairs * self.dh}

    def flops(self) -> dict:
        """Algorithmic FLOPs: projections and FFN dense; attention over the
        causal join (cells with t <= s)."""
        T, D, F = self.T, self.D, self.F
        proj = 2.0 * T * D * D * 4
        ffn = 2.0 * T * D * F * 3
        causal_pairs = self.b * self.H * self.s * (self.s + 1) / 2
        attn = 2.0 * causal_pairs * self.dh * 2
        return {"proj": proj, "ffn": ffn, "attn": attn, "total": proj + ffn + attn}
