"""Workload chains written as compositions of cell-level join-aggs.

TEST INFRASTRUCTURE (see the package docstring).

"Every Kernel Is a Join", Section 1: every operation of a transformer
(attention, softmax, normalisation, elementwise maps, matrix multiply) is a
relational join followed by an aggregation.  Each function below writes an
operation as exactly such join-aggs, in fp64, with no fusion or reordering.

Readings taken where the pages say nothing (each is listed in the design
notes):
  * softmax over t: m = MAX_t S; E = exp(S - m); l = SUM_t E; P = E / l.
  * SiLU(z) = z / (1 + exp(-z)).
  * RMSNorm: ms = SUM_d x^2 / D;  y = x / sqrt(ms + eps) * gamma.
  * RoPE: interleaved pairs (2i, 2i+1) of the head dimension rotated by the
    angle pos * theta^(-2i/d_head); written as the contraction
    "bshiq,sipq->bship" with the 2x2 rotation relation R[s, i, p, q].
  * causal attention: the cell predicate t <= s on the score join.

Dense storage order: a relation's letters may be stored in any order (the
relation is the same set of cells); weight and value relations are stored
with their aggregated letter last, which keeps the index-nested-loop join
on contiguous memory.
"""
from __future__ import annotations

import numpy as np

from . import joinagg


def softmax_attention(Q, K, V, scale: float = 1.0, causal: bool = False, qspec: str = "bhsd", kspec: str = "bhtd",
                      vspec: str = "bhtd", ospec: str = "bhsd", tier: str = "idx"):
    """Scores, row max, row sum, probabilities and output of attention.

    Returns dict S, m, l, P, O (NaN marks cells removed by the predicate).
    """
    pred = "ts" if causal else None
    S = joinagg(f"{qspec},{kspec}->bhst", [Q, K], "product", "sum", scale=scale, pred=pred, tier=tier)
    m = joinagg("bhst->bhs", [S], "identity", "max", tier=tier)
    E = joinagg("bhst,bhs->bhst", [S, m], "exp_sub", "none", tier=tier)
    l = joinagg("bhst->bhs", [E], "identity", "sum", tier=tier)
    P = joinagg("bhst,bhs->bhst", [E, l], "div", "none", tier=tier)
    Vt = np.ascontiguousarray(np.transpose(V, [vspec.index(c) for c in "bhdt"]))
    O = joinagg(f"bhst,bhdt->{ospec}", [P, Vt], "product", "sum", tier=tier)
    return {"S": S, "m": m, "l": l, "E": E, "P": P, "O": O}


def flash_attention(Q, K, V, group: int = 1, scale: float = 1.0, causal: bool = False, seq_ends=None,
                    layout: str = "bhsd", tier: str = "idx"):
    """Flash attention with grouped-query heads and packed sequences
    ("Every Kernel Is a Join", Example 3.10), as the attention join-aggs of
    ``softmax_attention``.

    Q: [b, h_q, s, d] (layout "bhsd") or [b, s, h_q, d] ("bshd"); K, V the
    same with h_kv = h_q / group heads and t in place of s.  Query head h
    reads key-value head h // group (heads g*m .. g*m+g-1 share head m).
    ``seq_ends``: increasing positions at which the packed sequences end (the
    last equals the sequence extent); a query attends only to keys of its own
    sequence, so the join is taken separately on each sequence's positions.
    Causal keeps t <= s.  Returns dict O (in ``layout``), m and l ([b, h_q, s];
    m is the row maximum of the scaled scores, l the row sum of exp(S - m)).
    """
    if layout not in ("bhsd", "bshd"):
        raise ValueError(layout)
    to_bhsd = (lambda x: x) if layout == "bhsd" else (lambda x: np.transpose(x, (0, 2, 1, 3)))
    q, k, v = (np.ascontiguousarray(to_bhsd(np.asarray(x, dtype=np.float64))) for x in (Q, K, V))
    b, hq, s, d = q.shape
    hk, t = k.shape[1], k.shape[2]
    if hq != group * hk:
        raise ValueError("query heads must be group x key-value heads")
    heads = np.arange(hq) // group
    kq, vq = k[:, heads], v[:, heads]
    ends = [s] if seq_ends is None else [int(e) for e in seq_ends]
    if seq_ends is not None and s != t:
        raise ValueError("packed sequences need s == t")
    O = np.zeros((b, hq, s, d))
    m = np.full((b, hq, s), -np.inf)
    ell = np.zeros((b, hq, s))
    lo = 0
    for e in ends:
        qs = slice(lo, e)
        ks = slice(lo, e) if seq_ends is not None else slice(0, t)
        if e > lo and ks.stop > ks.start:
            r = softmax_attention(q[:, :, qs], kq[:, :, ks], vq[:, :, ks], scale=scale, causal=causal, tier=tier)
            O[:, :, qs], m[:, :, qs], ell[:, :, qs] = r["O"], r["m"], r["l"]
        lo = e
    O = O if layout == "bhsd" else np.transpose(O, (0, 2, 1, 3))
    return {"O": np.ascontiguousarray(O), "m": m, "l": ell}


def matrix_chain(mats, paren, tier: str = "idx"):
    """The product of a chain of matrices in a fixed parenthesization ("Every
    Kernel Is a Join", Section 7: the matrix-chain workloads), every multiply
    the contraction join-agg "ij,jk->ik".

    mats: list of 2-D arrays M1..Mn; paren: nested pairs of 1-based matrix
    indices, e.g. ((1, 2), 3).  Returns the product (fp64).
    """
    def ev(node):
        if isinstance(node, int):
            return np.asarray(mats[node - 1], dtype=np.float64)
        left, right = ev(node[0]), ev(node[1])
        return joinagg("ij,kj->ik", [left, np.ascontiguousarray(right.T)], "product", "sum", tier=tier)
    return ev(paren)


def swiglu_ffn(x, w_gate, w_up, w_down, tier: str = "idx"):
    """G = x w_gate, U = x w_up (SUM over the model dimension),
    H = SiLU(G) * U (elementwise join), Y = H w_down."""
    G = joinagg("ij,kj->ik", [x, np.ascontiguousarray(w_gate.T)], "product", "sum", tier=tier)
    U = joinagg("ij,kj->ik", [x, np.ascontiguousarray(w_up.T)], "product", "sum", tier=tier)
    H = joinagg("ik,ik->ik", [G, U], "silu_mul", "none", tier=tier)
    Y = joinagg("ik,jk->ij", [H, np.ascontiguousarray(w_down.T)], "product", "sum", tier=tier)
    return {"G": G, "U": U, "H": H, "Y": Y}


def rmsnorm(x, gamma, eps: float, tier: str = "idx"):
    """x: [t, d]; gamma: [d]."""
    D = x.shape[1]
    ms = joinagg("td->t", [x], "square", "sum", scale=1.0 / D, tier=tier)
    y = joinagg("td,t,d->td", [x, ms, gamma], "rms_apply", "none", eps=eps, tier=tier)
    return {"ms": ms, "y": y}


def rope_rotation(n_pos: int, d_head: int, theta: float) -> np.ndarray:
    """R[s, i, p, q]: rotation of pair i at position s (fp64)."""
    i = np.arange(d_head // 2, dtype=np.float64)
    inv = theta ** (-2.0 * i / d_head)
    ang = np.arange(n_pos, dtype=np.float64)[:, None] * inv[None, :]
    c, s = np.cos(ang), np.sin(ang)
    R = np.empty((n_pos, d_head // 2, 2, 2))
    R[:, :, 0, 0] = c
    R[:, :, 0, 1] = -s
    R[:, :, 1, 0] = s
    R[:, :, 1, 1] = c
    return R


def rope(x, theta: float, tier: str = "idx"):
    """x: [b, s, h, d] with positions 0..s-1 along s."""
    b, s, h, d = x.shape
    xr = np.ascontiguousarray(x).reshape(b, s, h, d // 2, 2)
    R = rope_rotation(s, d, theta)
    y = joinagg("bshiq,sipq->bship", [xr, R], "product", "sum", tier=tier)
    return y.reshape(b, s, h, d)


def llama_block(x, W, n_heads: int, eps: float = 1e-6, theta: float = 10000.0, tier: str = "idx"):
    """Pre-norm LLaMA-style block (multi-head attention, no biases, causal).

    x: [b, s, D]; W: dict with wq, wk, wv, wo [D, D], w_gate, w_up [D, F],
    w_down [F, D], g1, g2 [D].  Projections are x W (row vector times matrix).
    Returns a dict with the intermediates and the block output ``y``.
    """
    b, s, D = x.shape
    dh = D // n_heads
    xt = x.reshape(b * s, D)
    n1 = rmsnorm(xt, W["g1"], eps, tier)["y"]
    proj = lambda a, w: joinagg("td,ed->te", [a, np.ascontiguousarray(w.T)], "product", "sum", tier=tier)  # noqa: E731
    q = proj(n1, W["wq"]).reshape(b, s, n_heads, dh)
    k = proj(n1, W["wk"]).reshape(b, s, n_heads, dh)
    v = proj(n1, W["wv"]).reshape(b, s, n_heads, dh)
    qr = rope(q, theta, tier)
    kr = rope(k, theta, tier)
    att = softmax_attention(qr, kr, v, scale=1.0 / np.sqrt(dh), causal=True, qspec="bshd", kspec="bthd",
                            vspec="bthd", ospec="bshd", tier=tier)
    o = att["O"].reshape(b * s, D)
    a = proj(o, W["wo"])
    h = joinagg("td,td->td", [xt, a], "add", "none", tier=tier)
    n2 = rmsnorm(h, W["g2"], eps, tier)["y"]
    f = swiglu_ffn(n2, W["w_gate"], W["w_up"], W["w_down"], tier)
    y = joinagg("td,td->td", [h, f["Y"]], "add", "none", tier=tier)
    return {"n1": n1, "q": qr, "k": kr, "v": v, "S": att["S"], "m": att["m"], "l": att["l"], "P": att["P"],
            "O": att["O"], "attn": a, "h": h, "n2": n2, "G": f["G"], "U": f["U"], "H": f["H"], "Y": f["Y"],
            "y": y.reshape(b, s, D)}
