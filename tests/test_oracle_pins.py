"""Pins for the fp64 oracle: things other than the oracle itself that fix
its results -- worked examples printed on the pages, closed forms, a library
routine on special cases (numpy.einsum), brute force on tiny inputs and
mathematical invariants.  CPU only.
"""
import itertools
import json
import os

import numpy as np
import pytest

import oracle
from oracle import blocked, chains, worklist

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def rng(seed=0):
    return np.random.default_rng(seed)


# ------------------------------------------------------------ worked examples

def test_ex38_worklist_matches_page():
    g = gold("ex3_8_matmul_worklist.json")
    wl = worklist.worklist(g["spec"], g["bounds"])
    assert len(wl["tuples"]) == g["n_function_specs"]
    assert len(wl["groups"]) == len(g["output_blocks"])
    # F_{m,n}: A block (m-th interval of i, n-th of j) = id (m-1)*2+(n-1); B block = n-1.
    for gi, members in enumerate(g["groups_as_mn"]):
        got = wl["tuples"][wl["grp_ptr"][gi]:wl["grp_ptr"][gi + 1]]
        want = [((m - 1) * 2 + (n - 1), n - 1) for m, n in members]
        assert got == want
    # output block keys: group id -> (i interval, k interval) -> lo/hi
    for gi, ob in enumerate(wl["groups"]):
        bi = ob  # k has one interval, so the output block id is the i interval
        lo = [g["bounds"]["i"][bi], 0]
        hi = [g["bounds"]["i"][bi + 1], 256]
        assert {"lo": lo, "hi": hi} == g["output_blocks"][gi]


@pytest.mark.parametrize("case", gold("matmul3d_volumes.json")["cases"])
def test_matmul3d_closed_forms(case):
    N, a, b, c = case["N"], case["a"], case["b"], case["c"]
    wl = worklist.worklist("ij,jk->ik", {"i": oracle.near_equal_bounds(N, a), "j": oracle.near_equal_bounds(N, b),
                                         "k": oracle.near_equal_bounds(N, c)})
    assert len(wl["tuples"]) == case["tuples"] == a * b * c
    assert wl["join_volume"] == case["join"] == (a + c) * N * N
    assert wl["agg_volume"] == case["agg"] == (b - 1) * N * N
    assert len(wl["groups"]) == a * c
    assert all(wl["grp_ptr"][i + 1] - wl["grp_ptr"][i] == b for i in range(a * c))


def test_ex54_overlay_atoms():
    g = gold("ex5_4_overlay.json")
    prod = [g["producer_row_bounds"], [0, g["cols"]]]
    cons = [g["consumer_row_bounds"], [0, g["cols"]]]
    ov = worklist.overlay(prod, cons)
    assert ov[0] == g["overlay_row_splits"]
    at = worklist.atoms(prod, cons)
    assert len(at) == g["n_atoms"]
    for i in range(len(g["producer_row_bounds"]) - 1):
        lo, hi = g["producer_row_bounds"][i], g["producer_row_bounds"][i + 1]
        inside = [a for a in at if a[0][0] >= lo and a[0][1] <= hi]
        assert len(inside) == g["atoms_per_producer_block"]
        assert sum(a[0][1] - a[0][0] for a in inside) == hi - lo


def test_function_spec_count_is_product_of_intervals():
    # Section 3.3: prod_s intervals[s] function specifications.
    b = {"b": [0, 1, 2], "h": [0, 2, 3, 4], "s": [0, 5], "t": [0, 2, 4, 7], "d": [0, 3, 6]}
    wl = worklist.worklist("bhsd,bhtd->bhst", b)
    assert len(wl["tuples"]) == 2 * 3 * 1 * 3 * 2
    assert len(wl["groups"]) == 2 * 3 * 1 * 3


# ------------------------------------------- library routine special cases

EINSUM_CASES = [
    ("ij,jk->ik", [(5, 7), (7, 3)]),
    ("ij,kj->ik", [(4, 6), (5, 6)]),
    ("bhsd,bhtd->bhst", [(2, 3, 4, 5), (2, 3, 6, 5)]),
    ("bhst,bhtd->bhsd", [(2, 2, 3, 4), (2, 2, 4, 5)]),
    ("ij,j->i", [(4, 9), (9,)]),
    ("i,j->ij", [(3,), (4,)]),
    ("ij->j", [(6, 4)]),
    ("ijk,kl,lm->im", [(2, 3, 4), (4, 5), (5, 2)]),
    ("ij,ij->", [(3, 4), (3, 4)]),
]


@pytest.mark.parametrize("tier", ["lit", "idx"])
@pytest.mark.parametrize("spec,shapes", EINSUM_CASES)
def test_sum_product_equals_numpy_einsum(tier, spec, shapes):
    r = rng(hash(spec) % 1000)
    arrs = [r.standard_normal(s) for s in shapes]
    got = oracle.joinagg(spec, arrs, "product", "sum", tier=tier)
    want = np.einsum(spec, *arrs)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("tier", ["lit", "idx"])
def test_max_aggregation_equals_numpy_max(tier):
    a = rng(3).standard_normal((4, 5, 7))
    got = oracle.joinagg("bst->bs", [a], "identity", "max", tier=tier)
    np.testing.assert_array_equal(got, a.max(axis=2))


def test_brute_force_dictionary_join_tiny():
    """A dictionary-of-cells join written out by hand (Section 1's
    degenerate relational form), independent of orc.c."""
    r = rng(4)
    A = r.integers(-3, 4, (3, 4)).astype(float)
    B = r.integers(-3, 4, (4, 2)).astype(float)
    RA = {(i, j): A[i, j] for i in range(3) for j in range(4)}
    RB = {(j, k): B[j, k] for j in range(4) for k in range(2)}
    groups = {}
    for (i, j), va in RA.items():
        for (j2, k), vb in RB.items():
            if j == j2:
                groups.setdefault((i, k), []).append(va * vb)
    want = np.zeros((3, 2))
    for (i, k), vals in groups.items():
        want[i, k] = sum(vals)
    for tier in ("lit", "idx"):
        assert np.array_equal(oracle.joinagg("ij,jk->ik", [A, B], tier=tier), want)


def test_integer_inputs_exact():
    r = rng(5)
    A = r.integers(-2, 3, (64, 96)).astype(float)
    B = r.integers(-2, 3, (96, 80)).astype(float)
    want = (A.astype(np.int64) @ B.astype(np.int64)).astype(float)
    assert np.array_equal(oracle.joinagg("ij,jk->ik", [A, B], tier="lit"), want)
    assert np.array_equal(oracle.joinagg("ij,jk->ik", [A, B], tier="idx"), want)


def test_literal_join_counts_joined_tuples():
    A = np.ones((3, 4))
    B = np.ones((4, 5))
    _, nj = oracle.joinagg("ij,jk->ik", [A, B], tier="lit", return_joined=True)
    assert nj == 3 * 4 * 5


# -------------------------------------------------- decomposition invariance

PARTITIONS = [
    {"i": [0, 10], "j": [0, 9], "k": [0, 8]},
    {"i": [0, 3, 10], "j": [0, 4, 5, 9], "k": [0, 8]},
    {"i": [0, 1, 2, 5, 10], "j": [0, 9], "k": [0, 2, 8]},
    {"i": [0, 5, 10], "j": [0, 3, 6, 9], "k": [0, 4, 8]},
]


@pytest.mark.parametrize("parts", PARTITIONS)
def test_block_decomposition_invariance_matmul(parts):
    r = rng(6)
    X = r.standard_normal((10, 9))
    Y = r.standard_normal((9, 8))
    cell = oracle.joinagg("ij,jk->ik", [X, Y])
    blk = blocked.joinagg_blocked("ij,jk->ik", [X, Y], parts)
    np.testing.assert_allclose(blk, cell, rtol=1e-12, atol=1e-12)
    Xi = r.integers(-2, 3, (10, 9)).astype(float)
    Yi = r.integers(-2, 3, (9, 8)).astype(float)
    assert np.array_equal(blocked.joinagg_blocked("ij,jk->ik", [Xi, Yi], parts), oracle.joinagg("ij,jk->ik", [Xi, Yi]))


def test_block_decomposition_invariance_max_and_causal():
    r = rng(7)
    Q = r.standard_normal((1, 2, 9, 3))
    K = r.standard_normal((1, 2, 9, 3))
    full = oracle.joinagg("bhsd,bhtd->bhst", [Q, K], pred="ts")
    parts = {"b": [0, 1], "h": [0, 1, 2], "s": [0, 4, 9], "t": [0, 2, 5, 9], "d": [0, 1, 3]}
    blk = blocked.joinagg_blocked("bhsd,bhtd->bhst", [Q, K], parts, pred="ts")
    np.testing.assert_allclose(blk, full, rtol=1e-12, atol=1e-12, equal_nan=True)
    m_full = oracle.joinagg("bhst->bhs", [full], "identity", "max")
    m_blk = blocked.joinagg_blocked("bhst->bhs", [full], {"b": [0, 1], "h": [0, 2], "s": [0, 9], "t": [0, 3, 6, 9]},
                                    "identity", "max")
    assert np.array_equal(m_full, m_blk)


# ------------------------------------------------------------- chain pins

def _ref_masked_attention(Q, K, V, scale, causal):
    S = np.einsum("bhsd,bhtd->bhst", Q, K) * scale
    if causal:
        n = S.shape[-1]
        S = np.where(np.tril(np.ones((S.shape[-2], n), bool)), S, -np.inf)
    P = np.exp(S - S.max(-1, keepdims=True))
    P /= P.sum(-1, keepdims=True)
    return P, np.einsum("bhst,bhtd->bhsd", P, V)


@pytest.mark.parametrize("causal", [False, True])
def test_attention_against_library_softmax(causal):
    r = rng(8)
    Q, K, V = (r.standard_normal((2, 2, 7, 5)) for _ in range(3))
    out = chains.softmax_attention(Q, K, V, scale=0.4, causal=causal)
    P, O = _ref_masked_attention(Q, K, V, 0.4, causal)
    np.testing.assert_allclose(out["O"], O, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(np.nan_to_num(out["P"]), P, rtol=1e-12, atol=1e-12)
    if causal:
        assert np.isnan(out["S"][0, 0, 0, 1]) and not np.isnan(out["S"][0, 0, 1, 0])


def test_attention_invariants():
    r = rng(9)
    Q, K, V = (r.standard_normal((1, 3, 6, 4)) for _ in range(3))
    out = chains.softmax_attention(Q, K, V)
    np.testing.assert_allclose(np.nansum(out["P"], axis=-1), 1.0, rtol=1e-14)
    ones = chains.softmax_attention(Q, K, np.ones_like(V))
    np.testing.assert_allclose(ones["O"], 1.0, rtol=1e-14)
    Ksame = np.repeat(K[:, :, :1, :], K.shape[2], axis=2)
    same = chains.softmax_attention(Q, Ksame, V)
    np.testing.assert_allclose(same["O"], np.broadcast_to(V.mean(axis=2, keepdims=True), V.shape), rtol=1e-12)


def _brute_flash(Q, K, V, group, scale, causal, ends):
    """Pure-Python loops over one (b, head, query) row at a time ([b, s, h, d])."""
    import math
    b, s, hq, d = Q.shape
    O = np.zeros_like(Q)
    starts = [0] + list(ends[:-1])
    for bi in range(b):
        for h in range(hq):
            for i in range(s):
                seg = max(j for j, a in enumerate(starts) if a <= i)
                keys = [j for j in range(starts[seg], ends[seg]) if not causal or j <= i]
                sc = [scale * sum(Q[bi, i, h, c] * K[bi, j, h // group, c] for c in range(d)) for j in keys]
                mx = max(sc)
                w = [math.exp(x - mx) for x in sc]
                tot = sum(w)
                for c in range(d):
                    O[bi, i, h, c] = sum(wj * V[bi, j, h // group, c] for wj, j in zip(w, keys)) / tot
    return O


@pytest.mark.parametrize("causal", [False, True])
def test_flash_attention_brute_force_gqa_packed(causal):
    r = rng(21)
    Q = r.standard_normal((2, 9, 4, 3))
    K, V = r.standard_normal((2, 9, 2, 3)), r.standard_normal((2, 9, 2, 3))
    ends = [4, 9]
    out = chains.flash_attention(Q, K, V, group=2, scale=0.7, causal=causal, seq_ends=ends, layout="bshd")
    np.testing.assert_allclose(out["O"], _brute_flash(Q, K, V, 2, 0.7, causal, ends), rtol=1e-12, atol=1e-13)
    # the same data in the head-major layout
    tr = lambda x: np.ascontiguousarray(np.transpose(x, (0, 2, 1, 3)))  # noqa: E731
    out2 = chains.flash_attention(tr(Q), tr(K), tr(V), group=2, scale=0.7, causal=causal, seq_ends=ends, layout="bhsd")
    np.testing.assert_allclose(out2["O"], tr(out["O"]), rtol=1e-14)


def test_flash_attention_head_groups_and_sequence_boundaries():
    r = rng(22)
    b, s, hk, g, d = 1, 10, 3, 4, 2
    Q = r.standard_normal((b, s, hk * g, d))
    K = r.standard_normal((b, s, hk, d))
    # value of key-value head m is the constant m + 1: query head h must read h // g + 1
    V = np.broadcast_to((np.arange(hk) + 1.0)[None, None, :, None], (b, s, hk, d)).copy()
    O = chains.flash_attention(Q, K, V, group=g, causal=True, seq_ends=[3, 10], layout="bshd")["O"]
    np.testing.assert_allclose(O, np.broadcast_to((np.arange(hk * g) // g + 1.0)[None, None, :, None], O.shape),
                               rtol=1e-13)
    # identical keys: every query gets the mean of its own sequence's values
    Ksame = np.zeros_like(K)
    V2 = r.standard_normal((b, s, hk, d))
    O2 = chains.flash_attention(Q, Ksame, V2, group=g, seq_ends=[3, 10], layout="bshd")["O"]
    for lo, hi in ((0, 3), (3, 10)):
        want = V2[:, lo:hi].mean(axis=1)[:, np.arange(hk * g) // g]
        np.testing.assert_allclose(O2[:, lo:hi], np.broadcast_to(want[:, None], O2[:, lo:hi].shape), rtol=1e-12)
    # causal with identical keys: the mean over the sequence's prefix up to the query
    O3 = chains.flash_attention(Q, Ksame, V2, group=g, causal=True, seq_ends=[3, 10], layout="bshd")["O"]
    for i in range(s):
        lo = 0 if i < 3 else 3
        want = V2[:, lo:i + 1].mean(axis=1)[:, np.arange(hk * g) // g]
        np.testing.assert_allclose(O3[:, i], want, rtol=1e-12)


def test_flash_attention_stats_close_forms():
    r = rng(23)
    Q, K = r.standard_normal((1, 2, 5, 3)), r.standard_normal((1, 2, 5, 3))
    V = r.standard_normal((1, 2, 5, 3))
    out = chains.flash_attention(Q, K, V, scale=0.5, causal=True)
    S = 0.5 * np.einsum("bhsd,bhtd->bhst", Q, K)
    S = np.where(np.tril(np.ones((5, 5), bool)), S, -np.inf)
    m = S.max(-1)
    np.testing.assert_allclose(out["m"], m, rtol=1e-14)
    np.testing.assert_allclose(out["l"], np.exp(S - m[..., None]).sum(-1), rtol=1e-13)
    # the first query sees only itself: l = 1, m = its own score
    np.testing.assert_allclose(out["l"][..., 0], 1.0, rtol=1e-15)


def test_matrix_chain_against_library_and_associativity():
    r = rng(31)
    dims = [5, 7, 3, 6, 4, 8]
    mats = [r.standard_normal((dims[i], dims[i + 1])) for i in range(5)]
    paren = ((1, 2), ((3, 4), 5))  # chain B's shape
    got = chains.matrix_chain(mats, paren)
    np.testing.assert_allclose(got, np.linalg.multi_dot(mats), rtol=1e-12, atol=1e-12)
    other = chains.matrix_chain(mats, ((((1, 2), 3), 4), 5))
    np.testing.assert_allclose(got, other, rtol=1e-12, atol=1e-12)
    # a transposed operand (a plausible mistake) changes the result
    bad = [m.copy() for m in mats]
    bad[2] = np.ascontiguousarray(mats[2][::-1])
    assert not np.allclose(chains.matrix_chain(bad, paren), got)


def test_silu_special_values():
    z = np.array([[0.0, 40.0, -40.0, 1.0]])
    one = np.ones_like(z)
    h = oracle.joinagg("ik,ik->ik", [z, one], "silu_mul", "none")
    assert h[0, 0] == 0.0
    assert abs(h[0, 1] - 40.0) < 1e-12 and abs(h[0, 2]) < 1e-15
    assert abs(h[0, 3] - 1.0 / (1.0 + np.exp(-1.0))) < 1e-15


def test_rmsnorm_invariant():
    r = rng(10)
    x = r.standard_normal((5, 16)) * 3.0
    eps = 1e-6
    out = chains.rmsnorm(x, np.ones(16), eps)
    ms = (x ** 2).mean(axis=1)
    np.testing.assert_allclose(out["ms"], ms, rtol=1e-14)
    np.testing.assert_allclose((out["y"] ** 2).mean(axis=1), ms / (ms + eps), rtol=1e-12)


def test_rmsnorm_gain_closed_form():
    """Rows whose cells all have magnitude c normalise (eps = 0) to
    sign(x) * gamma: with a gain far from 1 this fixes that the gain
    multiplies (a dropped or inverted gain fails)."""
    r = rng(42)
    D = 12
    g = 1.0 + 0.1 * r.standard_normal(D)
    signs = np.where(r.random((4, D)) < 0.5, -1.0, 1.0)
    c = np.array([[0.5], [1.0], [3.0], [7.25]])
    out = chains.rmsnorm(c * signs, g, 0.0)
    np.testing.assert_allclose(out["ms"], c[:, 0] ** 2, rtol=1e-15)
    np.testing.assert_allclose(out["y"], signs * g, rtol=1e-14)
    # with eps > 0 the same rows shrink by c / sqrt(c^2 + eps) exactly
    eps = 0.25
    out = chains.rmsnorm(c * signs, g, eps)
    np.testing.assert_allclose(out["y"], signs * g * c / np.sqrt(c ** 2 + eps), rtol=1e-14)


def test_rmsnorm_gain_random_rows():
    r = rng(43)
    x = r.standard_normal((6, 20)) * 2.0
    g = 1.0 + 0.1 * r.standard_normal(20)
    out = chains.rmsnorm(x, g, 1e-6)
    ms = np.mean(x * x, axis=1, keepdims=True)
    np.testing.assert_allclose(out["y"], x / np.sqrt(ms + 1e-6) * g[None, :], rtol=1e-13)


def test_add_join_values():
    """The residual ADD join on non-zero operands: IEEE fp64 sums cell by
    cell (a difference v0 - v1 fails the doubling check)."""
    r = rng(44)
    a, b = r.standard_normal((4, 5)), r.standard_normal((4, 5))
    np.testing.assert_array_equal(oracle.joinagg("td,td->td", [a, b], "add", "none"), a + b)
    np.testing.assert_array_equal(oracle.joinagg("td,td->td", [a, a], "add", "none"), 2.0 * a)
    np.testing.assert_array_equal(oracle.joinagg("td,td->td", [a, b], "add", "none", tier="lit"), a + b)


def _swiglu_closed_form_case():
    """Inputs whose SwiGLU output has a closed form: x in [0.5, 1.5), a gate
    of 50 x (SiLU(G) = G to 1e-10 since G >= 25), an up projection that
    copies column 0 of x into every column, and a down projection that is a
    6-cycle permutation (not its own transpose)."""
    r = rng(45)
    T, D = 5, 6
    x = 0.5 + r.random((T, D))
    w_gate = 50.0 * np.eye(D)
    w_up = np.zeros((D, D))
    w_up[0, :] = 1.0
    perm = np.array([1, 2, 3, 4, 5, 0])
    w_down = np.eye(D)[perm]              # row f is e_perm[f]: Y[:, perm[f]] = H[:, f]
    H = (50.0 * x) * x[:, :1]
    Y = np.empty_like(H)
    Y[:, perm] = H
    return x, w_gate, w_up, w_down, H, Y


def test_swiglu_ffn_closed_form():
    """H = SiLU(gate) * up and Y = H w_down: the closed form tells the gate
    from the up projection (the swapped map SiLU(U) * G gives
    SiLU(x0) * 50 x) and fixes w_down's orientation (its transpose is the
    inverse permutation)."""
    x, wg, wu, wd, H, Y = _swiglu_closed_form_case()
    out = chains.swiglu_ffn(x, wg, wu, wd)
    np.testing.assert_allclose(out["G"], 50.0 * x, rtol=1e-15)
    np.testing.assert_allclose(out["U"], np.repeat(x[:, :1], x.shape[1], axis=1), rtol=1e-15)
    np.testing.assert_allclose(out["H"], H, rtol=1e-9)
    np.testing.assert_allclose(out["Y"], Y, rtol=1e-9)


def test_swiglu_ffn_random_against_numpy():
    r = rng(46)
    x = r.standard_normal((7, 9))
    wg, wu = r.standard_normal((9, 11)), r.standard_normal((9, 11))
    wd = r.standard_normal((11, 9))
    out = chains.swiglu_ffn(x, wg, wu, wd)
    g = x @ wg
    h = g / (1.0 + np.exp(-g)) * (x @ wu)
    np.testing.assert_allclose(out["H"], h, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(out["Y"], h @ wd, rtol=1e-12, atol=1e-12)


def test_rope_invariants():
    r = rng(11)
    b, s, h, d = 1, 9, 2, 8
    q = r.standard_normal((b, s, h, d))
    k = r.standard_normal((b, s, h, d))
    qr = chains.rope(q, 10000.0)
    kr = chains.rope(k, 10000.0)
    # norm of every pair is preserved
    np.testing.assert_allclose(np.hypot(qr[..., 0::2], qr[..., 1::2]), np.hypot(q[..., 0::2], q[..., 1::2]), rtol=1e-12)
    # identity at position 0
    np.testing.assert_allclose(qr[:, 0], q[:, 0], rtol=0, atol=0)
    # the score of positions (m, n) depends only on m - n: rotate the same vectors at shifted positions
    qc = np.repeat(q[:, :1], s, axis=1)
    kc = np.repeat(k[:, :1], s, axis=1)
    qcr, kcr = chains.rope(qc, 10000.0), chains.rope(kc, 10000.0)
    sc = np.einsum("bmhd,bnhd->bhmn", qcr, kcr)
    for dlt in range(-3, 4):
        vals = [sc[0, 0, m, m - dlt] for m in range(s) if 0 <= m - dlt < s]
        np.testing.assert_allclose(vals, vals[0], rtol=1e-11)
    # pair (0, 1) of position 1 is rotated by exactly 1 radian (theta^0)
    want0 = q[0, 1, 0, 0] * np.cos(1.0) - q[0, 1, 0, 1] * np.sin(1.0)
    assert abs(qr[0, 1, 0, 0] - want0) < 1e-14


def _tiny_block_weights(D, F, seed, zero=()):
    r = rng(seed)
    W = {k: r.standard_normal(shape) * 0.2 for k, shape in
         [("wq", (D, D)), ("wk", (D, D)), ("wv", (D, D)), ("wo", (D, D)), ("w_gate", (D, F)), ("w_up", (D, F)),
          ("w_down", (F, D))]}
    W["g1"] = np.ones(D)
    W["g2"] = np.ones(D)
    for k in zero:
        W[k] = np.zeros_like(W[k])
    return W


def test_llama_block_residual_identity():
    x = rng(12).standard_normal((1, 5, 8))
    W = _tiny_block_weights(8, 12, 13, zero=("wo", "w_down"))
    out = chains.llama_block(x, W, n_heads=2)
    np.testing.assert_array_equal(out["y"], x)


def test_llama_block_is_causal():
    x = rng(14).standard_normal((1, 6, 8))
    W = _tiny_block_weights(8, 12, 15)
    y0 = chains.llama_block(x, W, n_heads=2)["y"]
    x2 = x.copy()
    x2[0, 4] += 1.0
    y1 = chains.llama_block(x2, W, n_heads=2)["y"]
    np.testing.assert_array_equal(y0[0, :4], y1[0, :4])
    assert np.abs(y0[0, 4:] - y1[0, 4:]).max() > 1e-3


def test_llama_block_prefix_sampling_is_exact():
    """A prefix of the tokens of one sequence gives the same outputs as the
    full sequence (causal attention only looks back) -- the property that
    lets full-size parity sample early tokens."""
    x = rng(16).standard_normal((2, 7, 8))
    W = _tiny_block_weights(8, 12, 17)
    full = chains.llama_block(x, W, n_heads=2)["y"]
    pre = chains.llama_block(x[1:2, :3], W, n_heads=2)["y"]
    np.testing.assert_allclose(pre[0], full[1, :3], rtol=1e-13, atol=1e-13)


# ------------------------------------------------------------------ exchange

def _dense_to_arena(a, bounds):
    """Brute-force arena construction: blocks in row-major id order, each
    block the row-major ravel of its slice."""
    parts = []
    for combo in itertools.product(*[range(len(b) - 1) for b in bounds]):
        sl = tuple(slice(b[i], b[i + 1]) for b, i in zip(bounds, combo))
        parts.append(a[sl].ravel())
    return np.concatenate(parts) if parts else a.ravel()


TILINGS = [
    [[0, 12], [0, 10]],
    [[0, 3, 6, 9, 12], [0, 10]],
    [[0, 12], [0, 5, 10]],
    [[0, 4, 8, 12], [0, 2, 7, 10]],
    [[0, 1, 12], [0, 9, 10]],
]


@pytest.mark.parametrize("src", range(len(TILINGS)))
@pytest.mark.parametrize("dst", range(len(TILINGS)))
def test_exchange_matches_slicing_definition(src, dst):
    a = np.arange(120, dtype=np.int32).reshape(12, 10) * 7 + 3
    sa = _dense_to_arena(a, TILINGS[src])
    got = oracle.exchange(sa, (12, 10), TILINGS[src], TILINGS[dst])
    assert np.array_equal(got, _dense_to_arena(a, TILINGS[dst]))
    perm = oracle.exchange_perm((12, 10), TILINGS[src], TILINGS[dst])
    assert np.array_equal(np.sort(perm), np.arange(120))
    assert np.array_equal(sa[perm], got)


def test_exchange_roundtrip_and_composition_rank3():
    a = np.arange(4 * 6 * 8, dtype=np.uint16).reshape(4, 6, 8)
    A = [[0, 2, 4], [0, 6], [0, 8]]
    B = [[0, 4], [0, 3, 6], [0, 2, 4, 8]]
    C = [[0, 1, 2, 3, 4], [0, 1, 6], [0, 8]]
    xa = _dense_to_arena(a, A)
    xb = oracle.exchange(xa, a.shape, A, B)
    assert np.array_equal(oracle.exchange(xb, a.shape, B, A), xa)
    assert np.array_equal(oracle.exchange(xb, a.shape, B, C), oracle.exchange(xa, a.shape, A, C))


# ---------------------------------------------- pins catch planted mistakes

def test_pins_catch_planted_mistakes():
    """Each pin must fail on a plausible oracle mistake planted here, on the
    CPU: a dropped term, a transposed operand, a sign error in the exp map,
    a missing causal predicate."""
    r = rng(18)
    A, B = r.standard_normal((5, 6)), r.standard_normal((6, 4))
    want = np.einsum("ij,jk->ik", A, B)
    dropped = oracle.joinagg("ij,jk->ik", [A[:, :5], B[:5, :]])
    assert not np.allclose(dropped, want)
    Bt = r.standard_normal((6, 6))
    transposed = oracle.joinagg("ij,kj->ik", [A, Bt])
    assert not np.allclose(transposed, np.einsum("ij,jk->ik", A, Bt))
    Q, K, V = (r.standard_normal((1, 1, 5, 3)) for _ in range(3))
    S = oracle.joinagg("bhsd,bhtd->bhst", [Q, K])
    m = oracle.joinagg("bhst->bhs", [S], "identity", "max")
    E_bad = np.exp(m[..., None] - S)  # exp(m - S) instead of exp(S - m)
    P_ref, _ = _ref_masked_attention(Q, K, V, 1.0, False)
    assert not np.allclose(E_bad / E_bad.sum(-1, keepdims=True), P_ref)
    # without the predicate, a later token changes an earlier output
    x = rng(19).standard_normal((1, 1, 4, 2))
    x2 = x.copy()
    x2[0, 0, 3] += 1.0
    o1 = chains.softmax_attention(x, x, x, causal=False)["O"]
    o2 = chains.softmax_attention(x2, x2, x2, causal=False)["O"]
    assert not np.array_equal(o1[0, 0, 0], o2[0, 0, 0])
    c1 = chains.softmax_attention(x, x, x, causal=True)["O"]
    c2 = chains.softmax_attention(x2, x2, x2, causal=True)["O"]
    assert np.array_equal(c1[0, 0, :3], c2[0, 0, :3])
    # SwiGLU with gate and up swapped (SiLU(U) * G) misses the closed form
    xs, wg, wu, wd, H, _ = _swiglu_closed_form_case()
    G = oracle.joinagg("ij,kj->ik", [xs, np.ascontiguousarray(wg.T)])
    U = oracle.joinagg("ij,kj->ik", [xs, np.ascontiguousarray(wu.T)])
    assert not np.allclose(oracle.joinagg("ik,ik->ik", [U, G], "silu_mul", "none"), H, rtol=1e-3)
    # ... and a transposed w_down misses Y
    assert not np.allclose(chains.swiglu_ffn(xs, wg, wu, np.ascontiguousarray(wd.T))["Y"],
                           _swiglu_closed_form_case()[5], rtol=1e-3)
    # RMSNorm with the gain dropped, or divided instead of multiplied
    g = 1.0 + 0.1 * rng(20).standard_normal(8)
    xr = np.where(rng(21).random((3, 8)) < 0.5, -2.0, 2.0)
    want = np.sign(xr) * g
    assert not np.allclose(chains.rmsnorm(xr, np.ones(8), 0.0)["y"], want, rtol=1e-3)
    assert not np.allclose(chains.rmsnorm(xr, 1.0 / g, 0.0)["y"], want, rtol=1e-3)
    # ADD written as a difference misses the doubling
    a = rng(22).standard_normal((2, 3))
    assert not np.array_equal(a - a, 2.0 * a)


# -------------------------------------------- partial copies and their (+)

def test_ex54_preamble_partials():
    """Example 5.4: the copies the producer's GPUs hold and the preamble's
    X_j + Y_j, written out with numpy matmul on the page's slices."""
    g = gold("ex5_4_preamble.json")
    r = rng(54)
    A = r.standard_normal((g["i"], g["j"]))
    B = r.standard_normal((g["j"], g["k"]))
    ib, jb = g["i_bounds"], g["j_bounds"]
    P = blocked.joinagg_partials("ij,jk->ik", [A, B], {"i": ib, "j": jb, "k": g["k_bounds"]})
    assert P.shape == (2, g["i"], g["k"])

    def held(gpu):  # the output block F(m,n) writes, computed from its slices alone
        m, n = g["spec_of_gpu"][gpu]
        rows = slice(ib[m - 1], ib[m])
        cols = slice(jb[n - 1], jb[n])
        return rows, n - 1, A[rows, cols] @ B[cols, :]

    for gpu in range(4):
        rows, copy, val = held(gpu)
        assert np.allclose(P[copy, rows], val, rtol=1e-12, atol=1e-12)
    cb = g["consumer_i_bounds"]
    S = blocked.aggregate_copies(P, "sum")
    for j, (x, y) in enumerate(g["out"]):
        rows = slice(cb[j], cb[j + 1])
        parts = []
        for atom in (x, y):
            prow, copy, val = held(g["in"][atom])
            parts.append(val[cb[j] - prow.start:cb[j + 1] - prow.start])
        assert np.allclose(S[rows], parts[0] + parts[1], rtol=1e-12, atol=1e-12)
    assert np.allclose(S, A @ B, rtol=1e-10, atol=1e-10)


@pytest.mark.parametrize("spec,shapes,bounds", [
    ("ij,jk->ik", [(7, 9), (9, 6)], {"i": [0, 3, 7], "j": [0, 2, 5, 9], "k": [0, 4, 6]}),
    ("bij,bjk->bik", [(2, 5, 8), (2, 8, 3)], {"b": [0, 1, 2], "i": [0, 5], "j": [0, 1, 4, 6, 8], "k": [0, 3]}),
    ("ij,kj->ik", [(4, 10), (3, 10)], {"i": [0, 2, 4], "j": [0, 5, 10], "k": [0, 1, 3]}),
])
def test_partials_brute_force_and_sum(spec, shapes, bounds):
    """Copy q of every block is the contraction over the q-th block of the
    aggregated letter alone (brute force over cells); SUM over the copies is
    numpy.einsum of the whole; MAX over the copies is numpy's max."""
    r = rng(7)
    arrs = [r.standard_normal(s) for s in shapes]
    P = blocked.joinagg_partials(spec, arrs, bounds)
    agg_letter = "j"
    nq = len(bounds[agg_letter]) - 1
    assert P.shape[0] == nq
    ins, out = spec.split("->")
    ta, tb = ins.split(",")
    for q in range(nq):
        lo, hi = bounds[agg_letter][q], bounds[agg_letter][q + 1]
        want = np.zeros(P.shape[1:])
        ext = dict(zip(ta, arrs[0].shape)) | dict(zip(tb, arrs[1].shape))
        for cell in itertools.product(*[range(ext[l]) for l in out]):
            env = dict(zip(out, cell))
            s = 0.0
            for jj in range(lo, hi):
                env[agg_letter] = jj
                s += arrs[0][tuple(env[l] for l in ta)] * arrs[1][tuple(env[l] for l in tb)]
            want[cell] = s
        assert np.allclose(P[q], want, rtol=1e-12, atol=1e-12)
    assert np.allclose(blocked.aggregate_copies(P, "sum"), np.einsum(spec, *arrs), rtol=1e-12, atol=1e-12)
    assert np.array_equal(blocked.aggregate_copies(P, "max"), P.max(axis=0))


def test_aggregate_copies_order_and_single_copy():
    x = rng(3).standard_normal((1, 4, 5))
    assert np.array_equal(blocked.aggregate_copies(x, "sum"), x[0])
    # copy order: ((a + b) + c), visible where it changes the fp64 rounding
    P = np.array([[1e16], [1.0], [-1e16]])
    assert blocked.aggregate_copies(P, "sum")[0] == (1e16 + 1.0) - 1e16
