"""GPU parity: libea.so's kernels against the fp64 oracle, element by
element, on seeded inputs at sizes that span several tiles with ragged
tails.  Bars: bit-exact for the exchange and for integer-valued inputs;
max relative Frobenius error 1e-5 (fp32) and 2e-2 (bf16 inputs, fp32
accumulation) otherwise."""
import numpy as np
import pytest

import oracle
import synth
from oracle import chains

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from tensor_relational_einsum_gb300.build import build
    build()
    assert torch.cuda.is_available(), "the GPU parity tests need a CUDA device"
    yield
    from tensor_relational_einsum_gb300.relation import check
    check()


from gpu_util import (BF16_TOL, FP32_TOL, arena_bits, bounds_of, dense64, exchange, joinagg, last,  # noqa: E402
                      max_block_rel_frob, rel, rel_frob, synth_bounds)


# ------------------------------------------------------------------ exchange

X_CASES = [
    ("bf16", (256, 384), [4, 1], [1, 3]),
    ("bf16", (256, 384), [4, 1], [16, 6]),
    ("f32", (200, 136), [[0, 8, 100, 200], [0, 136]], [[0, 64, 200], [0, 8, 72, 136]]),
    ("bf16", (12, 10), [[0, 3, 6, 9, 12], [0, 10]], [[0, 4, 8, 12], [0, 2, 7, 10]]),   # 2-byte runs: scalar path
    ("bf16", (2, 64, 4, 128), [2, 1, 1, 1], [2, 1, 4, 1]),                              # tokens -> heads
    ("f32", (3, 5, 7, 9), [3, 1, 7, 1], [1, 5, 1, 3]),
    ("bf16", (1, 70000), [1, 1], [1, 7]),                                               # one long row
]


@pytest.mark.parametrize("dtype,dims,src,dst", X_CASES)
def test_exchange_bit_exact(dtype, dims, src, dst):
    t = synth.make(dtype, dims, "uniform", seed=11, a=-1, b=1)
    R = rel(t, src)
    flat = t.host.reshape(-1)
    whole = [[0, n] for n in dims]
    want_src = oracle.exchange(flat, dims, whole, bounds_of(dims, src))
    assert np.array_equal(arena_bits(R).view(flat.dtype), want_src)
    X = exchange(R, dst)
    assert last()["kernel"] == "exchange"
    want_dst = oracle.exchange(flat, dims, whole, bounds_of(dims, dst))
    assert np.array_equal(arena_bits(X).view(flat.dtype), want_dst)
    back = exchange(X, src)
    assert np.array_equal(arena_bits(back).view(flat.dtype), want_src)
    # composition: src -> dst -> a third tiling equals src -> the third tiling
    third = [[0, n // 3, n] if n >= 3 else 1 for n in dims]
    via = exchange(X, third)
    direct = exchange(R, third)
    assert np.array_equal(arena_bits(via), arena_bits(direct))
    assert np.array_equal(arena_bits(direct).view(flat.dtype), oracle.exchange(flat, dims, whole, bounds_of(dims, third)))


# ------------------------------------------------------- fp32 contraction (C1)

def test_matmul_fp32_full_config():
    """fp32 A[256,256] B[256,256] U[-1,1], every index in 4 blocks: 64
    function specifications in 16 groups of 4, SUM over j-blocks."""
    A = synth.make("f32", (256, 256), "uniform", 1, -1, 1)
    B = synth.make("f32", (256, 256), "uniform", 2, -1, 1)
    RA, RB = rel(A, [4, 4]), rel(B, [4, 4])
    C = joinagg("ij,jk->ik", [RA, RB])
    info = last()
    assert info["kernel"] == "contract_simt" and info["groups"] == 16 and info["tuples"] == 64
    want = oracle.joinagg("ij,jk->ik", [A.to_f64(), B.to_f64()], tier="lit")
    err = max_block_rel_frob(dense64(C), want, [synth_bounds(256, 4)] * 2)
    assert err <= FP32_TOL, err


def test_matmul_fp32_integer_exact_any_partition():
    A = synth.make("f32", (130, 97), "int", 3, -2, 2)
    B = synth.make("f32", (97, 75), "int", 4, -2, 2)
    want = oracle.joinagg("ij,jk->ik", [A.to_f64(), B.to_f64()], tier="lit")
    for pa, pb in [([1, 1], [1, 1]), ([3, 4], [4, 2]), ([[0, 1, 130], [0, 50, 97]], [[0, 50, 97], [0, 70, 75]])]:
        C = joinagg("ij,jk->ik", [rel(A, pa), rel(B, pb)])
        assert np.array_equal(dense64(C), want)


# ----------------------------------------------------- bf16 tensor-core path

_LAST_CASE = {}


def _bf16_case(spec, shapes, parts_per_input, out_dtype, seeds=(5, 6), dist=("normal", 0.0, 1.0), pred=None,
               scale=1.0, expect="contract_tc", simt_bf16=False):
    ts = [synth.make("bf16", s, dist[0], sd, dist[1], dist[2]) for s, sd in zip(shapes, seeds)]
    rs = [rel(t, p) for t, p in zip(ts, parts_per_input)]
    C = joinagg(spec, rs, out_dtype=out_dtype, pred=pred, scale=scale, simt_bf16=simt_bf16)
    info = last()
    _LAST_CASE.clear()
    _LAST_CASE.update(info)  # reading C back runs an exchange, which replaces last()
    assert info["kernel"] == expect, info
    want = oracle.joinagg(spec, [t.to_f64() for t in ts], scale=scale, pred=pred)
    return dense64(C), want, C


@pytest.mark.parametrize("out_dtype", ["f32", "bf16"])
def test_tc_matmul_ragged_k_major_a_mn_major_b(out_dtype):
    # M = 320 (3 m-tiles, ragged), K = 200 in blocks 64/72/64, N = 520 (3 n-tiles of 256, ragged)
    got, want, C = _bf16_case("ij,jk->ik", [(320, 200), (200, 520)], [[1, [0, 64, 136, 200]], [[0, 64, 136, 200], 1]],
                              out_dtype)
    err = rel_frob(got, want)
    assert err <= (1e-5 if out_dtype == "f32" else 5e-3), err


def test_tc_integer_exact():
    got, want, _ = _bf16_case("ij,jk->ik", [(256, 320), (320, 384)], [[2, 5], [5, 3]], "f32", dist=("int", -2, 2))
    assert np.array_equal(got, want)


def test_tc_scores_k_major_both_and_causal_mask():
    # "bhsd,bhtd->bhst": both operands K-major (d contiguous); t in 3 blocks -> BN 128
    shapes = [(1, 2, 384, 128), (1, 2, 384, 128)]
    parts = [[1, 2, 1, 1], [1, 2, 3, 1]]
    got, want, _ = _bf16_case("bhsd,bhtd->bhst", shapes, parts, "f32", scale=0.125)
    assert rel_frob(got, want) <= 1e-5
    got, want, _ = _bf16_case("bhsd,bhtd->bhst", shapes, [[1, 2, 3, 1], [1, 2, 3, 1]], "f32", scale=0.125, pred="ts")
    present = ~np.isnan(want)
    assert rel_frob(got, want) <= 1e-5
    # blocks above the diagonal are not computed; masked cells of diagonal blocks hold -inf
    for s0 in range(0, 384, 128):
        blk = got[0, :, s0:s0 + 128, s0:s0 + 128]
        assert np.all(np.isneginf(blk[~present[0, :, s0:s0 + 128, s0:s0 + 128]]))


def test_tc_pv_mn_major_b():
    # "bhst,bhtd->bhsd": A = P (t contiguous, K-major), B = V (d contiguous, MN-major), 3 t-blocks summed
    got, want, _ = _bf16_case("bhst,bhtd->bhsd", [(1, 2, 256, 384), (1, 2, 384, 128)],
                              [[1, 2, 1, 3], [1, 2, 3, 1]], "bf16")
    assert rel_frob(got, want) <= 5e-3


def test_tc_batch_inside_block_and_swapped_roles():
    # heads in blocks of 2 -> batch dimension of extent 2 inside each block
    got, want, _ = _bf16_case("bhsd,bhtd->bhst", [(1, 4, 256, 64), (1, 4, 256, 64)], [[1, 2, 1, 1], [1, 2, 2, 1]],
                              "f32")
    assert rel_frob(got, want) <= 1e-5
    # output's contiguous letter comes from input 0 -> operands swap roles
    got, want, _ = _bf16_case("ij,jk->ki", [(384, 192), (192, 256)], [[1, 3], [3, 1]], "f32")
    assert rel_frob(got, want) <= 1e-5


@pytest.mark.parametrize("spec,bshape", [("bij,bjk->bik", (24, 256, 1096)), ("bij,bkj->bik", (24, 1096, 256))])
def test_tc_cta_pairs_with_padding_tiles(spec, bshape):
    # 24 groups of M = 300 (three m-tiles: a padding tile completes each CTA
    # pair), N = 1096 (five 256-wide tiles, ragged), K = 256: 360 tiles, at
    # least two per SM, so the launch runs in CTA pairs (one 256-row MMA over
    # two SMs, each loading half of the B tile) (B MN-major in the first
    # case, K-major in the second)
    got, want, _ = _bf16_case(spec, [(24, 300, 256), bshape], [[24, 1, 1], [24, 1, 1]], "f32")
    assert _LAST_CASE["cta_pair"]
    assert rel_frob(got, want) <= 1e-5
    got, want, _ = _bf16_case(spec, [(24, 300, 256), bshape], [[24, 1, 1], [24, 1, 1]], "f32",
                              dist=("int", -2, 2))
    assert np.array_equal(got, want)


@pytest.mark.parametrize("spec,ashape,bshape", [
    ("bji,bjk->bik", (24, 256, 320), (24, 256, 1096)),   # A MN-major (m contiguous), B MN-major
    ("bji,bkj->bik", (24, 256, 320), (24, 1096, 256)),   # A MN-major, B K-major
    ("bij,bkj->bik", (104, 300, 192), (104, 120, 192)),  # N = 120: 128-wide tiles in pairs (M = 256, N = 128)
])
def test_tc_cta_pairs_operand_majors(spec, ashape, bshape):
    # every operand layout through the CTA-pair launch, with padding tiles,
    # ragged N and a K that is not a multiple of the 64-wide chunk (192 = 3
    # chunks); integer inputs make the result exact
    parts = [[ashape[0], 1, 1], [bshape[0], 1, 1]]
    got, want, _ = _bf16_case(spec, [ashape, bshape], parts, "f32", dist=("int", -2, 2))
    assert _LAST_CASE["kernel"] == "contract_tc" and _LAST_CASE["cta_pair"]
    assert np.array_equal(got, want)
    got, want, _ = _bf16_case(spec, [ashape, bshape], parts, "bf16")
    assert rel_frob(got, want) <= 5e-3


@pytest.mark.parametrize("out_dtype", ["f32", "bf16"])
def test_tc_epilogue_add(out_dtype):
    # C = A B + R with the residual join fused: ragged M, K in blocks, ragged N
    A = synth.make("bf16", (320, 200), "normal", 61, 0, 1)
    B = synth.make("bf16", (200, 520), "normal", 62, 0, 1)
    R = synth.make(out_dtype, (320, 520), "normal", 63, 0, 1)
    C = joinagg("ij,jk->ik", [rel(A, [1, [0, 64, 136, 200]]), rel(B, [[0, 64, 136, 200], 1])], out_dtype=out_dtype,
                epi_map="add", epi_in=rel(R, [1, 1]))
    assert last()["kernel"] == "contract_tc"
    P = oracle.joinagg("ij,jk->ik", [A.to_f64(), B.to_f64()])
    want = oracle.joinagg("ik,ik->ik", [P, R.to_f64()], "add", "none")
    assert rel_frob(dense64(C), want) <= (1e-5 if out_dtype == "f32" else 5e-3)


def test_tc_epilogue_add_cta_pairs_integer_exact():
    # 24 groups (CTA pairs, padding tiles): C = A B + R exactly in integer mode
    A = synth.make("bf16", (24, 300, 256), "int", 64, -2, 2)
    B = synth.make("bf16", (24, 256, 1096), "int", 65, -2, 2)
    R = synth.make("f32", (24, 300, 1096), "int", 66, -100, 100)
    RA, RB, RR = rel(A, [24, 1, 1]), rel(B, [24, 1, 1]), rel(R, [24, 1, 1])
    C = joinagg("bij,bjk->bik", [RA, RB], out_dtype="f32", epi_map="add", epi_in=RR)
    assert last()["cta_pair"]
    P = oracle.joinagg("bij,bjk->bik", [A.to_f64(), B.to_f64()])
    want = oracle.joinagg("bik,bik->bik", [P, R.to_f64()], "add", "none")
    assert np.array_equal(dense64(C), want)


def _swiglu_pair_case(T, D, F, xp, wp, hp, rows=None):
    x = synth.make("bf16", (T, D), "normal", 67, 0, 1)
    w = synth.make("bf16", (D, F, 2), "normal", 68, 0, 0.05)
    H = joinagg("td,dfc->tf", [rel(x, xp), rel(w, wp)], epi_map="silu_mul", epi_pair="c")
    assert last()["kernel"] == "contract_tc"
    xs = x.to_f64() if rows is None else x.to_f64()[rows]
    wf = w.to_f64()
    G = oracle.joinagg("td,fd->tf", [xs, np.ascontiguousarray(wf[:, :, 0].T)])
    U = oracle.joinagg("td,fd->tf", [xs, np.ascontiguousarray(wf[:, :, 1].T)])
    want = oracle.joinagg("tf,tf->tf", [G, U], "silu_mul", "none")
    got = dense64(H) if rows is None else dense64(H)[rows]
    return got, want


def test_tc_epilogue_silu_pairs():
    # H = SiLU(x Wg) * (x Wu) with gate and up interleaved along c: ragged T, F in 3 blocks
    got, want = _swiglu_pair_case(300, 256, 600, [1, 2], [2, 3, 1], None)
    assert rel_frob(got, want) <= BF16_TOL


def test_tc_epilogue_silu_pairs_clustered_sampled_rows():
    # 4096 tokens x 1536 FFN columns: a clustered launch; 64 seeded rows against the oracle
    rows = [int(r) for r in synth.subset_rows(404, 4096, 64)]
    got, want = _swiglu_pair_case(4096, 512, 1536, [2, 2], [2, 4, 1], rows)
    assert rel_frob(got, want) <= BF16_TOL


@pytest.mark.parametrize("layout", [0, 1])
def test_tc_epilogue_rope(layout):
    # Q,K projection with RoPE in the epilogue: 2 sequences x 160 positions
    # (tokens in one block per sequence), 2 heads of 128, model dim 128 in 2
    # blocks; the table position-major (layout 0) or pair-major (layout 1)
    from tensor_relational_einsum_gb300.graphs import rope_table
    S, NS, H, DH, DM = 160, 2, 2, 128, 128
    T, E = NS * S, H * DH
    x = synth.make("bf16", (T, DM), "normal", 71, 0, 1)
    w = synth.make("bf16", (DM, 2, E), "normal", 72, 0, 0.1)
    tab = rope_table(S, DH, 10000.0)
    if layout == 1:
        tab = tab.transpose(0, 1).contiguous()
    out = joinagg("td,dce->cte", [rel(x, [NS, 2]), rel(w, [2, 2, 1])], epi_map="rope", rope_table=tab, rope_pos="t",
                  rope_dim=DH, rope_layout=layout)
    assert last()["kernel"] == "contract_tc"
    got = dense64(out)
    for c in range(2):
        P = oracle.joinagg("td,ed->te", [x.to_f64(), np.ascontiguousarray(w.to_f64()[:, c, :].T)])
        want = chains.rope(P.reshape(NS, S, H, DH), 10000.0).reshape(T, E)
        assert rel_frob(got[c], want) <= BF16_TOL, c


@pytest.mark.parametrize("epi", [None, "silu_mul"])
def test_tc_row_rms(epi):
    # RMSNorm's apply pushed through the contraction: rows scaled by rsqrt(ms + eps)
    # (ms from the oracle, passed as an f32 relation over the row letter)
    eps = 1e-6
    x = synth.make("bf16", (300, 256), "normal", 73, 0, 1)
    xo = x.to_f64()
    ms = oracle.joinagg("td->t", [xo], "square", "sum", scale=1.0 / 256)
    ms_rel = rel(synth.Tensor(ms.astype(np.float32), "f32", (300,)), [2])
    n = oracle.joinagg("td,t,d->td", [xo, ms, np.ones(256)], "rms_apply", "none", eps=eps)
    if epi is None:
        w = synth.make("bf16", (256, 384), "normal", 74, 0, 0.1)
        out = joinagg("td,de->te", [rel(x, [2, 2]), rel(w, [2, 1])], row_rms=ms_rel, eps=eps, out_dtype="f32")
        want = oracle.joinagg("td,ed->te", [n, np.ascontiguousarray(w.to_f64().T)])
        tol = 1e-5
    else:
        w = synth.make("bf16", (256, 192, 2), "normal", 74, 0, 0.1)
        out = joinagg("td,dfc->tf", [rel(x, [2, 2]), rel(w, [2, 1, 1])], row_rms=ms_rel, eps=eps,
                      epi_map="silu_mul", epi_pair="c")
        wf = w.to_f64()
        G = oracle.joinagg("td,fd->tf", [n, np.ascontiguousarray(wf[:, :, 0].T)])
        U = oracle.joinagg("td,fd->tf", [n, np.ascontiguousarray(wf[:, :, 1].T)])
        want = oracle.joinagg("tf,tf->tf", [G, U], "silu_mul", "none")
        tol = BF16_TOL
    assert last()["kernel"] == "contract_tc"
    assert rel_frob(dense64(out), want) <= tol


def test_tc_unaligned_bf16_needs_explicit_simt():
    # block rows of 45 and 33 bf16 elements are not 16-byte aligned, so TMA
    # cannot tile the operands: refused unless the SIMT kernel is asked for
    from tensor_relational_einsum_gb300._abi import EaError
    A = synth.make("bf16", (70, 45), "normal", 5, 0, 1)
    B = synth.make("bf16", (45, 33), "normal", 6, 0, 1)
    with pytest.raises(EaError, match="simt_bf16"):
        joinagg("ij,jk->ik", [rel(A, [2, 3]), rel(B, [3, 1])], out_dtype="f32")
    got, want, _ = _bf16_case("ij,jk->ik", [(70, 45), (45, 33)], [[2, 3], [3, 1]], "f32", expect="contract_simt",
                              simt_bf16=True)
    assert rel_frob(got, want) <= 1e-5


# -------------------------------------------------------------- elementwise

def test_ewise_silu_mul_and_add():
    G = synth.make("bf16", (96, 1040), "normal", 7, 0, 1)
    U = synth.make("bf16", (96, 1040), "normal", 8, 0, 1)
    H = joinagg("ik,ik->ik", [rel(G, [2, 4]), rel(U, [2, 4])], agg="none", map="silu_mul")
    assert last()["kernel"] == "elementwise"
    want = oracle.joinagg("ik,ik->ik", [G.to_f64(), U.to_f64()], "silu_mul", "none")
    assert rel_frob(dense64(H), want) <= 5e-3
    S = joinagg("ik,ik->ik", [rel(G, [3, 1]), rel(U, [3, 1])], agg="none", map="add", out_dtype="f32")
    want = oracle.joinagg("ik,ik->ik", [G.to_f64(), U.to_f64()], "add", "none")
    assert rel_frob(dense64(S), want) <= 1e-6


def test_ewise_rms_apply_broadcast_and_scalar_path():
    x = synth.make("bf16", (64, 264), "normal", 9, 0, 1)
    ms = synth.make("f32", (64,), "uniform", 10, 0.5, 2.0)
    g = synth.make("bf16", (264,), "normal", 11, 1, 0.1)
    want = oracle.joinagg("td,t,d->td", [x.to_f64(), ms.to_f64(), g.to_f64()], "rms_apply", "none", eps=1e-6)
    for parts in ([2, 1], [[0, 10, 64], [0, 5, 264]]):   # second: 5-wide blocks -> scalar path
        y = joinagg("td,t,d->td", [rel(x, parts), rel(ms, [parts[0]]), rel(g, [parts[1]])], agg="none",
                    map="rms_apply", eps=1e-6)
        assert rel_frob(dense64(y), want) <= 5e-3


def test_ewise_softmax_normalise_with_predicate():
    S = synth.make("f32", (1, 2, 64, 96), "normal", 12, 0, 2)
    m = synth.make("f32", (1, 2, 64), "normal", 13, 3, 0.1)
    l = synth.make("f32", (1, 2, 64), "uniform", 14, 5, 9)
    # cells with t > s are removed: the join keeps t <= s
    P = joinagg("bhst,bhs,bhs->bhst", [rel(S, [1, 2, 2, 3]), rel(m, [1, 2, 2]), rel(l, [1, 2, 2])], agg="none",
                map="exp_sub_div", pred="ts")
    E = oracle.joinagg("bhst,bhs->bhst", [S.to_f64(), m.to_f64()], "exp_sub", "none")
    want = oracle.joinagg("bhst,bhs->bhst", [E, l.to_f64()], "div", "none")
    s_idx = np.arange(64)[:, None]
    t_idx = np.arange(96)[None, :]
    got = dense64(P)
    # cells the predicate removes are absent; blocks with no kept cell are not written
    assert rel_frob(got, np.where(t_idx <= s_idx, want, np.nan)) <= 1e-6
    # removed cells inside a written block hold 0: s-block [32, 64) x t-block [32, 64)
    blk = got[..., 32:64, 32:64]
    assert np.all(blk[..., (t_idx[:, 32:64] > s_idx[32:64, :])] == 0.0)


def test_ewise_rope_against_rotation_relation():
    import torch as T
    b, s, h, d = 2, 48, 3, 64
    x = synth.make("bf16", (b, s, h, d), "normal", 15, 0, 1)
    i = np.arange(d // 2, dtype=np.float64)
    ang = np.arange(s, dtype=np.float64)[:, None] * (10000.0 ** (-2 * i / d))[None, :]
    tab = T.tensor(np.stack([np.cos(ang), np.sin(ang)], -1).astype(np.float32), device="cuda")
    y = joinagg("bshd->bshd", [rel(x, [2, 3, 1, 1])], agg="none", map="rope", rope_table=tab, rope_pos="s")
    want = chains.rope(x.to_f64(), 10000.0)
    assert rel_frob(dense64(y), want) <= 5e-3


# ------------------------------------------------------------ row reduction

def test_rowreduce_max_sum_square():
    S = synth.make("f32", (1, 3, 40, 300), "normal", 16, 0, 3)
    RS = rel(S, [1, 3, 2, [0, 100, 200, 300]])
    m = joinagg("bhst->bhs", [RS], agg="max", map="identity")
    assert last()["kernel"] == "rowreduce" and last()["tuples"] == 3 * 2 * 3
    want_m = oracle.joinagg("bhst->bhs", [S.to_f64()], "identity", "max")
    assert np.array_equal(dense64(m), want_m)
    l = joinagg("bhst,bhs->bhs", [RS, m], agg="sum", map="exp_sub")
    want_l = oracle.joinagg("bhst->bhs", [oracle.joinagg("bhst,bhs->bhst", [S.to_f64(), want_m], "exp_sub", "none")],
                            "identity", "sum")
    assert rel_frob(dense64(l), want_l) <= 1e-5
    x = synth.make("bf16", (70, 264), "normal", 17, 0, 1)
    ms = joinagg("td->t", [rel(x, [2, 3])], agg="sum", map="square", scale=1.0 / 264, out_dtype="f32")
    want = oracle.joinagg("td->t", [x.to_f64()], "square", "sum", scale=1.0 / 264)
    assert rel_frob(dense64(ms), want) <= 1e-5


@pytest.mark.parametrize("parts,pred", [([1, 3, 2, [0, 100, 200, 300]], None), ([1, 3, 2, [0, 100, 200, 300]], "ts"),
                                        ([1, 1, 1, [0, 37, 300]], "ts")])
def test_rowreduce_fused_softmax_stats(parts, pred):
    """MAX_SUMEXP against the oracle's two join-aggs: m = MAX_t S and
    l = SUM_t exp(S - m) (cells with t > s removed when pred is set); the
    last case has 37-wide blocks (scalar path)."""
    from tensor_relational_einsum_gb300.relation import Relation
    S = synth.make("f32", (1, 3, 40, 300), "normal", 19, 0, 3)
    RS = rel(S, parts)
    m = Relation("f32", (1, 3, 40), [parts[0], parts[1], parts[2]])
    l = Relation("f32", (1, 3, 40), [parts[0], parts[1], parts[2]])
    joinagg("bhst->bhs", [RS], agg="max_sumexp", map="identity", out=m, out2=l, pred=pred)
    assert last()["kernel"] == "rowreduce"
    want_m = oracle.joinagg("bhst->bhs", [S.to_f64()], "identity", "max", pred=pred)
    E = oracle.joinagg("bhst,bhs->bhst", [S.to_f64(), want_m], "exp_sub", "none", pred=pred)
    want_l = oracle.joinagg("bhst->bhs", [E], "identity", "sum")
    assert np.array_equal(dense64(m), want_m)
    assert rel_frob(dense64(l), want_l) <= 1e-5


@pytest.mark.parametrize("dtype,shape,parts", [("f32", (2, 3, 40, 512), [2, 3, 2, 4]),
                                               ("bf16", (1, 2, 50, 256), [1, 2, [0, 16, 33, 50], 4])])
def test_rowreduce_rowbatch_stats(dtype, shape, parts):
    """The softmax statistics over rows cut into four equal, vectorisable
    blocks (the row-batch kernel): ragged tiles, and for bf16 64-wide
    segments with sixteen rows per warp pass."""
    from tensor_relational_einsum_gb300.relation import Relation
    S = synth.make(dtype, shape, "normal", 23, 0, 3)
    m = Relation("f32", shape[:3], parts[:3])
    l = Relation("f32", shape[:3], parts[:3])
    joinagg("bhst->bhs", [rel(S, parts)], agg="max_sumexp", map="identity", out=m, out2=l)
    assert last()["kernel"] == "rowreduce"
    want_m = oracle.joinagg("bhst->bhs", [S.to_f64()], "identity", "max")
    E = oracle.joinagg("bhst,bhs->bhst", [S.to_f64(), want_m], "exp_sub", "none")
    want_l = oracle.joinagg("bhst->bhs", [E], "identity", "sum")
    assert np.array_equal(dense64(m), want_m)
    assert rel_frob(dense64(l), want_l) <= 1e-5


def test_rowreduce_scaled_softmax_stats():
    """MAX_SUMEXP of scale * S with scale 0.25 over row-batch-shaped blocks:
    m = MAX_t (scale S), l = SUM_t exp(scale S - m) against the oracle."""
    from tensor_relational_einsum_gb300.relation import Relation
    S = synth.make("f32", (2, 3, 40, 512), "normal", 27, 0, 3)
    m = Relation("f32", (2, 3, 40), [2, 3, 2])
    l = Relation("f32", (2, 3, 40), [2, 3, 2])
    joinagg("bhst->bhs", [rel(S, [2, 3, 2, 4])], agg="max_sumexp", map="identity", out=m, out2=l, scale=0.25)
    assert last()["kernel"] == "rowreduce"
    want_m = oracle.joinagg("bhst->bhs", [S.to_f64()], "identity", "max", scale=0.25)
    E = oracle.joinagg("bhst,bhs->bhst", [0.25 * S.to_f64(), want_m], "exp_sub", "none")
    want_l = oracle.joinagg("bhst->bhs", [E], "identity", "sum")
    assert rel_frob(dense64(m), want_m) <= 1e-6
    assert rel_frob(dense64(l), want_l) <= 1e-5


def test_rowreduce_rowbatch_sum_of_squares_four_pass_tiles():
    """40960 rows of 4096 bf16 in 8 x 4 blocks (2 KB row segments stored
    back to back: the bulk-copy kernel): enough rows that the planner cuts
    tiles of 32 rows, four 8-row chunks per block; 64 sampled rows against
    the oracle."""
    from tensor_relational_einsum_gb300.relation import Relation
    x = synth.make_torch("bf16", (40960, 4096), "normal", 24, 0, 1, device="cuda")
    ms = joinagg("td->t", [Relation.from_dense(x, [8, 4])], agg="sum", map="square", scale=1.0 / 4096,
                 out_dtype="f32")
    assert last()["kernel"] == "rowreduce" and last()["tiles"] == 8 * (5120 // 32)
    rows = [int(i) for i in synth.subset_rows(25, 40960, 64)]
    xs = x[rows].double().cpu().numpy()
    want = oracle.joinagg("td->t", [xs], "square", "sum", scale=1.0 / 4096)
    got = ms.to_dense()[rows].double().cpu().numpy()
    assert rel_frob(got, want) <= 1e-5


@pytest.mark.parametrize("dtype,map_,shape,parts", [
    ("bf16", "square", (300, 1024), [[0, 100, 213, 300], 4]),   # 512-byte segments, ragged 8-row chunks
    ("f32", "identity", (77, 2048), [[0, 40, 77], 4]),           # 2 KB fp32 segments, one block of odd rows
    ("bf16", "identity", (90, 8192), [3, 4]),                    # 4 KB segments: the row-batch kernel
    ("f32", "square", (50, 4096), [2, 2]),                       # 8 KB segments: the row-batch kernel
    ("f32", "identity", (64, 4096), [2, 8]),                     # eight blocks a row: the tile kernel
])
def test_rowreduce_rowbatch_sum_paths(dtype, map_, shape, parts):
    """SUM (of scale x or scale x^2) over whole rows, every row against the
    oracle: in at most four equal blocks with row segments of at most 2 KB
    stored back to back the bulk-copy kernel serves it (chunks of 8 rows of
    one block, the last chunk of a block ragged), with longer segments the
    row-batch kernel, with eight blocks the tile kernel's packed row sums.
    The scale is not 1, so each path must apply it for both maps."""
    x = synth.make(dtype, shape, "normal", 26, 0, 1)
    got = joinagg("td->t", [rel(x, parts)], agg="sum", map=map_, scale=1.0 / shape[1], out_dtype="f32")
    assert last()["kernel"] == "rowreduce"
    want = oracle.joinagg("td->t", [x.to_f64()], map_, "sum", scale=1.0 / shape[1])
    assert rel_frob(dense64(got), want) <= 1e-5


def test_rowreduce_causal_predicate():
    S = synth.make("f32", (1, 2, 64, 64), "normal", 18, 0, 2)
    RS = rel(S, [1, 2, 4, 4])
    m = joinagg("bhst->bhs", [RS], agg="max", map="identity", pred="ts")
    assert last()["tuples"] == 2 * (1 + 2 + 3 + 4)
    Sm = np.where(np.tril(np.ones((64, 64), bool)), S.to_f64(), np.nan)
    want = oracle.joinagg("bhst->bhs", [Sm], "identity", "max")
    assert np.array_equal(dense64(m), want)


# ------------------------------------------------------------ device checks

def test_no_device_error_raised():
    from tensor_relational_einsum_gb300.relation import check
    check()


# ----------------------------------------------------- host load / offload

@pytest.mark.parametrize("dtype,dims,parts", [
    ("bf16", (300, 200), [[0, 100, 300], [0, 72, 200]]),
    ("f32", (64, 8192), [4, 1]),
    ("bf16", (3, 5, 7, 9), [3, 1, 7, 1]),
    ("f32", (2, 64, 4, 128), [2, 4, 2, 1]),
    ("bf16", (1000,), [[0, 7, 1000]]),
])
def test_copy_host_bit_exact(dtype, dims, parts):
    """A relation loaded from a dense host tensor holds the oracle's arena
    of that tensor bit for bit, and offloading it gives the tensor back."""
    from tensor_relational_einsum_gb300.relation import Relation
    t = synth.make(dtype, dims, "uniform", 91, -1, 1)
    if dtype == "bf16":
        host = torch.from_numpy(t.host.view(np.int16).copy()).view(torch.bfloat16).reshape(dims)
    else:
        host = torch.from_numpy(t.host.copy()).reshape(dims)
    host = host.contiguous().pin_memory()
    R = Relation(dtype, dims, parts, device="cuda")
    R.copy_host(host, to_device=True)
    torch.cuda.synchronize()
    flat = t.host.reshape(-1)
    want = oracle.exchange(flat, dims, [[0, n] for n in dims], bounds_of(dims, parts))
    assert np.array_equal(arena_bits(R).view(flat.dtype), want)
    back = torch.empty_like(host).pin_memory()
    R.copy_host(back, to_device=False)
    torch.cuda.synchronize()
    bits = (lambda x: x.view(torch.int16)) if dtype == "bf16" else (lambda x: x.view(torch.int32))
    assert torch.equal(bits(back), bits(host))
