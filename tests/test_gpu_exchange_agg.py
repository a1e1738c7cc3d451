"""GPU parity of the exchange with aggregation ("Every Kernel Is a Join",
Section 5.3, Example 5.4): a contraction run without its aggregation step
leaves m unaggregated copies of each output block (the partials option), and
ea_exchange_agg combines the copies of every atom in copy order while it
re-blocks them into the consumer's tiling.

Bars: integer-valued inputs make every partial and every sum exact, so the
re-blocked arena must equal the oracle's bit for bit; MAX is exact for any
values; a SUM of m fp32 copies in fp32 is within 1e-5 relative Frobenius.
"""
import numpy as np
import pytest

import oracle
import synth
from oracle import blocked

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

from gpu_util import FP32_TOL, arena_bits, bounds_of, dense64, last, rel, rel_frob  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    from tensor_relational_einsum_gb300.build import build
    build()
    yield
    from tensor_relational_einsum_gb300.relation import check
    check()


def _arena_of(dense: np.ndarray, dtype: str, bounds) -> np.ndarray:
    """The oracle's arena of ``dense`` under ``bounds``, as raw element bits."""
    if dtype == "bf16":
        flat = synth.f32_to_bf16_bits(dense.astype(np.float32).reshape(-1))
    else:
        flat = dense.astype(np.float32).reshape(-1).view(np.int32)
    whole = [[0, n] for n in dense.shape]
    return oracle.exchange(flat, dense.shape, whole, bounds)


@pytest.mark.parametrize("agg", ["sum", "max"])
def test_example_5_4_partials_then_exchange_agg(agg):
    """The producer of Example 5.4: i = k = 256, j = 512, i and j in two
    intervals each, so each of C1 and C2 has two unaggregated copies (X, Y).
    The consumer takes four 64-row blocks: S_j = X_j (+) Y_j."""
    from tensor_relational_einsum_gb300.relation import exchange_agg, joinagg
    A = synth.make("bf16", (256, 512), "int", 541, -3, 3)
    B = synth.make("bf16", (512, 256), "int", 542, -3, 3)
    P = joinagg("ij,jk->ik", [rel(A, [2, 2]), rel(B, [2, 1])], partials=True, out_dtype="f32")
    info = last()
    assert info["groups"] == 4 and info["tuples"] == 4
    bnd = {"i": [0, 128, 256], "j": [0, 256, 512], "k": [0, 256]}
    want_p = blocked.joinagg_partials("ij,jk->ik", [A.to_f64(), B.to_f64()], bnd)
    assert P.dims == (2, 256, 256)
    assert np.array_equal(dense64(P), want_p)
    S = exchange_agg(P, agg, [4, 1])
    assert last()["kernel"] == "exchange_agg"
    want = blocked.aggregate_copies(want_p, agg)
    assert np.array_equal(arena_bits(S), _arena_of(want, "f32", bounds_of((256, 256), [4, 1])))


CASES = [
    # dims (copies first), source tiling, destination tiling
    ((2, 256, 256), [2, 2, 1], [4, 1]),                             # Example 5.4's shape
    ((4, 300, 200), [4, [0, 100, 300], [0, 72, 200]], [[0, 64, 128, 250, 300], [0, 40, 200]]),
    ((3, 130, 96), [3, 3, 2], [2, 4]),                               # ragged overlays both ways
    ((2, 7, 5), [2, 1, 1], [[0, 3, 7], [0, 2, 5]]),                  # copy stride of 35 elements: no vector path
    ((5, 64, 1000), [5, 2, 3], [1, 1]),                              # gather into one block
    ((1, 50, 40), [1, 2, 2], [3, 3]),                                # a single copy is a plain exchange
    ((2, 3, 9000), [2, 1, 1], [1, [0, 4500, 9000]]),                 # long runs: cut into 8 KiB rows + a tail
]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("agg", ["sum", "max"])
@pytest.mark.parametrize("dims,src,dst", CASES)
def test_exchange_agg_integer_bit_exact(dtype, agg, dims, src, dst):
    from tensor_relational_einsum_gb300.relation import exchange_agg
    t = synth.make(dtype, dims, "int", 77, -20, 20)
    X = exchange_agg(rel(t, src), agg, dst)
    want = blocked.aggregate_copies(t.to_f64(), agg)
    assert np.array_equal(arena_bits(X), _arena_of(want, dtype, bounds_of(dims[1:], dst)))


@pytest.mark.parametrize("dims,src,dst", CASES[:3])
def test_exchange_agg_fp32_sum_and_max(dims, src, dst):
    from tensor_relational_einsum_gb300.relation import exchange_agg
    t = synth.make("f32", dims, "normal", 78, 0, 1)
    want = blocked.aggregate_copies(t.to_f64(), "sum")
    assert rel_frob(dense64(exchange_agg(rel(t, src), "sum", dst)), want) <= FP32_TOL
    X = exchange_agg(rel(t, src), "max", dst)
    mx = blocked.aggregate_copies(t.to_f64(), "max")
    assert np.array_equal(arena_bits(X), _arena_of(mx, "f32", bounds_of(dims[1:], dst)))


def test_exchange_agg_into_given_output_and_repeat():
    from tensor_relational_einsum_gb300.relation import Relation, exchange_agg
    t = synth.make("f32", (3, 200, 128), "normal", 79, 0, 1)
    P = rel(t, [3, 4, 2])
    out = Relation("f32", (200, 128), [[0, 50, 150, 200], 1], device="cuda")
    exchange_agg(P, "sum", out=out)
    a = out.arena().clone()
    exchange_agg(P, "sum", out=out)
    torch.cuda.synchronize()
    assert torch.equal(a, out.arena())


def test_partials_bf16_output_then_sum():
    """bf16 partial copies: each copy is a bf16 rounding of an exact fp32
    value; the fp32 sum of the copies, rounded once, is within the bf16
    bar of the oracle's aggregate."""
    from tensor_relational_einsum_gb300.relation import exchange_agg, joinagg
    A = synth.make("bf16", (384, 1024), "normal", 543, 0, 1)
    B = synth.make("bf16", (1024, 256), "normal", 544, 0, 1)
    P = joinagg("ij,jk->ik", [rel(A, [3, 4]), rel(B, [4, 2])], partials=True)
    assert P.dims == (4, 384, 256)
    bnd = {"i": [0, 128, 256, 384], "j": [0, 256, 512, 768, 1024], "k": [0, 128, 256]}
    want_p = blocked.joinagg_partials("ij,jk->ik", [A.to_f64(), B.to_f64()], bnd)
    assert rel_frob(dense64(P), want_p) <= 2e-2
    S = exchange_agg(P, "sum", [[0, 100, 384], 1])
    assert rel_frob(dense64(S), A.to_f64() @ B.to_f64()) <= 2e-2


def test_full_size_ffn_down_partials_sampled_rows():
    """The FFN's down projection h[8192, 11008] x w_down[11008, 4096], bf16,
    with the contracted dim in 4 blocks run as 4 unaggregated fp32 copies,
    then SUM-exchanged into 16 x 16 tiles: sampled rows against the oracle's
    per-copy partial products and their sum."""
    from tensor_relational_einsum_gb300.relation import Relation, exchange_agg, joinagg
    h = synth.make_torch("bf16", (8192, 11008), "normal", 21, 0.0, 1.0, device="cpu")
    w = synth.make_torch("bf16", (11008, 4096), "normal", 22, 0.0, 0.02, device="cpu")
    H = Relation.from_dense(h.cuda(), [1, 4])
    W = Relation.from_dense(w.cuda(), [4, 1])
    P = joinagg("ij,jk->ik", [H, W], partials=True, out_dtype="f32")
    S = exchange_agg(P, "sum", [16, 16])
    got_p = P.to_dense()
    got = S.to_dense()
    torch.cuda.synchronize()
    jb = oracle.near_equal_bounds(11008, 4)
    wd = w.double().numpy()
    for r in synth.subset_rows(103, 8192, 3):
        r = int(r)
        hd = {r: h[r].double().numpy()}
        parts = np.stack([hd[r][jb[q]:jb[q + 1]] @ wd[jb[q]:jb[q + 1]] for q in range(4)])
        assert rel_frob(got_p[:, r].double().cpu().numpy(), parts) <= FP32_TOL
        assert rel_frob(got[r].double().cpu().numpy(), blocked.aggregate_copies(parts[:, None], "sum")[0]) <= FP32_TOL
