"""GPU parity of the fused attention join-agg (ea_attention_run) against the
oracle's flash attention ("Every Kernel Is a Join", Example 3.10): heads
grouped g to 1, packed sequences, causal predicate, ragged query and key
tiles, head dims 64 and 128, rank-3 and rank-4 terms, and the full-size
attention shapes on sampled heads.

Tolerances: O is bf16 from bf16 inputs with the probabilities rounded to
bf16 before the second product: 2e-2 relative Frobenius.  The row maximum m
is a max of fp32 dot products of bf16 values (exact products, fp32 sums) and
l a sum of fp32 exponentials: 1e-5.
"""
import numpy as np
import pytest

import synth
from oracle import chains

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

from gpu_util import BF16_TOL, FP32_TOL, dense64, rel, rel_frob  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    from tensor_relational_einsum_gb300.build import build
    build()
    yield
    from tensor_relational_einsum_gb300.relation import check
    check()


def _stats(q_rel):
    from tensor_relational_einsum_gb300.relation import Relation
    dims, bounds = q_rel.dims[:-1], q_rel.bounds[:-1]
    return (Relation("f32", dims, bounds, device="cuda"), Relation("f32", dims, bounds, device="cuda"))


def _to_bhs(x, layout):
    """[b, s, h] (bshd stats) -> [b, h, s]."""
    return x if layout == "bhsd" else np.transpose(x, (0, 2, 1))


def _run(spec, Q, K, V, qp, kp, layout, group=1, scale=0.0, causal=False, seq_ends=None, stats=True):
    from tensor_relational_einsum_gb300 import _abi
    from tensor_relational_einsum_gb300.relation import attention
    q, k, v = rel(Q, qp), rel(K, kp), rel(V, kp)
    m, l = _stats(q) if stats else (None, None)
    O = attention(spec, q, k, v, scale=scale, causal=causal, seq_ends=seq_ends, m_out=m, l_out=l)
    torch.cuda.synchronize()
    assert _abi.last_plan()["kernel"] == "attention"
    d = Q.shape[-1]
    sc = scale if scale > 0 else 1.0 / np.sqrt(d)
    want = chains.flash_attention(Q.to_f64(), K.to_f64(), V.to_f64(), group=group, scale=sc, causal=causal,
                                  seq_ends=seq_ends, layout=layout)
    got = dense64(O)
    assert np.isfinite(got).all()
    assert rel_frob(got, want["O"]) <= BF16_TOL
    if stats:
        assert rel_frob(_to_bhs(dense64(m), layout), want["m"]) <= FP32_TOL
        assert rel_frob(_to_bhs(dense64(l), layout), want["l"]) <= FP32_TOL
    return O


def test_mha_head_major_ragged_tiles():
    # s = t = 300: query tiles of 128, 128, 44; t in 3 blocks of 100 keys (one partial tile each)
    shp = (1, 2, 300, 128)
    Q, K, V = (synth.make("bf16", shp, "normal", sd, 0, 1) for sd in (41, 42, 43))
    _run("bhsd,bhtd,bhtd->bhsd", Q, K, V, [1, 2, 1, 1], [1, 2, 3, 1], "bhsd", scale=1.0)


@pytest.mark.parametrize("causal", [False, True])
def test_grouped_heads_token_major(causal):
    # 8 query heads over 2 key-value heads (g = 4), s in 3 blocks, t in 2
    Q = synth.make("bf16", (2, 384, 8, 128), "normal", 44, 0, 1)
    K, V = (synth.make("bf16", (2, 384, 2, 128), "normal", sd, 0, 1) for sd in (45, 46))
    _run("bshd,bthd,bthd->bshd", Q, K, V, [2, 3, 1, 1], [2, 2, 1, 1], "bshd", group=4, causal=causal)


def test_grouped_heads_in_head_blocks():
    # query heads in blocks [0, 4), [4, 8) over key-value heads [0, 1), [1, 2)
    Q = synth.make("bf16", (1, 256, 8, 128), "normal", 47, 0, 1)
    K, V = (synth.make("bf16", (1, 256, 2, 128), "normal", sd, 0, 1) for sd in (48, 49))
    _run("bshd,bthd,bthd->bshd", Q, K, V, [1, 2, [0, 4, 8], 1], [1, 4, [0, 1, 2], 1], "bshd", group=4, causal=True)


@pytest.mark.parametrize("causal", [False, True])
def test_packed_sequences_head_dim_64(causal):
    # three packed sequences ending at 100, 260 and 512; g = 2; d = 64
    Q = synth.make("bf16", (1, 512, 4, 64), "normal", 50, 0, 1)
    K, V = (synth.make("bf16", (1, 512, 2, 64), "normal", sd, 0, 1) for sd in (51, 52))
    _run("bshd,bthd,bthd->bshd", Q, K, V, [1, 2, 1, 1], [1, [0, 100, 300, 512], 1, 1], "bshd", group=2,
         causal=causal, seq_ends=[100, 260, 512])


@pytest.mark.parametrize("causal", [False, True])
def test_packed_sequences_head_dim_128(causal):
    # CTA pairs (d = 128): sequences ending at 100, 260, 333 and 512, so the
    # boundaries fall inside 32-key chunks and inside warps (rows 96-127 hold
    # the end of the first sequence and the start of the second); g = 2
    Q = synth.make("bf16", (1, 512, 4, 128), "normal", 56, 0, 1)
    K, V = (synth.make("bf16", (1, 512, 2, 128), "normal", sd, 0, 1) for sd in (57, 58))
    _run("bshd,bthd,bthd->bshd", Q, K, V, [1, 2, 1, 1], [1, [0, 100, 300, 512], 1, 1], "bshd", group=2,
         causal=causal, seq_ends=[100, 260, 333, 512])


def test_rank3_terms():
    from tensor_relational_einsum_gb300.relation import attention
    Q, K, V = (synth.make("bf16", (200, 3, 128), "normal", sd, 0, 1) for sd in (53, 54, 55))
    q, k, v = rel(Q, [2, 1, 1]), rel(K, [1, 1, 1]), rel(V, [1, 1, 1])
    O = attention("shd,thd,thd->shd", q, k, v, causal=True)
    want = chains.flash_attention(Q.to_f64()[None], K.to_f64()[None], V.to_f64()[None], scale=1 / np.sqrt(128),
                                  causal=True, layout="bshd")
    assert rel_frob(dense64(O)[None], want["O"]) <= BF16_TOL


def test_repeat_is_bit_identical_and_plan_cached():
    from tensor_relational_einsum_gb300.relation import attention
    Q, K, V = (synth.make("bf16", (1, 2, 256, 128), "normal", sd, 0, 1) for sd in (56, 57, 58))
    q, k, v = rel(Q, [1, 2, 1, 1]), rel(K, [1, 2, 2, 1]), rel(V, [1, 2, 2, 1])
    O1 = attention("bhsd,bhtd,bhtd->bhsd", q, k, v, causal=True)
    a = O1.arena().clone()
    attention("bhsd,bhtd,bhtd->bhsd", q, k, v, causal=True, out=O1)
    torch.cuda.synchronize()
    assert torch.equal(a, O1.arena())


@pytest.mark.parametrize("causal,want", [(True, 2 * 3 * (4 + 3 + 2 + 1)), (False, 2 * 3 * 4 * 4)])
def test_causal_pairs_run_only_kept_key_tiles(causal, want):
    """s = t = 512 (four tiles of 128), 2 x 3 heads, t in 2 blocks: with the
    causal predicate a query tile runs only the key tiles up to its
    diagonal -- the earlier tile of a pair skips the later one's diagonal
    tile, all masked for it -- so the (query tile, key tile) steps are
    4 + 3 + 2 + 1 per head instead of 4 + 4 + 2 + 2; without it, all 16."""
    from tensor_relational_einsum_gb300 import _abi
    from tensor_relational_einsum_gb300.relation import attention
    Q, K, V = (synth.make("bf16", (2, 3, 512, 128), "normal", sd, 0, 1) for sd in (64, 65, 66))
    q, k, v = rel(Q, [2, 3, 1, 1]), rel(K, [2, 3, 2, 1]), rel(V, [2, 3, 2, 1])
    attention("bhsd,bhtd,bhtd->bhsd", q, k, v, causal=causal)
    plan = _abi.last_plan()  # read before anything else launches
    assert plan["kernel"] == "attention" and plan["tuples"] == want
    _run("bhsd,bhtd,bhtd->bhsd", Q, K, V, [2, 3, 1, 1], [2, 3, 2, 1], "bhsd", causal=causal, stats=False)


def test_value_closed_forms():
    # V = 1 everywhere: every kept row averages ones, O = 1 exactly up to bf16
    from tensor_relational_einsum_gb300.relation import Relation, attention
    Q, K = (synth.make("bf16", (1, 4, 300, 128), "normal", sd, 0, 1) for sd in (59, 60))
    ones = Relation.from_dense(torch.ones(1, 4, 300, 128, dtype=torch.bfloat16, device="cuda"), [1, 4, 3, 1])
    O = attention("bhsd,bhtd,bhtd->bhsd", rel(Q, [1, 4, 1, 1]), rel(K, [1, 4, 3, 1]), ones, causal=True)
    torch.cuda.synchronize()
    assert torch.allclose(O.to_dense().float(), torch.ones(1, 4, 300, 128, device="cuda"), atol=2e-3)


@pytest.mark.parametrize("d", [64, 128])
def test_reference_maximum_moves(d):
    """Key rows grow along t (key t scaled by 1 + t/64, scale 1): a query row's
    maximum score rises from key tile to key tile by tens of units, more than
    2^64 in exp every tile or two, so the lazily kept reference maximum moves
    and each chain's row of A is rescaled in TMEM many times (head dim 64 on
    the single-CTA kernel, 128 on CTA pairs).  Ragged query and key tiles."""
    Q = synth.make("bf16", (1, 4, 300, d), "normal", 81, 0, 1)
    K0 = synth.make("bf16", (1, 4, 700, d), "normal", 82, 0, 1)
    V = synth.make("bf16", (1, 4, 700, d), "normal", 83, 0, 1)
    grow = 1.0 + np.arange(700) / 64.0
    k = K0.to_f64() * grow[None, None, :, None]
    K = synth.Tensor(synth.f32_to_bf16_bits(synth.f64_to_f32(k)).ravel(), "bf16", K0.shape)
    _run("bhsd,bhtd,bhtd->bhsd", Q, K, V, [1, 4, 1, 1], [1, 4, 2, 1], "bhsd", scale=1.0)


def test_full_size_head_major_sampled_heads():
    """Q, K, V bf16 [4, 32, 2048, 128], (b, h) unit intervals, t in 4 blocks,
    scale 1, no mask: two seeded (b, h) pairs in full against the oracle."""
    from tensor_relational_einsum_gb300.relation import Relation, attention
    shape = (4, 32, 2048, 128)
    q, k, v = (synth.make_torch("bf16", shape, "normal", sd, 0.0, 1.0, device="cpu") for sd in (11, 12, 13))
    O = attention("bhsd,bhtd,bhtd->bhsd", Relation.from_dense(q.cuda(), [4, 32, 1, 1]),
                  Relation.from_dense(k.cuda(), [4, 32, 4, 1]), Relation.from_dense(v.cuda(), [4, 32, 4, 1]),
                  scale=1.0)
    got = O.to_dense()
    torch.cuda.synchronize()
    assert torch.isfinite(got).all()
    for pair in synth.subset_rows(101, 4 * 32, 2):
        b, h = divmod(int(pair), 32)
        sl = (slice(b, b + 1), slice(h, h + 1))
        want = chains.softmax_attention(q[sl].double().numpy(), k[sl].double().numpy(), v[sl].double().numpy())
        assert rel_frob(got[sl].double().cpu().numpy(), want["O"]) <= BF16_TOL


def test_full_size_token_major_causal_sampled_heads():
    """The block's attention: bf16 [8, 2048, 32, 128] token-major, sequences
    in 4 blocks of 512, causal, scale 1/sqrt(128): two seeded (b, h) pairs."""
    from tensor_relational_einsum_gb300.relation import Relation, attention
    shape = (8, 2048, 32, 128)
    q, k, v = (synth.make_torch("bf16", shape, "normal", sd, 0.0, 1.0, device="cpu") for sd in (61, 62, 63))
    O = attention("bshd,bthd,bthd->bshd", Relation.from_dense(q.cuda(), [8, 4, 1, 1]),
                  Relation.from_dense(k.cuda(), [8, 4, 1, 1]), Relation.from_dense(v.cuda(), [8, 4, 1, 1]),
                  causal=True)
    got = O.to_dense()
    torch.cuda.synchronize()
    assert torch.isfinite(got).all()
    for pair in synth.subset_rows(102, 8 * 32, 2):
        b, h = divmod(int(pair), 32)
        sl = (slice(b, b + 1), slice(None), slice(h, h + 1))
        want = chains.flash_attention(q[sl].double().numpy(), k[sl].double().numpy(), v[sl].double().numpy(),
                                      scale=1 / np.sqrt(128), causal=True, layout="bshd")
        assert rel_frob(got[sl].double().cpu().numpy(), want["O"]) <= BF16_TOL
