"""GPU parity at the workloads' full sizes, in the configurations bench.py
times, on outputs the oracle can compute one by one:

* attention b4 h32 s=t=2048 d128 (t in 4 blocks): eight seeded (b, h)
  pairs in full, S, m, l, P and O (an attention output depends only on its
  own (b, h) inputs);
* SwiGLU FFN x[8192, 4096] with 4096 x 11008 weights (contracted dims in 4
  blocks; SiLU * up fused into the gate+up epilogue): 64 seeded token
  rows (the FFN is row-wise);
* the exchange of bf16 8192^2 from 8x1 row blocks to 1x8, 4x2 and 16x16:
  every element, bit-exact;
* the LLaMA-7B-shaped block (b8, s2048): a 16-token prefix of one seeded
  sequence -- causal attention only looks back, so the prefix outputs of
  the full-size run equal the oracle's block on the prefix alone.

Inputs are drawn once on the host with the seeded generator; the GPU gets
the same bits, the oracle the same values in fp64.
"""
import numpy as np
import pytest

import oracle
import synth
from oracle import chains

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

from gpu_util import BF16_TOL, FP32_TOL, rel_frob  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    from tensor_relational_einsum_gb300.build import build
    build()
    yield
    from tensor_relational_einsum_gb300.relation import check
    check()
    torch.cuda.empty_cache()


def host(dtype, shape, dist, seed, a, b):
    return synth.make_torch(dtype, shape, dist, seed, a, b, device="cpu")


def f64(t):
    return t.double().numpy()


def pick(seed, n_total, n):
    return [int(i) for i in synth.subset_rows(seed, n_total, n)]


def test_attention_chain_full_size_sampled_heads():
    from tensor_relational_einsum_gb300.graphs import AttentionChain
    from tensor_relational_einsum_gb300.relation import Relation
    shape = (4, 32, 2048, 128)
    q, k, v = (host("bf16", shape, "normal", sd, 0.0, 1.0) for sd in (11, 12, 13))
    ch = AttentionChain(Relation.from_dense(q.cuda(), [4, 32, 1, 1]), Relation.from_dense(k.cuda(), [4, 32, 4, 1]),
                        Relation.from_dense(v.cuda(), [4, 32, 4, 1]))
    ch.run()
    torch.cuda.synchronize()
    S, m, l, P, O = (x.to_dense() for x in (ch.S, ch.m, ch.l, ch.P, ch.O))
    for pair in pick(101, 4 * 32, 8):
        b, h = divmod(pair, 32)
        sl = (slice(b, b + 1), slice(h, h + 1))
        want = chains.softmax_attention(f64(q[sl]), f64(k[sl]), f64(v[sl]))
        assert rel_frob(S[sl].double().cpu().numpy(), want["S"]) <= FP32_TOL
        assert rel_frob(m[sl].double().cpu().numpy(), want["m"]) <= FP32_TOL
        assert rel_frob(l[sl].double().cpu().numpy(), want["l"]) <= FP32_TOL
        assert rel_frob(P[sl].double().cpu().numpy(), want["P"]) <= BF16_TOL
        assert rel_frob(O[sl].double().cpu().numpy(), want["O"]) <= BF16_TOL
    assert torch.isfinite(O).all()
    del ch, S, P


def test_swiglu_ffn_full_size_sampled_rows():
    from tensor_relational_einsum_gb300.graphs import SwigluFFN
    from tensor_relational_einsum_gb300.relation import Relation
    x = host("bf16", (8192, 4096), "normal", 21, 0.0, 1.0)
    wg = host("bf16", (4096, 11008), "normal", 22, 0.0, 0.02)
    wu = host("bf16", (4096, 11008), "normal", 23, 0.0, 0.02)
    wd = host("bf16", (11008, 4096), "normal", 24, 0.0, 0.02)
    ffn = SwigluFFN(Relation.from_dense(x.cuda(), [1, 4]), wg.cuda(), wu.cuda(), wd.cuda(), k_blocks=4)
    ffn.run()
    torch.cuda.synchronize()
    rows = pick(202, 8192, 64)
    want = chains.swiglu_ffn(f64(x[rows]), f64(wg), f64(wu), f64(wd))
    # the bench's configuration: SiLU * up fused into the gate+up epilogue (G, U never written)
    got = {k: getattr(ffn, k).to_dense()[rows].double().cpu().numpy() for k in ("H", "Y")}
    for k in ("H", "Y"):
        assert rel_frob(got[k], want[k]) <= BF16_TOL, k
    assert torch.isfinite(ffn.Y.to_dense()).all()
    del ffn


@pytest.mark.parametrize("dst", [[1, 8], [4, 2], [16, 16]])
def test_exchange_full_size_bit_exact(dst):
    from tensor_relational_einsum_gb300.relation import Relation, exchange
    X = host("bf16", (8192, 8192), "uniform", 31, -1.0, 1.0)
    R = Relation.from_dense(X.cuda(), [8, 1])
    Y = exchange(R, dst)
    torch.cuda.synchronize()
    bits = X.view(torch.int16).numpy().view(np.uint16).reshape(-1)
    want = oracle.exchange(bits, (8192, 8192), [[0, 8192], [0, 8192]],
                           [oracle.near_equal_bounds(8192, dst[0]), oracle.near_equal_bounds(8192, dst[1])])
    got = Y.arena().cpu().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, want)


def test_llama_block_full_size_prefix_sample():
    from tensor_relational_einsum_gb300.graphs import LlamaBlock
    B, S, D, NH, FF = 8, 2048, 4096, 32, 11008
    seeds = {"wq": 101, "wk": 102, "wv": 103, "wo": 104, "w_gate": 105, "w_up": 106, "w_down": 107}
    shapes = {"wq": (D, D), "wk": (D, D), "wv": (D, D), "wo": (D, D), "w_gate": (D, FF), "w_up": (D, FF),
              "w_down": (FF, D)}
    W = {k: host("bf16", shapes[k], "normal", seeds[k], 0.0, 0.02) for k in seeds}
    x = host("bf16", (B * S, D), "normal", 100, 0.0, 1.0)
    Wg = {k: v.cuda() for k, v in W.items()}
    # RMSNorm gains ~ N(1, 0.1) (folded into the projection weights by the block)
    gains = {k: host("bf16", (D,), "normal", sd, 1.0, 0.1) for k, sd in (("g1", 108), ("g2", 109))}
    Wg["g1"] = gains["g1"].cuda()
    Wg["g2"] = gains["g2"].cuda()
    blk = LlamaBlock(B, S, D, NH, FF, Wg, eps=1e-6, theta=10000.0)
    del Wg
    blk.x.load(x.cuda())
    blk.run()
    torch.cuda.synchronize()
    y = blk.y.to_dense()
    assert torch.isfinite(y).all()
    seq = pick(303, B, 1)[0]
    n = 16
    Wd = {k: f64(v) for k, v in W.items()}
    Wd["g1"] = f64(gains["g1"])
    Wd["g2"] = f64(gains["g2"])
    xs = f64(x[seq * S: seq * S + n]).reshape(1, n, D)
    want = chains.llama_block(xs, Wd, n_heads=NH, eps=1e-6, theta=10000.0)
    got_y = y[seq * S: seq * S + n].double().cpu().numpy().reshape(1, n, D)
    assert rel_frob(got_y, want["y"]) <= BF16_TOL
    got_h = blk.h.to_dense()[seq * S: seq * S + n].double().cpu().numpy()
    assert rel_frob(got_h, want["h"]) <= BF16_TOL
    got_o = blk.attn.O.to_dense()[seq, :n].double().cpu().numpy()
    assert rel_frob(got_o, want["O"][0]) <= BF16_TOL
    del blk
