"""GPU parity of the workload graphs (attention chain, SwiGLU FFN, LLaMA
block) against the oracle's join-agg compositions, at reduced sizes where
the oracle covers every output cell."""
import numpy as np
import pytest

import synth
from oracle import chains

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

from gpu_util import BF16_TOL, dense64, rel, rel_frob, to_device  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    from tensor_relational_einsum_gb300.build import build
    build()
    yield
    from tensor_relational_einsum_gb300.relation import check
    check()


def test_attention_chain_small():
    from tensor_relational_einsum_gb300.graphs import AttentionChain
    b, h, s, d = 1, 2, 256, 128
    Q, K, V = (synth.make("bf16", (b, h, s, d), "normal", sd, 0, 1) for sd in (21, 22, 23))
    ch = AttentionChain(rel(Q, [1, 2, 1, 1]), rel(K, [1, 2, 4, 1]), rel(V, [1, 2, 4, 1]))
    ch.run()
    want = chains.softmax_attention(Q.to_f64(), K.to_f64(), V.to_f64())
    assert rel_frob(dense64(ch.S), want["S"]) <= 1e-5
    assert rel_frob(dense64(ch.m), want["m"]) <= 1e-6
    assert rel_frob(dense64(ch.l), want["l"]) <= 1e-5
    assert rel_frob(dense64(ch.P), want["P"]) <= BF16_TOL
    assert rel_frob(dense64(ch.O), want["O"]) <= BF16_TOL


def test_attention_chain_causal_small():
    from tensor_relational_einsum_gb300.graphs import AttentionChain
    b, h, s, d = 2, 2, 256, 128
    Q, K, V = (synth.make("bf16", (b, h, s, d), "normal", sd, 0, 1) for sd in (24, 25, 26))
    ch = AttentionChain(rel(Q, [2, 2, 4, 1]), rel(K, [2, 2, 4, 1]), rel(V, [2, 2, 4, 1]), scale=1 / np.sqrt(d),
                        causal=True)
    ch.run()
    want = chains.softmax_attention(Q.to_f64(), K.to_f64(), V.to_f64(), scale=1 / np.sqrt(d), causal=True)
    assert rel_frob(dense64(ch.m), want["m"]) <= 1e-6
    assert rel_frob(dense64(ch.O), want["O"]) <= BF16_TOL


@pytest.mark.parametrize("fused", [True, False])
def test_swiglu_ffn_small(fused):
    from tensor_relational_einsum_gb300.graphs import SwigluFFN
    T, D, F = 256, 512, 768
    x = synth.make("bf16", (T, D), "normal", 31, 0, 1)
    wg, wu = (synth.make("bf16", (D, F), "normal", sd, 0, 0.02) for sd in (32, 33))
    wd = synth.make("bf16", (F, D), "normal", 34, 0, 0.02)
    ffn = SwigluFFN(rel(x, [1, 4]), to_device(wg), to_device(wu), to_device(wd), k_blocks=4, fused=fused)
    ffn.run()
    want = chains.swiglu_ffn(x.to_f64(), wg.to_f64(), wu.to_f64(), wd.to_f64())
    # fused: G and U are never written (SiLU * up runs in the contraction's epilogue)
    for k in (("H", "Y") if fused else ("G", "U", "H", "Y")):
        assert rel_frob(dense64(getattr(ffn, k)), want[k]) <= BF16_TOL, k


def _block_weights(D, F, seed0):
    W = {}
    for i, (k, shp) in enumerate([("wq", (D, D)), ("wk", (D, D)), ("wv", (D, D)), ("wo", (D, D)),
                                  ("w_gate", (D, F)), ("w_up", (D, F)), ("w_down", (F, D))]):
        W[k] = synth.make("bf16", shp, "normal", seed0 + i, 0, 0.02)
    # RMSNorm gains ~ N(1, 0.1): far enough from 1 that a dropped, inverted
    # or misplaced gain (the fused path folds it into the projection
    # weights) breaks the tolerance
    for i, k in enumerate(("g1", "g2")):
        W[k] = synth.make("bf16", (D,), "normal", seed0 + 20 + i, 1.0, 0.1)
    return W


@pytest.mark.parametrize("fused", [True, False])
def test_llama_block_small(fused):
    from tensor_relational_einsum_gb300.graphs import LlamaBlock
    b, s, D, H, F = 2, 256, 256, 2, 512
    W = _block_weights(D, F, 40)
    x = synth.make("bf16", (b * s, D), "normal", 50, 0, 1)
    blk = LlamaBlock(b, s, D, H, F, {k: to_device(v) for k, v in W.items()}, fused_attention=fused,
                     fused_epilogues=fused)
    blk.x.load(to_device(x))
    blk.run()
    Wd = {k: v.to_f64() for k, v in W.items()}
    want = chains.llama_block(x.to_f64().reshape(b, s, D), Wd, n_heads=H, eps=1e-6, theta=10000.0)
    if not fused:  # fused: RMSNorm's apply runs in the projections' epilogues (n1 is never written)
        assert rel_frob(dense64(blk.n1), want["n1"]) <= BF16_TOL
    assert rel_frob(dense64(blk.qr), want["q"]) <= BF16_TOL
    assert rel_frob(dense64(blk.attn.O), want["O"]) <= BF16_TOL
    assert rel_frob(dense64(blk.h), want["h"]) <= BF16_TOL
    assert rel_frob(dense64(blk.y).reshape(b, s, D), want["y"]) <= BF16_TOL


def test_llama_block_cuda_graph_replay_matches_eager():
    """The block captured into one CUDA graph replays the same kernels with
    the same arguments: its output equals the eager run bit for bit."""
    from tensor_relational_einsum_gb300.graphs import LlamaBlock, capture
    b, s, D, H, F = 2, 256, 256, 2, 512
    W = _block_weights(D, F, 60)
    x = synth.make("bf16", (b * s, D), "normal", 61, 0, 1)
    blk = LlamaBlock(b, s, D, H, F, {k: to_device(v) for k, v in W.items()})
    blk.x.load(to_device(x))
    blk.run()
    torch.cuda.synchronize()
    eager = blk.y.arena().clone()
    blk.y.arena().zero_()
    g = capture(blk.run)
    blk.y.arena().zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(blk.y.arena(), eager)
    # a new input loaded into the same relation flows through the replay
    x2 = synth.make("bf16", (b * s, D), "normal", 62, 0, 1)
    blk.x.load(to_device(x2))
    g.replay()
    torch.cuda.synchronize()
    Wd = {k: v.to_f64() for k, v in W.items()}
    want = chains.llama_block(x2.to_f64().reshape(b, s, D), Wd, n_heads=H, eps=1e-6, theta=10000.0)
    assert rel_frob(dense64(blk.y).reshape(b, s, D), want["y"]) <= BF16_TOL
