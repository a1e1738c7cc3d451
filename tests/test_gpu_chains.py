"""GPU parity of the matrix-chain workloads ("Every Kernel Is a Join",
Section 7, chains A-E): every chain in its fixed parenthesization at about
1/128 of the pages' dimensions (the same shapes of plan, every dimension still in
several blocks) against the oracle's chain of contraction join-aggs, and
chain C at full size on sampled rows (a row of the product is the row of M1
carried through the chain, in fp64).

Tolerance: bf16 inputs, fp32 accumulation, every intermediate product
rounded to bf16 (at most 12 roundings of 2^-9): 2e-2 relative Frobenius.
"""
import numpy as np
import pytest

import synth
from oracle import chains

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

from gpu_util import BF16_TOL, dense64, rel_frob, to_device  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    from tensor_relational_einsum_gb300.build import build
    build()
    yield
    from tensor_relational_einsum_gb300.relation import check
    check()


def _mats(dims, seed0, host=True):
    out = []
    for i in range(len(dims) - 1):
        sd = 1.0 if i == 0 else 1.0 / np.sqrt(dims[i])
        out.append(synth.make("bf16", (dims[i], dims[i + 1]), "normal", seed0 + i, 0.0, sd))
    return out


@pytest.mark.parametrize("name", ["A", "B", "C", "D", "E"])
def test_chain_scaled(name):
    from tensor_relational_einsum_gb300.graphs import CHAINS, MatrixChain
    dims, paren = CHAINS[name]
    # 1/128 of each dimension, rounded up to whole 32-wide blocks (64-byte
    # bf16 rows, which the tensor-core kernel's TMA loads need)
    dims = [max(32, -(-(d // 128) // 32) * 32) for d in dims]
    mats = _mats(dims, 200)
    ch = MatrixChain([to_device(m) for m in mats], paren, block=32)
    out = ch.run()
    torch.cuda.synchronize()
    want = chains.matrix_chain([m.to_f64() for m in mats], paren)
    got = dense64(out)
    assert np.isfinite(got).all()
    assert rel_frob(got, want) <= BF16_TOL


def test_chain_c_full_size_sampled_rows():
    from tensor_relational_einsum_gb300.graphs import CHAINS, MatrixChain
    dims, paren = CHAINS["C"]
    mats = [synth.make_torch("bf16", (dims[i], dims[i + 1]), "normal", 300 + i, 0.0,
                             1.0 if i == 0 else 1.0 / np.sqrt(dims[i]), device="cpu") for i in range(3)]
    ch = MatrixChain([m.cuda() for m in mats], paren)
    out = ch.run().to_dense()
    torch.cuda.synchronize()
    for r in synth.subset_rows(77, dims[0], 2):
        v = mats[0][int(r)].double().numpy()
        for m in mats[1:]:
            v = v @ m.double().numpy()
        assert rel_frob(out[int(r)].double().cpu().numpy(), v) <= BF16_TOL
