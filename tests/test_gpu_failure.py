"""Failure detection on the GPU without a fault: a bounded mbarrier wait
that nothing ends gives up after its limit, raises the device error word,
and ea_check reports it; the context stays usable and the word is cleared."""
import time

import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

from gpu_util import dense64, rel  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    from tensor_relational_einsum_gb300.build import build
    build()
    yield


def test_bounded_wait_gives_up_and_reports():
    from tensor_relational_einsum_gb300 import _abi
    from tensor_relational_einsum_gb300.relation import check, joinagg
    L = _abi.lib()
    check()  # a clean word before the test
    t0 = time.time()
    _abi.check_status(L.ea_selftest_wait_timeout(20000, None))  # 20 ms
    rc = L.ea_check(None)
    dt = time.time() - t0
    assert rc == 9, rc  # EA_ERR_DEVICE
    assert b"self-test" in L.ea_last_error()
    assert dt < 10.0
    # the context is still usable and the word was cleared
    A = synth.make("f32", (64, 48), "int", 3, -3, 3)
    B = synth.make("f32", (48, 32), "int", 4, -3, 3)
    C = joinagg("ij,jk->ik", [rel(A, [2, 2]), rel(B, [2, 1])])
    assert L.ea_check(None) == 0
    assert np.array_equal(dense64(C), A.to_f64() @ B.to_f64())
