"""The library's own device memory through torch's caching allocator
(ea_set_allocator): plans and library-created relations are charged to
torch's pool, work as before, and go back to it when freed."""
import ctypes

import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

from gpu_util import arena_bits, dense64, rel  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    from tensor_relational_einsum_gb300.build import build
    build()
    yield
    from tensor_relational_einsum_gb300.relation import check, use_torch_allocator
    use_torch_allocator(False)
    check()


def test_plans_and_library_relations_use_torch_pool():
    from tensor_relational_einsum_gb300 import _abi
    from tensor_relational_einsum_gb300.relation import exchange, joinagg, plan_cache_clear, use_torch_allocator
    L = _abi.lib()
    A = synth.make("f32", (96, 80), "int", 5, -3, 3)
    B = synth.make("f32", (80, 48), "int", 6, -3, 3)
    RA, RB = rel(A, [3, 2]), rel(B, [2, 3])
    torch.cuda.synchronize()
    plan_cache_clear()
    use_torch_allocator(True)
    try:
        before = torch.cuda.memory_allocated()
        C = joinagg("ij,jk->ik", [RA, RB])          # a new plan: its device copy comes from torch's pool
        torch.cuda.synchronize()
        with_plan = torch.cuda.memory_allocated()
        assert with_plan > before + C.storage.numel() * 4
        assert np.array_equal(dense64(C), A.to_f64() @ B.to_f64())
        # a relation the library creates itself (no storage given)
        dims = (96, 48)
        arr, keep, _ = _abi.dim_parts(dims, [[0, 50, 96], 1])
        h = ctypes.c_void_p()
        _abi.check_status(L.ea_relation_create(0, 2, _abi.i64(dims), arr, None, ctypes.byref(h)))
        assert torch.cuda.memory_allocated() >= with_plan + 96 * 48 * 4
        X = exchange(C, [[0, 50, 96], 1])
        out = ctypes.c_void_p(h.value)
        _abi.check_status(L.ea_exchange(C.handle, None, None, ctypes.byref(out)))
        torch.cuda.synchronize()
        ptr, nbytes = ctypes.c_void_p(), ctypes.c_size_t()
        _abi.check_status(L.ea_relation_data(h, ctypes.byref(ptr), ctypes.byref(nbytes)))
        from tensor_relational_einsum_gb300.relation import Relation
        view = Relation("f32", dims, [[0, 50, 96], 1], device="cuda")
        _abi.check_status(L.ea_exchange(h, None, None, ctypes.byref(ctypes.c_void_p(view.handle.value))))
        torch.cuda.synchronize()
        assert nbytes.value == 96 * 48 * 4
        assert np.array_equal(arena_bits(view), arena_bits(X))
        held = torch.cuda.memory_allocated()
        _abi.check_status(L.ea_relation_destroy(h))
        torch.cuda.synchronize()
        assert torch.cuda.memory_allocated() <= held - 96 * 48 * 4   # the arena went back to torch's pool
    finally:
        use_torch_allocator(False)
    # plans taken from torch's pool go back to it, through torch, after the switch
    torch.cuda.synchronize()
    held = torch.cuda.memory_allocated()
    plan_cache_clear()
    assert torch.cuda.memory_allocated() < held
