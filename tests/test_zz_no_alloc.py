"""ea_exchange_noalloc: the exchange for callers that cannot allocate device
memory (a process whose device memory belongs to its own pool, a path that
cannot take cudaMalloc's device-wide synchronisation).  Its plan lives in a
static 1 MiB device array inside libea.so instead of memory from
cudaMalloc.  Checked through the C ABI against ea_exchange, bit for bit,
on two calls in a row (the second call must replace the first call's plan
in the shared array).  Kept in a file that pytest collects last."""
import ctypes

import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def L():
    from tensor_relational_einsum_gb300 import _abi
    from tensor_relational_einsum_gb300.build import build
    build()
    assert torch.cuda.is_available()
    return _abi


def _rel(abi, dtype_code, dims, parts, buf):
    arr, keep, _ = abi.dim_parts(dims, parts)
    h = ctypes.c_void_p()
    abi.check_status(abi.lib().ea_relation_create(dtype_code, len(dims), abi.i64(dims), arr,
                                                  ctypes.c_void_p(buf.data_ptr()), ctypes.byref(h)))
    return h


def _bits(t):
    return t.cpu().view(torch.int16).numpy() if t.dtype == torch.bfloat16 else t.cpu().view(torch.int32).numpy()


CASES = [
    ("bf16", (1024, 768), [8, 1], [4, 2], 41),
    ("f32", (96, 40, 24), [[0, 5, 96], [0, 40], [0, 8, 24]], [[0, 48, 96], [0, 10, 20, 40], [0, 24]], 42),
]


def test_noalloc_exchange_matches_ea_exchange_twice(L):
    lib = L.lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for dtype, dims, src, dst, seed in CASES:
        code = 1 if dtype == "bf16" else 0
        t = synth.make_torch(dtype, dims, "uniform", seed, -1.0, 1.0, device="cuda")
        n = t.numel()
        src_buf = torch.empty(n, dtype=t.dtype, device="cuda")
        whole = _rel(L, code, dims, [1] * len(dims), t.reshape(-1))
        h_src = _rel(L, code, dims, src, src_buf)
        L.check_status(lib.ea_exchange(whole, None, stream, ctypes.byref(h_src)))
        ref_buf = torch.empty(n, dtype=t.dtype, device="cuda")
        out_buf = torch.full((n,), 7.0, dtype=t.dtype, device="cuda")
        h_ref = _rel(L, code, dims, dst, ref_buf)
        h_out = _rel(L, code, dims, dst, out_buf)
        L.check_status(lib.ea_exchange(h_src, None, stream, ctypes.byref(h_ref)))
        L.check_status(lib.ea_exchange_noalloc(h_src, h_out, stream))
        L.check_status(lib.ea_check(stream))
        assert np.array_equal(_bits(out_buf), _bits(ref_buf))
        # and back again through the same static array
        back_buf = torch.empty(n, dtype=t.dtype, device="cuda")
        h_back = _rel(L, code, dims, src, back_buf)
        L.check_status(lib.ea_exchange_noalloc(h_out, h_back, stream))
        L.check_status(lib.ea_check(stream))
        assert np.array_equal(_bits(back_buf), _bits(src_buf))
        for h in (whole, h_src, h_ref, h_out, h_back):
            lib.ea_relation_destroy(h)


def test_noalloc_rejects_plans_beyond_its_scratch(L):
    lib = L.lib()
    dims = (4096, 4096)
    buf_a = torch.empty(dims[0] * dims[1], dtype=torch.bfloat16, device="cuda")
    buf_b = torch.empty_like(buf_a)
    a = _rel(L, 1, dims, [1, 1], buf_a)
    b = _rel(L, 1, dims, [256, 256], buf_b)   # 65536 atoms: far beyond 1 MiB of plan
    rc = lib.ea_exchange_noalloc(a, b, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 8 and b"static scratch" in lib.ea_last_error()
    lib.ea_relation_destroy(a)
    lib.ea_relation_destroy(b)
