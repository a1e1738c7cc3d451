"""ea_exchange_noalloc: the exchange for callers that cannot allocate device
memory (a process whose device memory belongs to its own pool, a path that
cannot take cudaMalloc's device-wide synchronisation).  Its plan lives in a
static 1 MiB device array inside libea.so instead of memory from
cudaMalloc.

Checked through the C ABI against the oracle's re-blocking, bit for bit, on
two calls in a row (the second call must replace the first call's plan in
the shared array), including the planner's long-row and rank > 5 branches;
a counting allocator installed with ea_set_allocator must see no call, and
the device's free memory must not move across the calls.  Kept in a file
that pytest collects last."""
import ctypes

import numpy as np
import pytest

import oracle
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


def _rel(abi, dtype_code, dims, bounds, buf):
    arr, keep, _ = abi.dim_parts(dims, bounds)
    h = ctypes.c_void_p()
    abi.check_status(abi.lib().ea_relation_create(dtype_code, len(dims), abi.i64(dims), arr,
                                                  ctypes.c_void_p(buf.data_ptr()), ctypes.byref(h)))
    return h


def _bounds(dims, parts):
    return [oracle.near_equal_bounds(n, p) if isinstance(p, int) else list(p) for n, p in zip(dims, parts)]


def _raw(t):
    """Element bits of a tensor as an unsigned numpy array."""
    if t.dtype == torch.bfloat16:
        return t.cpu().view(torch.int16).numpy().view(np.uint16)
    return t.cpu().view(torch.int32).numpy().view(np.uint32)


def _upload(bits, dtype):
    t = torch.from_numpy(bits.view(np.int16 if dtype == "bf16" else np.int32).copy()).cuda()
    return t.view(torch.bfloat16 if dtype == "bf16" else torch.float32)


CASES = [
    # bf16 8 row blocks -> 4 x 2 tiles
    ("bf16", (1024, 768), [8, 1], [4, 2], 41),
    # ragged tilings of a rank-3 fp32 tensor
    ("f32", (96, 40, 24), [[0, 5, 96], [0, 40], [0, 8, 24]], [[0, 48, 96], [0, 10, 20, 40], [0, 24]], 42),
    # whole rows of 128 KiB contiguous on both sides: tiles that cut a row into 64 KiB pieces
    ("f32", (64, 32768), [1, 1], [2, 1], 43),
    # rank 6, every outer dimension split at 3 on one side and at 1 on the
    # other: atoms with five outer dimensions that do not merge (the planner
    # peels the outermost)
    ("f32", (4, 4, 4, 4, 4, 8), [[0, 3, 4]] * 5 + [[0, 8]], [[0, 1, 4]] * 5 + [[0, 8]], 44),
]


def test_noalloc_exchange_matches_oracle_twice_without_allocating(L):
    lib = L.lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    # Any allocation the library makes on its own behalf from here on goes
    # through these callbacks (and fails: they return NULL).
    calls = {"alloc": 0, "free": 0}

    def _alloc(nbytes, ctx):
        calls["alloc"] += 1
        return None

    def _free(ptr, ctx):
        calls["free"] += 1

    alloc_cb, free_cb = L.ALLOC_FN(_alloc), L.FREE_FN(_free)
    prepared = []
    for dtype, dims, src, dst, seed in CASES:
        code = 1 if dtype == "bf16" else 0
        t = synth.make_torch(dtype, dims, "uniform", seed, -1.0, 1.0, device="cpu")
        flat = _raw(t.reshape(-1))
        whole = [[0, n] for n in dims]
        sb, db = _bounds(dims, src), _bounds(dims, dst)
        want_src = oracle.exchange(flat, dims, whole, sb)
        want_dst = oracle.exchange(flat, dims, whole, db)
        src_buf = _upload(want_src, dtype)
        out_buf = torch.full_like(src_buf, 7.0)
        back_buf = torch.full_like(src_buf, -3.0)
        hs, ho, hb = (_rel(L, code, dims, b, buf) for b, buf in ((sb, src_buf), (db, out_buf), (sb, back_buf)))
        # the relations borrow these buffers: keep every one alive until the end
        prepared.append((hs, ho, hb, src_buf, out_buf, back_buf, want_src, want_dst))
    torch.cuda.synchronize()
    L.check_status(lib.ea_set_allocator(alloc_cb, free_cb, None))
    try:
        free_before = None
        for i, (hs, ho, hb, _src, out_buf, back_buf, want_src, want_dst) in enumerate(prepared):
            L.check_status(lib.ea_exchange_noalloc(hs, ho, stream))        # first call: src -> dst
            L.check_status(lib.ea_check(stream))
            if free_before is None:
                # the first call may load the kernel's module (lazy loading);
                # from here on the device's free memory must not move
                free_before = torch.cuda.mem_get_info()[0]
            assert np.array_equal(_raw(out_buf), want_dst), CASES[i]
            L.check_status(lib.ea_exchange_noalloc(ho, hb, stream))        # second call: dst -> src
            L.check_status(lib.ea_check(stream))
            assert np.array_equal(_raw(back_buf), want_src), CASES[i]
        torch.cuda.synchronize()
        assert torch.cuda.mem_get_info()[0] == free_before
        assert calls == {"alloc": 0, "free": 0}
    finally:
        L.check_status(lib.ea_set_allocator(L.ALLOC_FN(), L.FREE_FN(), None))
    for hs, ho, hb, *_ in prepared:
        for h in (hs, ho, hb):
            lib.ea_relation_destroy(h)


def test_noalloc_rejects_plans_beyond_its_scratch(L):
    lib = L.lib()
    dims = (4096, 4096)
    buf_a = torch.empty(dims[0] * dims[1], dtype=torch.bfloat16, device="cuda")
    buf_b = torch.empty_like(buf_a)
    a = _rel(L, 1, dims, _bounds(dims, [1, 1]), buf_a)
    b = _rel(L, 1, dims, _bounds(dims, [256, 256]), buf_b)   # 65536 atoms: far beyond 1 MiB of plan
    rc = lib.ea_exchange_noalloc(a, b, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 8 and b"static scratch" in lib.ea_last_error()
    lib.ea_relation_destroy(a)
    lib.ea_relation_destroy(b)


def test_noalloc_refuses_a_capturing_stream(L):
    """A captured plan copy would read the static host buffer at replay
    time, after later calls changed it: the call is refused while its
    stream is being captured, and works again afterwards."""
    lib = L.lib()
    dims = (256, 512)
    t = synth.make_torch("bf16", dims, "uniform", 45, -1.0, 1.0, device="cuda")
    out_buf = torch.empty_like(t.reshape(-1))
    a = _rel(L, 1, dims, _bounds(dims, [1, 1]), t.reshape(-1))
    b = _rel(L, 1, dims, _bounds(dims, [2, 4]), out_buf)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        g.capture_begin()
        rc = lib.ea_exchange_noalloc(a, b, ctypes.c_void_p(side.cuda_stream))
        msg = lib.ea_last_error()
        g.capture_end()
    assert rc == 8 and b"captured" in msg
    L.check_status(lib.ea_exchange_noalloc(a, b, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)))
    L.check_status(lib.ea_check(None))
    flat = _raw(t.reshape(-1).cpu())
    want = oracle.exchange(flat, dims, [[0, 256], [0, 512]], _bounds(dims, [2, 4]))
    assert np.array_equal(_raw(out_buf), want)
    lib.ea_relation_destroy(a)
    lib.ea_relation_destroy(b)
