"""CPU tests of libea.so: it loads and exports every symbol include/ea.h
declares, and its host planner (no GPU involved) matches the oracle's
independent enumerators bit-exactly: work lists, exchange permutations,
overlay atom counts, near-equal tilings, error codes."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
from oracle import worklist as owl
from tensor_relational_einsum_gb300 import _abi
from tensor_relational_einsum_gb300.build import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    build()
    return _abi.lib()


def test_exports_every_declared_symbol(L):
    hdr = open(os.path.join(ROOT, "include", "ea.h")).read()
    names = set(re.findall(r"^(?:ea_status|int|const char \*)\s*(ea_[a-z_]+)\s*\(", hdr, re.M))
    assert {"ea_relation_create", "ea_joinagg_run", "ea_exchange"} <= names
    for n in sorted(names):
        assert hasattr(L, n), n
    assert L.ea_abi_version() == 5


def plan(L, spec, shapes, parts, pred=None):
    ip, n, keep = _abi.index_parts(parts)
    sh = _abi.i64([x for s in shapes for x in s])
    ng, nt, jv, av = (ctypes.c_int64() for _ in range(4))
    pl, ph = (pred[0].encode(), pred[1].encode()) if pred else (b"\0", b"\0")
    _abi.check_status(L.ea_plan_worklist(spec.encode(), sh, ip, n, pl, ph, 0, 0, None, None, None, ctypes.byref(ng),
                                         ctypes.byref(nt), ctypes.byref(jv), ctypes.byref(av)))
    n_in = len(spec.split("->")[0].split(","))
    g = np.zeros(max(1, ng.value), dtype=np.int64)
    gp = np.zeros(ng.value + 1, dtype=np.int64)
    tp = np.zeros(max(1, nt.value * n_in), dtype=np.int64)
    _abi.check_status(L.ea_plan_worklist(spec.encode(), sh, ip, n, pl, ph, ng.value, nt.value,
                                         g.ctypes.data_as(_abi.P64), gp.ctypes.data_as(_abi.P64),
                                         tp.ctypes.data_as(_abi.P64), ctypes.byref(ng), ctypes.byref(nt),
                                         ctypes.byref(jv), ctypes.byref(av)))
    tuples = [tuple(int(x) for x in tp[i * n_in:(i + 1) * n_in]) for i in range(nt.value)]
    return {"groups": [int(x) for x in g[:ng.value]], "grp_ptr": [int(x) for x in gp], "tuples": tuples,
            "join_volume": jv.value, "agg_volume": av.value}


WL_CASES = [
    ("ij,jk->ik", [(256, 512), (512, 256)], {"i": [0, 128, 256], "j": [0, 256, 512]}, None),
    ("ij,jk->ik", [(256, 256), (256, 256)], {"i": 4, "j": 4, "k": 4}, None),
    ("ij,jk->ik", [(10, 9), (9, 8)], {"i": [0, 3, 10], "j": [0, 4, 5, 9], "k": [0, 2, 8]}, None),
    ("bhsd,bhtd->bhst", [(4, 32, 2048, 128), (4, 32, 2048, 128)], {"b": 4, "h": 32, "t": 4}, None),
    ("bhst,bhtd->bhsd", [(4, 32, 2048, 2048), (4, 32, 2048, 128)], {"b": 4, "h": 32, "t": 4}, None),
    ("bshd,bthd->bhst", [(2, 64, 2, 8), (2, 64, 2, 8)], {"b": 2, "h": 2, "s": 4, "t": 4}, "ts"),
    ("bhst,bthd->bshd", [(2, 2, 64, 64), (2, 64, 2, 8)], {"b": 2, "h": 2, "s": 4, "t": 4}, "ts"),
    ("bhst->bhs", [(2, 3, 10, 12)], {"h": [0, 1, 3], "t": [0, 5, 12], "s": [0, 7, 10]}, None),
    ("td,t,d->td", [(12, 8), (12,), (8,)], {"t": 3, "d": 2}, None),
    ("ijk,kl->ijl", [(3, 4, 5), (5, 6)], {"i": 3, "k": [0, 1, 5], "l": 2}, None),
]


@pytest.mark.parametrize("spec,shapes,parts,pred", WL_CASES)
def test_worklist_matches_oracle_enumerator(L, spec, shapes, parts, pred):
    got = plan(L, spec, shapes, parts, pred)
    ext = oracle.letter_extents(spec, shapes)
    bounds = {}
    for l, n in ext.items():
        p = parts.get(l, 1)
        bounds[l] = oracle.near_equal_bounds(n, p) if isinstance(p, int) else list(p)
    want = owl.worklist(spec, bounds, pred)
    assert got["groups"] == want["groups"]
    assert got["grp_ptr"] == want["grp_ptr"]
    assert got["tuples"] == [tuple(t) for t in want["tuples"]]
    assert got["join_volume"] == want["join_volume"]
    assert got["agg_volume"] == want["agg_volume"]


def test_worklist_golden_example_3_8(L):
    import json
    g = json.load(open(os.path.join(ROOT, "tests", "golden", "ex3_8_matmul_worklist.json")))
    got = plan(L, g["spec"], [(256, 512), (512, 256)], g["bounds"])
    assert len(got["tuples"]) == g["n_function_specs"]
    assert got["tuples"] == [((m - 1) * 2 + (n - 1), n - 1) for grp in g["groups_as_mn"] for m, n in grp]


def test_matmul3d_closed_forms_from_planner(L):
    import json
    for c in json.load(open(os.path.join(ROOT, "tests", "golden", "matmul3d_volumes.json")))["cases"]:
        N = c["N"]
        got = plan(L, "ij,jk->ik", [(N, N), (N, N)], {"i": c["a"], "j": c["b"], "k": c["c"]})
        assert len(got["tuples"]) == c["tuples"]
        assert got["join_volume"] == c["join"] and got["agg_volume"] == c["agg"]


def perm(L, dims, src, dst):
    sa, k1, _ = _abi.dim_parts(dims, src)
    da, k2, _ = _abi.dim_parts(dims, dst)
    out = np.empty(int(np.prod(dims)), dtype=np.int64)
    _abi.check_status(L.ea_exchange_permutation(len(dims), _abi.i64(dims), sa, da, out.ctypes.data_as(_abi.P64)))
    return out


X_CASES = [
    ((64, 64), [8, 1], [1, 8]),
    ((64, 64), [8, 1], [4, 2]),
    ((64, 64), [8, 1], [16, 16]),
    ((64, 64), [1, 1], [16, 16]),
    ((12, 10), [[0, 3, 6, 9, 12], [0, 10]], [[0, 4, 8, 12], [0, 2, 7, 10]]),
    ((4, 6, 8), [[0, 2, 4], [0, 6], [0, 8]], [[0, 4], [0, 3, 6], [0, 2, 4, 8]]),
    ((2, 16, 4, 8), [2, 1, 1, 1], [2, 1, 4, 1]),
    ((2, 3, 5, 7, 3), [2, 3, 1, 2, 1], [1, 1, 5, 1, 3]),
    ((8192, 8), [8, 1], [16, 1]),
    ((4, 50000), [2, 1], [1, 1]),                                   # long runs: cut into rows + a tail
    ((3, 40000), [1, [0, 17000, 40000]], [[0, 1, 3], 1]),
]


@pytest.mark.parametrize("dims,src,dst", X_CASES)
def test_exchange_permutation_matches_oracle(L, dims, src, dst):
    got = perm(L, dims, src, dst)
    sb = [oracle.near_equal_bounds(n, p) if isinstance(p, int) else p for n, p in zip(dims, src)]
    db = [oracle.near_equal_bounds(n, p) if isinstance(p, int) else p for n, p in zip(dims, dst)]
    want = oracle.exchange_perm(dims, sb, db)
    assert np.array_equal(got, want)
    n = ctypes.c_int64()
    sa, k1, _ = _abi.dim_parts(dims, sb)
    da, k2, _ = _abi.dim_parts(dims, db)
    _abi.check_status(L.ea_overlay_atoms(len(dims), _abi.i64(dims), sa, da, ctypes.byref(n)))
    assert n.value == len(owl.atoms(sb, db))


def test_exchange_full_config_permutation(L):
    """The 8192 x 8192 re-blockings of the exchange workload, bit-exact."""
    dims = (8192, 8192)
    for dst in ([1, 8], [4, 2], [16, 16]):
        got = perm(L, dims, [8, 1], dst)
        want = oracle.exchange_perm(dims, [oracle.near_equal_bounds(8192, 8), [0, 8192]],
                                    [oracle.near_equal_bounds(8192, dst[0]), oracle.near_equal_bounds(8192, dst[1])])
        assert np.array_equal(got, want)


def test_near_equal_tiling_of_relations(L):
    for n, k in [(10, 3), (7, 7), (8192, 8), (11008, 4), (5, 2)]:
        arr, keep, _ = _abi.dim_parts([n], [k])
        arr[0].bounds = None  # ask the library for its near-equal split
        h = ctypes.c_void_p()
        _abi.check_status(L.ea_relation_create(0, 1, _abi.i64([n]), arr, ctypes.c_void_p(256), ctypes.byref(h)))
        nb = ctypes.c_int32()
        b = (ctypes.c_int64 * (k + 1))()
        _abi.check_status(L.ea_relation_bounds(h, 0, ctypes.byref(nb), b))
        assert list(b) == oracle.near_equal_bounds(n, k)
        L.ea_relation_destroy(h)


def _fake_rel(L, dtype, dims, parts, addr=4096):
    arr, keep, _ = _abi.dim_parts(dims, parts)
    h = ctypes.c_void_p()
    rc = L.ea_relation_create(dtype, len(dims), _abi.i64(dims), arr, ctypes.c_void_p(addr), ctypes.byref(h))
    return rc, h


def test_error_codes_without_gpu(L):
    assert _fake_rel(L, 0, (10,), [[0, 5, 4, 10]])[0] == 3          # bounds not a tiling
    assert _fake_rel(L, 0, (10,), [[0, 5, 11]])[0] == 3             # past the extent
    assert _fake_rel(L, 0, (3,), [5])[0] == 3                        # empty blocks
    assert _fake_rel(L, 7, (3,), [1])[0] == 4                        # dtype
    assert _fake_rel(L, 0, (3,), [1], addr=4097)[0] == 7             # misaligned arena
    rc, a = _fake_rel(L, 0, (8, 6), [2, 1], 4096)
    rc2, b = _fake_rel(L, 0, (6, 4), [3, 1], 1 << 20)                # j tiled 3 ways here, 1 way in a
    rc3, c = _fake_rel(L, 0, (8, 4), [2, 1], 1 << 21)
    assert rc == rc2 == rc3 == 0
    hs = (ctypes.c_void_p * 2)(a.value, b.value)
    out = ctypes.c_void_p(c.value)
    err = L.ea_joinagg_run(b"ij,jk->ik", hs, 2, None, 0, 1, 0, None, None, ctypes.byref(out))
    assert err == 3 and b"re-block" in L.ea_last_error()
    rc5, b1 = _fake_rel(L, 0, (6, 4), [1, 1], 1 << 23)
    hs = (ctypes.c_void_p * 2)(a.value, b1.value)
    assert L.ea_joinagg_run(b"ij,jk->", hs, 2, None, 0, 1, 0, None, None, ctypes.byref(out)) == 8
    assert L.ea_joinagg_run(b"ij,jk-ik", hs, 2, None, 0, 1, 0, None, None, ctypes.byref(out)) == 1
    assert L.ea_joinagg_run(b"ii,jk->ik", hs, 2, None, 0, 1, 0, None, None, ctypes.byref(out)) == 1
    assert L.ea_joinagg_run(b"ij,jk->ik", hs, 1, None, 0, 1, 0, None, None, ctypes.byref(out)) == 7
    assert L.ea_joinagg_run(b"ij,jk->ik", hs, 2, None, 0, 5, 0, None, None, ctypes.byref(out)) == 7
    rc4, d = _fake_rel(L, 0, (7, 4), [1, 1], 1 << 22)
    hs2 = (ctypes.c_void_p * 2)(a.value, d.value)
    assert L.ea_joinagg_run(b"ij,jk->ik", hs2, 2, None, 0, 1, 0, None, None, ctypes.byref(out)) == 2  # j: 6 vs 7
    for h in (a, b, c, d, b1):
        L.ea_relation_destroy(h)


def test_attention_errors_without_gpu(L):
    """ea_attention_run validates roles, extents, tilings and options before
    it touches the GPU."""
    BF, F32 = 1, 0
    _, q = _fake_rel(L, BF, (2, 256, 8, 128), [2, 2, 1, 1], 1 << 24)
    _, k = _fake_rel(L, BF, (2, 256, 2, 128), [2, 4, 1, 1], 1 << 25)
    _, v = _fake_rel(L, BF, (2, 256, 2, 128), [2, 4, 1, 1], 1 << 26)
    out = ctypes.c_void_p()
    o = _abi.AttnOpts()

    def run(spec, a=q, b=k, c=v, opts=o):
        return L.ea_attention_run(spec, a, b, c, ctypes.byref(opts), None, ctypes.byref(out))

    assert run(b"bshd,bthd,bthd") == 1                     # no output term
    assert run(b"bshd,bthd,bthd->bhsd") == 1               # O must have Q's term
    assert run(b"bshd,bthd,btdh->bshd") == 1               # V must have K's term
    assert run(b"bshd,bshd,bshd->bshd") == 1               # no key letter
    assert run(b"bshd,bthd,bthd->bshd", b=q) == 2          # K extents differ from V
    _, k3 = _fake_rel(L, BF, (2, 256, 3, 128), [2, 4, 1, 1], 1 << 27)
    _, v3 = _fake_rel(L, BF, (2, 256, 3, 128), [2, 4, 1, 1], 1 << 28)
    assert run(b"bshd,bthd,bthd->bshd", b=k3, c=v3) == 2   # 8 query heads over 3 kv heads
    _, kf = _fake_rel(L, F32, (2, 256, 2, 128), [2, 4, 1, 1], 1 << 27)
    assert run(b"bshd,bthd,bthd->bshd", b=kf, c=kf) == 4  # K, V not bf16
    _, kb = _fake_rel(L, BF, (2, 256, 2, 128), [1, 4, 1, 1], 1 << 27)
    _, vb = _fake_rel(L, BF, (2, 256, 2, 128), [1, 4, 1, 1], 1 << 28)
    assert run(b"bshd,bthd,bthd->bshd", b=kb, c=vb) == 3   # b tiled differently in Q and K
    _, kh = _fake_rel(L, BF, (2, 256, 2, 128), [2, 4, 2, 1], 1 << 27)
    _, vh = _fake_rel(L, BF, (2, 256, 2, 128), [2, 4, 2, 1], 1 << 28)
    assert run(b"bshd,bthd,bthd->bshd", b=kh, c=vh) == 3   # heads: 2 kv blocks vs 1 query block
    _, q96 = _fake_rel(L, BF, (2, 256, 8, 96), [2, 2, 1, 1], 1 << 29)
    _, k96 = _fake_rel(L, BF, (2, 256, 2, 96), [2, 4, 1, 1], 1 << 30)
    assert run(b"bshd,bthd,bthd->bshd", a=q96, b=k96, c=k96) == 8   # head dim 96
    bad = _abi.AttnOpts()
    ends = _abi.i64([100, 90, 256])
    bad.n_seq_ends, bad.seq_ends = 3, ctypes.cast(ends, ctypes.c_void_p)
    assert run(b"bshd,bthd,bthd->bshd", opts=bad) == 7     # ends not increasing
    ends2 = _abi.i64([100, 200])
    bad.n_seq_ends, bad.seq_ends = 2, ctypes.cast(ends2, ctypes.c_void_p)
    assert run(b"bshd,bthd,bthd->bshd", opts=bad) == 7     # last end != extent
    neg = _abi.AttnOpts()
    neg.scale = -1.0
    assert run(b"bshd,bthd,bthd->bshd", opts=neg) == 7
    _, m = _fake_rel(L, F32, (2, 256, 8), [2, 2, 1], 1 << 31)
    one = _abi.AttnOpts()
    one.m_out = m.value
    assert run(b"bshd,bthd,bthd->bshd", opts=one) == 7     # m_out without l_out
    _, mb = _fake_rel(L, BF, (2, 256, 8), [2, 2, 1], 1 << 32)
    both = _abi.AttnOpts()
    both.m_out, both.l_out = mb.value, mb.value
    assert run(b"bshd,bthd,bthd->bshd", opts=both) == 4    # stats must be f32
    for h in (q, k, v, k3, v3, kf, kb, vb, kh, vh, q96, k96, m, mb):
        L.ea_relation_destroy(h)


def test_epilogue_join_errors_without_gpu(L):
    """The epilogue options of a contraction are validated before any GPU
    work: ADD needs epi_in of the output's shape and tiling; SILU_MUL needs
    a pair letter of the second input only, extent 2, one block."""
    BF = 1
    _, x = _fake_rel(L, BF, (256, 128), [2, 1], 1 << 24)
    _, w = _fake_rel(L, BF, (128, 64, 2), [1, 1, 1], 1 << 25)
    _, h = _fake_rel(L, BF, (256, 64), [2, 1], 1 << 26)
    _, wrong = _fake_rel(L, BF, (256, 64), [4, 1], 1 << 27)
    hs = (ctypes.c_void_p * 2)(x.value, w.value)
    out = ctypes.c_void_p(h.value)
    o = _abi.Opts()
    o.epi_map = _abi.MAPS["silu_mul"]
    o.epi_pair = b"z"  # not a letter of the spec
    assert L.ea_joinagg_run(b"td,dfc->tf", hs, 2, None, 0, 1, 0, ctypes.byref(o), None, ctypes.byref(out)) == 1
    o.epi_pair = b"d"  # the contracted letter: in both inputs
    assert L.ea_joinagg_run(b"td,dfc->tf", hs, 2, None, 0, 1, 0, ctypes.byref(o), None, ctypes.byref(out)) == 1
    o2 = _abi.Opts()
    o2.epi_map = _abi.MAPS["add"]
    assert L.ea_joinagg_run(b"td,dfc->tfc", hs, 2, None, 0, 1, 0, ctypes.byref(o2), None,
                            ctypes.byref(ctypes.c_void_p())) == 7  # ADD without epi_in
    _, h3 = _fake_rel(L, BF, (256, 64, 2), [2, 1, 1], 1 << 28)
    _, r3 = _fake_rel(L, BF, (256, 64, 2), [4, 1, 1], 1 << 29)
    o2.epi_in = r3.value
    out3 = ctypes.c_void_p(h3.value)
    assert L.ea_joinagg_run(b"td,dfc->tfc", hs, 2, None, 0, 1, 0, ctypes.byref(o2), None, ctypes.byref(out3)) == 3
    o3 = _abi.Opts()
    o3.epi_map = _abi.MAPS["exp_sub"]
    assert L.ea_joinagg_run(b"td,dfc->tfc", hs, 2, None, 0, 1, 0, ctypes.byref(o3), None, ctypes.byref(out3)) == 8
    for r in (x, w, h, wrong, h3, r3):
        L.ea_relation_destroy(r)


def test_exchange_agg_and_partials_errors_without_gpu(L):
    """ea_exchange_agg checks the copy dimension, the aggregation and the
    output before any GPU work; a contraction's partials option checks its
    output's leading copy dimension and refuses epilogues."""
    F32 = 0
    _, p = _fake_rel(L, F32, (2, 256, 64), [2, 2, 1], 1 << 24)
    _, o = _fake_rel(L, F32, (256, 64), [4, 1], 1 << 26)
    out = ctypes.c_void_p(o.value)
    assert L.ea_exchange_agg(None, 1, None, None, ctypes.byref(out)) == 7
    assert L.ea_exchange_agg(p, 0, None, None, ctypes.byref(out)) == 7           # NONE is no aggregation
    assert L.ea_exchange_agg(p, 3, None, None, ctypes.byref(out)) == 7           # MAX_SUMEXP neither
    _, blocked = _fake_rel(L, F32, (2, 256, 64), [1, 2, 1], 1 << 27)
    assert L.ea_exchange_agg(blocked, 1, None, None, ctypes.byref(out)) == 3     # copies not in unit blocks
    _, flat = _fake_rel(L, F32, (256,), [2], 1 << 28)
    assert L.ea_exchange_agg(flat, 1, None, None, ctypes.byref(out)) == 2        # no dimension besides the copies
    _, wide = _fake_rel(L, F32, (256, 65), [4, 1], 1 << 29)
    w = ctypes.c_void_p(wide.value)
    assert L.ea_exchange_agg(p, 1, None, None, ctypes.byref(w)) == 2             # extents differ
    _, bf = _fake_rel(L, 1, (256, 64), [4, 1], 1 << 30)
    b = ctypes.c_void_p(bf.value)
    assert L.ea_exchange_agg(p, 1, None, None, ctypes.byref(b)) == 2             # dtype differs
    _, ov = _fake_rel(L, F32, (256, 64), [4, 1], (1 << 24) + 4096)
    v = ctypes.c_void_p(ov.value)
    assert L.ea_exchange_agg(p, 1, None, None, ctypes.byref(v)) == 7             # arenas overlap
    # partials of "ij,jk->ik" with j in 2 blocks: output [2, i, k], copies in unit blocks
    _, a = _fake_rel(L, 1, (256, 128), [2, 2], 1 << 31)
    _, bb = _fake_rel(L, 1, (128, 64), [2, 1], 1 << 32)
    hs = (ctypes.c_void_p * 2)(a.value, bb.value)
    po = _abi.Opts()
    po.partials = 1
    none = ctypes.c_void_p()
    assert L.ea_joinagg_run(b"ij,jk->ik", hs, 2, None, 0, 1, 0, ctypes.byref(po), None, ctypes.byref(none)) == 7
    _, o2 = _fake_rel(L, F32, (256, 64), [2, 1], 1 << 33)
    x = ctypes.c_void_p(o2.value)
    assert L.ea_joinagg_run(b"ij,jk->ik", hs, 2, None, 0, 1, 0, ctypes.byref(po), None, ctypes.byref(x)) == 2
    _, o3 = _fake_rel(L, F32, (2, 256, 64), [1, 2, 1], 1 << 34)
    x = ctypes.c_void_p(o3.value)
    assert L.ea_joinagg_run(b"ij,jk->ik", hs, 2, None, 0, 1, 0, ctypes.byref(po), None, ctypes.byref(x)) == 3
    _, o4 = _fake_rel(L, F32, (2, 256, 64), [2, 2, 1], 1 << 35)
    x = ctypes.c_void_p(o4.value)
    assert L.ea_joinagg_run(b"ij,jk->ik", hs, 2, None, 0, 2, 0, ctypes.byref(po), None, ctypes.byref(x)) == 8  # MAX
    po.epi_map = 3  # an epilogue join (ADD)
    assert L.ea_joinagg_run(b"ij,jk->ik", hs, 2, None, 0, 1, 0, ctypes.byref(po), None, ctypes.byref(x)) == 8
    for h in (p, o, blocked, flat, wide, bf, ov, a, bb, o2, o3, o4):
        L.ea_relation_destroy(h)


def test_set_allocator_routes_library_arenas_without_gpu(L):
    """ea_set_allocator: relations the library creates take their arena from
    the given allocator and give it back through the matching free, even
    after the allocator has been switched back; a NULL or misaligned block
    is EA_ERR_ALLOC.  ea_relation_create touches no memory, so fake device
    addresses serve here."""
    calls = []

    def fake_alloc(n, ctx):
        calls.append(("alloc", n))
        return 1 << 40

    def fake_free(p, ctx):
        calls.append(("free", p))

    a, f = _abi.ALLOC_FN(fake_alloc), _abi.FREE_FN(fake_free)
    assert L.ea_set_allocator(a, _abi.FREE_FN(), None) == 7          # one of the two missing
    assert L.ea_set_allocator(a, f, None) == 0
    dims = (64, 32)
    arr, keep, _ = _abi.dim_parts(dims, [2, 1])
    h = ctypes.c_void_p()
    assert L.ea_relation_create(0, 2, _abi.i64(dims), arr, None, ctypes.byref(h)) == 0
    ptr, nbytes = ctypes.c_void_p(), ctypes.c_size_t()
    assert L.ea_relation_data(h, ctypes.byref(ptr), ctypes.byref(nbytes)) == 0
    assert ptr.value == 1 << 40 and nbytes.value == 64 * 32 * 4
    assert calls == [("alloc", 64 * 32 * 4)]
    assert L.ea_set_allocator(_abi.ALLOC_FN(), _abi.FREE_FN(), None) == 0   # back to cudaMalloc
    assert L.ea_relation_destroy(h) == 0
    assert calls[-1] == ("free", 1 << 40)                              # released by the pair that took it

    def bad_alloc(n, ctx):
        calls.append(("bad", n))
        return (1 << 40) + 8

    def null_alloc(n, ctx):
        return None

    b = _abi.ALLOC_FN(bad_alloc)
    assert L.ea_set_allocator(b, f, None) == 0
    h2 = ctypes.c_void_p()
    assert L.ea_relation_create(0, 2, _abi.i64(dims), arr, None, ctypes.byref(h2)) == 5
    assert b"aligned" in L.ea_last_error() and calls[-1] == ("free", (1 << 40) + 8)
    n = _abi.ALLOC_FN(null_alloc)
    assert L.ea_set_allocator(n, f, None) == 0
    assert L.ea_relation_create(0, 2, _abi.i64(dims), arr, None, ctypes.byref(h2)) == 5
    assert L.ea_set_allocator(_abi.ALLOC_FN(), _abi.FREE_FN(), None) == 0


def test_rope_layout_errors_without_gpu(L):
    """rope_layout: 0 or 1 (else EA_ERR_ARG); the elementwise ROPE join
    reads only the position-major table (EA_ERR_UNSUPPORTED for 1)."""
    BF = 1
    _, x = _fake_rel(L, BF, (4, 64, 2, 128), [1, 1, 1, 1], 1 << 24)
    _, y = _fake_rel(L, BF, (4, 64, 2, 128), [1, 1, 1, 1], 1 << 26)
    hs = (ctypes.c_void_p * 1)(x.value)
    out = ctypes.c_void_p(y.value)
    o = _abi.Opts()
    o.rope_table = 1 << 28
    o.rope_npos = 64
    o.rope_pos = b"s"
    o.rope_layout = 2
    assert L.ea_joinagg_run(b"bshd->bshd", hs, 1, None, 0, 0, 9, ctypes.byref(o), None, ctypes.byref(out)) == 7
    o.rope_layout = 1
    assert L.ea_joinagg_run(b"bshd->bshd", hs, 1, None, 0, 0, 9, ctypes.byref(o), None, ctypes.byref(out)) == 8
    for h in (x, y):
        L.ea_relation_destroy(h)


def test_copy_host_errors_without_gpu(L):
    """ea_relation_copy_host checks its arguments before any copy."""
    _, r = _fake_rel(L, 0, (8, 6), [2, 2], 1 << 24)
    host = ctypes.create_string_buffer(8 * 6 * 4)
    assert L.ea_relation_copy_host(None, host, 1, None) == 7
    assert L.ea_relation_copy_host(r, None, 1, None) == 7
    assert L.ea_relation_copy_host(r, host, 2, None) == 7
    assert L.ea_relation_copy_host(r, host, -1, None) == 7
    L.ea_relation_destroy(r)


def test_selftest_wait_timeout_argument_check_without_gpu(L):
    assert L.ea_selftest_wait_timeout(0, None) == 7
    assert L.ea_selftest_wait_timeout(2000000, None) == 7


# ---------------------------------------------------------- the plan check

def _check_exchange(L, segs, tiles, src_elems, dst_elems):
    import numpy as np
    from tensor_relational_einsum_gb300 import _abi
    sw = np.array([w for s in segs for w in s], dtype=np.int64) if segs else np.zeros(1, np.int64)
    tw = np.array([w for t in tiles for w in t], dtype=np.int64) if tiles else np.zeros(1, np.int64)
    P = ctypes.POINTER(ctypes.c_int64)
    return L.ea_plan_check_exchange(sw.ctypes.data_as(P), len(segs), tw.ctypes.data_as(P), len(tiles),
                                    src_elems, dst_elems)


def _seg(src, dst, inner, ext=(), sstr=(), dstr=()):
    nd = len(ext)
    pad = lambda v, fill: list(v) + [fill] * (4 - nd)  # noqa: E731
    return [src, dst, inner, nd] + pad(ext, 1) + pad(sstr, 0) + pad(dstr, 0)


def test_plan_check_accepts_a_valid_exchange_plan(L):
    # the re-blocking of a [4, 6] tensor from 2 row blocks to 2 column blocks:
    # each atom is [2, 3], rows of 3 elements; arenas of 24 elements
    segs = [_seg(0, 0, 3, (2,), (6,), (3,)), _seg(3, 12, 3, (2,), (6,), (3,)),
            _seg(12, 6, 3, (2,), (6,), (3,)), _seg(15, 18, 3, (2,), (6,), (3,))]
    tiles = [[i, 0, 2, 0, 3] for i in range(4)]
    assert _check_exchange(L, segs, tiles, 24, 24) == 0
    # the same plan with one element too few in either arena
    assert _check_exchange(L, segs, tiles, 23, 24) == 10
    assert _check_exchange(L, segs, tiles, 24, 23) == 10


@pytest.mark.parametrize("bad,what", [
    (lambda s, t: (s[:1] + [_seg(22, 0, 3, (2,), (6,), (3,))] + s[2:], t), "source offset past the end"),
    (lambda s, t: ([_seg(0, 0, 3, (2,), (22,), (3,))] + s[1:], t), "a source stride that walks off the arena"),
    (lambda s, t: (s[:3] + [_seg(15, -1, 3, (2,), (6,), (3,))], t), "a negative destination offset"),
    (lambda s, t: (s, t[:1] + [[1, 1, 2, 0, 3]] + t[2:]), "a tile past its segment's rows"),
    (lambda s, t: (s, t[:1] + [[1, 0, 2, 1, 3]] + t[2:]), "a tile past its segment's run"),
    (lambda s, t: (s, t + [[4, 0, 1, 0, 1]]), "a tile naming no segment"),
    (lambda s, t: ([[0, 0, 3, 5, 2, 1, 1, 1, 6, 0, 0, 0, 3, 0, 0, 0]] + s[1:], t),
     "a segment with more than four outer dimensions"),
])
def test_plan_check_rejects_hand_made_bad_descriptors(L, bad, what):
    segs = [_seg(0, 0, 3, (2,), (6,), (3,)), _seg(3, 12, 3, (2,), (6,), (3,)),
            _seg(12, 6, 3, (2,), (6,), (3,)), _seg(15, 18, 3, (2,), (6,), (3,))]
    tiles = [[i, 0, 2, 0, 3] for i in range(4)]
    s2, t2 = bad(segs, tiles)
    assert _check_exchange(L, s2, t2, 24, 24) == 10, what
    assert b"plan check" in L.ea_last_error()


def test_plan_check_argument_errors(L):
    assert _check_exchange(L, [], [], -1, 0) == 7
    assert _check_exchange(L, [], [], 0, 0) == 0


def test_bounds_checking_build_exports_the_abi():
    """The EA_DEBUG_BOUNDS build (every kernel checks each tile against its
    arena) compiles, loads, exports every symbol the header declares, and
    says which build it is; the default build says it is not."""
    from tensor_relational_einsum_gb300.build import LIB
    path = build(bounds=True)
    assert path.endswith("libea_bounds.so")
    B = ctypes.CDLL(path)
    hdr = open(os.path.join(ROOT, "include", "ea.h")).read()
    names = set(re.findall(r"^(?:ea_status|int|const char \*)\s*(ea_[a-z_]+)\s*\(", hdr, re.M))
    assert "ea_debug_bounds" in names
    for n in sorted(names):
        assert hasattr(B, n), n
    B.ea_abi_version.restype = ctypes.c_int
    assert B.ea_abi_version() == 5
    assert B.ea_debug_bounds() == 1
    build(bounds=False)
    assert ctypes.CDLL(LIB).ea_debug_bounds() == 0
