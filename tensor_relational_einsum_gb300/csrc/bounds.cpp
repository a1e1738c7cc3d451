// bounds.cpp -- the plan check: before a plan is uploaded, every descriptor
// a kernel will follow is checked against the arenas it addresses.
//
// The kernels index memory only through descriptors the host planner
// builds (segment offsets and strides of an exchange, strided views of an
// elementwise join or a row reduction, operand blocks of a contraction,
// output rows of the attention join-agg).  Each descriptor names an
// element range of a block arena; a plan whose ranges all lie inside their
// arenas cannot make a kernel read or write outside them.  A plan that
// fails is rejected with EA_ERR_BOUNDS before anything is launched.  The
// same ranges are re-checked on the device, access by access, in a library
// built with EA_DEBUG_BOUNDS (the kernels then raise the device error word
// and skip the access).
#include <string.h>

#include "host.h"
#include "plan.h"

namespace ea {

namespace {

typedef __int128 i128;

// The element range [lo, hi) of base + sum_i c_i str_i (0 <= c_i < ext_i)
// + c len_str (0 <= c < len); empty (lo == hi) when any extent is 0.
struct Range {
    i128 lo, hi;
};

Range strided(int64_t base, int n, const int64_t *ext, const int64_t *str, int64_t len, int64_t len_str) {
    Range r{base, base};
    if (len <= 0) return r;
    for (int i = 0; i < n; i++)
        if (ext[i] <= 0) return r;
    i128 lo = base, hi = base;
    for (int i = 0; i < n; i++) {
        const i128 span = (i128)(ext[i] - 1) * str[i];
        if (span < 0) lo += span;
        else hi += span;
    }
    const i128 span = (i128)(len - 1) * len_str;
    if (span < 0) lo += span;
    else hi += span;
    r.lo = lo;
    r.hi = hi + 1;
    return r;
}

ea_status in_arena(Range r, int64_t elems, const char *what, size_t index) {
    if (r.lo == r.hi) return EA_OK;
    if (r.lo < 0 || r.hi > elems)
        return set_error(EA_ERR_BOUNDS, "plan check: %s %zu addresses elements [%lld, %lld) of an arena of %lld",
                         what, index, (long long)r.lo, (long long)r.hi, (long long)elems);
    return EA_OK;
}

}  // namespace

ea_status check_exchange_plan(const XSeg *segs, size_t nseg, const XTile *tiles, size_t ntiles, int64_t src_elems,
                              int64_t dst_elems, int64_t copies, int64_t copy_stride) {
    for (size_t i = 0; i < nseg; i++) {
        const XSeg &g = segs[i];
        if (g.nd < 0 || g.nd > 4 || g.inner < 0) return set_error(EA_ERR_BOUNDS, "plan check: exchange segment %zu is malformed", i);
        int64_t rows = 1;
        for (int d = 0; d < g.nd; d++) rows *= g.ext[d];
        if (rows != g.rows) return set_error(EA_ERR_BOUNDS, "plan check: exchange segment %zu has %lld rows, not %lld", i,
                                             (long long)g.rows, (long long)rows);
        Range s = strided(g.src_off, g.nd, g.ext, g.sstr, g.inner, 1);
        if (copies > 1 && s.lo != s.hi) s.hi += (i128)(copies - 1) * copy_stride;
        ea_status st = in_arena(s, src_elems, "exchange segment (source)", i);
        if (st) return st;
        st = in_arena(strided(g.dst_off, g.nd, g.ext, g.dstr, g.inner, 1), dst_elems, "exchange segment (destination)", i);
        if (st) return st;
    }
    for (size_t t = 0; t < ntiles; t++) {
        const XTile &T = tiles[t];
        if (T.seg < 0 || (size_t)T.seg >= nseg)
            return set_error(EA_ERR_BOUNDS, "plan check: exchange tile %zu names segment %d of %zu", t, T.seg, nseg);
        const XSeg &g = segs[T.seg];
        if (T.row0 < 0 || T.nrows < 0 || T.row0 + T.nrows > g.rows || T.col0 < 0 || T.ncols < 0 ||
            T.col0 + T.ncols > g.inner)
            return set_error(EA_ERR_BOUNDS, "plan check: exchange tile %zu (rows %lld+%lld, columns %lld+%lld) leaves "
                                            "its segment (%lld x %lld)",
                             t, (long long)T.row0, (long long)T.nrows, (long long)T.col0, (long long)T.ncols,
                             (long long)g.rows, (long long)g.inner);
    }
    return EA_OK;
}

ea_status check_view_items(const EwItem *items, size_t n, int n_in, const int64_t *in_elems, int64_t out_elems,
                           const char *what) {
    for (size_t i = 0; i < n; i++) {
        const EwItem &it = items[i];
        if (it.nd < 0 || it.nd > kViewDims) return set_error(EA_ERR_BOUNDS, "plan check: %s view %zu is malformed", what, i);
        ea_status st = in_arena(strided(it.out_base, it.nd, it.ext, it.ostr, it.len, it.out_inner), out_elems, what, i);
        if (st) return st;
        for (int k = 0; k < n_in; k++) {
            st = in_arena(strided(it.in_base[k], it.nd, it.ext, it.istr[k], it.len, it.in_inner[k]), in_elems[k], what, i);
            if (st) return st;
        }
    }
    return EA_OK;
}

ea_status check_ew_tiles(const EwTile *tiles, size_t nt, const EwItem *items, size_t n) {
    for (size_t t = 0; t < nt; t++) {
        const EwTile &T = tiles[t];
        if (T.item < 0 || (size_t)T.item >= n) return set_error(EA_ERR_BOUNDS, "plan check: elementwise tile %zu names no view", t);
        const EwItem &it = items[T.item];
        if (T.row0 < 0 || T.nrows < 0 || T.row0 + T.nrows > it.rows || T.col0 < 0 || T.ncols < 0 ||
            T.col0 + T.ncols > it.len)
            return set_error(EA_ERR_BOUNDS, "plan check: elementwise tile %zu leaves its view", t);
    }
    return EA_OK;
}

ea_status check_rr_tiles(const RrTile *tiles, size_t nt, const RrGroup *groups, size_t ng, const EwItem *items,
                         size_t n) {
    for (size_t g = 0; g < ng; g++)
        if (groups[g].i0 < 0 || groups[g].i1 < groups[g].i0 || (size_t)groups[g].i1 > n)
            return set_error(EA_ERR_BOUNDS, "plan check: row-reduction group %zu names views outside the plan", g);
    for (size_t t = 0; t < nt; t++) {
        const RrTile &T = tiles[t];
        if (T.group < 0 || (size_t)T.group >= ng) return set_error(EA_ERR_BOUNDS, "plan check: row-reduction tile %zu names no group", t);
        const RrGroup &G = groups[T.group];
        for (int32_t i = G.i0; i < G.i1; i++)
            if (T.row0 < 0 || T.nrows < 0 || T.row0 + T.nrows > items[i].rows)
                return set_error(EA_ERR_BOUNDS, "plan check: row-reduction tile %zu leaves view %d", t, i);
    }
    return EA_OK;
}

ea_status check_rb_desc(const int64_t *w, size_t ntiles, int64_t in_elems, int64_t out_elems) {
    for (size_t t = 0; t < ntiles; t++, w += kRbWords) {
        const int64_t rows = (int64_t)(uint32_t)(w[11] & 0xFFFFFFFF), nb = w[11] >> 32, len = w[10];
        if (nb < 1 || nb > 4) return set_error(EA_ERR_BOUNDS, "plan check: row-batch tile %zu has %lld blocks", t, (long long)nb);
        const int64_t e1[1] = {rows};
        for (int64_t b = 0; b < nb; b++) {
            const int64_t s1[1] = {w[4 + b]};
            ea_status st = in_arena(strided(w[b], 1, e1, s1, len, 1), in_elems, "row-batch tile (input)", t);
            if (st) return st;
        }
        const int64_t s1[1] = {w[9]};
        ea_status st = in_arena(strided(w[8], 1, e1, s1, 1, 0), out_elems, "row-batch tile (output)", t);
        if (st) return st;
    }
    return EA_OK;
}

ea_status check_simt_plan(const CtGroup *groups, size_t ng, const CtTuple *tuples, size_t nt, int64_t a_elems,
                          int64_t b_elems, int64_t c_elems) {
    for (size_t g = 0; g < ng; g++) {
        const CtGroup &G = groups[g];
        const int64_t ce[3] = {G.M, G.N, G.nb}, cs[3] = {G.c_sm, G.c_sn, G.c_sb};
        ea_status st = in_arena(strided(G.c_base, 3, ce, cs, 1, 0), c_elems, "contraction output block", g);
        if (st) return st;
        if (G.t0 < 0 || G.t1 < G.t0 || (size_t)G.t1 > nt)
            return set_error(EA_ERR_BOUNDS, "plan check: contraction group %zu names tuples outside the plan", g);
        for (int32_t t = G.t0; t < G.t1; t++) {
            const CtTuple &U = tuples[t];
            const int64_t ae[3] = {G.M, U.K, G.nb}, as[3] = {U.a_sm, U.a_sk, U.a_sb};
            const int64_t be[3] = {U.K, G.N, G.nb}, bs[3] = {U.b_sk, U.b_sn, U.b_sb};
            st = in_arena(strided(U.a_base, 3, ae, as, 1, 0), a_elems, "contraction operand A block", (size_t)t);
            if (st) return st;
            st = in_arena(strided(U.b_base, 3, be, bs, 1, 0), b_elems, "contraction operand B block", (size_t)t);
            if (st) return st;
        }
    }
    return EA_OK;
}

ea_status check_block(int64_t base, int n, const int64_t *ext, const int64_t *str, int64_t elems, const char *what,
                      size_t index) {
    return in_arena(strided(base, n, ext, str, 1, 0), elems, what, index);
}

}  // namespace ea

using namespace ea;

extern "C" ea_status ea_plan_check_exchange(const int64_t *seg_words, int64_t nseg, const int64_t *tile_words,
                                            int64_t ntiles, int64_t src_elems, int64_t dst_elems) {
    set_error(EA_OK, "");
    if (nseg < 0 || ntiles < 0 || (nseg > 0 && !seg_words) || (ntiles > 0 && !tile_words) || src_elems < 0 ||
        dst_elems < 0)
        return set_error(EA_ERR_ARG, "ea_plan_check_exchange: bad arguments");
    std::vector<XSeg> segs((size_t)nseg);
    for (int64_t i = 0; i < nseg; i++) {
        const int64_t *w = seg_words + 16 * i;
        XSeg &g = segs[(size_t)i];
        memset(&g, 0, sizeof g);
        g.src_off = w[0];
        g.dst_off = w[1];
        g.inner = w[2];
        g.nd = (int32_t)w[3];
        if (w[3] < 0 || w[3] > 4) return set_error(EA_ERR_BOUNDS, "plan check: exchange segment %lld is malformed", (long long)i);
        g.rows = 1;
        for (int d = 0; d < 4; d++) {
            g.ext[d] = d < g.nd ? w[4 + d] : 1;
            g.sstr[d] = d < g.nd ? w[8 + d] : 0;
            g.dstr[d] = d < g.nd ? w[12 + d] : 0;
            g.rows *= g.ext[d];
        }
    }
    std::vector<XTile> tiles((size_t)ntiles);
    for (int64_t t = 0; t < ntiles; t++) {
        const int64_t *w = tile_words + 5 * t;
        XTile &T = tiles[(size_t)t];
        memset(&T, 0, sizeof T);
        if (w[0] < 0 || w[0] > INT32_MAX) return set_error(EA_ERR_BOUNDS, "plan check: exchange tile %lld names no segment", (long long)t);
        T.seg = (int32_t)w[0];
        T.row0 = w[1];
        T.nrows = w[2];
        T.col0 = w[3];
        T.ncols = w[4];
    }
    return check_exchange_plan(segs.data(), segs.size(), tiles.data(), tiles.size(), src_elems, dst_elems, 1, 0);
}

extern "C" int ea_debug_bounds(void) {
#ifdef EA_DEBUG_BOUNDS
    return 1;
#else
    return 0;
#endif
}
