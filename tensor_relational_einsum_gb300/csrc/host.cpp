// host.cpp -- relations, spec parsing, letter tilings, the canonical join
// work list and the exchange overlay of libea.so (host code, no kernels).
//
// Semantics follow "Every Kernel Is a Join" (Einsummable):
//   tensor types and tilings        Definitions 3.1, 3.2
//   function specs / join-agg spec  Definitions 3.5, 3.6; Section 3.3
//   join -> aggregate -> recompose  Definition 3.7
//   overlay atoms of an exchange    Section 5.3
#include "host.h"

#include <stdio.h>
#include <string.h>

#include <algorithm>

namespace ea {

std::mutex g_mu;

// ------------------------------------------------------------- allocator

namespace {
std::mutex g_alloc_mu;
ea_alloc_fn g_alloc_fn = nullptr;
ea_free_fn g_free_fn = nullptr;
void *g_alloc_ctx = nullptr;
}  // namespace

ea_status dev_alloc(size_t bytes, void **ptr, DevFree *rel, const char *what) {
    ea_alloc_fn fa;
    DevFree r;
    {
        std::lock_guard<std::mutex> lk(g_alloc_mu);
        fa = g_alloc_fn;
        r.fn = g_free_fn;
        r.ctx = g_alloc_ctx;
    }
    *ptr = nullptr;
    if (!fa) {
        r = DevFree{};
        cudaError_t e = cudaMalloc(ptr, bytes);
        if (e != cudaSuccess) {
            cudaGetLastError();
            *ptr = nullptr;
            return set_error(EA_ERR_ALLOC, "%s: cudaMalloc(%zu) failed: %s", what, bytes, cudaGetErrorString(e));
        }
    } else {
        *ptr = fa(bytes, r.ctx);
        if (!*ptr) return set_error(EA_ERR_ALLOC, "%s: the allocator returned NULL for %zu bytes", what, bytes);
        if ((uintptr_t)*ptr % 16) {
            r.fn(*ptr, r.ctx);
            *ptr = nullptr;
            return set_error(EA_ERR_ALLOC, "%s: the allocator returned memory not 16-byte aligned", what);
        }
    }
    *rel = r;
    return EA_OK;
}

void dev_free(void *ptr, const DevFree &rel) {
    if (!ptr) return;
    if (rel.fn) rel.fn(ptr, rel.ctx);
    else cudaFree(ptr);
}
static thread_local char t_err[1024];

ea_status set_error(ea_status code, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(t_err, sizeof t_err, fmt, ap);
    va_end(ap);
    return code;
}

ea_status cuda_error(cudaError_t e, const char *what) {
    return set_error(EA_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorString(e), cudaGetErrorName(e));
}

size_t elem_size(int dtype) { return dtype == EA_F32 ? 4 : 2; }

ea_status make_tiling(int64_t extent, int32_t nblocks, const int64_t *bounds, Tiling *t) {
    if (extent < 0) return set_error(EA_ERR_SHAPE, "negative extent %lld", (long long)extent);
    if (nblocks < 1) return set_error(EA_ERR_PARTITION, "nblocks must be >= 1 (got %d)", nblocks);
    if (extent == 0 && nblocks != 1)
        return set_error(EA_ERR_PARTITION, "an empty dimension takes exactly one (empty) block");
    if (extent > 0 && nblocks > extent)
        return set_error(EA_ERR_PARTITION, "%d blocks over an extent of %lld leave empty blocks", nblocks,
                         (long long)extent);
    t->extent = extent;
    t->b.resize(nblocks + 1);
    for (int i = 0; i <= nblocks; i++) t->b[i] = bounds ? bounds[i] : (int64_t)((i * (__int128)extent) / nblocks);
    if (t->b[0] != 0 || t->b[nblocks] != extent)
        return set_error(EA_ERR_PARTITION, "bounds must run from 0 to the extent %lld", (long long)extent);
    for (int i = 0; i < nblocks; i++)
        if (t->b[i + 1] <= t->b[i] && extent > 0)
            return set_error(EA_ERR_PARTITION, "bounds must increase strictly (block %d is empty)", i);
    return EA_OK;
}

void row_major_strides(int rank, const int64_t *ext, int64_t *str) {
    int64_t s = 1;
    for (int d = rank - 1; d >= 0; d--) {
        str[d] = s;
        s *= ext[d];
    }
}

void tiling_offsets(int rank, const Tiling *t, std::vector<int64_t> *off) {
    int64_t nb = 1;
    for (int d = 0; d < rank; d++) nb *= t[d].nblocks();
    off->assign(nb + 1, 0);
    int64_t iv[kMaxRank] = {0};
    int64_t acc = 0;
    for (int64_t id = 0; id < nb; id++) {
        (*off)[id] = acc;
        int64_t sz = 1;
        for (int d = 0; d < rank; d++) sz *= t[d].b[iv[d] + 1] - t[d].b[iv[d]];
        acc += sz;
        for (int d = rank - 1; d >= 0; d--) {
            if (++iv[d] < t[d].nblocks()) break;
            iv[d] = 0;
        }
    }
    (*off)[nb] = acc;
}

void block_coords(const ea_relation_s *r, int64_t bid, int64_t *iv) {
    for (int d = r->rank - 1; d >= 0; d--) {
        int64_t n = (int64_t)r->bounds[d].size() - 1;
        iv[d] = bid % n;
        bid /= n;
    }
}

void block_box(const ea_relation_s *r, const int64_t *iv, int64_t *lo, int64_t *ext) {
    for (int d = 0; d < r->rank; d++) {
        lo[d] = r->bounds[d][iv[d]];
        ext[d] = r->bounds[d][iv[d] + 1] - lo[d];
    }
}

// ------------------------------------------------------------------ spec

ea_status parse_spec(const char *s, Spec *sp) {
    if (!s) return set_error(EA_ERR_ARG, "spec is NULL");
    const char *arrow = strstr(s, "->");
    if (!arrow) return set_error(EA_ERR_SPEC, "spec \"%s\": missing '->'", s);
    std::string lhs(s, arrow - s), out(arrow + 2);
    sp->n_in = 0;
    size_t pos = 0;
    for (;;) {
        size_t comma = lhs.find(',', pos);
        std::string term = lhs.substr(pos, comma == std::string::npos ? std::string::npos : comma - pos);
        if (sp->n_in == kMaxIn) return set_error(EA_ERR_SPEC, "spec \"%s\": more than %d inputs", s, kMaxIn);
        sp->term[sp->n_in++] = term;
        if (comma == std::string::npos) break;
        pos = comma + 1;
    }
    sp->out = out;
    auto check_term = [&](const std::string &t) -> ea_status {
        if ((int)t.size() > kMaxRank) return set_error(EA_ERR_SPEC, "spec \"%s\": a term has more than 8 letters", s);
        for (size_t i = 0; i < t.size(); i++) {
            if (t[i] < 'a' || t[i] > 'z') return set_error(EA_ERR_SPEC, "spec \"%s\": letters must be a-z", s);
            if (t.find(t[i]) != i) return set_error(EA_ERR_SPEC, "spec \"%s\": letter '%c' repeated in a term", s, t[i]);
        }
        return EA_OK;
    };
    for (int k = 0; k < sp->n_in; k++) {
        ea_status st = check_term(sp->term[k]);
        if (st) return st;
    }
    ea_status st = check_term(sp->out);
    if (st) return st;
    sp->order.clear();
    sp->contracted.clear();
    for (const char *p = s; *p; p++)
        if (*p >= 'a' && *p <= 'z' && sp->order.find(*p) == std::string::npos) sp->order.push_back(*p);
    for (char c : sp->out) {
        bool found = false;
        for (int k = 0; k < sp->n_in; k++) found |= sp->term[k].find(c) != std::string::npos;
        if (!found) return set_error(EA_ERR_SPEC, "spec \"%s\": output letter '%c' is in no input", s, c);
    }
    for (char c : sp->order)
        if (sp->out.find(c) == std::string::npos) sp->contracted.push_back(c);
    return EA_OK;
}

// ------------------------------------------------------------- work list

// Tuples are enumerated directly in canonical order: output blocks in
// row-major id order; for each, the contracted letters' intervals in
// row-major order over the contracted letters (first-appearance order).
ea_status plan_worklist(const Spec &sp, const LetterTilings &lt, char pred_lo, char pred_hi, WorkList *wl) {
    wl->groups.clear();
    wl->grp_ptr.assign(1, 0);
    wl->tuples.clear();
    wl->tuple_iv.clear();
    wl->join_volume = 0;
    wl->agg_volume = 0;
    for (char c : sp.order)
        if (lt.t[c - 'a'].extent < 0) return set_error(EA_ERR_SHAPE, "letter '%c' has no extent", c);
    auto nb = [&](char c) { return (int64_t)lt.t[c - 'a'].nblocks(); };
    auto sz = [&](char c, int64_t i) { return lt.t[c - 'a'].b[i + 1] - lt.t[c - 'a'].b[i]; };
    int64_t n_out = 1, n_con = 1;
    for (char c : sp.out) n_out *= nb(c);
    for (char c : sp.contracted) n_con *= nb(c);
    int64_t iv[26] = {0};
    for (int64_t ob = 0; ob < n_out; ob++) {
        int64_t r = ob;
        for (int d = (int)sp.out.size() - 1; d >= 0; d--) {
            iv[sp.out[d] - 'a'] = r % nb(sp.out[d]);
            r /= nb(sp.out[d]);
        }
        int64_t members = 0;
        for (int64_t cb = 0; cb < n_con; cb++) {
            int64_t q = cb;
            for (int d = (int)sp.contracted.size() - 1; d >= 0; d--) {
                iv[sp.contracted[d] - 'a'] = q % nb(sp.contracted[d]);
                q /= nb(sp.contracted[d]);
            }
            if (pred_lo) {
                const Tiling &A = lt.t[pred_lo - 'a'], &B = lt.t[pred_hi - 'a'];
                // keep iff some cell of the two intervals has value(lo) <= value(hi)
                if (!(A.b[iv[pred_lo - 'a']] <= B.b[iv[pred_hi - 'a'] + 1] - 1)) continue;
            }
            for (int k = 0; k < sp.n_in; k++) {
                int64_t bid = 0, cells = 1;
                for (char c : sp.term[k]) {
                    bid = bid * nb(c) + iv[c - 'a'];
                    cells *= sz(c, iv[c - 'a']);
                }
                wl->tuples.push_back(bid);
                wl->join_volume += cells;
            }
            wl->tuple_iv.insert(wl->tuple_iv.end(), iv, iv + 26);
            members++;
        }
        if (members == 0) continue;
        int64_t ocells = 1;
        for (char c : sp.out) ocells *= sz(c, iv[c - 'a']);
        wl->agg_volume += (members - 1) * ocells;
        wl->groups.push_back(ob);
        wl->grp_ptr.push_back((int64_t)wl->tuples.size() / sp.n_in);
    }
    return EA_OK;
}

// -------------------------------------------------------------- exchange

static int interval_of(const Tiling &t, int64_t x) {
    // the block [b_i, b_i+1) holding x (x < extent)
    int lo = 0, hi = t.nblocks() - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) / 2;
        if (t.b[mid] <= x) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

static void emit_segment(XSeg seg, int nd, const int64_t *ext, const int64_t *ss, const int64_t *ds, int esize,
                         ExchangePlan *xp) {
    // A run of 16 KiB or more, contiguous on both sides, is cut into rows of
    // 8 KiB (plus its tail), so that its tiles hold many rows and every warp
    // of a CTA takes part in copying it.
    const int64_t w = 8192 / esize;
    if (seg.inner >= 2 * w && nd < kMaxRank) {
        const int64_t q = seg.inner / w, rem = seg.inner - q * w;
        int64_t e2[kMaxRank + 1], s2[kMaxRank + 1], d2[kMaxRank + 1];
        for (int i = 0; i < nd; i++) {
            e2[i] = ext[i];
            s2[i] = ss[i];
            d2[i] = ds[i];
        }
        e2[nd] = q;
        s2[nd] = w;
        d2[nd] = w;
        XSeg body = seg;
        body.inner = w;
        emit_segment(body, nd + 1, e2, s2, d2, esize, xp);
        if (rem > 0) {
            XSeg tail = seg;
            tail.inner = rem;
            tail.src_off += q * w;
            tail.dst_off += q * w;
            emit_segment(tail, nd, ext, ss, ds, esize, xp);
        }
        return;
    }
    // Up to 4 outer dims fit one segment; peel the outermost otherwise.
    if (nd > 4) {
        for (int64_t i = 0; i < ext[0]; i++) {
            XSeg s2 = seg;
            s2.src_off += i * ss[0];
            s2.dst_off += i * ds[0];
            emit_segment(s2, nd - 1, ext + 1, ss + 1, ds + 1, esize, xp);
        }
        return;
    }
    seg.nd = nd;
    seg.rows = 1;
    for (int i = 0; i < 4; i++) {
        seg.ext[i] = i < nd ? ext[i] : 1;
        seg.sstr[i] = i < nd ? ss[i] : 0;
        seg.dstr[i] = i < nd ? ds[i] : 0;
        seg.rows *= seg.ext[i];
    }
    bool vec = (seg.src_off * esize) % 16 == 0 && (seg.dst_off * esize) % 16 == 0 && (seg.inner * esize) % 16 == 0;
    for (int i = 0; i < nd; i++) vec = vec && (ss[i] * esize) % 16 == 0 && (ds[i] * esize) % 16 == 0;
    seg.vec = vec ? 1 : 0;
    if (seg.rows == 0 || seg.inner == 0) return;
    int32_t sid = (int32_t)xp->segs.size();
    xp->segs.push_back(seg);
    // Tiles of about 64 KiB.
    const int64_t target = 64 * 1024;
    int64_t row_bytes = seg.inner * esize;
    if (row_bytes >= target) {
        int64_t cols = std::max<int64_t>(16 / esize, (target / esize) / (16 / esize) * (16 / esize));
        for (int64_t r = 0; r < seg.rows; r++)
            for (int64_t c = 0; c < seg.inner; c += cols)
                xp->tiles.push_back(XTile{sid, 0, r, 1, c, std::min(cols, seg.inner - c)});
    } else {
        int64_t per = std::max<int64_t>(1, target / row_bytes);
        for (int64_t r = 0; r < seg.rows; r += per)
            xp->tiles.push_back(XTile{sid, 0, r, std::min(per, seg.rows - r), 0, seg.inner});
    }
}

ea_status plan_exchange(int rank, const int64_t *dims, const Tiling *src, const Tiling *dst, int esize,
                        ExchangePlan *xp) {
    xp->segs.clear();
    xp->tiles.clear();
    xp->n_atoms = 0;
    std::vector<int64_t> soff, doff;
    tiling_offsets(rank, src, &soff);
    tiling_offsets(rank, dst, &doff);
    // Overlay: per dimension the union of both families' split points.
    std::vector<int64_t> ov[kMaxRank];
    int64_t natoms = 1;
    for (int d = 0; d < rank; d++) {
        ov[d] = src[d].b;
        ov[d].insert(ov[d].end(), dst[d].b.begin(), dst[d].b.end());
        std::sort(ov[d].begin(), ov[d].end());
        ov[d].erase(std::unique(ov[d].begin(), ov[d].end()), ov[d].end());
        natoms *= (int64_t)ov[d].size() - 1;
        if (dims[d] == 0) natoms = 0;
    }
    xp->n_atoms = natoms;
    int64_t ai[kMaxRank] = {0};
    for (int64_t a = 0; a < natoms; a++) {
        int64_t lo[kMaxRank], ext[kMaxRank];
        int64_t sid = 0, did = 0;
        int64_t sblo[kMaxRank], sbext[kMaxRank], dblo[kMaxRank], dbext[kMaxRank];
        for (int d = 0; d < rank; d++) {
            lo[d] = ov[d][ai[d]];
            ext[d] = ov[d][ai[d] + 1] - lo[d];
            int si = interval_of(src[d], lo[d]), di = interval_of(dst[d], lo[d]);
            sid = sid * src[d].nblocks() + si;
            did = did * dst[d].nblocks() + di;
            sblo[d] = src[d].b[si];
            sbext[d] = src[d].b[si + 1] - sblo[d];
            dblo[d] = dst[d].b[di];
            dbext[d] = dst[d].b[di + 1] - dblo[d];
        }
        int64_t sstr[kMaxRank], dstr[kMaxRank];
        row_major_strides(rank, sbext, sstr);
        row_major_strides(rank, dbext, dstr);
        XSeg seg;
        memset(&seg, 0, sizeof seg);
        seg.src_off = soff[sid];
        seg.dst_off = doff[did];
        for (int d = 0; d < rank; d++) {
            seg.src_off += (lo[d] - sblo[d]) * sstr[d];
            seg.dst_off += (lo[d] - dblo[d]) * dstr[d];
        }
        // Merge trailing dims into one contiguous run while both sides agree.
        int last = rank - 1;
        seg.inner = ext[last];
        while (last > 0 && sstr[last - 1] == seg.inner && dstr[last - 1] == seg.inner) {
            last--;
            seg.inner *= ext[last];
        }
        // Outer dims: drop extent-1 dims, merge neighbours with compatible strides.
        int64_t oe[kMaxRank], os[kMaxRank], od[kMaxRank];
        int nd = 0;
        for (int d = 0; d < last; d++) {
            if (ext[d] == 1) continue;
            if (nd > 0 && os[nd - 1] == ext[d] * sstr[d] && od[nd - 1] == ext[d] * dstr[d]) {
                oe[nd - 1] *= ext[d];
                os[nd - 1] = sstr[d];
                od[nd - 1] = dstr[d];
                continue;
            }
            oe[nd] = ext[d];
            os[nd] = sstr[d];
            od[nd] = dstr[d];
            nd++;
        }
        emit_segment(seg, nd, oe, os, od, esize, xp);
        for (int d = rank - 1; d >= 0; d--) {
            if (++ai[d] < (int64_t)ov[d].size() - 1) break;
            ai[d] = 0;
        }
    }
    if (xp->tiles.size() > (size_t)INT32_MAX || xp->segs.size() > (size_t)INT32_MAX)
        return set_error(EA_ERR_UNSUPPORTED, "exchange plan too large");
    return EA_OK;
}

}  // namespace ea

using namespace ea;

// =================================================================== C ABI

extern "C" {

ea_status ea_set_allocator(ea_alloc_fn alloc, ea_free_fn free_fn, void *ctx) {
    t_err[0] = 0;
    if ((alloc == nullptr) != (free_fn == nullptr))
        return set_error(EA_ERR_ARG, "ea_set_allocator: give both functions or neither");
    std::lock_guard<std::mutex> lk(ea::g_alloc_mu);
    ea::g_alloc_fn = alloc;
    ea::g_free_fn = free_fn;
    ea::g_alloc_ctx = alloc ? ctx : nullptr;
    return EA_OK;
}

int ea_abi_version(void) { return EA_ABI_VERSION; }

const char *ea_last_error(void) { return t_err; }

ea_status ea_relation_create(ea_dtype dtype, int rank, const int64_t *dims, const ea_dim_part *parts, void *dev_ptr,
                             ea_relation *out) {
    t_err[0] = 0;
    if (!out || !dims || !parts) return set_error(EA_ERR_ARG, "ea_relation_create: NULL argument");
    if (dtype != EA_F32 && dtype != EA_BF16) return set_error(EA_ERR_DTYPE, "ea_relation_create: unknown dtype %d", dtype);
    if (rank < 1 || rank > kMaxRank) return set_error(EA_ERR_ARG, "ea_relation_create: rank %d out of [1, 8]", rank);
    if (dev_ptr && ((uintptr_t)dev_ptr % 16) != 0)
        return set_error(EA_ERR_ARG, "ea_relation_create: arena must be 16-byte aligned");
    ea_relation_s *r = new ea_relation_s();
    r->dtype = dtype;
    r->rank = rank;
    Tiling t[kMaxRank];
    for (int d = 0; d < rank; d++) {
        r->dims[d] = dims[d];
        ea_status st = make_tiling(dims[d], parts[d].nblocks, parts[d].bounds, &t[d]);
        if (st) {
            delete r;
            return st;
        }
        r->bounds[d] = t[d].b;
    }
    tiling_offsets(rank, t, &r->blk_off);
    r->nblocks = (int64_t)r->blk_off.size() - 1;
    r->bytes = (size_t)r->blk_off.back() * elem_size(dtype);
    if (dev_ptr) {
        r->arena = (char *)dev_ptr;
    } else if (r->bytes > 0) {
        ea_status st = dev_alloc(r->bytes, (void **)&r->arena, &r->release, "ea_relation_create");
        if (st) {
            delete r;
            return st;
        }
        r->owned = true;
    }
    *out = r;
    return EA_OK;
}

ea_status ea_relation_copy_host(ea_relation rel, void *host, int direction, void *stream) {
    t_err[0] = 0;
    if (!rel || (!host && rel->bytes)) return set_error(EA_ERR_ARG, "ea_relation_copy_host: NULL argument");
    if (direction != EA_TO_HOST && direction != EA_TO_DEVICE)
        return set_error(EA_ERR_ARG, "ea_relation_copy_host: direction must be EA_TO_HOST or EA_TO_DEVICE");
    const int r = rel->rank;
    const size_t es = elem_size(rel->dtype);
    int64_t hstr[kMaxRank];  // row-major strides of the dense host tensor (elements)
    hstr[r - 1] = 1;
    for (int d = r - 2; d >= 0; d--) hstr[d] = hstr[d + 1] * rel->dims[d + 1];
    cudaStream_t st = (cudaStream_t)stream;
    char *hbase = (char *)host;
    for (int64_t b = 0; b < rel->nblocks; b++) {
        int64_t iv[kMaxRank], lo[kMaxRank], ext[kMaxRank];
        block_coords(rel, b, iv);
        block_box(rel, iv, lo, ext);
        // k: the innermost dim the block does not span whole (or 0); the
        // block's cells over dims k.. are then one run, contiguous in the host
        // tensor and in the block alike
        int k = r - 1;
        while (k > 0 && ext[k] == rel->dims[k]) k--;
        int64_t run = 1;
        for (int d = k; d < r; d++) run *= ext[d];
        if (run == 0) continue;
        // one strided copy per index of dims < k - 1; dim k - 1 (if any) is
        // the copy's height at the host stride of that dim
        const int64_t height = k >= 1 ? ext[k - 1] : 1;
        const int64_t hpitch = k >= 1 ? hstr[k - 1] : 0;
        const int nout = k >= 1 ? k - 1 : 0;
        int64_t nouter = 1;
        for (int d = 0; d < nout; d++) nouter *= ext[d];
        const size_t wbytes = (size_t)run * es;
        char *dblock = rel->arena + rel->blk_off[b] * es;
        for (int64_t o = 0; o < nouter; o++) {
            int64_t rem = o, hoff = 0;
            for (int d = nout - 1; d >= 0; d--) {
                hoff += (lo[d] + rem % ext[d]) * hstr[d];
                rem /= ext[d];
            }
            for (int d = nout; d < r; d++) hoff += lo[d] * hstr[d];
            char *hp = hbase + hoff * es;
            char *dp = dblock + (size_t)(o * height * run) * es;
            cudaError_t e;
            if (height == 1)
                e = direction == EA_TO_DEVICE ? cudaMemcpyAsync(dp, hp, wbytes, cudaMemcpyHostToDevice, st)
                                              : cudaMemcpyAsync(hp, dp, wbytes, cudaMemcpyDeviceToHost, st);
            else
                e = direction == EA_TO_DEVICE
                        ? cudaMemcpy2DAsync(dp, wbytes, hp, (size_t)hpitch * es, wbytes, (size_t)height,
                                            cudaMemcpyHostToDevice, st)
                        : cudaMemcpy2DAsync(hp, (size_t)hpitch * es, dp, wbytes, wbytes, (size_t)height,
                                            cudaMemcpyDeviceToHost, st);
            if (e != cudaSuccess) return cuda_error(e, "ea_relation_copy_host");
        }
    }
    return EA_OK;
}

ea_status ea_relation_destroy(ea_relation rel) {
    t_err[0] = 0;
    if (!rel) return EA_OK;
    if (rel->owned && rel->arena) dev_free(rel->arena, rel->release);
    delete rel;
    return EA_OK;
}

ea_status ea_relation_info(ea_relation rel, int32_t *dtype, int32_t *rank, int64_t *dims, int64_t *nblocks) {
    if (!rel) return set_error(EA_ERR_ARG, "ea_relation_info: NULL relation");
    if (dtype) *dtype = rel->dtype;
    if (rank) *rank = rel->rank;
    if (dims)
        for (int d = 0; d < rel->rank; d++) dims[d] = rel->dims[d];
    if (nblocks) *nblocks = rel->nblocks;
    return EA_OK;
}

ea_status ea_relation_block(ea_relation rel, int64_t block_id, void **dev_ptr, int64_t *lo, int64_t *hi) {
    if (!rel) return set_error(EA_ERR_ARG, "ea_relation_block: NULL relation");
    if (block_id < 0 || block_id >= rel->nblocks) return set_error(EA_ERR_ARG, "ea_relation_block: id out of range");
    int64_t iv[kMaxRank], l[kMaxRank], e[kMaxRank];
    block_coords(rel, block_id, iv);
    block_box(rel, iv, l, e);
    if (dev_ptr) *dev_ptr = rel->arena + rel->blk_off[block_id] * elem_size(rel->dtype);
    for (int d = 0; d < rel->rank; d++) {
        if (lo) lo[d] = l[d];
        if (hi) hi[d] = l[d] + e[d];
    }
    return EA_OK;
}

ea_status ea_relation_data(ea_relation rel, void **arena, size_t *bytes) {
    if (!rel) return set_error(EA_ERR_ARG, "ea_relation_data: NULL relation");
    if (arena) *arena = rel->arena;
    if (bytes) *bytes = rel->bytes;
    return EA_OK;
}

ea_status ea_relation_bounds(ea_relation rel, int dim, int32_t *nblocks, int64_t *bounds) {
    if (!rel || dim < 0 || dim >= rel->rank) return set_error(EA_ERR_ARG, "ea_relation_bounds: bad relation or dim");
    if (nblocks) *nblocks = (int32_t)rel->bounds[dim].size() - 1;
    if (bounds)
        for (size_t i = 0; i < rel->bounds[dim].size(); i++) bounds[i] = rel->bounds[dim][i];
    return EA_OK;
}

ea_status ea_plan_worklist(const char *spec, const int64_t *shapes, const ea_index_part *parts, int n_parts,
                           char pred_lo, char pred_hi, int64_t cap_groups, int64_t cap_tuples, int64_t *groups,
                           int64_t *grp_ptr, int64_t *tuples, int64_t *n_groups, int64_t *n_tuples,
                           int64_t *join_volume, int64_t *agg_volume) {
    t_err[0] = 0;
    Spec sp;
    ea_status st = parse_spec(spec, &sp);
    if (st) return st;
    if (!shapes) return set_error(EA_ERR_ARG, "ea_plan_worklist: shapes is NULL");
    LetterTilings lt;
    int si = 0;
    for (int k = 0; k < sp.n_in; k++)
        for (char c : sp.term[k]) {
            int64_t e = shapes[si++];
            Tiling &t = lt.t[c - 'a'];
            if (t.extent >= 0 && t.extent != e)
                return set_error(EA_ERR_SHAPE, "letter '%c' has extents %lld and %lld", c, (long long)t.extent,
                                 (long long)e);
            if (t.extent < 0) {
                st = make_tiling(e, 1, nullptr, &t);
                if (st) return st;
            }
        }
    for (int i = 0; i < n_parts; i++) {
        char c = parts[i].index;
        if (c < 'a' || c > 'z' || lt.t[c - 'a'].extent < 0)
            return set_error(EA_ERR_SPEC, "partition names letter '%c' that the spec does not use", c);
        st = make_tiling(lt.t[c - 'a'].extent, parts[i].nblocks, parts[i].bounds, &lt.t[c - 'a']);
        if (st) return st;
    }
    if ((pred_lo != 0) != (pred_hi != 0)) return set_error(EA_ERR_ARG, "predicate needs two letters");
    if (pred_lo && (lt.t[pred_lo - 'a'].extent < 0 || lt.t[pred_hi - 'a'].extent < 0))
        return set_error(EA_ERR_SPEC, "predicate letter not in the spec");
    WorkList wl;
    st = plan_worklist(sp, lt, pred_lo, pred_hi, &wl);
    if (st) return st;
    int64_t ng = (int64_t)wl.groups.size(), nt = (int64_t)wl.tuples.size() / sp.n_in;
    if (n_groups) *n_groups = ng;
    if (n_tuples) *n_tuples = nt;
    if (join_volume) *join_volume = wl.join_volume;
    if (agg_volume) *agg_volume = wl.agg_volume;
    if (groups || grp_ptr || tuples) {
        if (cap_groups < ng || cap_tuples < nt) return set_error(EA_ERR_ARG, "ea_plan_worklist: capacity too small");
        if (groups) memcpy(groups, wl.groups.data(), sizeof(int64_t) * ng);
        if (grp_ptr) memcpy(grp_ptr, wl.grp_ptr.data(), sizeof(int64_t) * (ng + 1));
        if (tuples) memcpy(tuples, wl.tuples.data(), sizeof(int64_t) * nt * sp.n_in);
    }
    return EA_OK;
}

static ea_status tilings_from_parts(int rank, const int64_t *dims, const ea_dim_part *parts, Tiling *t) {
    if (!dims || !parts) return set_error(EA_ERR_ARG, "NULL dims or parts");
    if (rank < 1 || rank > kMaxRank) return set_error(EA_ERR_ARG, "rank %d out of [1, 8]", rank);
    for (int d = 0; d < rank; d++) {
        ea_status st = make_tiling(dims[d], parts[d].nblocks, parts[d].bounds, &t[d]);
        if (st) return st;
    }
    return EA_OK;
}

ea_status ea_exchange_permutation(int rank, const int64_t *dims, const ea_dim_part *src_parts,
                                  const ea_dim_part *dst_parts, int64_t *perm) {
    t_err[0] = 0;
    Tiling s[kMaxRank], d[kMaxRank];
    ea_status st = tilings_from_parts(rank, dims, src_parts, s);
    if (st) return st;
    st = tilings_from_parts(rank, dims, dst_parts, d);
    if (st) return st;
    if (!perm) return set_error(EA_ERR_ARG, "perm is NULL");
    ExchangePlan xp;
    st = plan_exchange(rank, dims, s, d, 1, &xp);
    if (st) return st;
    // Walk the planned segments exactly as the kernel does.
    for (const XTile &t : xp.tiles) {
        const XSeg &g = xp.segs[t.seg];
        for (int64_t r = t.row0; r < t.row0 + t.nrows; r++) {
            int64_t rem = r, so = g.src_off, dof = g.dst_off;
            for (int i = g.nd - 1; i >= 0; i--) {
                int64_t c = rem % g.ext[i];
                rem /= g.ext[i];
                so += c * g.sstr[i];
                dof += c * g.dstr[i];
            }
            for (int64_t c = t.col0; c < t.col0 + t.ncols; c++) perm[dof + c] = so + c;
        }
    }
    return EA_OK;
}

ea_status ea_overlay_atoms(int rank, const int64_t *dims, const ea_dim_part *src_parts, const ea_dim_part *dst_parts,
                           int64_t *n_atoms) {
    t_err[0] = 0;
    Tiling s[kMaxRank], d[kMaxRank];
    ea_status st = tilings_from_parts(rank, dims, src_parts, s);
    if (st) return st;
    st = tilings_from_parts(rank, dims, dst_parts, d);
    if (st) return st;
    if (!n_atoms) return set_error(EA_ERR_ARG, "n_atoms is NULL");
    ExchangePlan xp;
    st = plan_exchange(rank, dims, s, d, 1, &xp);
    if (st) return st;
    *n_atoms = xp.n_atoms;
    return EA_OK;
}

}  // extern "C"
