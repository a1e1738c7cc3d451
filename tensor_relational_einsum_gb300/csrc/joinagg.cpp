// joinagg.cpp -- ea_joinagg_run and ea_exchange: plan a join-agg (or an
// exchange) on the host, upload the plan once, cache it, launch the kernel.
//
// A join-agg ("Every Kernel Is a Join", Definition 3.7) is executed as:
//   join       the canonical work list (plan_worklist): one function
//              specification per combination of letter intervals, grouped
//              by output block;
//   aggregate  fused into the kernel that runs the group (the accumulator
//              of a contraction, the warp reduction of a row reduction);
//   recompose  zero-copy: the output relation is stored as its blocks.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <map>
#include <unordered_map>

#include "plan.h"

namespace ea {

// ----------------------------------------------------------- device context

DevCtx g_ctx[64];

ea_status get_ctx(DevCtx **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_error(e, "cudaGetDevice");
    if (dev < 0 || dev >= 64) return set_error(EA_ERR_ARG, "device index %d out of range", dev);
    DevCtx &c = g_ctx[dev];
    if (!c.init) {
        e = cudaDeviceGetAttribute(&c.num_sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return cuda_error(e, "cudaDeviceGetAttribute");
        e = cudaMalloc((void **)&c.err, 256);
        if (e != cudaSuccess) return cuda_error(e, "cudaMalloc(error word)");
        e = cudaMemset(c.err, 0, 256);
        if (e != cudaSuccess) return cuda_error(e, "cudaMemset(error word)");
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
        if (e == cudaSuccess && q == cudaDriverEntryPointSuccess) c.encode = (PFN_cuTensorMapEncodeTiled_v12000)fn;
        else cudaGetLastError();
        c.init = true;
    }
    *out = &c;
    return EA_OK;
}

// --------------------------------------------------------------- plan blob

thread_local LastPlan t_last;

std::unordered_map<std::string, DevPlan *> g_cache;

ea_status upload(const Blob &b, cudaStream_t st, DevPlan *p) {
    p->bytes = b.h.size();
    ea_status s = dev_alloc(p->bytes, (void **)&p->dev, &p->dev_release, "plan upload");
    if (s) return s;
    cudaError_t e = cudaMallocHost((void **)&p->pinned, p->bytes);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return set_error(EA_ERR_ALLOC, "plan upload: cudaMallocHost(%zu): %s", p->bytes, cudaGetErrorString(e));
    }
    memcpy(p->pinned, b.h.data(), p->bytes);
    e = cudaMemcpyAsync(p->dev, p->pinned, p->bytes, cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) return cuda_error(e, "plan upload: cudaMemcpyAsync");
    e = cudaEventCreateWithFlags(&p->ready, cudaEventDisableTiming);
    if (e != cudaSuccess) return cuda_error(e, "cudaEventCreate");
    e = cudaEventRecord(p->ready, st);
    if (e != cudaSuccess) return cuda_error(e, "cudaEventRecord");
    p->made_on = st;
    return EA_OK;
}

void free_plan(DevPlan *p) {
    if (!p) return;
    if (p->dev) dev_free(p->dev, p->dev_release);
    if (p->pinned) cudaFreeHost(p->pinned);
    if (p->ready) cudaEventDestroy(p->ready);
    delete p;
}

// Order the plan's upload before work on `st`.  Once the upload is known to
// have completed (queried on any later use), no CUDA call is made at all, so
// a cached plan can be launched inside a CUDA-graph capture.
ea_status plan_ready_on(DevPlan *p, cudaStream_t st) {
    if (p->uploaded) return EA_OK;
    cudaError_t q = cudaEventQuery(p->ready);
    if (q == cudaSuccess) {
        p->uploaded = true;
        return EA_OK;
    }
    if (q != cudaErrorNotReady) return cuda_error(q, "cudaEventQuery(plan upload)");
    if (st != p->made_on) {
        cudaError_t e = cudaStreamWaitEvent(st, p->ready, 0);
        if (e != cudaSuccess) return cuda_error(e, "cudaStreamWaitEvent(plan upload)");
    }
    return EA_OK;
}

// ----------------------------------------------------------- block views

struct BlockView {
    int64_t base = 0;  // element offset of the block in its arena
    int64_t lo[26], ext[26], str[26];
    bool has[26];
};

static void view_of(const ea_relation_s *r, const std::string &term, int64_t bid, BlockView *v) {
    int64_t iv[kMaxRank], lo[kMaxRank], ext[kMaxRank], str[kMaxRank];
    block_coords(r, bid, iv);
    block_box(r, iv, lo, ext);
    row_major_strides(r->rank, ext, str);
    for (int l = 0; l < 26; l++) {
        v->has[l] = false;
        v->lo[l] = 0;
        v->ext[l] = 1;
        v->str[l] = 0;
    }
    for (int d = 0; d < r->rank; d++) {
        int l = term[d] - 'a';
        v->has[l] = true;
        v->lo[l] = lo[d];
        v->ext[l] = ext[d];
        v->str[l] = str[d];
    }
    v->base = r->blk_off[bid];
}

// Merge a group of letters (outer first) into one dimension for every
// operand that holds them.  Extent-1 letters are dropped.
struct Merged {
    int64_t ext = 1;
    int64_t str[3] = {0, 0, 0};
    int single = -1;  // the only letter of extent > 1, if exactly one
};

static bool merge_letters(const std::string &letters, const BlockView *const *vs, int nv, Merged *m) {
    std::string keep;
    const BlockView *ref = nullptr;
    for (int i = 0; i < nv; i++)
        if (vs[i]) {
            ref = vs[i];
            break;
        }
    m->ext = 1;
    for (int i = 0; i < 3; i++) m->str[i] = 0;
    for (char c : letters) {
        if (ref->ext[c - 'a'] == 0) {
            m->ext = 0;  // empty block: nothing to merge
            return true;
        }
        if (ref->ext[c - 'a'] > 1) keep.push_back(c);
    }
    m->single = keep.size() == 1 ? keep[0] - 'a' : -1;
    if (keep.empty()) return true;
    for (char c : keep) m->ext *= ref->ext[c - 'a'];
    for (int i = 0; i < nv; i++) {
        const BlockView *v = vs[i];
        if (!v) continue;
        for (size_t j = 0; j + 1 < keep.size(); j++) {
            int a = keep[j] - 'a', b = keep[j + 1] - 'a';
            if (v->str[a] != v->ext[b] * v->str[b]) return false;
        }
        m->str[i] = v->str[keep.back() - 'a'];
    }
    return true;
}

// ---------------------------------------------------------- tensor maps

static ea_status encode_map(DevCtx *c, CUtensorMap *map, int dtype, const void *base, uint64_t d0, uint64_t d1,
                            uint64_t d2, uint64_t s1_bytes, uint64_t s2_bytes, uint32_t b0, uint32_t b1) {
    if (!c->encode) return set_error(EA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    cuuint64_t dims[3] = {d0, d1, d2};
    cuuint64_t strides[2] = {s1_bytes, s2_bytes};
    cuuint32_t box[3] = {b0, b1, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = c->encode(map, dtype == EA_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                           const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return set_error(EA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return EA_OK;
}

static bool al16(int64_t elems, size_t es) { return ((uint64_t)elems * es) % 16 == 0; }

// --------------------------------------------------------------- classes

struct JoinCtx {
    Spec sp;
    const ea_relation_s *in[kMaxIn];
    ea_relation_s *out;
    LetterTilings lt;
    WorkList wl;
    ea_agg agg;
    ea_map map;
    float scale, eps;
    char pred_lo, pred_hi;
    const float *rope_table;
    int64_t rope_npos;
    char rope_pos;
    ea_relation_s *out2;
    int epi_map;                 // epilogue join of a contraction: 0, EA_MAP_ADD or EA_MAP_SILU_MUL
    const ea_relation_s *epi_in; // EA_MAP_ADD: the joined relation (output's extents and tiling)
    int rope_dim;                // ROPE: pair period along the last letter (0 = its extent)
    int rope_layout;             // ROPE table: 0 position-major, 1 pair-major
    const ea_relation_s *row_rms;  // contraction row scale rsqrt(row_rms[row] + eps), or null
    char row_letter;             // the output letter of input 0 only (rows of the contraction)
    char copy_letter;            // partials: the letter of the copies (leading output letter), or 0
    char epi_pair;               // EA_MAP_SILU_MUL: the paired letter (innermost in the planned output)
    int simt_bf16;               // a bf16 contraction may run on the SIMT kernel
    ea_relation_s *user_out;     // the output relation (out is its pre-epilogue view when paired)
};

// Special letters of an elementwise / row-reduction view.
static void set_special(EwItem *it, int slot, char letter, const BlockView &ov, const int *dim_of_letter,
                        int inner_letter) {
    if (!letter) {
        it->sdim[slot] = -1;
        it->slo[slot] = 0;
        return;
    }
    int l = letter - 'a';
    it->slo[slot] = ov.lo[l];
    if (l == inner_letter) it->sdim[slot] = kViewDims;
    else if (dim_of_letter[l] >= 0) it->sdim[slot] = dim_of_letter[l];
    else it->sdim[slot] = -1;
}

// Elementwise join: agg NONE, every tuple is one output block.
static ea_status build_ewise(JoinCtx &j, DevCtx *c, cudaStream_t st, DevPlan *p) {
    const Spec &sp = j.sp;
    int n_in = sp.n_in;
    std::vector<EwItem> items;
    std::vector<EwTile> tiles;
    size_t es_out = elem_size(j.out->dtype);
    for (size_t g = 0; g < j.wl.groups.size(); g++) {
        int64_t t = j.wl.grp_ptr[g];
        if (j.wl.grp_ptr[g + 1] - t != 1) return set_error(EA_ERR_SPEC, "agg NONE needs one tuple per output block");
        BlockView ov, iv[kMaxIn];
        view_of(j.out, sp.out, j.wl.groups[g], &ov);
        for (int k = 0; k < n_in; k++) view_of(j.in[k], sp.term[k], j.wl.tuples[t * n_in + k], &iv[k]);
        EwItem it;
        memset(&it, 0, sizeof it);
        int inner = sp.out.back() - 'a';
        it.out_base = ov.base;
        it.len = ov.ext[inner];
        it.out_inner = ov.str[inner];
        for (int k = 0; k < n_in; k++) {
            it.in_base[k] = iv[k].base;
            it.in_inner[k] = iv[k].has[inner] ? iv[k].str[inner] : 0;
        }
        // Row dims: the other output letters with extent > 1; merge neighbours
        // when every operand agrees; never merge a special letter.
        int dim_of_letter[26];
        for (int l = 0; l < 26; l++) dim_of_letter[l] = -1;
        int nd = 0;
        char last_c = 0;
        for (size_t d = 0; d + 1 < sp.out.size(); d++) {
            char ch = sp.out[d];
            int l = ch - 'a';
            if (ov.ext[l] == 1) continue;
            bool special = ch == j.pred_lo || ch == j.pred_hi || (j.map == EA_MAP_ROPE && ch == j.rope_pos);
            bool prev_special = last_c && (last_c == j.pred_lo || last_c == j.pred_hi ||
                                           (j.map == EA_MAP_ROPE && last_c == j.rope_pos));
            bool can = nd > 0 && !special && !prev_special && it.ostr[nd - 1] == ov.ext[l] * ov.str[l];
            for (int k = 0; k < n_in && can; k++) {
                int64_t s = iv[k].has[l] ? iv[k].str[l] : 0;
                can = it.istr[k][nd - 1] == ov.ext[l] * s;
            }
            if (can) {
                it.ext[nd - 1] *= ov.ext[l];
                it.ostr[nd - 1] = ov.str[l];
                for (int k = 0; k < n_in; k++) it.istr[k][nd - 1] = iv[k].has[l] ? iv[k].str[l] : 0;
            } else {
                if (nd == kViewDims) return set_error(EA_ERR_UNSUPPORTED, "elementwise view needs more than 6 row dims");
                it.ext[nd] = ov.ext[l];
                it.ostr[nd] = ov.str[l];
                for (int k = 0; k < n_in; k++) it.istr[k][nd] = iv[k].has[l] ? iv[k].str[l] : 0;
                dim_of_letter[l] = nd;
                nd++;
            }
            last_c = ch;
        }
        for (int d = nd; d < kViewDims; d++) it.ext[d] = 1;
        it.nd = (int16_t)nd;
        it.inner_lo = ov.lo[inner];
        it.rows = 1;
        for (int d = 0; d < kViewDims; d++) it.rows *= it.ext[d];
        set_special(&it, 0, j.pred_lo, ov, dim_of_letter, inner);
        set_special(&it, 1, j.pred_hi, ov, dim_of_letter, inner);
        set_special(&it, 2, j.map == EA_MAP_ROPE ? j.rope_pos : 0, ov, dim_of_letter, inner);
        bool vec = it.len % 8 == 0 && it.out_inner == 1 && it.out_base % 8 == 0;
        for (int d = 0; d < nd; d++) vec = vec && it.ostr[d] % 8 == 0;
        for (int k = 0; k < n_in; k++) {
            if (it.in_inner[k] == 1) {
                vec = vec && it.in_base[k] % 8 == 0;
                for (int d = 0; d < nd; d++) vec = vec && it.istr[k][d] % 8 == 0;
            } else if (it.in_inner[k] != 0) {
                vec = false;
            }
        }
        it.vec = vec ? 1 : 0;
        if (j.map == EA_MAP_ROPE) {
            if (it.in_inner[0] != 1 || it.len % 2 != 0 || ov.lo[inner] % 2 != 0)
                return set_error(EA_ERR_UNSUPPORTED, "ROPE needs the pair letter last, contiguous, with even blocks");
            if (!j.rope_table || it.sdim[2] == kViewDims)
                return set_error(EA_ERR_ARG, "ROPE needs rope_table and a position letter other than the pair letter");
            int64_t pos_hi = it.slo[2] + (it.sdim[2] >= 0 ? it.ext[it.sdim[2]] : 1);
            int64_t pair_hi = (ov.lo[inner] + it.len) / 2;
            if (pos_hi > j.rope_npos) return set_error(EA_ERR_ARG, "ROPE position beyond rope_npos");
            (void)pair_hi;
        }
        int32_t id = (int32_t)items.size();
        items.push_back(it);
        if (it.rows == 0 || it.len == 0) continue;
        // tiles of about 32K cells whose row count is a whole number of the
        // CTA's row passes (8 warps x rows per warp, as the kernel packs them)
        const int64_t target = 32768;
        if (it.len >= target) {
            for (int64_t r = 0; r < it.rows; r++)
                for (int64_t c0 = 0; c0 < it.len; c0 += target)
                    tiles.push_back(EwTile{id, 0, r, 1, c0, std::min(target, it.len - c0)});
        } else {
            const int64_t cpr = it.vec ? it.len / 8 : it.len;
            int ns = 0, bytes = 16;
            for (int k = 0; k < n_in; k++)
                if (sp.term[k].find(sp.out.back()) != std::string::npos) {
                    ns++;
                    if (j.in[k]->dtype == EA_F32) bytes = 32;
                }
            // the kernel's batch: about 128 bytes of streamed inputs per lane
            // (RoPE batches 4 chunks: it also loads the (cos, sin) table)
            const int64_t u = !it.vec || j.map == EA_MAP_ROPE ? 4 : std::max<int64_t>(1, (128 / bytes) / std::max(1, ns));
            int64_t lpr = 32;
            while (lpr > 1 && lpr * u > cpr) lpr /= 2;
            const int64_t pass = 8 * (32 / lpr);
            int64_t per = std::max<int64_t>(1, target / it.len);
            per = std::max<int64_t>(pass, per / pass * pass);
            // A tile either stays inside one run of the innermost row dim, or
            // covers whole runs inside one run of the second-innermost dim; the
            // kernel then addresses its rows with two strides.
            const int64_t run = it.nd > 0 ? it.ext[it.nd - 1] : 1;
            const int64_t run2 = it.nd > 1 ? run * it.ext[it.nd - 2] : run;
            if (run >= per) {
                for (int64_t r0 = 0; r0 < it.rows; r0 += run)
                    for (int64_t r = r0; r < r0 + run; r += per)
                        tiles.push_back(EwTile{id, 0, r, std::min(per, r0 + run - r), 0, it.len});
            } else {
                const int64_t perr = std::max<int64_t>(run, per / run * run);
                for (int64_t r0 = 0; r0 < it.rows; r0 += run2)
                    for (int64_t r = r0; r < r0 + run2; r += perr)
                        tiles.push_back(EwTile{id, 0, r, std::min(perr, r0 + run2 - r), 0, it.len});
            }
        }
    }
    (void)es_out;
    (void)c;
    int64_t in_el[kMaxIn];
    for (int k = 0; k < n_in; k++) in_el[k] = rel_elems(j.in[k]);
    ea_status cs = check_view_items(items.data(), items.size(), n_in, in_el, rel_elems(j.out), "elementwise view");
    if (!cs) cs = check_ew_tiles(tiles.data(), tiles.size(), items.data(), items.size());
    if (cs) return cs;
    Blob b;
    size_t oi = b.add_vec(items), ot = b.add_vec(tiles);
    ea_status s = upload(b, st, p);
    if (s) return s;
    p->kind = kEwise;
    EwParams &e = p->ew;
    e.items = (const EwItem *)(p->dev + oi);
    e.tiles = (const EwTile *)(p->dev + ot);
    e.ntiles = (int64_t)tiles.size();
    for (int k = 0; k < n_in; k++) {
        e.in[k] = j.in[k]->arena;
        e.in_dtype[k] = j.in[k]->dtype;
    }
    e.out = j.out->arena;
    e.out_dtype = j.out->dtype;
    e.out_elems = rel_elems(j.out);
    for (int k = 0; k < n_in; k++) e.in_elems[k] = rel_elems(j.in[k]);
    e.n_in = n_in;
    e.map = j.map;
    e.scale = j.scale;
    e.eps = j.eps;
    e.pred = j.pred_lo ? 1 : 0;
    e.rope_table = j.rope_table;
    e.rope_npos = j.rope_npos;
    e.rope_half = j.lt.t[sp.out.back() - 'a'].extent / 2;
    e.has_vec = e.has_scalar = 0;
    e.stream_mask = 0;
    for (int k = 0; k < n_in; k++) {
        bool runs = sp.term[k].find(sp.out.back()) != std::string::npos;
        if (runs) e.stream_mask |= 1 << k;
    }
    for (const EwItem &x : items) {
        if (x.rows == 0 || x.len == 0) continue;
        if (x.vec) e.has_vec = 1;
        else e.has_scalar = 1;
    }
    return EA_OK;
}

// Row reduction: the aggregated letters are the trailing letters of input 0.
static ea_status build_rowreduce(JoinCtx &j, DevCtx *c, cudaStream_t st, DevPlan *p) {
    const Spec &sp = j.sp;
    int n_in = sp.n_in;
    const std::string &red = sp.contracted;
    const std::string &t0 = sp.term[0];
    if (t0.size() < red.size() || t0.substr(t0.size() - red.size()) != red)
        return set_error(EA_ERR_UNSUPPORTED, "row reduction needs the aggregated letters last in input 0 (\"%s\")",
                         t0.c_str());
    for (int k = 1; k < n_in; k++) {
        const std::string &tk = sp.term[k];
        bool any = false;
        for (char ch : red) any |= tk.find(ch) != std::string::npos;
        if (any && (tk.size() < red.size() || tk.substr(tk.size() - red.size()) != red))
            return set_error(EA_ERR_UNSUPPORTED, "row reduction: input %d must hold the aggregated letters last", k);
    }
    if ((j.pred_lo && red.find(j.pred_lo) != std::string::npos && red.size() != 1) ||
        (j.pred_hi && red.find(j.pred_hi) != std::string::npos && red.size() != 1))
        return set_error(EA_ERR_UNSUPPORTED, "a predicate on an aggregated letter needs a single aggregated letter");
    std::vector<EwItem> items;
    std::vector<RrGroup> groups;
    std::vector<RrTile> tiles;
    struct GroupRows {
        int32_t gid;
        int64_t rows, run, per;
    };
    std::vector<GroupRows> grows;
    int64_t max_items = 0;
    int inner_letter = red.size() == 1 ? red[0] - 'a' : -2;
    for (size_t g = 0; g < j.wl.groups.size(); g++) {
        BlockView ov;
        view_of(j.out, sp.out, j.wl.groups[g], &ov);
        RrGroup G{(int32_t)items.size(), 0, 0, 0};
        int64_t rows = 1;
        for (int64_t t = j.wl.grp_ptr[g]; t < j.wl.grp_ptr[g + 1]; t++) {
            BlockView iv[kMaxIn];
            for (int k = 0; k < n_in; k++) view_of(j.in[k], sp.term[k], j.wl.tuples[t * n_in + k], &iv[k]);
            EwItem it;
            memset(&it, 0, sizeof it);
            it.out_base = ov.base;
            it.len = 1;
            for (char ch : red) it.len *= iv[0].ext[ch - 'a'];
            it.out_inner = 0;
            for (int k = 0; k < n_in; k++) {
                it.in_base[k] = iv[k].base;
                it.in_inner[k] = iv[k].has[red.back() - 'a'] ? 1 : 0;
            }
            int dim_of_letter[26];
            for (int l = 0; l < 26; l++) dim_of_letter[l] = -1;
            int nd = 0;
            for (char ch : sp.out) {
                int l = ch - 'a';
                if (ov.ext[l] == 1) continue;
                if (nd == kViewDims) return set_error(EA_ERR_UNSUPPORTED, "row reduction with more than 6 row dims");
                it.ext[nd] = ov.ext[l];
                it.ostr[nd] = ov.str[l];
                for (int k = 0; k < n_in; k++) it.istr[k][nd] = iv[k].has[l] ? iv[k].str[l] : 0;
                dim_of_letter[l] = nd;
                nd++;
            }
            for (int d = nd; d < kViewDims; d++) it.ext[d] = 1;
            it.nd = (int16_t)nd;
            it.inner_lo = iv[0].lo[red.back() - 'a'];
            it.rows = 1;
            for (int d = 0; d < kViewDims; d++) it.rows *= it.ext[d];
            rows = it.rows;
            // predicate letters may live in the input only (the reduced letter)
            BlockView pv = iv[0];
            for (int l = 0; l < 26; l++)
                if (!pv.has[l] && ov.has[l]) pv.lo[l] = ov.lo[l];
            set_special(&it, 0, j.pred_lo, pv, dim_of_letter, inner_letter);
            set_special(&it, 1, j.pred_hi, pv, dim_of_letter, inner_letter);
            it.sdim[2] = -1;
            bool vec = it.len % 8 == 0;
            for (int k = 0; k < n_in; k++)
                if (it.in_inner[k] == 1) {
                    vec = vec && it.in_base[k] % 8 == 0;
                    for (int d = 0; d < nd; d++) vec = vec && it.istr[k][d] % 8 == 0;
                }
            it.vec = vec ? 1 : 0;
            items.push_back(it);
        }
        G.i1 = (int32_t)items.size();
        int32_t gid = (int32_t)groups.size();
        groups.push_back(G);
        // rows per tile: four passes of the CTA's 8 warps, each pass packing
        // as many rows per warp as the kernel does for this segment length;
        // a tile never crosses a run of the innermost row dimension, so the
        // offsets inside it are linear in the row index
        const EwItem &first = items[G.i0];
        const int64_t chunks = first.vec ? first.len / 8 : first.len;
        int ns = 0, bytes = 16, dts = 0;
        for (int k = 0; k < n_in; k++)
            if (sp.term[k].find(red.back()) != std::string::npos) {
                ns++;
                bytes = j.in[k]->dtype == EA_F32 ? std::max(bytes, 32) : bytes;
                dts |= 1 << j.in[k]->dtype;
            }
        if (dts == 3) bytes = 32;  // mixed dtypes: the generic instance batches like fp32
        // the kernel's batch: about 128 bytes of streamed inputs per lane
        const int64_t u = std::max<int64_t>(1, (128 / bytes) / std::max(1, ns));
        int64_t lpr = 32;
        while (lpr > 1 && lpr * u > chunks) lpr /= 2;
        // four CTA passes per tile, or one when the whole reduction has few rows
        const int64_t pass = 8 * (32 / lpr);
        const int64_t per = rows * (int64_t)j.wl.groups.size() >= 4 * pass * 8 * c->num_sms ? 4 * pass : pass;
        const int64_t run = first.nd > 0 ? first.ext[first.nd - 1] : 1;
        grows.push_back(GroupRows{gid, rows, run, per});
        max_items = std::max<int64_t>(max_items, G.i1 - G.i0);
    }
    // The row-batch kernels (one streamed input, SUM of x or x^2, or the
    // softmax statistics; at most four blocks of one length per row, no
    // predicate) take flat tile descriptors: per tile the element offset of
    // its first row and the row stride in each block, the output offset and
    // stride, the length and the rows -- a warp reads one with a single load
    // and needs no CTA barrier.
    bool rb = !j.pred_lo && max_items <= 4 && n_in == 1 &&
              ((j.agg == EA_AGG_SUM && (j.map == EA_MAP_SQUARE || j.map == EA_MAP_IDENTITY)) ||
               (j.agg == EA_AGG_MAX_SUMEXP && j.map == EA_MAP_IDENTITY && j.scale == 1.0f));  // its kernel takes v as is
    for (const RrGroup &G : groups)
        for (int32_t i = G.i0; i < G.i1 && rb; i++) {
            const EwItem &it = items[i];
            rb = it.vec && it.len == items[G.i0].len;
            if (it.nd > 0)  // row strides held in 32 bits
                rb = rb && std::llabs(it.istr[0][it.nd - 1]) < (1ll << 31) && std::llabs(it.ostr[it.nd - 1]) < (1ll << 31);
        }
    // The bulk-copy path of the row-batch SUM: every block's rows stored back
    // to back (innermost row stride = segment length), every offset and
    // stride 16-byte aligned, a row segment at most 2 KB (a chunk of 8 rows
    // of one block fits a 16 KB stage).  Its tiles are cut to about six per
    // CTA, in multiples of 8 rows.
    const int64_t esz = j.in[0]->dtype == EA_BF16 ? 2 : 4;
    bool bulk = rb && j.agg == EA_AGG_SUM;
    for (const RrGroup &G : groups)
        for (int32_t i = G.i0; i < G.i1 && bulk; i++) {
            const EwItem &it = items[i];
            const int64_t rowb = it.len * esz;
            bulk = it.nd >= 1 && it.istr[0][it.nd - 1] == it.len && rowb % 16 == 0 &&
                   rowb <= kRbBulkBytes / kRbBulkRows && (it.in_base[0] * esz) % 16 == 0;
            for (int d = 0; d < it.nd && bulk; d++) bulk = (it.istr[0][d] * esz) % 16 == 0;
        }
    int64_t bulk_rows = kRbBulkRows;
    if (bulk) {
        int64_t all_rows = 0;
        for (const GroupRows &gr : grows) all_rows += gr.rows;
        while (bulk_rows < 64 && all_rows / (2 * bulk_rows) >= 6 * (int64_t)c->num_sms) bulk_rows *= 2;
    }
    for (const GroupRows &gr : grows) {
        int64_t per = gr.per;
        if (bulk) {
            per = bulk_rows;
        } else if (rb) {
            const int64_t row_u = j.in[0]->dtype == EA_BF16 ? 4 : 2;  // 8-element chunks per lane per block
            const int64_t chunks = items[groups[gr.gid].i0].len / 8;
            int64_t lpb = 32;
            while (lpb > 1 && lpb * row_u > chunks) lpb /= 2;
            // one row pass of the 8 warp slots, or four when there are many rows
            const int64_t pass = 8 * (32 / lpb);
            per = gr.rows * (int64_t)groups.size() >= 4 * pass * 8 * c->num_sms ? 4 * pass : pass;
        }
        for (int64_t r0 = 0; r0 < gr.rows; r0 += gr.run)
            for (int64_t r = r0; r < r0 + gr.run; r += per)
                tiles.push_back(RrTile{gr.gid, 0, r, std::min(per, r0 + gr.run - r)});
    }
    std::vector<int64_t> rbd;
    if (rb) {
        rbd.assign(tiles.size() * kRbWords, 0);
        for (size_t t = 0; t < tiles.size(); t++) {
            const RrTile &T = tiles[t];
            const RrGroup &G = groups[T.group];
            int64_t *w = &rbd[t * kRbWords];
            for (int32_t i = G.i0; i < G.i1; i++) {
                const EwItem &it = items[i];
                int64_t cd[kViewDims] = {0, 0, 0, 0, 0, 0};
                int64_t r = T.row0;
                for (int d = it.nd - 1; d >= 1; d--) {
                    cd[d] = r % it.ext[d];
                    r /= it.ext[d];
                }
                if (it.nd > 0) cd[0] = r;
                const int last = it.nd - 1;
                int64_t o = it.in_base[0];
                for (int d = 0; d < it.nd; d++) o += cd[d] * it.istr[0][d];
                w[i - G.i0] = o;
                w[4 + i - G.i0] = last >= 0 ? it.istr[0][last] : 0;
                if (i == G.i0) {
                    int64_t oo = it.out_base;
                    for (int d = 0; d < it.nd; d++) oo += cd[d] * it.ostr[d];
                    w[8] = oo;
                    w[9] = last >= 0 ? it.ostr[last] : 0;
                    w[10] = it.len;
                }
            }
            w[11] = (int64_t)(uint32_t)T.nrows | ((int64_t)(G.i1 - G.i0) << 32);
        }
    }
    int64_t in_el[kMaxIn];
    for (int k = 0; k < n_in; k++) in_el[k] = rel_elems(j.in[k]);
    ea_status cs = check_view_items(items.data(), items.size(), n_in, in_el, rel_elems(j.out), "row-reduction view");
    if (!cs) cs = check_rr_tiles(tiles.data(), tiles.size(), groups.data(), groups.size(), items.data(), items.size());
    if (!cs && rb) cs = check_rb_desc(rbd.data(), tiles.size(), in_el[0], rel_elems(j.out));
    if (cs) return cs;
    Blob b;
    size_t oi = b.add_vec(items), og = b.add_vec(groups), ot = b.add_vec(tiles), orb = b.add_vec(rbd);
    ea_status s = upload(b, st, p);
    if (s) return s;
    p->kind = kRowReduce;
    RrParams &r = p->rr;
    r.items = (const EwItem *)(p->dev + oi);
    r.groups = (const RrGroup *)(p->dev + og);
    r.tiles = (const RrTile *)(p->dev + ot);
    r.rb_desc = rb ? (const int64_t *)(p->dev + orb) : nullptr;
    r.ntiles = (int64_t)tiles.size();
    for (int k = 0; k < n_in; k++) {
        r.in[k] = j.in[k]->arena;
        r.in_dtype[k] = j.in[k]->dtype;
    }
    r.out = j.out->arena;
    r.out_dtype = j.out->dtype;
    r.out_elems = rel_elems(j.out);
    for (int k = 0; k < n_in; k++) r.in_elems[k] = rel_elems(j.in[k]);
    r.out2 = j.out2 ? j.out2->arena : nullptr;
    r.out2_dtype = j.out2 ? j.out2->dtype : 0;
    r.n_in = n_in;
    r.map = j.map;
    r.agg = j.agg;
    r.scale = j.scale;
    r.eps = j.eps;
    r.pred = j.pred_lo ? 1 : 0;
    r.max_items = (int)max_items;
    r.tile_linear = 1;
    r.row_batch = rb ? 1 : 0;
    r.row_bulk = bulk ? 1 : 0;
    r.stream_mask = 0;
    for (int k = 0; k < n_in; k++)
        if (sp.term[k].find(red.back()) != std::string::npos) r.stream_mask |= 1 << k;
    return EA_OK;
}

// Contraction: letters grouped as batch (A, B, C), M (A, C), N (B, C), K (A, B).
struct ContractionViews {
    std::string batch, M, N, K;
};

static ea_status contraction_roles(const Spec &sp, ContractionViews *cv) {
    const std::string &A = sp.term[0], &B = sp.term[1], &C = sp.out;
    for (char ch : C) {
        bool a = A.find(ch) != std::string::npos, b = B.find(ch) != std::string::npos;
        if (a && b) cv->batch.push_back(ch);
        else if (a) cv->M.push_back(ch);
        else cv->N.push_back(ch);
    }
    for (char ch : A) {
        bool b = B.find(ch) != std::string::npos, c = C.find(ch) != std::string::npos;
        if (!c && b) cv->K.push_back(ch);
        if (!c && !b) return set_error(EA_ERR_UNSUPPORTED, "letter '%c' is aggregated within input 0 only", ch);
    }
    for (char ch : B)
        if (C.find(ch) == std::string::npos && A.find(ch) == std::string::npos)
            return set_error(EA_ERR_UNSUPPORTED, "letter '%c' is aggregated within input 1 only", ch);
    return EA_OK;
}

struct TupleGeom {
    Merged bt, m, n, k;
    BlockView a, b, c;
};

static ea_status tuple_geom(const JoinCtx &j, const ContractionViews &cv, int64_t g, int64_t t, TupleGeom *tg) {
    view_of(j.in[0], j.sp.term[0], j.wl.tuples[t * 2 + 0], &tg->a);
    view_of(j.in[1], j.sp.term[1], j.wl.tuples[t * 2 + 1], &tg->b);
    view_of(j.out, j.sp.out, j.wl.groups[g], &tg->c);
    const BlockView *abc[3] = {&tg->a, &tg->b, &tg->c};
    const BlockView *ac[3] = {&tg->a, nullptr, &tg->c};
    const BlockView *bc[3] = {nullptr, &tg->b, &tg->c};
    const BlockView *ab[3] = {&tg->a, &tg->b, nullptr};
    if (!merge_letters(cv.batch, abc, 3, &tg->bt) || !merge_letters(cv.M, ac, 3, &tg->m) ||
        !merge_letters(cv.N, bc, 3, &tg->n) || !merge_letters(cv.K, ab, 3, &tg->k))
        return set_error(EA_ERR_UNSUPPORTED, "contraction: a letter group is not contiguous in every operand");
    return EA_OK;
}

static int pred_mode_of(const JoinCtx &j, const ContractionViews &cv, int *kpred) {
    *kpred = 0;
    if (!j.pred_lo) return 0;
    auto in = [](const std::string &s, char ch) { return s.find(ch) != std::string::npos; };
    if (in(cv.K, j.pred_lo) || in(cv.K, j.pred_hi)) {
        *kpred = 1;  // block filter only; removed cells must hold 0 in the operand
        return 0;
    }
    if (in(cv.N, j.pred_lo) && in(cv.M, j.pred_hi)) return 1;  // mask cells with n > m
    if (in(cv.M, j.pred_lo) && in(cv.N, j.pred_hi)) return 2;  // mask cells with m > n
    return -1;
}

static ea_status build_simt(JoinCtx &j, const ContractionViews &cv, DevCtx *c, cudaStream_t st, DevPlan *p) {
    int kpred = 0;
    int mode = pred_mode_of(j, cv, &kpred);
    if (mode < 0) return set_error(EA_ERR_UNSUPPORTED, "contraction: predicate letters must be output letters");
    std::vector<CtGroup> groups;
    std::vector<CtTuple> tuples;
    std::vector<CtTile> tiles;
    std::vector<std::pair<int32_t, CtGroup>> gtiles;  // groups with work, for the tiles
    for (size_t g = 0; g < j.wl.groups.size(); g++) {
        CtGroup G;
        memset(&G, 0, sizeof G);
        G.t0 = (int32_t)tuples.size();
        for (int64_t t = j.wl.grp_ptr[g]; t < j.wl.grp_ptr[g + 1]; t++) {
            TupleGeom tg;
            ea_status s = tuple_geom(j, cv, (int64_t)g, t, &tg);
            if (s) return s;
            if (t == j.wl.grp_ptr[g]) {
                G.c_base = tg.c.base;
                G.M = tg.m.ext;
                G.N = tg.n.ext;
                G.nb = tg.bt.ext;
                G.c_sm = tg.m.str[2];
                G.c_sn = tg.n.str[2];
                G.c_sb = tg.bt.str[2];
                if (mode) {
                    int lm = mode == 1 ? j.pred_hi - 'a' : j.pred_lo - 'a';
                    int ln = mode == 1 ? j.pred_lo - 'a' : j.pred_hi - 'a';
                    if ((tg.m.single >= 0 && tg.m.single != lm) || (tg.n.single >= 0 && tg.n.single != ln) ||
                        (tg.m.single < 0 && tg.m.ext > 1) || (tg.n.single < 0 && tg.n.ext > 1))
                        return set_error(EA_ERR_UNSUPPORTED, "contraction predicate needs single-letter M and N");
                    G.m_lo = tg.c.lo[lm];
                    G.n_lo = tg.c.lo[ln];
                }
            }
            CtTuple T;
            T.a_base = tg.a.base;
            T.b_base = tg.b.base;
            T.K = tg.k.ext;
            T.a_sm = tg.m.str[0];
            T.a_sk = tg.k.str[0];
            T.a_sb = tg.bt.str[0];
            T.b_sk = tg.k.str[1];
            T.b_sn = tg.n.str[1];
            T.b_sb = tg.bt.str[1];
            tuples.push_back(T);
        }
        G.t1 = (int32_t)tuples.size();
        int32_t gid = (int32_t)groups.size();
        groups.push_back(G);
        gtiles.push_back({gid, G});
    }
    // 64-wide output tiles, or 32-wide when the 64-wide ones would leave SMs idle
    int64_t n64 = 0;
    for (auto &g : gtiles) n64 += g.second.nb * ((g.second.M + 63) / 64) * ((g.second.N + 63) / 64);
    const int tsz = n64 < 2 * (int64_t)c->num_sms ? 32 : 64;
    for (auto &g : gtiles)
        for (int64_t bb = 0; bb < g.second.nb; bb++)
            for (int64_t n0 = 0; n0 < g.second.N; n0 += tsz)
                for (int64_t m0 = 0; m0 < g.second.M; m0 += tsz)
                    tiles.push_back(CtTile{g.first, (int32_t)bb, (int32_t)m0, (int32_t)n0});
    ea_status cs = check_simt_plan(groups.data(), groups.size(), tuples.data(), tuples.size(), rel_elems(j.in[0]),
                                   rel_elems(j.in[1]), rel_elems(j.out));
    if (cs) return cs;
    Blob b;
    size_t og = b.add_vec(groups), ou = b.add_vec(tuples), ot = b.add_vec(tiles);
    ea_status s = upload(b, st, p);
    if (s) return s;
    p->kind = kSimt;
    CtParams &q = p->ct;
    q.groups = (const CtGroup *)(p->dev + og);
    q.tuples = (const CtTuple *)(p->dev + ou);
    q.tiles = (const CtTile *)(p->dev + ot);
    q.ntiles = (int64_t)tiles.size();
    q.a = j.in[0]->arena;
    q.b = j.in[1]->arena;
    q.c = j.out->arena;
    q.a_elems = rel_elems(j.in[0]);
    q.b_elems = rel_elems(j.in[1]);
    q.c_elems = rel_elems(j.out);
    q.err = c->err;
    q.a_dtype = j.in[0]->dtype;
    q.b_dtype = j.in[1]->dtype;
    q.c_dtype = j.out->dtype;
    q.scale = j.scale;
    q.pred_mode = mode;
    q.tile = tsz;
    // small groups of fp32 blocks: every tuple of a group at once (split)
    bool split = tsz == 32 && q.a_dtype == EA_F32 && q.b_dtype == EA_F32;
    for (const CtGroup &G : groups) split = split && G.t1 - G.t0 <= 4;
    for (const CtTuple &T : tuples) split = split && T.K <= 64;
    q.split = split ? 1 : 0;
    return EA_OK;
}

// tcgen05 path: bf16 operands whose blocks TMA can tile.  Returns
// EA_ERR_UNSUPPORTED (no message) when the SIMT kernel has to run instead.
struct TcOp {
    int64_t base, M, K, nb, s_m, s_k, s_b;  // viewed as [nb][M][K] (M = N for operand B)
    const ea_relation_s *rel;
};

static int64_t outer_stride(const TcOp &o, int mn) {
    // stride of the non-contiguous dimension of a 2-D tile, packed if extent 1
    if (!mn) return o.s_m ? o.s_m : o.K;
    return o.s_k ? o.s_k : o.M;
}

static ea_status build_tc(JoinCtx &j, const ContractionViews &cv, DevCtx *c, cudaStream_t st, DevPlan *p) {
    if (j.in[0]->dtype != EA_BF16 || j.in[1]->dtype != EA_BF16) return EA_ERR_UNSUPPORTED;
    if (!c->encode) return EA_ERR_UNSUPPORTED;
    int kpred = 0;
    int mode = pred_mode_of(j, cv, &kpred);
    if (mode < 0) return EA_ERR_UNSUPPORTED;
    const size_t es = 2, esc = elem_size(j.out->dtype);
    struct GroupGeom {
        int64_t c_base, M, N, nb, c_sm, c_sb, m_lo, n_lo, r_lo, e_lo;
        int64_t t0, t1;
    };
    std::vector<GroupGeom> gg;
    std::vector<std::pair<TcOp, TcOp>> tg_ops;
    bool swap = false;
    int a_mn = -1, b_mn = -1;
    int64_t maxN = 0;
    // ---- pass 1: geometry of every tuple; roles and majorness must agree
    for (size_t g = 0; g < j.wl.groups.size(); g++) {
        GroupGeom G{};
        G.t0 = (int64_t)tg_ops.size();
        for (int64_t t = j.wl.grp_ptr[g]; t < j.wl.grp_ptr[g + 1]; t++) {
            TupleGeom tg;
            if (tuple_geom(j, cv, (int64_t)g, t, &tg)) return EA_ERR_UNSUPPORTED;
            if (tg.k.ext == 0) return EA_ERR_UNSUPPORTED;
            TcOp A{tg.a.base, tg.m.ext, tg.k.ext, tg.bt.ext, tg.m.str[0], tg.k.str[0], tg.bt.str[0], j.in[0]};
            TcOp B{tg.b.base, tg.n.ext, tg.k.ext, tg.bt.ext, tg.n.str[1], tg.k.str[1], tg.bt.str[1], j.in[1]};
            int64_t M = tg.m.ext, N = tg.n.ext, c_sm = tg.m.str[2], c_sn = tg.n.str[2];
            int64_t m_lo = 0, n_lo = 0;
            if (mode) {
                int lm = mode == 1 ? j.pred_hi - 'a' : j.pred_lo - 'a';
                int ln = mode == 1 ? j.pred_lo - 'a' : j.pred_hi - 'a';
                if ((tg.m.single >= 0 && tg.m.single != lm) || (tg.n.single >= 0 && tg.n.single != ln) ||
                    (tg.m.single < 0 && tg.m.ext > 1) || (tg.n.single < 0 && tg.n.ext > 1))
                    return EA_ERR_UNSUPPORTED;
                m_lo = tg.c.lo[lm];
                n_lo = tg.c.lo[ln];
            }
            bool sw = !(c_sn == 1 || N == 1);
            if (sw && !(c_sm == 1 || M == 1)) return EA_ERR_UNSUPPORTED;
            if (tg_ops.empty()) swap = sw;
            if (sw != swap) return EA_ERR_UNSUPPORTED;
            if (swap) {
                std::swap(A, B);
                std::swap(M, N);
                std::swap(c_sm, c_sn);
                std::swap(m_lo, n_lo);
            }
            auto major = [](const TcOp &o) -> int {
                if (o.s_k == 1 || o.K == 1) return 0;
                if (o.s_m == 1 || o.M == 1) return 1;
                return -1;
            };
            int am = major(A), bm = major(B);
            if (am < 0 || bm < 0) return EA_ERR_UNSUPPORTED;
            if (a_mn < 0) {
                a_mn = am;
                b_mn = bm;
            }
            if (am != a_mn || bm != b_mn) return EA_ERR_UNSUPPORTED;
            auto tma_ok = [&](const TcOp &o, int mn) {
                int64_t row = outer_stride(o, mn);
                int64_t bstr = o.nb > 1 ? o.s_b : row * (mn ? o.K : o.M);
                return al16(o.base, es) && al16(row, es) && al16(bstr, es);
            };
            if (!tma_ok(A, a_mn) || !tma_ok(B, b_mn)) return EA_ERR_UNSUPPORTED;
            int64_t crow = c_sm ? c_sm : N;
            int64_t cb = A.nb > 1 ? tg.bt.str[2] : crow * M;
            if (!al16(tg.c.base, esc) || !al16(crow, esc) || !al16(cb, esc)) return EA_ERR_UNSUPPORTED;
            int64_t r_lo = 0, e_lo = 0;
            if (j.epi_map == EA_MAP_ROPE) {
                // rows: the position letter; columns: the output's last letter
                const int lr = j.rope_pos - 'a', le = j.sp.out.back() - 'a';
                if (swap || (tg.m.single != lr && M > 1) || (tg.n.single != le && N > 1)) return EA_ERR_UNSUPPORTED;
                r_lo = tg.c.lo[lr];
                e_lo = tg.c.lo[le];
            }
            if (j.row_rms) {
                // rows: the row letter, global index = the row_rms element (a rank-1 arena is dense)
                const int lr = j.row_letter - 'a';
                if (swap || (tg.m.single != lr && M > 1)) return EA_ERR_UNSUPPORTED;
                if (j.epi_map == EA_MAP_ROPE && j.rope_pos != j.row_letter) return EA_ERR_UNSUPPORTED;
                r_lo = tg.c.lo[lr];
            }
            if (t == j.wl.grp_ptr[g]) {
                G.r_lo = r_lo;
                G.e_lo = e_lo;
                G.c_base = tg.c.base;
                G.M = M;
                G.N = N;
                G.nb = A.nb;
                G.c_sm = crow;
                G.c_sb = cb;
                G.m_lo = m_lo;
                G.n_lo = n_lo;
            }
            tg_ops.push_back({A, B});
            maxN = std::max(maxN, N);
        }
        G.t1 = (int64_t)tg_ops.size();
        gg.push_back(G);
    }
    if (tg_ops.empty()) return EA_ERR_UNSUPPORTED;
    const int bn = maxN <= 128 ? 128 : 256;
    if (mode && swap) mode = 3 - mode;  // the mask is stated in the swapped roles
    // CTA pairs (one 256-row MMA over two SMs, each loading half of the B
    // tile) when there are enough tiles to keep every SM busy in pairs.
    int64_t est_tiles = 0;
    for (const GroupGeom &G : gg) est_tiles += G.nb * ((G.M + 127) / 128) * ((G.N + bn - 1) / bn);
    const int cl = est_tiles >= 2 * (int64_t)c->num_sms ? 2 : 1;
    // ---- pass 2: tensor maps, tuples, tiles
    std::vector<CUtensorMap> maps;
    struct Rast {
        int32_t gid;
        int64_t nb, nm, nn, band;
        std::vector<int32_t> key;   // M, batch count, first row, the A tensor map of each tuple
        std::vector<int32_t> ckey;  // N, batch count, first column, the B tensor map of each tuple
    };
    std::vector<Rast> rast;
    std::vector<TcGroup> groups;
    std::vector<TcTuple> tuples;
    std::vector<TcTile> tiles;
    std::unordered_map<int64_t, int32_t> cache_a, cache_b;
    auto op_map = [&](const TcOp &o, int mn, int box_rows, std::unordered_map<int64_t, int32_t> &cache,
                      int32_t *id) -> ea_status {
        auto it = cache.find(o.base);
        if (it != cache.end()) {
            *id = it->second;
            return EA_OK;
        }
        {
            const int64_t e[3] = {o.M, o.K, o.nb}, st3[3] = {o.s_m, o.s_k, o.s_b};
            ea_status cs = check_block(o.base, 3, e, st3, rel_elems(o.rel), "contraction operand block", maps.size());
            if (cs) return cs;
        }
        CUtensorMap m;
        int64_t row = outer_stride(o, mn);
        int64_t bstr = o.nb > 1 ? o.s_b : row * (mn ? o.K : o.M);
        const void *ptr = o.rel->arena + o.base * es;
        ea_status s = !mn ? encode_map(c, &m, EA_BF16, ptr, o.K, o.M, o.nb, row * es, bstr * es, 64, box_rows)
                          : encode_map(c, &m, EA_BF16, ptr, o.M, o.K, o.nb, row * es, bstr * es, 64, 64);
        if (s) return s;
        *id = (int32_t)maps.size();
        maps.push_back(m);
        cache[o.base] = *id;
        return EA_OK;
    };
    for (size_t g = 0; g < gg.size(); g++) {
        const GroupGeom &G = gg[g];
        TcGroup TG;
        memset(&TG, 0, sizeof TG);
        TG.t0 = (int32_t)tuples.size();
        int64_t k_total = 0;  // the group's contracted extent (all its tuples)
        TG.m_lo = G.m_lo;
        TG.n_lo = G.n_lo;
        bool empty = G.M == 0 || G.N == 0 || G.nb == 0;
        for (int64_t t = G.t0; t < G.t1 && !empty; t++) {
            const TcOp &A = tg_ops[t].first, &B = tg_ops[t].second;
            TcTuple T;
            memset(&T, 0, sizeof T);
            ea_status s = op_map(A, a_mn, 128, cache_a, &T.a_map);
            if (s) return s;
            s = op_map(B, b_mn, bn / cl, cache_b, &T.b_map);
            if (s) return s;
            T.kchunks = (int32_t)((A.K + 63) / 64);
            k_total += A.K;
            tuples.push_back(T);
        }
        TG.t1 = (int32_t)tuples.size();
        TG.n_ext = (int32_t)G.N;
        TG.m_ext = (int32_t)G.M;
        if (empty) continue;
        // the stored output: the planned one, or its pairs halved (one cell per pair)
        const int64_t h = j.epi_pair ? 2 : 1;
        if (j.epi_pair && (G.N % 2 || G.c_base % 2 || G.c_sm % 2 || G.c_sb % 2 || !al16(G.c_base / 2, esc) ||
                           !al16(G.c_sm / 2, esc) || !al16(G.c_sb / 2, esc)))
            return EA_ERR_UNSUPPORTED;
        TG.e_base = G.c_base / h;
        TG.e_sm = G.c_sm / h;
        TG.e_sb = G.c_sb / h;
        TG.r_lo = G.r_lo;
        TG.c_lo = G.e_lo;
        {
            // the stored output block, the residual block read by an ADD
            // epilogue (same geometry) and the rows of the row scale
            const int64_t e[3] = {G.N / h, G.M, G.nb}, st3[3] = {1, G.c_sm / h, G.c_sb / h};
            ea_status cs = check_block(G.c_base / h, 3, e, st3, rel_elems(j.user_out), "contraction output block", g);
            if (!cs && j.epi_in) cs = check_block(TG.e_base, 3, e, st3, rel_elems(j.epi_in), "epilogue input block", g);
            const int64_t re[1] = {G.M}, rs[1] = {1};
            if (!cs && j.row_rms) cs = check_block(G.r_lo, 1, re, rs, rel_elems(j.row_rms), "row-scale block", g);
            if (cs) return cs;
        }
        CUtensorMap m;
        const void *cptr = j.out->arena + (G.c_base / h) * esc;
        ea_status s = encode_map(c, &m, j.out->dtype, cptr, G.N / h, G.M, G.nb, (G.c_sm / h) * esc,
                                 (G.c_sb / h) * esc, (uint32_t)(128 / esc), 128);
        if (s) return s;
        TG.out_map = (int32_t)maps.size();
        maps.push_back(m);
        int32_t gid = (int32_t)groups.size();
        groups.push_back(TG);
        // The group's raster: bands of `band` m-tiles (about 32 MiB of A rows:
        // B is re-read once per band, and a larger band no longer stays in
        // L2 beside the B columns in flight -- FFN gate+up, 8192 tokens: DRAM
        // reads 907 MB with bands of 16, 668 MB with 32, 1271 MB with 64);
        // the tiles are laid out below, once every group is known.
        const int64_t a_row_bytes = 128 * std::max<int64_t>(1, k_total) * (int64_t)elem_size(j.in[0]->dtype);
        Rast R;
        R.gid = gid;
        R.nb = G.nb;
        R.nm = (G.M + 127) / 128;
        R.nn = (G.N + bn - 1) / bn;
        R.band = std::max<int64_t>(8, std::min<int64_t>(64, ((32ll << 20) / a_row_bytes) & ~1ll));
        R.key.assign(1, (int32_t)G.M);
        R.key.push_back((int32_t)G.nb);
        R.key.push_back((int32_t)G.m_lo);
        for (int32_t t = TG.t0; t < TG.t1; t++) R.key.push_back(tuples[t].a_map);
        R.ckey.assign(1, (int32_t)G.N);
        R.ckey.push_back((int32_t)G.nb);
        R.ckey.push_back((int32_t)G.n_lo);
        for (int32_t t = TG.t0; t < TG.t1; t++) R.ckey.push_back(tuples[t].b_map);
        rast.push_back(R);
    }
    // Grouped raster over the grid of groups: a group's row key is what it
    // reads of A (its tuples' A blocks), its column key what it reads of B.
    // Row keys are taken in order into bands of about 32 MiB of A rows
    // (whole row keys while they fit, a long one cut into several bands);
    // each band is swept across every column key's n-tiles with m fastest,
    // so the tiles in flight at once share a band of A rows and a few B
    // columns that stay in L2: A is read from DRAM about once, and B once per
    // band instead of once per row key (FFN gate+up of the block, x in 8 row
    // blocks: W read 4 times, not 8).  With CTA pairs the tiles come in pairs
    // of the same n-tile (consecutive m-tiles of one row key; a segment with
    // an odd count gets a padding tile past the block's rows).
    {
        std::map<std::vector<int32_t>, int32_t> row_of, col_of;
        std::vector<std::vector<size_t>> rows_g;  // row key -> its groups
        std::vector<int64_t> col_nn;              // column key -> n-tiles
        std::vector<int32_t> gcol(rast.size());
        for (size_t r = 0; r < rast.size(); r++) {
            auto ir = row_of.find(rast[r].key);
            if (ir == row_of.end()) {
                row_of.emplace(rast[r].key, (int32_t)rows_g.size());
                rows_g.push_back(std::vector<size_t>(1, r));
            } else {
                rows_g[ir->second].push_back(r);
            }
            auto ic = col_of.find(rast[r].ckey);
            if (ic == col_of.end()) {
                gcol[r] = (int32_t)col_nn.size();
                col_of.emplace(rast[r].ckey, gcol[r]);
                col_nn.push_back(rast[r].nn);
            } else {
                gcol[r] = ic->second;
            }
        }
        struct Seg {
            int32_t row;     // row key
            int64_t m0, m1;  // its m-tiles [m0, m1)
        };
        std::vector<std::vector<Seg>> bands;
        {
            std::vector<Seg> cur;
            int64_t used = 0, budget = 0;
            for (size_t rk = 0; rk < rows_g.size(); rk++) {
                const Rast &R = rast[rows_g[rk][0]];
                for (int64_t m0 = 0; m0 < R.nm;) {
                    if (cur.empty()) budget = R.band;
                    int64_t take = std::min(R.nm - m0, budget - used);
                    // with CTA pairs a segment that stops inside the row key has
                    // an even count (its padding tile would be a real tile)
                    if (cl == 2 && m0 + take < R.nm) take &= ~1ll;
                    if (take <= 0) {
                        bands.push_back(cur);
                        cur.clear();
                        used = 0;
                        continue;
                    }
                    cur.push_back(Seg{(int32_t)rk, m0, m0 + take});
                    used += take;
                    m0 += take;
                }
            }
            if (!cur.empty()) bands.push_back(cur);
        }
        // (row key, column key) -> the group; per band, the column keys its
        // groups use, in order of first appearance
        const int64_t ncol = (int64_t)col_nn.size();
        std::unordered_map<int64_t, std::vector<size_t>> at;
        for (size_t rk = 0; rk < rows_g.size(); rk++)
            for (size_t r : rows_g[rk]) at[(int64_t)rk * ncol + gcol[r]].push_back(r);
        int64_t nb_max = 0;
        for (const Rast &R : rast) nb_max = std::max(nb_max, R.nb);
        std::vector<char> seen(col_nn.size(), 0);
        std::vector<int32_t> cols;
        for (int64_t bb = 0; bb < nb_max; bb++)
            for (const std::vector<Seg> &band : bands) {
                cols.clear();
                for (const Seg &sg : band)
                    for (size_t r : rows_g[sg.row])
                        if (bb < rast[r].nb && !seen[gcol[r]]) {
                            seen[gcol[r]] = 1;
                            cols.push_back(gcol[r]);
                        }
                for (int32_t ck : cols) {
                    seen[ck] = 0;
                    for (int64_t ni = 0; ni < col_nn[ck]; ni++)
                        for (const Seg &sg : band) {
                            const auto it = at.find((int64_t)sg.row * ncol + ck);
                            if (it == at.end()) continue;
                            for (size_t r : it->second) {
                                if (bb >= rast[r].nb) continue;
                                const int32_t gid = rast[r].gid;
                                for (int64_t mi = sg.m0; mi < sg.m1; mi++)
                                    tiles.push_back(TcTile{gid, (int32_t)bb, (int32_t)(mi * 128), (int32_t)(ni * bn)});
                                if (cl == 2 && ((sg.m1 - sg.m0) & 1))
                                    tiles.push_back(TcTile{gid, (int32_t)bb, (int32_t)(sg.m1 * 128), (int32_t)(ni * bn)});
                            }
                        }
                }
            }
        // every group's tiles are laid out exactly once (padding tiles aside)
        std::vector<int64_t> got(groups.size(), 0);
        for (const TcTile &T : tiles)
            if (T.m0 < groups[T.group].m_ext) got[T.group]++;
        for (const Rast &R : rast)
            if (got[R.gid] != R.nb * R.nm * R.nn)
                return set_error(EA_ERR_UNSUPPORTED, "contraction: raster covers group %d with %lld of %lld tiles",
                                 R.gid, (long long)got[R.gid], (long long)(R.nb * R.nm * R.nn));
    }
    if (tiles.size() > (size_t)INT32_MAX) return EA_ERR_UNSUPPORTED;
    if (cl == 2) {
        // a CTA pair computes tiles 2u and 2u + 1 as one 256-row MMA tile
        if (tiles.size() % 2) return set_error(EA_ERR_UNSUPPORTED, "contraction: odd tile count for CTA pairs");
        for (size_t u = 0; u < tiles.size(); u += 2) {
            const TcTile &t0 = tiles[u], &t1 = tiles[u + 1];
            if (t0.group != t1.group || t0.batch != t1.batch || t0.n0 != t1.n0 || t1.m0 != t0.m0 + 128)
                return set_error(EA_ERR_UNSUPPORTED, "contraction: tiles of a CTA pair are not M-adjacent");
        }
    }
    Blob b;
    size_t om = b.add(maps.data(), maps.size() * sizeof(CUtensorMap), 128);
    size_t og = b.add_vec(groups), ou = b.add_vec(tuples), ot = b.add_vec(tiles);
    ea_status s = upload(b, st, p);
    if (s) return s;
    p->kind = kTc;
    TcParams &q = p->tc;
    q.tmaps = p->dev + om;
    q.groups = (const TcGroup *)(p->dev + og);
    q.tuples = (const TcTuple *)(p->dev + ou);
    q.tiles = (const TcTile *)(p->dev + ot);
    q.ntiles = (int32_t)tiles.size();
    q.a_mn_major = a_mn;
    q.b_mn_major = b_mn;
    q.out_f32 = j.out->dtype == EA_F32;
    q.scale = j.scale;
    q.pred_mode = mode;
    q.bn = bn;
    q.cluster = cl;
    q.epi = j.epi_map == EA_MAP_ADD ? 1 : j.epi_map == EA_MAP_SILU_MUL ? 2 : j.epi_map == EA_MAP_ROPE ? 3 : 0;
    q.epi_in = j.epi_in ? j.epi_in->arena : nullptr;
    q.row_rms = j.row_rms ? (const float *)j.row_rms->arena : nullptr;
    q.epi_elems = j.epi_in ? rel_elems(j.epi_in) : 0;
    q.rms_elems = j.row_rms ? rel_elems(j.row_rms) : 0;
    q.eps = j.eps;
    q.rope_table = j.rope_table;
    q.rope_npos = j.rope_npos;
    q.rope_half = (int32_t)((j.rope_dim ? j.rope_dim : j.lt.t[j.sp.out.back() - 'a'].extent) / 2);
    q.rope_pm = j.rope_layout;
    q.err = c->err;
    return EA_OK;
}

// ------------------------------------------------------------ launching

ea_status launch_plan(DevPlan *p, DevCtx *c, cudaStream_t st) {
    ea_status s = plan_ready_on(p, st);
    if (s) return s;
    cudaError_t e = cudaSuccess;
    t_last = LastPlan{};
    t_last.kind = p->kind;
    t_last.groups = p->n_groups;
    t_last.tuples = p->n_tuples;
    switch (p->kind) {
    case kExchange: t_last.tiles = p->nxtiles; t_last.launches = p->nxtiles > 0; break;
    case kEwise: t_last.tiles = p->ew.ntiles; t_last.launches = p->ew.has_vec + p->ew.has_scalar; break;
    case kRowReduce: t_last.tiles = p->rr.ntiles; t_last.launches = p->rr.ntiles > 0; break;
    case kSimt: t_last.tiles = p->ct.ntiles; t_last.launches = p->ct.ntiles > 0; break;
    case kTc:
        t_last.tiles = p->tc.ntiles;
        t_last.launches = p->tc.ntiles > 0;
        t_last.cluster = p->tc.cluster;
        break;
    case kAttn: t_last.tiles = p->n_groups; t_last.launches = p->at.ncta > 0; break;
    case kExchangeAgg: t_last.tiles = p->nxtiles; t_last.launches = p->nxtiles > 0; break;
    }
    switch (p->kind) {
    case kExchange:
        if (p->nxtiles)
            e = launch_exchange(p->segs, p->xtiles, p->nxtiles, p->xsrc, p->xdst, p->esize, c->num_sms, st,
                                p->xsrc_elems, p->xdst_elems, c->err);
        break;
    case kEwise:
        p->ew.err = c->err;
        if (p->ew.ntiles) e = launch_ewise(p->ew, c->num_sms, st);
        break;
    case kRowReduce:
        p->rr.err = c->err;
        if (p->rr.ntiles) e = launch_rowreduce(p->rr, c->num_sms, st);
        break;
    case kSimt:
        p->ct.err = c->err;
        if (p->ct.ntiles) e = launch_contract_simt(p->ct, st);
        break;
    case kTc:
        p->tc.err = c->err;
        if (p->tc.ntiles) e = launch_contract_tc(p->tc, c->num_sms, st);
        break;
    case kAttn:
        p->at.err = c->err;
        if (p->at.ncta) e = launch_attention(p->at, st);
        break;
    case kExchangeAgg:
        if (p->nxtiles)
            e = launch_exchange_agg(p->segs, p->xtiles, p->nxtiles, p->xsrc, p->xdst, p->xdtype, p->xagg, p->xcopies,
                                    p->xcopy_stride, c->num_sms, st, p->xsrc_elems, p->xdst_elems, c->err);
        break;
    }
    if (e != cudaSuccess) return cuda_error(e, "kernel launch");
    return EA_OK;
}

static bool same_tiling(const ea_relation_s *r, int d, const Tiling &t) { return r->bounds[d] == t.b; }

// Partials: the copy letter leads the output and joins with every tuple, so
// group (q, b) lists all the function specifications of output block b; it
// keeps only the q-th (canonical order), whose output block copy q receives.
static ea_status keep_copy_tuples(JoinCtx &j) {
    const WorkList &w = j.wl;
    const int n_in = j.sp.n_in;
    const int64_t m = j.lt.t[j.copy_letter - 'a'].extent;
    int64_t per_copy = 1;  // output blocks per copy
    for (size_t d = 1; d < j.sp.out.size(); d++) per_copy *= j.lt.t[j.sp.out[d] - 'a'].nblocks();
    WorkList nw;
    nw.grp_ptr.push_back(0);
    for (size_t g = 0; g < w.groups.size(); g++) {
        const int64_t q = w.groups[g] / per_copy;
        const int64_t nt = w.grp_ptr[g + 1] - w.grp_ptr[g];
        if (nt != m)
            return set_error(EA_ERR_SHAPE, "partials: an output block has %lld function specifications, not %lld",
                             (long long)nt, (long long)m);
        const int64_t t = w.grp_ptr[g] + q;
        nw.groups.push_back(w.groups[g]);
        for (int k = 0; k < n_in; k++) nw.tuples.push_back(w.tuples[t * n_in + k]);
        for (int l = 0; l < 26; l++) nw.tuple_iv.push_back(w.tuple_iv[t * 26 + l]);
        nw.grp_ptr.push_back((int64_t)nw.groups.size());
    }
    j.wl.groups.swap(nw.groups);
    j.wl.grp_ptr.swap(nw.grp_ptr);
    j.wl.tuples.swap(nw.tuples);
    j.wl.tuple_iv.swap(nw.tuple_iv);
    return EA_OK;
}

}  // namespace ea

using namespace ea;

// =================================================================== C ABI

extern "C" {

ea_status ea_exchange(ea_relation in, const ea_dim_part *new_parts, void *stream, ea_relation *out) {
    set_error(EA_OK, "");
    if (!in || !out) return set_error(EA_ERR_ARG, "ea_exchange: NULL argument");
    std::lock_guard<std::mutex> lk(g_mu);
    ea_status s = EA_OK;
    Tiling src[kMaxRank], dst[kMaxRank];
    for (int d = 0; d < in->rank; d++) {
        src[d].extent = in->dims[d];
        src[d].b = in->bounds[d];
    }
    if (new_parts) {
        for (int d = 0; d < in->rank; d++) {
            s = make_tiling(in->dims[d], new_parts[d].nblocks, new_parts[d].bounds, &dst[d]);
            if (s) return s;
        }
    } else {
        if (!*out) return set_error(EA_ERR_ARG, "ea_exchange: need new_parts or an output relation");
        for (int d = 0; d < in->rank; d++) {
            dst[d].extent = (*out)->dims[d];
            dst[d].b = (*out)->bounds[d];
        }
    }
    ea_relation o = *out;
    if (o) {
        if (o->dtype != in->dtype || o->rank != in->rank) return set_error(EA_ERR_SHAPE, "ea_exchange: output dtype/rank differ");
        for (int d = 0; d < in->rank; d++) {
            if (o->dims[d] != in->dims[d]) return set_error(EA_ERR_SHAPE, "ea_exchange: output extents differ");
            if (!same_tiling(o, d, dst[d])) return set_error(EA_ERR_PARTITION, "ea_exchange: output tiling differs from new_parts");
        }
        if (o->bytes && in->bytes && o->arena < in->arena + in->bytes && in->arena < o->arena + o->bytes)
            return set_error(EA_ERR_ARG, "ea_exchange: input and output arenas overlap");
    } else {
        ea_dim_part parts[kMaxRank];
        for (int d = 0; d < in->rank; d++) parts[d] = ea_dim_part{dst[d].nblocks(), 0, dst[d].b.data()};
        s = ea_relation_create((ea_dtype)in->dtype, in->rank, in->dims, parts, nullptr, &o);
        if (s) return s;
    }
    DevCtx *c;
    s = get_ctx(&c);
    if (s) {
        if (!*out) ea_relation_destroy(o);
        return s;
    }
    Key k;
    k.str("X");
    k.rel(in);
    k.rel(o);
    cudaStream_t st = (cudaStream_t)stream;
    DevPlan *p;
    auto it = g_cache.find(k.s);
    if (it != g_cache.end()) {
        p = it->second;
    } else {
        ExchangePlan xp;
        s = plan_exchange(in->rank, in->dims, src, dst, (int)elem_size(in->dtype), &xp);
        if (!s) s = check_exchange_plan(xp.segs.data(), xp.segs.size(), xp.tiles.data(), xp.tiles.size(), rel_elems(in),
                                        rel_elems(o), 1, 0);
        if (!s) {
            p = new DevPlan();
            Blob b;
            size_t os = b.add_vec(xp.segs), ot = b.add_vec(xp.tiles);
            s = upload(b, st, p);
            if (!s) {
                p->kind = kExchange;
                p->segs = (XSeg *)(p->dev + os);
                p->xtiles = (XTile *)(p->dev + ot);
                p->nxtiles = (int64_t)xp.tiles.size();
                p->xsrc = in->arena;
                p->xdst = o->arena;
                p->xsrc_elems = rel_elems(in);
                p->xdst_elems = rel_elems(o);
                p->esize = (int)elem_size(in->dtype);
                g_cache[k.s] = p;
            } else {
                free_plan(p);
            }
        }
        if (s) {
            if (!*out) ea_relation_destroy(o);
            return s;
        }
    }
    s = launch_plan(p, c, st);
    if (s) {
        if (!*out) ea_relation_destroy(o);
        return s;
    }
    *out = o;
    return EA_OK;
}

ea_status ea_exchange_agg(ea_relation in, ea_agg agg, const ea_dim_part *new_parts, void *stream, ea_relation *out) {
    set_error(EA_OK, "");
    if (!in || !out) return set_error(EA_ERR_ARG, "ea_exchange_agg: NULL argument");
    if (agg != EA_AGG_SUM && agg != EA_AGG_MAX) return set_error(EA_ERR_ARG, "ea_exchange_agg: agg must be SUM or MAX");
    if (in->rank < 2) return set_error(EA_ERR_SHAPE, "ea_exchange_agg: the input needs a copy dimension and one more");
    const int rank = in->rank - 1;
    const int64_t m = in->dims[0];
    if ((int64_t)in->bounds[0].size() != m + 1)
        return set_error(EA_ERR_PARTITION, "ea_exchange_agg: the copy dimension must be tiled into unit blocks");
    std::lock_guard<std::mutex> lk(g_mu);
    ea_status s = EA_OK;
    Tiling src[kMaxRank], dst[kMaxRank];
    int64_t dims[kMaxRank];
    for (int d = 0; d < rank; d++) {
        dims[d] = in->dims[d + 1];
        src[d].extent = dims[d];
        src[d].b = in->bounds[d + 1];
    }
    ea_relation o = *out;
    if (new_parts) {
        for (int d = 0; d < rank; d++) {
            s = make_tiling(dims[d], new_parts[d].nblocks, new_parts[d].bounds, &dst[d]);
            if (s) return s;
        }
    } else {
        if (!o) return set_error(EA_ERR_ARG, "ea_exchange_agg: need new_parts or an output relation");
        if (o->rank != rank) return set_error(EA_ERR_SHAPE, "ea_exchange_agg: output rank");
        for (int d = 0; d < rank; d++) {
            dst[d].extent = o->dims[d];
            dst[d].b = o->bounds[d];
        }
    }
    if (o) {
        if (o->dtype != in->dtype || o->rank != rank) return set_error(EA_ERR_SHAPE, "ea_exchange_agg: output dtype/rank");
        for (int d = 0; d < rank; d++) {
            if (o->dims[d] != dims[d]) return set_error(EA_ERR_SHAPE, "ea_exchange_agg: output extents differ");
            if (!same_tiling(o, d, dst[d])) return set_error(EA_ERR_PARTITION, "ea_exchange_agg: output tiling differs");
        }
        if (o->bytes && in->bytes && o->arena < in->arena + in->bytes && in->arena < o->arena + o->bytes)
            return set_error(EA_ERR_ARG, "ea_exchange_agg: input and output arenas overlap");
    } else {
        ea_dim_part parts[kMaxRank];
        for (int d = 0; d < rank; d++) parts[d] = ea_dim_part{dst[d].nblocks(), 0, dst[d].b.data()};
        s = ea_relation_create((ea_dtype)in->dtype, rank, dims, parts, nullptr, &o);
        if (s) return s;
    }
    DevCtx *c;
    s = get_ctx(&c);
    if (s) {
        if (!*out) ea_relation_destroy(o);
        return s;
    }
    Key k;
    k.str("XA");
    k.rel(in);
    k.rel(o);
    k.v((int)agg);
    cudaStream_t st = (cudaStream_t)stream;
    DevPlan *p;
    auto it = g_cache.find(k.s);
    if (it != g_cache.end()) {
        p = it->second;
    } else {
        ExchangePlan xp;
        s = plan_exchange(rank, dims, src, dst, (int)elem_size(in->dtype), &xp);
        // copy q lies q * copy_stride elements on: 16-byte chunks stay aligned
        // in every copy only if that stride is a multiple of 16 bytes
        if (((in->blk_off.back() / m) * (int64_t)elem_size(in->dtype)) % 16)
            for (XSeg &g : xp.segs) g.vec = 0;
        if (!s) s = check_exchange_plan(xp.segs.data(), xp.segs.size(), xp.tiles.data(), xp.tiles.size(), rel_elems(in),
                                        rel_elems(o), m, in->blk_off.back() / m);
        if (!s) {
            p = new DevPlan();
            Blob b;
            size_t os = b.add_vec(xp.segs), ot = b.add_vec(xp.tiles);
            s = upload(b, st, p);
            if (!s) {
                p->kind = kExchangeAgg;
                p->segs = (XSeg *)(p->dev + os);
                p->xtiles = (XTile *)(p->dev + ot);
                p->nxtiles = (int64_t)xp.tiles.size();
                p->xsrc = in->arena;
                p->xdst = o->arena;
                p->xsrc_elems = rel_elems(in);
                p->xdst_elems = rel_elems(o);
                p->esize = (int)elem_size(in->dtype);
                p->xdtype = in->dtype;
                p->xagg = agg;
                p->xcopies = (int)m;
                p->xcopy_stride = in->blk_off.back() / m;
                g_cache[k.s] = p;
            } else {
                free_plan(p);
            }
        }
        if (s) {
            if (!*out) ea_relation_destroy(o);
            return s;
        }
    }
    s = launch_plan(p, c, st);
    if (s) {
        if (!*out) ea_relation_destroy(o);
        return s;
    }
    *out = o;
    return EA_OK;
}

ea_status ea_joinagg_run(const char *spec, const ea_relation *inputs, int n_inputs, const ea_index_part *parts,
                         int n_parts, ea_agg agg, ea_map map, const ea_opts *opts, void *stream, ea_relation *out) {
    set_error(EA_OK, "");
    if (!spec || !inputs || !out) return set_error(EA_ERR_ARG, "ea_joinagg_run: NULL argument");
    if (n_parts < 0 || (n_parts > 0 && !parts)) return set_error(EA_ERR_ARG, "ea_joinagg_run: bad parts");
    if (agg < EA_AGG_NONE || agg > EA_AGG_MAX_SUMEXP) return set_error(EA_ERR_ARG, "ea_joinagg_run: unknown agg %d", agg);
    if (map < EA_MAP_PRODUCT || map > EA_MAP_ROPE) return set_error(EA_ERR_ARG, "ea_joinagg_run: unknown map %d", map);
    std::lock_guard<std::mutex> lk(g_mu);
    JoinCtx j;
    ea_status s = parse_spec(spec, &j.sp);
    if (s) return s;
    if (n_inputs != j.sp.n_in) return set_error(EA_ERR_ARG, "spec \"%s\" has %d inputs, got %d", spec, j.sp.n_in, n_inputs);
    static const int arity[] = {-2, 1, 2, 2, 2, 2, 1, 3, 3, 1};  // -2: two or three
    if ((arity[map] == -2 && n_inputs < 2) || (arity[map] > 0 && arity[map] != n_inputs))
        return set_error(EA_ERR_ARG, "map %d does not take %d inputs", map, n_inputs);
    for (int k = 0; k < n_inputs; k++) {
        if (!inputs[k]) return set_error(EA_ERR_ARG, "input %d is NULL", k);
        j.in[k] = inputs[k];
        if ((int)j.sp.term[k].size() != inputs[k]->rank)
            return set_error(EA_ERR_SHAPE, "input %d has rank %d but term \"%s\"", k, inputs[k]->rank,
                             j.sp.term[k].c_str());
    }
    ea_opts o{};
    if (opts) o = *opts;
    j.agg = agg;
    j.map = map;
    j.scale = o.scale == 0.0f ? 1.0f : o.scale;
    j.eps = o.eps;
    j.pred_lo = o.pred_lo;
    j.pred_hi = o.pred_hi;
    j.rope_table = o.rope_table;
    j.rope_npos = o.rope_npos;
    j.rope_layout = o.rope_layout;
    if (o.rope_layout != 0 && o.rope_layout != 1) return set_error(EA_ERR_ARG, "rope_layout must be 0 or 1");
    if (map == EA_MAP_ROPE && o.rope_layout != 0)
        return set_error(EA_ERR_UNSUPPORTED, "the elementwise ROPE join reads a position-major table (rope_layout 0)");
    j.rope_pos = o.rope_pos;
    j.rope_dim = o.rope_dim;
    j.simt_bf16 = o.simt_bf16 != 0;
    j.out2 = agg == EA_AGG_MAX_SUMEXP ? o.out2 : nullptr;
    if (agg == EA_AGG_MAX_SUMEXP && !j.out2) return set_error(EA_ERR_ARG, "MAX_SUMEXP needs opts->out2");
    // Letter tilings: from the inputs, which must agree; explicit parts must match.
    for (int k = 0; k < n_inputs; k++)
        for (int d = 0; d < inputs[k]->rank; d++) {
            char ch = j.sp.term[k][d];
            Tiling &t = j.lt.t[ch - 'a'];
            if (t.extent >= 0) {
                if (t.extent != inputs[k]->dims[d])
                    return set_error(EA_ERR_SHAPE, "letter '%c' has extents %lld and %lld", ch, (long long)t.extent,
                                     (long long)inputs[k]->dims[d]);
                if (t.b != inputs[k]->bounds[d])
                    return set_error(EA_ERR_PARTITION,
                                     "letter '%c' is tiled differently by two inputs; re-block one with ea_exchange", ch);
            } else {
                t.extent = inputs[k]->dims[d];
                t.b = inputs[k]->bounds[d];
            }
        }
    for (int i = 0; i < n_parts; i++) {
        char ch = parts[i].index;
        if (ch < 'a' || ch > 'z' || j.lt.t[ch - 'a'].extent < 0)
            return set_error(EA_ERR_SPEC, "partition for letter '%c' that the spec does not use", ch);
        Tiling t;
        s = make_tiling(j.lt.t[ch - 'a'].extent, parts[i].nblocks, parts[i].bounds, &t);
        if (s) return s;
        if (t.b != j.lt.t[ch - 'a'].b)
            return set_error(EA_ERR_PARTITION, "letter '%c': the inputs are not tiled as requested; re-block with ea_exchange",
                             ch);
    }
    if ((j.pred_lo != 0) != (j.pred_hi != 0)) return set_error(EA_ERR_ARG, "predicate needs two letters");
    if (j.pred_lo && (j.pred_lo < 'a' || j.pred_lo > 'z' || j.pred_hi < 'a' || j.pred_hi > 'z' ||
                      j.lt.t[j.pred_lo - 'a'].extent < 0 || j.lt.t[j.pred_hi - 'a'].extent < 0))
        return set_error(EA_ERR_SPEC, "predicate letters must be letters of the spec");
    if (map == EA_MAP_ROPE && (j.rope_pos < 'a' || j.rope_pos > 'z' || j.lt.t[j.rope_pos - 'a'].extent < 0))
        return set_error(EA_ERR_ARG, "ROPE needs rope_pos, a letter of the spec");
    if (map == EA_MAP_ROPE && j.rope_dim && j.rope_dim != j.lt.t[j.sp.out.back() - 'a'].extent)
        return set_error(EA_ERR_UNSUPPORTED, "the elementwise ROPE join takes pairs over the whole last letter");
    // Partials: the output gains a leading copy letter (unit blocks), and each
    // group keeps only its copy's function specification (see below).
    j.copy_letter = 0;
    if (o.partials) {
        if (!(map == EA_MAP_PRODUCT && agg == EA_AGG_SUM && n_inputs == 2))
            return set_error(EA_ERR_UNSUPPORTED, "partials need a contraction (SUM of PRODUCT, two inputs)");
        if (o.epi_map || o.row_rms || j.pred_lo)
            return set_error(EA_ERR_UNSUPPORTED, "partials do not combine with an epilogue, row_rms or a predicate");
        if (!*out) return set_error(EA_ERR_ARG, "partials need the output relation (its first extent is the copy count)");
        for (char ch = 'a'; ch <= 'z' && !j.copy_letter; ch++)
            if (j.lt.t[ch - 'a'].extent < 0) j.copy_letter = ch;
        if (!j.copy_letter) return set_error(EA_ERR_SPEC, "partials: no letter left for the copies");
        const ea_relation_s *ro = *out;
        const int64_t m = ro->rank > 0 ? ro->dims[0] : 0;
        if (ro->rank != (int)j.sp.out.size() + 1 || m < 1)
            return set_error(EA_ERR_SHAPE, "partials: the output needs a leading copy dimension");
        if ((int64_t)ro->bounds[0].size() != m + 1)
            return set_error(EA_ERR_PARTITION, "partials: the copy dimension must be tiled into unit blocks");
        Tiling tc;
        make_tiling(m, (int32_t)m, nullptr, &tc);
        j.lt.t[j.copy_letter - 'a'] = tc;
        j.sp.out.insert(j.sp.out.begin(), j.copy_letter);
    }
    // Output relation.
    int odt = o.out_dtype == 0 ? inputs[0]->dtype : o.out_dtype - 1;
    if (odt != EA_F32 && odt != EA_BF16) return set_error(EA_ERR_DTYPE, "unknown out_dtype %d", o.out_dtype);
    int64_t odims[kMaxRank];
    ea_dim_part oparts[kMaxRank];
    int orank = (int)j.sp.out.size();
    if (orank == 0) return set_error(EA_ERR_UNSUPPORTED, "a rank-0 output is not supported");
    for (int d = 0; d < orank; d++) {
        const Tiling &t = j.lt.t[j.sp.out[d] - 'a'];
        odims[d] = t.extent;
        oparts[d] = ea_dim_part{t.nblocks(), 0, t.b.data()};
    }
    ea_relation orel = *out;
    bool created = false;
    if (orel) {
        if (orel->rank != orank) return set_error(EA_ERR_SHAPE, "output relation has rank %d, spec wants %d", orel->rank, orank);
        for (int d = 0; d < orank; d++) {
            if (orel->dims[d] != odims[d]) return set_error(EA_ERR_SHAPE, "output extent mismatch in dim %d", d);
            if (!same_tiling(orel, d, j.lt.t[j.sp.out[d] - 'a']))
                return set_error(EA_ERR_PARTITION, "output relation is tiled differently from the output letters");
        }
        for (int k = 0; k < n_inputs; k++)
            if (orel->bytes && inputs[k]->bytes && orel->arena < inputs[k]->arena + inputs[k]->bytes &&
                inputs[k]->arena < orel->arena + orel->bytes && orel->arena != inputs[k]->arena)
                return set_error(EA_ERR_ARG, "output arena partially overlaps input %d", k);
    }
    // Row scale of a contraction.
    j.row_rms = o.row_rms;
    j.row_letter = 0;
    if (o.row_rms) {
        if (!(map == EA_MAP_PRODUCT && agg == EA_AGG_SUM && n_inputs == 2))
            return set_error(EA_ERR_UNSUPPORTED, "row_rms needs a contraction (SUM of PRODUCT, two inputs)");
        for (char ch : j.sp.out)
            if (j.sp.term[0].find(ch) != std::string::npos && j.sp.term[1].find(ch) == std::string::npos) {
                if (j.row_letter) return set_error(EA_ERR_UNSUPPORTED, "row_rms needs exactly one row letter");
                j.row_letter = ch;
            }
        if (!j.row_letter) return set_error(EA_ERR_SPEC, "row_rms: the output has no letter of input 0 only");
        const ea_relation_s *r = o.row_rms;
        const Tiling &tr = j.lt.t[j.row_letter - 'a'];
        if (r->rank != 1 || r->dtype != EA_F32) return set_error(EA_ERR_SHAPE, "row_rms must be a rank-1 f32 relation");
        if (r->dims[0] != tr.extent) return set_error(EA_ERR_SHAPE, "row_rms extent differs from letter '%c'", j.row_letter);
        if (r->bounds[0] != tr.b) return set_error(EA_ERR_PARTITION, "row_rms is tiled unlike letter '%c'", j.row_letter);
        if (j.pred_lo) return set_error(EA_ERR_UNSUPPORTED, "row_rms with a predicate is not supported");
    }
    // Epilogue join of a contraction.
    j.epi_map = o.epi_map;
    j.epi_in = o.epi_in;
    j.epi_pair = 0;
    if (o.epi_map != 0) {
        if (!(map == EA_MAP_PRODUCT && agg == EA_AGG_SUM && n_inputs == 2))
            return set_error(EA_ERR_UNSUPPORTED, "an epilogue join needs a contraction (SUM of PRODUCT, two inputs)");
        if (j.pred_lo) return set_error(EA_ERR_UNSUPPORTED, "an epilogue join with a predicate is not supported");
        if (o.epi_map == EA_MAP_ADD) {
            const ea_relation_s *r = o.epi_in;
            if (!r) return set_error(EA_ERR_ARG, "epilogue ADD needs epi_in");
            if (r->rank != orank || r->dtype != (orel ? orel->dtype : odt))
                return set_error(EA_ERR_SHAPE, "epi_in must have the output's rank and dtype");
            if (((uintptr_t)r->arena & 15) != 0) return set_error(EA_ERR_UNSUPPORTED, "epi_in arena not 16-byte aligned");
            for (int d = 0; d < orank; d++) {
                if (r->dims[d] != odims[d]) return set_error(EA_ERR_SHAPE, "epi_in extent mismatch in dim %d", d);
                if (!same_tiling(r, d, j.lt.t[j.sp.out[d] - 'a']))
                    return set_error(EA_ERR_PARTITION, "epi_in is tiled differently from the output letters");
            }
        } else if (o.epi_map == EA_MAP_ROPE) {
            const char last = j.sp.out.back();
            const int64_t ext = j.lt.t[last - 'a'].extent;
            const int64_t period = o.rope_dim ? o.rope_dim : ext;
            if (!o.rope_table || o.rope_npos <= 0 || j.rope_pos < 'a' || j.rope_pos > 'z' ||
                j.sp.out.find(j.rope_pos) == std::string::npos || j.rope_pos == last)
                return set_error(EA_ERR_ARG, "epilogue ROPE needs rope_table, rope_npos and rope_pos, an output letter "
                                             "other than the last");
            if (period <= 0 || period % 2 || ext % period)
                return set_error(EA_ERR_ARG, "rope_dim must be even and divide the last letter's extent");
        } else if (o.epi_map == EA_MAP_SILU_MUL) {
            const char pc = o.epi_pair;
            if (pc < 'a' || pc > 'z') return set_error(EA_ERR_ARG, "epilogue SILU_MUL needs epi_pair, a letter");
            const Tiling &tp = j.lt.t[pc - 'a'];
            if (tp.extent != 2 || tp.nblocks() != 1 || j.sp.term[0].find(pc) != std::string::npos ||
                j.sp.term[1].find(pc) == std::string::npos || j.sp.out.find(pc) != std::string::npos)
                return set_error(EA_ERR_SPEC, "epi_pair '%c' must be a letter of the second input only, extent 2, one block",
                                 pc);
            if ((orel ? orel->dtype : odt) != EA_BF16) return set_error(EA_ERR_DTYPE, "epilogue SILU_MUL writes bf16 only");
            j.epi_pair = pc;
            // plan with the paired letter as the innermost output letter
            j.sp.out.push_back(pc);
            j.sp.contracted.erase(j.sp.contracted.find(pc), 1);
        } else {
            return set_error(EA_ERR_UNSUPPORTED, "epilogue map %d (ADD or SILU_MUL only)", o.epi_map);
        }
    }
    // Classify.
    int kind;
    ContractionViews cv;
    if (agg == EA_AGG_NONE) {
        if (!j.sp.contracted.empty())
            return set_error(EA_ERR_SPEC, "agg NONE but letters \"%s\" are aggregated", j.sp.contracted.c_str());
        kind = kEwise;
    } else {
        if (j.sp.contracted.empty())
            return set_error(EA_ERR_SPEC, "agg %d needs an aggregated letter (use EA_AGG_NONE for a join)", agg);
        if (map == EA_MAP_PRODUCT && agg == EA_AGG_SUM && n_inputs == 2) {
            s = contraction_roles(j.sp, &cv);
            if (s) return s;
            kind = kSimt;  // or kTc, decided below
        } else {
            if (map != EA_MAP_IDENTITY && map != EA_MAP_SQUARE && map != EA_MAP_EXP_SUB && map != EA_MAP_PRODUCT)
                return set_error(EA_ERR_UNSUPPORTED, "row reduction supports IDENTITY, SQUARE, EXP_SUB, PRODUCT maps");
            kind = kRowReduce;
        }
    }
    if (j.out2) {
        if (j.out2->rank != orank) return set_error(EA_ERR_SHAPE, "out2 has rank %d, the output %d", j.out2->rank, orank);
        for (int d = 0; d < orank; d++) {
            if (j.out2->dims[d] != odims[d]) return set_error(EA_ERR_SHAPE, "out2 extent mismatch in dim %d", d);
            if (!same_tiling(j.out2, d, j.lt.t[j.sp.out[d] - 'a']))
                return set_error(EA_ERR_PARTITION, "out2 is tiled differently from the output letters");
        }
    }
    if (!orel) {
        s = ea_relation_create((ea_dtype)odt, orank, odims, oparts, nullptr, &orel);
        if (s) return s;
        created = true;
    }
    j.out = orel;
    j.user_out = orel;
    // A paired epilogue is planned against the output's pre-epilogue view:
    // the paired letter appended as the innermost output letter (every cell
    // doubled, blocks at twice the offsets), which the kernel stores halved.
    ea_relation_s vout;
    if (j.epi_pair) {
        if (orank + 1 > kMaxRank) {
            if (created) ea_relation_destroy(orel);
            return set_error(EA_ERR_UNSUPPORTED, "output rank too large for a paired epilogue");
        }
        vout.dtype = orel->dtype;
        vout.rank = orank + 1;
        for (int d = 0; d < orank; d++) {
            vout.dims[d] = orel->dims[d];
            vout.bounds[d] = orel->bounds[d];
        }
        vout.dims[orank] = 2;
        vout.bounds[orank] = {0, 2};
        vout.nblocks = orel->nblocks;
        vout.blk_off.resize(orel->blk_off.size());
        for (size_t i = 0; i < orel->blk_off.size(); i++) vout.blk_off[i] = 2 * orel->blk_off[i];
        vout.arena = orel->arena;
        vout.bytes = 2 * orel->bytes;
        vout.owned = false;
        j.out = &vout;
    }
    DevCtx *c;
    s = get_ctx(&c);
    if (s) {
        if (created) ea_relation_destroy(orel);
        return s;
    }
    Key key;
    key.str("J");
    key.str(spec);
    for (int k = 0; k < n_inputs; k++) key.rel(inputs[k]);
    key.rel(orel);
    key.v((int)agg);
    key.v((int)map);
    key.v(j.scale);
    key.v(j.eps);
    key.v(j.pred_lo);
    key.v(j.pred_hi);
    key.v(j.rope_pos);
    key.v(j.rope_table);
    key.v(j.rope_npos);
    key.v(j.rope_layout);
    if (j.out2) key.rel(j.out2);
    key.v(j.epi_map);
    key.v(j.epi_pair);
    key.v(j.rope_dim);
    if (j.row_rms) key.rel(j.row_rms);
    key.v(j.copy_letter);
    key.v(j.simt_bf16);
    if (j.epi_in) key.rel(j.epi_in);
    cudaStream_t st = (cudaStream_t)stream;
    DevPlan *p = nullptr;
    auto it = g_cache.find(key.s);
    if (it != g_cache.end()) {
        p = it->second;
    } else {
        s = plan_worklist(j.sp, j.lt, j.pred_lo, j.pred_hi, &j.wl);
        if (!s && j.copy_letter) s = keep_copy_tuples(j);
        if (!s) {
            p = new DevPlan();
            if (kind == kEwise) s = build_ewise(j, c, st, p);
            else if (kind == kRowReduce) s = build_rowreduce(j, c, st, p);
            else {
                s = build_tc(j, cv, c, st, p);
                if (s == EA_ERR_UNSUPPORTED && (j.epi_map || j.row_rms)) {
                    s = set_error(EA_ERR_UNSUPPORTED, "an epilogue join needs the tcgen05 contraction path "
                                                      "(bf16 operands that TMA can tile)");
                } else if (s == EA_ERR_UNSUPPORTED && !j.simt_bf16 &&
                           std::all_of(j.in, j.in + j.sp.n_in,
                                       [](const ea_relation_s *r) { return r->dtype == EA_BF16; })) {
                    s = set_error(EA_ERR_UNSUPPORTED, "this bf16 contraction cannot run on the tcgen05 kernel "
                                                      "(operand rows TMA cannot tile); opts->simt_bf16 lets it run "
                                                      "on the SIMT kernel");
                } else if (s == EA_ERR_UNSUPPORTED) {
                    free_plan(p);
                    p = new DevPlan();
                    set_error(EA_OK, "");
                    s = build_simt(j, cv, c, st, p);
                }
            }
            if (s) {
                free_plan(p);
                p = nullptr;
            } else {
                p->n_groups = (int64_t)j.wl.groups.size();
                p->n_tuples = (int64_t)j.wl.tuples.size() / j.sp.n_in;
                g_cache[key.s] = p;
            }
        }
        if (s) {
            if (created) ea_relation_destroy(orel);
            return s;
        }
    }
    s = launch_plan(p, c, st);
    if (s) {
        if (created) ea_relation_destroy(orel);
        return s;
    }
    *out = orel;
    return EA_OK;
}

ea_status ea_last_plan(int32_t *kernel_class, int32_t *launches, int64_t *tiles, int64_t *groups, int64_t *tuples) {
    if (kernel_class) *kernel_class = t_last.kind;
    if (launches) *launches = t_last.launches;
    if (tiles) *tiles = t_last.tiles;
    if (groups) *groups = t_last.groups;
    if (tuples) *tuples = t_last.tuples;
    return EA_OK;
}

ea_status ea_last_plan_cluster(int32_t *ctas) {
    if (!ctas) return set_error(EA_ERR_ARG, "ea_last_plan_cluster: NULL pointer");
    *ctas = t_last.cluster;
    return EA_OK;
}

ea_status ea_check(void *stream) {
    set_error(EA_OK, "");
    DevCtx *c;
    ea_status s;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        s = get_ctx(&c);
    }
    if (s) return s;
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_error(e, "ea_check: cudaStreamSynchronize");
    int flag = 0;
    e = cudaMemcpy(&flag, c->err, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_error(e, "ea_check: reading the device error word");
    if (flag) {
        int zero = 0;
        cudaMemcpy(c->err, &zero, sizeof(int), cudaMemcpyHostToDevice);
        return set_error(EA_ERR_DEVICE, "a kernel raised device error %d (%s)", flag,
                         flag == kDevTimeoutProducer   ? "bounded wait ran out in the TMA producer"
                         : flag == kDevTimeoutMma      ? "bounded wait ran out in the MMA issuer"
                         : flag == kDevTimeoutEpilogue ? "bounded wait ran out in the epilogue"
                         : flag == kDevBounds          ? "bounds check"
                         : flag == kDevTimeoutSoftmax  ? "bounded wait ran out in the attention softmax warps"
                         : flag == kDevTimeoutCorrection ? "bounded wait ran out in the attention output warps"
                         : flag == kDevTimeoutSelftest ? "bounded wait ran out in the wait self-test (expected)"
                         : flag == kDevTimeoutReduce   ? "bounded wait ran out in the row-reduction warps"
                                                       : "unknown");
    }
    return EA_OK;
}

ea_status ea_selftest_wait_timeout(int64_t limit_us, void *stream) {
    set_error(EA_OK, "");
    if (limit_us < 1 || limit_us > 1000000)
        return set_error(EA_ERR_ARG, "ea_selftest_wait_timeout: limit_us must be in [1, 1000000]");
    std::lock_guard<std::mutex> lk(g_mu);
    DevCtx *c;
    ea_status s = get_ctx(&c);
    if (s) return s;
    cudaError_t e = launch_wait_timeout(c->err, (uint64_t)limit_us * 1000ull, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_error(e, "ea_selftest_wait_timeout");
    return EA_OK;
}

ea_status ea_plan_cache_clear(void) {
    set_error(EA_OK, "");
    std::lock_guard<std::mutex> lk(g_mu);
    cudaError_t e = cudaDeviceSynchronize();
    for (auto &kv : g_cache) free_plan(kv.second);
    g_cache.clear();
    if (e != cudaSuccess) return cuda_error(e, "ea_plan_cache_clear: cudaDeviceSynchronize");
    return EA_OK;
}

}  // extern "C"
