// attention.cpp -- ea_attention_run: flash attention with grouped-query
// heads and packed sequences ("Every Kernel Is a Join", Example 3.10),
// planned on the host as one join-agg and run by one tcgen05 kernel.
//
// The plan: for every query block, every (shared-letter) position inside
// it and every tile of 128 query positions, one aggregation group; its
// tuples are the key tiles of the matching K/V blocks (same shared-letter
// intervals; key-value head floor(h / g)) that the predicate keeps, stored
// as runs of consecutive tiles of one block.  Two neighbouring query tiles
// of one head form a work item over the union of their key tiles (a tile
// only one of them keeps is fully masked for the other; the trailing tiles
// a query tile keeps none of -- under the causal predicate, the later
// tile's diagonal tile for the earlier one -- are not run for it).  Items
// are weighted by the key tiles each query tile runs, and dealt
// to the CTAs by list scheduling in block order: each goes to the CTA with
// the least work so far, which balances the causal triangle and keeps the
// items that read the same K/V blocks running at the same time (their
// tiles then come from L2); the last few rounds of items go out largest
// first.
#include <algorithm>
#include <cmath>
#include <queue>

#include "plan.h"

namespace ea {

namespace {

constexpr int kTileRows = 128;

struct AttnRoles {
    std::string qt, kt;  // terms of Q (and O) and of K (and V)
    char s = 0, t = 0, d = 0;
    std::string shared;  // letters in all terms besides d, in Q order (1 or 2)
    char head = 0;       // the grouped letter, or 0
    int64_t group = 1;
};

int pos_in(const std::string &term, char ch) { return (int)term.find(ch); }

ea_status roles_of(const Spec &sp, const ea_relation_s *q, const ea_relation_s *k, const ea_relation_s *v,
                   AttnRoles *a) {
    if (sp.n_in != 3) return set_error(EA_ERR_SPEC, "attention spec needs three inputs (Q, K, V)");
    a->qt = sp.term[0];
    a->kt = sp.term[1];
    if (sp.term[2] != a->kt) return set_error(EA_ERR_SPEC, "attention: V must have K's term");
    if (sp.out != a->qt) return set_error(EA_ERR_SPEC, "attention: O must have Q's term");
    const int r = (int)a->qt.size();
    if (r < 3 || r > 4 || (int)a->kt.size() != r)
        return set_error(EA_ERR_SPEC, "attention: terms must have 3 or 4 letters");
    a->d = a->qt.back();
    if (a->kt.back() != a->d) return set_error(EA_ERR_SPEC, "attention: the last letter (head dim) must be shared");
    for (char ch : a->qt)
        if (ch != a->d && a->kt.find(ch) == std::string::npos) {
            if (a->s) return set_error(EA_ERR_SPEC, "attention: more than one letter of Q is not in K");
            a->s = ch;
        }
    for (char ch : a->kt)
        if (ch != a->d && a->qt.find(ch) == std::string::npos) {
            if (a->t) return set_error(EA_ERR_SPEC, "attention: more than one letter of K is not in Q");
            a->t = ch;
        }
    if (!a->s || !a->t) return set_error(EA_ERR_SPEC, "attention: need a query letter and a key letter");
    for (char ch : a->qt)
        if (ch != a->d && ch != a->s) a->shared.push_back(ch);
    if (q->rank != r || k->rank != r || v->rank != r) return set_error(EA_ERR_SHAPE, "attention: ranks differ from the spec");
    for (char ch : a->shared) {
        const int64_t nq = q->dims[pos_in(a->qt, ch)], nk = k->dims[pos_in(a->kt, ch)];
        if (nq == nk) continue;
        if (nk <= 0 || nq % nk != 0 || a->head)
            return set_error(EA_ERR_SHAPE, "attention: letter '%c' has %lld values in Q and %lld in K", ch,
                             (long long)nq, (long long)nk);
        a->head = ch;
        a->group = nq / nk;
    }
    for (int i = 0; i < r; i++)
        if (k->dims[i] != v->dims[i]) return set_error(EA_ERR_SHAPE, "attention: K and V extents differ");
    if (q->dims[pos_in(a->qt, a->d)] != k->dims[pos_in(a->kt, a->d)])
        return set_error(EA_ERR_SHAPE, "attention: head dims of Q and K differ");
    return EA_OK;
}

// A 4-D tensor map over one block: dim 0 the head dim (box 64), dims 1-3
// the position letter and the shared letters ordered by stride.  slot[role]
// gives the map dim - 1 of role 0 (position), 1 (first shared letter), 2
// (second shared letter, or a dummy of extent 1).
struct BlockMap {
    CUtensorMap map;
    int slot[3];
};

ea_status encode_block(DevCtx *c, const ea_relation_s *r, int64_t bid, const std::string &term, char pos,
                       const std::string &shared, BlockMap *bm, int box_rows = kTileRows) {
    const int rank = r->rank;
    int64_t iv[kMaxRank], lo[kMaxRank], ext[kMaxRank], str[kMaxRank];
    block_coords(r, bid, iv);
    block_box(r, iv, lo, ext);
    row_major_strides(rank, ext, str);
    int64_t total = 1;
    for (int d = 0; d < rank; d++) total *= ext[d];
    const char *base = r->arena + r->blk_off[bid] * 2;
    if (((uintptr_t)base & 15) != 0) return set_error(EA_ERR_UNSUPPORTED, "attention: a block is not 16-byte aligned");
    struct Dim {
        int role;
        int64_t ext, str;
    } dims[3];
    dims[0] = {0, ext[pos_in(term, pos)], str[pos_in(term, pos)]};
    dims[1] = {1, ext[pos_in(term, shared[0])], str[pos_in(term, shared[0])]};
    if (shared.size() > 1) dims[2] = {2, ext[pos_in(term, shared[1])], str[pos_in(term, shared[1])]};
    else dims[2] = {2, 1, std::max<int64_t>(total, 1)};
    std::stable_sort(dims, dims + 3, [](const Dim &x, const Dim &y) { return x.str < y.str; });
    const int64_t D = ext[rank - 1];
    cuuint64_t gdim[4] = {(cuuint64_t)D, 0, 0, 0};
    cuuint64_t gstr[3];
    cuuint32_t box[4] = {64, 1, 1, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    for (int i = 0; i < 3; i++) {
        gdim[i + 1] = (cuuint64_t)std::max<int64_t>(dims[i].ext, 1);
        gstr[i] = (cuuint64_t)(std::max<int64_t>(dims[i].str, 1) * 2);
        if (gstr[i] % 16) return set_error(EA_ERR_UNSUPPORTED, "attention: a block stride is not a multiple of 16 bytes");
        if (dims[i].role == 0) box[i + 1] = (cuuint32_t)box_rows;
        bm->slot[dims[i].role] = i;
    }
    if (!c->encode) return set_error(EA_ERR_UNSUPPORTED, "cuTensorMapEncodeTiled is not available from the driver");
    CUresult res = c->encode(&bm->map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<char *>(base), gdim, gstr, box,
                             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (res != CUDA_SUCCESS) return set_error(EA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)res);
    return EA_OK;
}

// Block id of interval indices iv (row-major over the block grid).
int64_t block_id(const ea_relation_s *r, const int64_t *iv) {
    int64_t id = 0;
    for (int d = 0; d < r->rank; d++) id = id * ((int64_t)r->bounds[d].size() - 1) + iv[d];
    return id;
}

struct AttnJob {
    AttnRoles a;
    const ea_relation_s *q, *k, *v, *o, *m, *l;
    bool causal;
    float scale;
    std::vector<int64_t> ends;
};

ea_status build_attention(const AttnJob &j, DevCtx *c, cudaStream_t st, DevPlan *p) {
    const AttnRoles &a = j.a;
    const ea_relation_s *q = j.q, *k = j.k;
    const int rank = q->rank;
    const int ds = pos_in(a.qt, a.s), dq_d = rank - 1;
    const int D = (int)q->dims[dq_d];
    // Head dim 128 runs on CTA pairs: each CTA of a pair loads half of every
    // K tile (64 keys: K maps with 64-key boxes) and half of every V tile's
    // head dims, and holds one query tile of the pair's two.
    const bool pair = D == 128;
    std::vector<BlockMap> maps;
    maps.reserve(2 * q->nblocks + 2 * k->nblocks);
    for (int64_t b = 0; b < q->nblocks; b++) {
        BlockMap bm;
        ea_status s = encode_block(c, q, b, a.qt, a.s, a.shared, &bm);
        if (s) return s;
        maps.push_back(bm);
    }
    const int kmap0 = (int)maps.size();
    for (const ea_relation_s *r : {j.k, j.v})
        for (int64_t b = 0; b < k->nblocks; b++) {
            BlockMap bm;
            ea_status s = encode_block(c, r, b, a.kt, a.t, a.shared, &bm, pair && r == j.k ? kTileRows / 2 : kTileRows);
            if (s) return s;
            maps.push_back(bm);
        }
    const int n_kv = (int)k->nblocks;
    // CTA pairs store the output through tensor maps over O's blocks (O has
    // Q's tiling): each softmax warp stores its 32 rows x 64 head dims
    const int o_map0 = (int)maps.size();
    if (pair)
        for (int64_t b = 0; b < q->nblocks; b++) {
            BlockMap bm;
            ea_status s = encode_block(c, j.o, b, a.qt, a.s, a.shared, &bm, kTileRows / 4);
            if (s) return s;
            maps.push_back(bm);
        }
    auto seg_of = [&](int64_t pos, int64_t *lo, int64_t *hi) {  // [lo, hi) of the sequence holding pos
        *lo = 0;
        *hi = INT64_MAX;
        if (j.ends.empty()) return;
        size_t i = std::upper_bound(j.ends.begin(), j.ends.end(), pos) - j.ends.begin();
        *lo = i ? j.ends[i - 1] : 0;
        *hi = j.ends[i];
    };

    std::vector<AtItem> items;
    std::vector<AtRun> runs;
    const int ksd = pos_in(a.kt, a.t);
    const int nsh = (int)a.shared.size();
    int qs_pos[2], ks_pos[2];
    for (int i = 0; i < nsh; i++) {
        qs_pos[i] = pos_in(a.qt, a.shared[i]);
        ks_pos[i] = pos_in(a.kt, a.shared[i]);
    }
    for (int64_t qb = 0; qb < q->nblocks; qb++) {
        int64_t iv[kMaxRank], lo[kMaxRank], ext[kMaxRank], str[kMaxRank];
        block_coords(q, qb, iv);
        block_box(q, iv, lo, ext);
        row_major_strides(rank, ext, str);
        const BlockMap &qm = maps[qb];
        // stats block and its strides
        int64_t ml_base = 0, ml_str[kMaxRank] = {0};
        if (j.m) {
            int64_t miv[kMaxRank], mext[kMaxRank];
            for (int d = 0; d < rank - 1; d++) {
                miv[d] = iv[d];
                mext[d] = ext[d];
            }
            ml_base = j.m->blk_off[block_id(j.m, miv)];
            row_major_strides(rank - 1, mext, ml_str);
        }
        const int64_t n0 = nsh > 0 ? ext[qs_pos[0]] : 1, n1 = nsh > 1 ? ext[qs_pos[1]] : 1;
        for (int64_t x0 = 0; x0 < n0; x0++)
            for (int64_t x1 = 0; x1 < n1; x1++) {
                // K/V blocks: same intervals of the shared letters; every interval of t
                int64_t kiv[kMaxRank] = {0};
                int64_t kc_shared[2] = {0, 0};
                for (int i = 0; i < nsh; i++) {
                    const int64_t xq = i == 0 ? x0 : x1;
                    const int64_t g_q = lo[qs_pos[i]] + xq;
                    const bool grouped = a.shared[i] == a.head;
                    const int64_t g_k = grouped ? g_q / a.group : g_q;
                    kiv[ks_pos[i]] = iv[qs_pos[i]];
                    kc_shared[i] = g_k - k->bounds[ks_pos[i]][iv[qs_pos[i]]];
                }
                int64_t q_off = 0;
                for (int i = 0; i < nsh; i++) q_off += (i == 0 ? x0 : x1) * str[qs_pos[i]];
                int64_t ml_off = ml_base;
                if (j.m)
                    for (int i = 0; i < nsh; i++) ml_off += (i == 0 ? x0 : x1) * ml_str[qs_pos[i]];
                // tiles of 128 query positions, last first inside the block, in pairs
                const int64_t ns = ext[ds];
                const int64_t ntile_q = (ns + kTileRows - 1) / kTileRows;
                for (int64_t qt = ntile_q - 1; qt >= 0; qt -= 2) {
                    AtItem it{};
                    it.nq = qt >= 1 ? 2 : 1;
                    int64_t klo = INT64_MAX, khi = INT64_MIN;  // keys either tile may see: one interval per tile
                    int64_t tlo_k[2], thi_k[2];
                    for (int xq = 0; xq < it.nq; xq++) {
                        AtQTile &Q = it.q[xq];
                        const int64_t s_loc = (qt - xq) * kTileRows;
                        Q.s_glob0 = lo[ds] + s_loc;
                        Q.nrows = (int32_t)std::min<int64_t>(kTileRows, ns - s_loc);
                        Q.o_off = j.o->blk_off[qb] + q_off + s_loc * str[ds];
                        Q.o_rstr = str[ds];
                        Q.ml_off = j.m ? ml_off + s_loc * ml_str[ds] : 0;
                        Q.ml_rstr = j.m ? ml_str[ds] : 0;
                        Q.q_map = (int32_t)qb;
                        int32_t qc[3] = {0, 0, 0};
                        qc[qm.slot[0]] = (int32_t)s_loc;
                        qc[qm.slot[1]] = (int32_t)(nsh > 0 ? x0 : 0);
                        qc[qm.slot[2]] = (int32_t)(nsh > 1 ? x1 : 0);
                        for (int i = 0; i < 3; i++) Q.q_c[i] = qc[i];
                        Q.pos_slot = qm.slot[0];
                        int64_t a0, a1, b0, b1;
                        seg_of(Q.s_glob0, &a0, &a1);
                        seg_of(Q.s_glob0 + Q.nrows - 1, &b0, &b1);
                        tlo_k[xq] = a0;
                        thi_k[xq] = b1 == INT64_MAX ? INT64_MAX : b1 - 1;
                        if (j.causal) thi_k[xq] = std::min<int64_t>(thi_k[xq], Q.s_glob0 + Q.nrows - 1);
                        klo = std::min(klo, tlo_k[xq]);
                        khi = std::max(khi, thi_k[xq]);
                    }
                    it.r0 = (int32_t)runs.size();
                    int64_t last_kept[2] = {-1, -1};  // per query slot: its last kept tile in the item
                    const int ntb = (int)k->bounds[ksd].size() - 1;
                    for (int tb = 0; tb < ntb; tb++) {
                        kiv[ksd] = tb;
                        const int64_t tlo = k->bounds[ksd][tb], thi = k->bounds[ksd][tb + 1];
                        if (thi <= tlo) continue;
                        const int64_t nkt = (thi - tlo + kTileRows - 1) / kTileRows;
                        int64_t first = -1, last = -2;
                        for (int64_t kt = 0; kt < nkt; kt++) {
                            const int64_t t0 = tlo + kt * kTileRows, t1 = std::min<int64_t>(thi, t0 + kTileRows) - 1;
                            bool keep = false;
                            for (int xq = 0; xq < it.nq; xq++) keep = keep || !(t1 < tlo_k[xq] || t0 > thi_k[xq]);
                            if (!keep) continue;
                            if (first < 0) first = kt;
                            last = kt;
                        }
                        if (first < 0) continue;
                        for (int64_t kt = first; kt <= last; kt++) {
                            const int64_t t0 = tlo + kt * kTileRows, t1 = std::min<int64_t>(thi, t0 + kTileRows) - 1;
                            for (int xq = 0; xq < it.nq; xq++)
                                if (!(t1 < tlo_k[xq] || t0 > thi_k[xq])) last_kept[xq] = it.ntiles + (kt - first);
                        }
                        const int64_t kb = block_id(k, kiv);
                        const BlockMap &km = maps[kmap0 + kb];
                        AtRun R{};
                        R.t_glob0 = tlo + first * kTileRows;
                        R.k_map = (int32_t)(kmap0 + kb);
                        int32_t kc[3] = {0, 0, 0};
                        kc[km.slot[0]] = (int32_t)(first * kTileRows);
                        kc[km.slot[1]] = (int32_t)(nsh > 0 ? kc_shared[0] : 0);
                        kc[km.slot[2]] = (int32_t)(nsh > 1 ? kc_shared[1] : 0);
                        for (int i = 0; i < 3; i++) R.k_c[i] = kc[i];
                        R.pos_slot = km.slot[0];
                        R.ntiles = (int32_t)(last - first + 1);
                        R.nkeys = (int32_t)std::min<int64_t>(thi - R.t_glob0, (int64_t)R.ntiles * kTileRows);
                        runs.push_back(R);
                        it.ntiles += R.ntiles;
                    }
                    (void)klo;
                    (void)khi;
                    it.r1 = (int32_t)runs.size();
                    // a query slot skips the trailing key tiles it keeps none of
                    for (int xq = 0; xq < it.nq; xq++)
                        it.nt[xq] = last_kept[xq] >= 0 ? (int32_t)(last_kept[xq] + 1) : it.ntiles;
                    if (pair && it.nq == 1) {
                        // the second CTA of the pair holds a padding tile: no rows,
                        // its Q box past the block's positions (read as zeros)
                        it.q[1] = it.q[0];
                        it.q[1].nrows = 0;
                        it.q[1].q_c[qm.slot[0]] = (int32_t)ns;
                        it.nt[1] = 0;
                    }
                    items.push_back(it);
                }
            }
    }
    // the plan check: every query tile's output rows and statistics rows
    // inside their arenas (Q, K and V are read through tensor maps over
    // whole blocks, which the block offsets keep inside the arenas)
    for (size_t i = 0; i < items.size(); i++)
        for (int x = 0; x < items[i].nq; x++) {
            const AtQTile &Q = items[i].q[x];
            const int64_t e[2] = {Q.nrows, D}, st2[2] = {Q.o_rstr, 1};
            ea_status cs = check_block(Q.o_off, 2, e, st2, rel_elems(j.o), "attention output rows", i);
            const int64_t me[1] = {Q.nrows}, ms[1] = {Q.ml_rstr};
            if (!cs && j.m) cs = check_block(Q.ml_off, 1, me, ms, rel_elems(j.m), "attention statistics rows", i);
            if (cs) return cs;
        }
    // List scheduling: each item, in order, to the CTA (or CTA pair) with
    // the least work so far.  The items of one query block (one head) stay
    // together, so the K and V tiles the CTAs read at a time are those of a
    // few heads and stay in L2; inside a block they are taken largest,
    // smallest, second largest, ... so that neighbours even out (causal
    // blocks run from 2 to 16 key tiles an item).  Work in units of half a
    // key tile of one query slot: a pair runs every key tile of its item
    // once for both query tiles (2 units each), and an item costs about 4.5
    // key tiles more for its set-up and output (timed on the GPU: causal
    // items cost 3.2 us + 0.69 us per key tile).
    const int ncta = (int)std::min<int64_t>(pair ? attention_pair_clusters(c->num_sms) : (int64_t)c->num_sms,
                                            (int64_t)items.size());
    std::vector<std::vector<int32_t>> per(std::max(ncta, 1));
    if (ncta > 0) {
        std::vector<int64_t> work(items.size());
        for (size_t i = 0; i < items.size(); i++)
            work[i] = pair ? 2 * (int64_t)items[i].ntiles + 9
                           : 2 * (int64_t)(items[i].nt[0] + (items[i].nq > 1 ? items[i].nt[1] : 0)) + 9;
        std::vector<int32_t> order;
        order.reserve(items.size());
        for (size_t a = 0; a < items.size();) {
            size_t b = a + 1;
            while (b < items.size() && items[b].q[0].q_map == items[a].q[0].q_map) b++;
            std::vector<int32_t> blk;
            for (size_t i = a; i < b; i++) blk.push_back((int32_t)i);
            std::stable_sort(blk.begin(), blk.end(), [&](int32_t x, int32_t y) { return work[x] > work[y]; });
            for (size_t lo = 0, hi = blk.size(); lo < hi;) {
                order.push_back(blk[lo++]);
                if (lo < hi) order.push_back(blk[--hi]);
            }
            a = b;
        }
        // The last few rounds of items go out largest first: list scheduling
        // in block order leaves the CTAs up to one large item apart at the
        // end (causal b4 s2048 h32: the busiest pair 4.7% above the mean);
        // filling the end largest first evens them out (0.6%), and the items
        // it moves are those of the last few query blocks, whose K and V are
        // in L2 together anyway.
        const size_t tail = std::min(order.size() / 2, (size_t)3 * (size_t)ncta);
        std::stable_sort(order.end() - (std::ptrdiff_t)tail, order.end(),
                         [&](int32_t x, int32_t y) { return work[x] > work[y]; });
        typedef std::pair<int64_t, int> Load;  // (work, cta)
        std::priority_queue<Load, std::vector<Load>, std::greater<Load>> heap;
        for (int x = 0; x < ncta; x++) heap.push(Load(0, x));
        for (int32_t i : order) {
            Load l = heap.top();
            heap.pop();
            per[l.second].push_back(i);
            l.first += work[i];
            heap.push(l);
        }
    }
    // items in the order each CTA (pair) runs them, their runs renumbered in
    // the same order: a CTA's runs are one contiguous range
    std::vector<AtItem> ordered;
    std::vector<AtRun> oruns;
    std::vector<int32_t> cta_ptr(1, 0);
    ordered.reserve(items.size());
    oruns.reserve(runs.size());
    for (int x = 0; x < ncta; x++) {
        for (int32_t i : per[x]) {
            AtItem it = items[i];
            const int32_t r0 = (int32_t)oruns.size();
            for (int32_t r = it.r0; r < it.r1; r++) oruns.push_back(runs[r]);
            it.r1 = r0 + (it.r1 - it.r0);
            it.r0 = r0;
            ordered.push_back(it);
        }
        cta_ptr.push_back((int32_t)ordered.size());
    }
    int64_t ntup = 0, ngroups = 0;
    for (const AtItem &it : items) {
        ntup += (int64_t)it.nt[0] + (it.nq > 1 ? it.nt[1] : 0);
        ngroups += it.nq;
    }

    std::vector<CUtensorMap> raw(maps.size());
    for (size_t i = 0; i < maps.size(); i++) raw[i] = maps[i].map;
    Blob b;
    const size_t om = b.add(raw.data(), raw.size() * sizeof(CUtensorMap), 128);
    const size_t oi = b.add_vec(ordered), op = b.add_vec(cta_ptr), orr = b.add_vec(oruns), oe = b.add_vec(j.ends);
    ea_status s = upload(b, st, p);
    if (s) return s;
    p->kind = kAttn;
    AtParams &P = p->at;
    P.tmaps = p->dev + om;
    P.items = (const AtItem *)(p->dev + oi);
    P.cta_ptr = (const int32_t *)(p->dev + op);
    P.runs = (const AtRun *)(p->dev + orr);
    P.seq_ends = j.ends.empty() ? nullptr : (const int64_t *)(p->dev + oe);
    P.o = j.o->arena;
    P.o_elems = rel_elems(j.o);
    P.ml_elems = j.m ? rel_elems(j.m) : 0;
    P.m_out = j.m ? (float *)j.m->arena : nullptr;
    P.l_out = j.l ? (float *)j.l->arena : nullptr;
    P.ncta = pair ? 2 * ncta : ncta;  // in pairs: cta_ptr indexes pairs
    P.pair = pair ? 1 : 0;
    P.n_kv = n_kv;
    P.o_map0 = o_map0;
    P.nseq = (int32_t)j.ends.size();
    P.causal = j.causal ? 1 : 0;
    P.scale = j.scale;
    P.scale_log2 = (float)((double)j.scale * 1.4426950408889634);
    P.d = (int32_t)q->dims[dq_d];
    p->n_groups = ngroups;
    p->n_tuples = ntup;
    return EA_OK;
}

ea_status check_same_tiling(const ea_relation_s *x, const ea_relation_s *y, const char *what) {
    if (x->rank != y->rank) return set_error(EA_ERR_SHAPE, "attention: %s ranks differ", what);
    for (int d = 0; d < x->rank; d++) {
        if (x->dims[d] != y->dims[d]) return set_error(EA_ERR_SHAPE, "attention: %s extents differ", what);
        if (x->bounds[d] != y->bounds[d]) return set_error(EA_ERR_PARTITION, "attention: %s tilings differ", what);
    }
    return EA_OK;
}

}  // namespace

}  // namespace ea

using namespace ea;

extern "C" ea_status ea_attention_run(const char *spec, ea_relation q, ea_relation k, ea_relation v,
                                      const ea_attn_opts *opts, void *stream, ea_relation *out) {
    set_error(EA_OK, "");
    if (!spec || !q || !k || !v || !out) return set_error(EA_ERR_ARG, "ea_attention_run: NULL argument");
    ea_attn_opts o{};
    if (opts) o = *opts;
    std::lock_guard<std::mutex> lk(g_mu);
    Spec sp;
    ea_status s = parse_spec(spec, &sp);
    if (s) return s;
    AttnJob j;
    s = roles_of(sp, q, k, v, &j.a);
    if (s) return s;
    const AttnRoles &a = j.a;
    const int rank = q->rank;
    if (q->dtype != EA_BF16 || k->dtype != EA_BF16 || v->dtype != EA_BF16)
        return set_error(EA_ERR_DTYPE, "attention: Q, K and V must be bf16");
    const int64_t D = q->dims[rank - 1];
    if (D != 64 && D != 128) return set_error(EA_ERR_UNSUPPORTED, "attention: head dim %lld (64 or 128 only)", (long long)D);
    // tilings
    if (q->bounds[rank - 1].size() != 2 || k->bounds[rank - 1].size() != 2)
        return set_error(EA_ERR_PARTITION, "attention: the head dim must be one block");
    s = check_same_tiling(k, v, "K and V");
    if (s) return s;
    for (char ch : a.shared) {
        const std::vector<int64_t> &bq = q->bounds[pos_in(a.qt, ch)], &bk = k->bounds[pos_in(a.kt, ch)];
        bool same = bq.size() == bk.size();
        for (size_t i = 0; same && i < bq.size(); i++) same = bq[i] == (ch == a.head ? a.group : 1) * bk[i];
        if (!same)
            return set_error(EA_ERR_PARTITION, "attention: letter '%c' is tiled differently in Q and K; re-block with ea_exchange", ch);
    }
    if (o.scale < 0.0f || !std::isfinite(o.scale)) return set_error(EA_ERR_ARG, "attention: scale must be > 0");
    j.scale = o.scale == 0.0f ? (float)(1.0 / std::sqrt((double)D)) : o.scale;
    j.causal = o.causal != 0;
    const int64_t ns = q->dims[pos_in(a.qt, a.s)], nt = k->dims[pos_in(a.kt, a.t)];
    if (o.n_seq_ends < 0 || (o.n_seq_ends > 0 && !o.seq_ends)) return set_error(EA_ERR_ARG, "attention: bad seq_ends");
    if (o.n_seq_ends > 0) {
        if (ns != nt) return set_error(EA_ERR_ARG, "attention: packed sequences need equal s and t extents");
        for (int i = 0; i < o.n_seq_ends; i++) {
            const int64_t e = o.seq_ends[i];
            if (e <= (i ? o.seq_ends[i - 1] : 0)) return set_error(EA_ERR_ARG, "attention: seq_ends must increase from > 0");
            j.ends.push_back(e);
        }
        if (j.ends.back() != ns) return set_error(EA_ERR_ARG, "attention: the last sequence end must equal the s extent");
    }
    if ((o.m_out != nullptr) != (o.l_out != nullptr)) return set_error(EA_ERR_ARG, "attention: give both m_out and l_out or neither");
    for (ea_relation st : {o.m_out, o.l_out}) {
        if (!st) continue;
        if (st->dtype != EA_F32) return set_error(EA_ERR_DTYPE, "attention: m_out and l_out must be f32");
        if (st->rank != rank - 1) return set_error(EA_ERR_SHAPE, "attention: m_out / l_out have Q's term without d");
        for (int d = 0; d < rank - 1; d++) {
            if (st->dims[d] != q->dims[d]) return set_error(EA_ERR_SHAPE, "attention: m_out / l_out extents differ from Q");
            if (st->bounds[d] != q->bounds[d]) return set_error(EA_ERR_PARTITION, "attention: m_out / l_out tiled unlike Q");
        }
    }
    ea_relation O = *out;
    if (O) {
        if (O->dtype != EA_BF16) return set_error(EA_ERR_DTYPE, "attention: O must be bf16");
        s = check_same_tiling(q, O, "Q and O");
        if (s) return s;
    }
    DevCtx *c;
    s = get_ctx(&c);
    if (s) return s;
    if (!O) {
        ea_dim_part parts[kMaxRank];
        for (int d = 0; d < rank; d++)
            parts[d] = ea_dim_part{(int32_t)q->bounds[d].size() - 1, 0, q->bounds[d].data()};
        s = ea_relation_create(EA_BF16, rank, q->dims, parts, nullptr, &O);
        if (s) return s;
    }
    j.q = q;
    j.k = k;
    j.v = v;
    j.o = O;
    j.m = o.m_out;
    j.l = o.l_out;
    Key key;
    key.str("A");
    key.str(spec);
    for (const ea_relation_s *r : {j.q, j.k, j.v, j.o}) key.rel(r);
    key.v(j.m ? j.m->arena : nullptr);
    key.v(j.l ? j.l->arena : nullptr);
    key.v(j.causal);
    key.v(j.scale);
    for (int64_t e : j.ends) key.v(e);
    cudaStream_t st = (cudaStream_t)stream;
    DevPlan *p;
    auto it = g_cache.find(key.s);
    if (it != g_cache.end()) {
        p = it->second;
    } else {
        p = new DevPlan();
        s = build_attention(j, c, st, p);
        if (s) {
            free_plan(p);
            if (!*out) ea_relation_destroy(O);
            return s;
        }
        g_cache[key.s] = p;
    }
    s = launch_plan(p, c, st);
    if (s) {
        if (!*out) ea_relation_destroy(O);
        return s;
    }
    *out = O;
    return EA_OK;
}
