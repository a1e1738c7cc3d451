// host.h -- host-side planner types of libea.so (relations, specs, tilings,
// work lists, exchange segments).  Internal.
#pragma once

#include <stdarg.h>

#include <mutex>
#include <string>
#include <vector>

#include "ea_internal.h"

namespace ea {
// How to release a block of device memory the library took: through the
// allocator pair that was current when it was taken (fn == NULL: cudaFree).
struct DevFree {
    ea_free_fn fn = nullptr;
    void *ctx = nullptr;
};
}  // namespace ea

struct ea_relation_s {
    int dtype = 0;
    int rank = 0;
    int64_t dims[ea::kMaxRank] = {0};
    std::vector<int64_t> bounds[ea::kMaxRank];  // per dim: nblocks + 1 values
    int64_t nblocks = 0;
    std::vector<int64_t> blk_off;                // element offset of each block (+ total)
    char *arena = nullptr;
    size_t bytes = 0;
    bool owned = false;
    ea::DevFree release;  // owned arenas: how to free them
};

namespace ea {

ea_status set_error(ea_status code, const char *fmt, ...);
// Device memory through the allocator of ea_set_allocator (else cudaMalloc);
// *rel receives the matching release.  EA_ERR_ALLOC on failure.
ea_status dev_alloc(size_t bytes, void **ptr, DevFree *rel, const char *what);
void dev_free(void *ptr, const DevFree &rel);
ea_status cuda_error(cudaError_t e, const char *what);
size_t elem_size(int dtype);

// Tiling of one dimension / letter.
struct Tiling {
    int64_t extent = -1;
    std::vector<int64_t> b;  // nblocks + 1 bounds
    int nblocks() const { return (int)b.size() - 1; }
};

ea_status make_tiling(int64_t extent, int32_t nblocks, const int64_t *bounds, Tiling *t);

// Block grid helpers for a relation.
void block_coords(const ea_relation_s *r, int64_t bid, int64_t *iv);  // interval index per dim
void block_box(const ea_relation_s *r, const int64_t *iv, int64_t *lo, int64_t *ext);
void row_major_strides(int rank, const int64_t *ext, int64_t *str);

// Parsed spec "ij,jk->ik".
struct Spec {
    int n_in = 0;
    std::string term[kMaxIn];
    std::string out;
    std::string order;       // letters in order of first appearance in the spec string
    std::string contracted;  // letters not in the output, in order of first appearance
};
ea_status parse_spec(const char *s, Spec *sp);

// Letter tilings (index 0..25); extent -1 = letter unused.
struct LetterTilings {
    Tiling t[26];
};

// Canonical work list of a join (Section 3.3 enumeration, Definition 3.7 grouping).
struct WorkList {
    std::vector<int64_t> groups;    // output block ids
    std::vector<int64_t> grp_ptr;   // CSR
    std::vector<int64_t> tuples;    // n_in ids per tuple
    std::vector<int64_t> tuple_iv;  // per tuple: interval index of every letter (26 per tuple)
    int64_t join_volume = 0;
    int64_t agg_volume = 0;
};
ea_status plan_worklist(const Spec &sp, const LetterTilings &lt, char pred_lo, char pred_hi, WorkList *wl);

// Exchange plan: overlay atoms as copy segments, split into tiles.
struct ExchangePlan {
    std::vector<XSeg> segs;
    std::vector<XTile> tiles;
    int64_t n_atoms = 0;
};
ea_status plan_exchange(int rank, const int64_t *dims, const Tiling *src, const Tiling *dst, int esize,
                        ExchangePlan *xp);

// The plan check (bounds.cpp): every descriptor's element range inside the
// arena it addresses, else EA_ERR_BOUNDS.  copies / copy_stride: the
// exchange with aggregation reads copy q at q * copy_stride elements on.
ea_status check_exchange_plan(const XSeg *segs, size_t nseg, const XTile *tiles, size_t ntiles, int64_t src_elems,
                              int64_t dst_elems, int64_t copies, int64_t copy_stride);
ea_status check_view_items(const EwItem *items, size_t n, int n_in, const int64_t *in_elems, int64_t out_elems,
                           const char *what);
ea_status check_ew_tiles(const EwTile *tiles, size_t nt, const EwItem *items, size_t n);
ea_status check_rr_tiles(const RrTile *tiles, size_t nt, const RrGroup *groups, size_t ng, const EwItem *items,
                         size_t n);
ea_status check_rb_desc(const int64_t *w, size_t ntiles, int64_t in_elems, int64_t out_elems);
ea_status check_simt_plan(const CtGroup *groups, size_t ng, const CtTuple *tuples, size_t nt, int64_t a_elems,
                          int64_t b_elems, int64_t c_elems);
inline int64_t rel_elems(const ea_relation_s *r) { return r->blk_off.empty() ? 0 : r->blk_off.back(); }
// base + sum_i c_i str_i (0 <= c_i < ext_i) inside [0, elems).
ea_status check_block(int64_t base, int n, const int64_t *ext, const int64_t *str, int64_t elems, const char *what,
                      size_t index);

// Arena offsets of a tiling (row-major blocks, consecutive).
void tiling_offsets(int rank, const Tiling *t, std::vector<int64_t> *off);

extern std::mutex g_mu;

}  // namespace ea
