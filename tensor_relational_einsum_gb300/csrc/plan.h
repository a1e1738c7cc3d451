// plan.h -- the device plans of libea.so: the per-device context, plan
// blobs uploaded once and cached, and the record of the last launch.
// Internal (shared by the join-agg, exchange and attention entry points).
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <string.h>

#include <algorithm>
#include <string>
#include <unordered_map>

#include "host.h"

namespace ea {

struct DevCtx {
    bool init = false;
    int num_sms = 0;
    int *err = nullptr;  // device error word (kernels raise it; ea_check reads it)
    PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
};
extern DevCtx g_ctx[64];
ea_status get_ctx(DevCtx **out);

struct Blob {
    std::vector<char> h;
    size_t add(const void *p, size_t n, size_t align = 128) {
        size_t off = (h.size() + align - 1) / align * align;
        h.resize(off + std::max<size_t>(n, 1));
        if (n) memcpy(h.data() + off, p, n);
        return off;
    }
    template <class T>
    size_t add_vec(const std::vector<T> &v) {
        return add(v.data(), v.size() * sizeof(T));
    }
};

enum PlanKind { kExchange = 0, kEwise, kRowReduce, kSimt, kTc, kAttn, kExchangeAgg };

struct DevPlan {
    int kind = 0;
    char *dev = nullptr;
    DevFree dev_release;  // how `dev` is freed (the allocator that took it)
    char *pinned = nullptr;
    size_t bytes = 0;
    cudaEvent_t ready = nullptr;
    cudaStream_t made_on = nullptr;
    bool uploaded = false;  // the upload is known complete: no stream needs to wait for it
    // exchange
    XSeg *segs = nullptr;
    XTile *xtiles = nullptr;
    int64_t nxtiles = 0;
    const char *xsrc = nullptr;
    char *xdst = nullptr;
    int64_t xsrc_elems = 0, xdst_elems = 0;  // arena sizes (EA_DEBUG_BOUNDS checks)
    int esize = 0;
    int xdtype = 0, xagg = 0, xcopies = 1;  // exchange with aggregation
    int64_t xcopy_stride = 0;
    // kernels
    EwParams ew{};
    RrParams rr{};
    CtParams ct{};
    TcParams tc{};
    AtParams at{};
    int64_t n_groups = 0, n_tuples = 0;
};

struct LastPlan {
    int32_t kind = -1, launches = 0;
    int64_t tiles = 0, groups = 0, tuples = 0;
    int32_t cluster = 1;  // CTAs that share one MMA tile (tcgen05 contraction: 2 = CTA pairs)
};
extern thread_local LastPlan t_last;

// Plans by key (spec, relations, options); owned here until ea_plan_cache_clear.
extern std::unordered_map<std::string, DevPlan *> g_cache;

ea_status upload(const Blob &b, cudaStream_t st, DevPlan *p);
void free_plan(DevPlan *p);
ea_status plan_ready_on(DevPlan *p, cudaStream_t st);
ea_status launch_plan(DevPlan *p, DevCtx *c, cudaStream_t st);

// A plan-cache key: the bytes of everything the plan depends on.
struct Key {
    std::string s;
    void raw(const void *p, size_t n) { s.append((const char *)p, n); }
    template <class T>
    void v(const T &x) {
        raw(&x, sizeof x);
    }
    void str(const char *c) {
        s.append(c);
        s.push_back(0);
    }
    void rel(const ea_relation_s *r) {
        v(r->dtype);
        v(r->rank);
        for (int d = 0; d < r->rank; d++) {
            v(r->dims[d]);
            int64_t n = (int64_t)r->bounds[d].size();
            v(n);
            raw(r->bounds[d].data(), n * sizeof(int64_t));
        }
        v(r->arena);
    }
};

}  // namespace ea
