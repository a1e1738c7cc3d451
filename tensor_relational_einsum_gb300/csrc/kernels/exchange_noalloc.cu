// exchange_noalloc.cu -- ea_exchange_noalloc: the re-blocking exchange for
// callers that must not allocate device memory.
//
// ea_exchange plans an exchange once, uploads the plan into memory it gets
// from cudaMalloc and caches it.  Some callers cannot allow that: a serving
// process whose device memory is carved up in advance by its own pool (a
// cudaMalloc outside the pool can fail or fragment it), code on a latency
// path where cudaMalloc's implicit device-wide synchronisation would stall
// other streams, or an embedding that forbids the library from owning any
// device memory at all.  This entry point keeps its plan in one
// file-scope __device__ array instead, so it allocates nothing: the caller
// brings the input and output relations (created over the caller's own
// memory with ea_relation_create(..., dev_ptr, ...)).
//
// The array is part of the module, so every GPU that loads libea.so holds
// kNoAllocScratchBytes of device memory until the process exits.  Host code
// cannot use the array's name as a device address; the first call on each
// device looks the address up with cudaGetSymbolAddress (with that device
// current) and keeps it.
//
// The plan is computed on the host without heap allocation, staged in a
// static host buffer and copied into the array with cudaMemcpyAsync on the
// caller's stream, right before the kernel.  Every call shares the array:
// two calls whose copies and kernels overlap on the GPU (different streams
// without ordering between them) race on it.  A call on a stream that is
// being captured into a CUDA graph is refused: a captured copy would read
// the static host buffer when the graph is replayed, by which time a later
// call may have put another plan there.
#include <string.h>

#include <mutex>

#include "../host.h"

namespace ea {

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(1) << 20;  // 1 MiB
constexpr int kMaxSplitsPerDim = 2048 + 2;                // union of two tilings' bounds
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

struct Staging {
    int64_t ov[kMaxRank][kMaxSplitsPerDim];
    int nov[kMaxRank];
    alignas(256) unsigned char plan[kNoAllocScratchBytes];
    XTile tiles[kNoAllocScratchBytes / sizeof(XTile)];
};

Staging g_stage;  // host staging, static: no heap
std::mutex g_na_mu;
void *g_scratch_dev[kMaxDevices];
int g_sms[kMaxDevices];
bool g_ready[kMaxDevices];

// Sorted union of two increasing bound lists into out; false if it does not fit.
bool merge_bounds(const std::vector<int64_t> &a, const std::vector<int64_t> &b, int64_t *out, int *n) {
    size_t i = 0, j = 0;
    int k = 0;
    while (i < a.size() || j < b.size()) {
        int64_t v;
        if (j >= b.size() || (i < a.size() && a[i] <= b[j])) v = a[i++];
        else v = b[j++];
        if (k > 0 && out[k - 1] == v) continue;
        if (k == kMaxSplitsPerDim) return false;
        out[k++] = v;
    }
    *n = k;
    return true;
}

int find_block(const std::vector<int64_t> &b, int64_t x) {
    int lo = 0, hi = (int)b.size() - 2;
    while (lo < hi) {
        int mid = (lo + hi + 1) / 2;
        if (b[mid] <= x) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

struct Emitter {
    XSeg *segs;
    size_t max_segs;
    size_t nseg = 0;
    size_t ntile = 0;
    int esize;
    bool overflow = false;

    void tile(XTile t) {
        if (ntile == sizeof(g_stage.tiles) / sizeof(XTile)) {
            overflow = true;
            return;
        }
        g_stage.tiles[ntile++] = t;
    }

    void emit(XSeg seg, int nd, const int64_t *ext, const int64_t *ss, const int64_t *ds) {
        if (nd > 4) {  // peel the outermost dimension
            for (int64_t i = 0; i < ext[0] && !overflow; i++) {
                XSeg s2 = seg;
                s2.src_off += i * ss[0];
                s2.dst_off += i * ds[0];
                emit(s2, nd - 1, ext + 1, ss + 1, ds + 1);
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
        if (nseg == max_segs) {
            overflow = true;
            return;
        }
        int32_t sid = (int32_t)nseg;
        segs[nseg++] = seg;
        const int64_t target = 64 * 1024;
        int64_t row_bytes = seg.inner * esize;
        if (row_bytes >= target) {
            int64_t cols = (target / esize) / (16 / esize) * (16 / esize);
            for (int64_t r = 0; r < seg.rows && !overflow; r++)
                for (int64_t c = 0; c < seg.inner && !overflow; c += cols)
                    tile(XTile{sid, 0, r, 1, c, seg.inner - c < cols ? seg.inner - c : cols});
        } else {
            int64_t per = target / row_bytes > 1 ? target / row_bytes : 1;
            for (int64_t r = 0; r < seg.rows && !overflow; r += per)
                tile(XTile{sid, 0, r, seg.rows - r < per ? seg.rows - r : per, 0, seg.inner});
        }
    }
};

}  // namespace

}  // namespace ea

using namespace ea;

extern "C" ea_status ea_exchange_noalloc(ea_relation in, ea_relation out, void *stream) {
    set_error(EA_OK, "");
    if (!in || !out) return set_error(EA_ERR_ARG, "ea_exchange_noalloc: NULL relation");
    if (in->dtype != out->dtype || in->rank != out->rank)
        return set_error(EA_ERR_SHAPE, "ea_exchange_noalloc: input and output differ in dtype or rank");
    for (int d = 0; d < in->rank; d++)
        if (in->dims[d] != out->dims[d]) return set_error(EA_ERR_SHAPE, "ea_exchange_noalloc: extents differ");
    if (in->bytes && out->bytes && out->arena < in->arena + in->bytes && in->arena < out->arena + out->bytes)
        return set_error(EA_ERR_ARG, "ea_exchange_noalloc: input and output arenas overlap");
    cudaStream_t st = (cudaStream_t)stream;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(st, &cap);
    if (e != cudaSuccess) return cuda_error(e, "ea_exchange_noalloc: cudaStreamIsCapturing");
    if (cap != cudaStreamCaptureStatusNone)
        return set_error(EA_ERR_UNSUPPORTED, "ea_exchange_noalloc: the stream is being captured; the plan copy "
                                             "reads a static host buffer that later calls overwrite");
    std::lock_guard<std::mutex> lk(g_na_mu);
    // -- set-up, once per device, with that device current
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_error(e, "ea_exchange_noalloc: cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return set_error(EA_ERR_ARG, "ea_exchange_noalloc: device %d out of range", dev);
    if (!g_ready[dev]) {
        e = cudaGetSymbolAddress(&g_scratch_dev[dev], g_noalloc_scratch);
        if (e != cudaSuccess) return cuda_error(e, "ea_exchange_noalloc: cudaGetSymbolAddress(scratch)");
        e = cudaDeviceGetAttribute(&g_sms[dev], cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return cuda_error(e, "ea_exchange_noalloc: cudaDeviceGetAttribute");
        g_ready[dev] = true;
    }
    // -- plan: overlay atoms of the two tilings, written into static staging
    const int rank = in->rank, esize = (int)elem_size(in->dtype);
    int64_t natoms = 1;
    for (int d = 0; d < rank; d++) {
        if (!merge_bounds(in->bounds[d], out->bounds[d], g_stage.ov[d], &g_stage.nov[d]))
            return set_error(EA_ERR_UNSUPPORTED, "ea_exchange_noalloc: more than %d split points in dimension %d",
                             kMaxSplitsPerDim, d);
        natoms *= g_stage.nov[d] - 1;
        if (in->dims[d] == 0) natoms = 0;
    }
    Emitter em;
    em.segs = reinterpret_cast<XSeg *>(g_stage.plan);
    em.max_segs = kNoAllocScratchBytes / sizeof(XSeg);
    em.esize = esize;
    int64_t ai[kMaxRank] = {0};
    for (int64_t a = 0; a < natoms && !em.overflow; a++) {
        int64_t lo[kMaxRank], ext[kMaxRank], sext[kMaxRank], dext[kMaxRank], slo[kMaxRank], dlo[kMaxRank];
        int64_t sid = 0, did = 0;
        for (int d = 0; d < rank; d++) {
            lo[d] = g_stage.ov[d][ai[d]];
            ext[d] = g_stage.ov[d][ai[d] + 1] - lo[d];
            int si = find_block(in->bounds[d], lo[d]), di = find_block(out->bounds[d], lo[d]);
            sid = sid * ((int64_t)in->bounds[d].size() - 1) + si;
            did = did * ((int64_t)out->bounds[d].size() - 1) + di;
            slo[d] = in->bounds[d][si];
            sext[d] = in->bounds[d][si + 1] - slo[d];
            dlo[d] = out->bounds[d][di];
            dext[d] = out->bounds[d][di + 1] - dlo[d];
        }
        int64_t sstr[kMaxRank], dstr[kMaxRank];
        row_major_strides(rank, sext, sstr);
        row_major_strides(rank, dext, dstr);
        XSeg seg;
        memset(&seg, 0, sizeof seg);
        seg.src_off = in->blk_off[sid];
        seg.dst_off = out->blk_off[did];
        for (int d = 0; d < rank; d++) {
            seg.src_off += (lo[d] - slo[d]) * sstr[d];
            seg.dst_off += (lo[d] - dlo[d]) * dstr[d];
        }
        int last = rank - 1;
        seg.inner = ext[last];
        while (last > 0 && sstr[last - 1] == seg.inner && dstr[last - 1] == seg.inner) {
            last--;
            seg.inner *= ext[last];
        }
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
        em.emit(seg, nd, oe, os, od);
        for (int d = rank - 1; d >= 0; d--) {
            if (++ai[d] < g_stage.nov[d] - 1) break;
            ai[d] = 0;
        }
    }
    const size_t seg_bytes = (em.nseg * sizeof(XSeg) + 255) / 256 * 256;
    const size_t total = seg_bytes + em.ntile * sizeof(XTile);
    if (em.overflow || total > kNoAllocScratchBytes)
        return set_error(EA_ERR_UNSUPPORTED,
                         "ea_exchange_noalloc: the plan needs more than the %zu bytes of static scratch (%lld atoms); "
                         "use ea_exchange",
                         kNoAllocScratchBytes, (long long)natoms);
    if (em.ntile == 0) return EA_OK;
    ea_status cs = check_exchange_plan(reinterpret_cast<const XSeg *>(g_stage.plan), em.nseg, g_stage.tiles, em.ntile,
                                       rel_elems(in), rel_elems(out), 1, 0);
    if (cs) return cs;
    memcpy(g_stage.plan + seg_bytes, g_stage.tiles, em.ntile * sizeof(XTile));
    // -- copy the plan into the device array and launch, both on the caller's stream
    char *scratch = static_cast<char *>(g_scratch_dev[dev]);
    e = cudaMemcpyAsync(scratch, g_stage.plan, total, cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) return cuda_error(e, "ea_exchange_noalloc: cudaMemcpyAsync(plan)");
    // (no device error word: the library's word is taken with cudaMalloc on
    // a device's first allocating call; the plan was checked above, and a
    // library built with EA_DEBUG_BOUNDS still skips an out-of-arena tile)
    e = launch_exchange(reinterpret_cast<const XSeg *>(scratch), reinterpret_cast<const XTile *>(scratch + seg_bytes),
                        (int64_t)em.ntile, in->arena, out->arena, esize, g_sms[dev], st, rel_elems(in),
                        rel_elems(out), nullptr);
    if (e != cudaSuccess) return cuda_error(e, "ea_exchange_noalloc: kernel launch");
    return EA_OK;
}
