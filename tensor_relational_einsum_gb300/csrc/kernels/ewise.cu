// ewise.cu -- elementwise join-agg kernel (aggregation NONE).
//
// "Every Kernel Is a Join", Section 1: elementwise operations (ReLU, SiLU,
// residual adds, normalisation steps) are joins of relations on equal keys
// -- or of a relation with a broadcast one, keyed by a subset of its
// letters -- followed by a map and no aggregation.  Each function
// specification of such a join-agg owns one output block; the host gives
// every block a strided view (EwItem) and cuts it into tiles of rows.
//
// The work is a pure HBM stream, so the kernel is built for bytes in flight
// and few instructions per byte: a row of the view is owned by a warp (or a
// slice of a warp when rows are short); its geometry (offsets, predicate
// range, rope position, broadcast operands) is decoded once per row; the
// row loop is instantiated per map and per set of streamed inputs, keeps
// several 16-byte loads per lane in flight, and needs no per-cell
// predicate test unless the row crosses the predicate's boundary.
#include <algorithm>
#include <type_traits>

#include "dev_common.cuh"

namespace ea {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

template <int NIN>
struct Row {
    int64_t ooff;         // output offset of column 0 of the tile
    int64_t ioff[NIN];    // input offsets of column 0
    int64_t iinn[NIN];    // input strides along the row
    float bc[NIN];        // broadcast operand values
    int cmin, cmax;       // kept columns (tile-local)
    const float2 *tab;    // rope: (cos, sin) row of this position
    int64_t pair0;        // rope: global pair index of column 0
};

// MAP < 0: the map is read at run time (generic kernel); MASK < 0: which
// inputs stream along the row is read at run time.
template <int MAP, int NIN, int MASK>
__device__ __forceinline__ float apply(const EwParams &p, float x0, float x1, float x2) {
    if constexpr (MAP >= 0) return fmap<MAP>(x0, x1, x2, p.scale, p.eps);
    else return cell_map(p.map, x0, x1, x2, p.scale, p.eps);
}

__device__ __forceinline__ bool streams(int mask, int k) { return (mask >> k) & 1; }

// Cells per chunk and chunks per batch: every lane keeps about 128 bytes of
// streamed inputs in flight (raw, converted only when used).
// RoPE also loads 32 bytes of (cos, sin) per chunk, so it batches 4 chunks.
template <bool kVec, int NS, int DT, int MAP>
struct Batch {
    static constexpr int V = kVec ? 8 : 1;
    static constexpr int BYTES = DT == 1 ? 16 : 32;  // one chunk of one input
    static constexpr int U = !kVec ? 4
                             : MAP == EA_MAP_ROPE ? 4
                             : (NS <= 1 ? 128 / BYTES : (128 / BYTES) / NS > 0 ? (128 / BYTES) / NS : 1);
};

// Stream one row: chunks sl, sl + lpr, ... of V cells, U chunks per batch.
// DT: 1 = streamed inputs are bf16, 2 = fp32, 0 = read at run time.
template <int MAP, bool kVec, int NIN, int MASK, int DT>
__device__ __forceinline__ void ew_row(const EwParams &p, const Row<NIN> &w, int cpr, int sl, int lpr, bool masked,
                                       int64_t out_inner) {
    constexpr int V = kVec ? 8 : 1;
    constexpr int NS = MASK < 0 ? NIN : ((MASK & 1) + ((MASK >> 1) & 1) + ((MASK >> 2) & 1));
    constexpr int NSV = NS > 0 ? NS : 1;
    constexpr int U = Batch<kVec, NS, DT, MAP>::U;
    constexpr bool kRaw = kVec && DT != 0 && MASK >= 0;
    constexpr bool kB16 = DT == 1;
    constexpr bool kTab = MAP == EA_MAP_ROPE && kVec;
    const int mask = MASK < 0 ? p.stream_mask : MASK;
    for (int c0 = sl; c0 < cpr; c0 += lpr * U) {
        uint4 raw[kRaw ? U : 1][kRaw ? NSV : 1][kB16 ? 1 : 2];
        float v[kRaw ? 1 : U][kRaw ? 1 : NSV][kRaw ? 1 : V];
        float4 tab[kTab ? U : 1][2];  // rope: (cos, sin) of the chunk's 4 pairs
#pragma unroll
        for (int u = 0; u < U; u++) {
            const int c = c0 + u * lpr;
            if (c >= cpr) continue;
            const int64_t col = (int64_t)c * V;
            if constexpr (kTab) {
                const float4 *tp = reinterpret_cast<const float4 *>(w.tab + w.pair0 + (col >> 1));
                tab[u][0] = __ldg(tp);
                tab[u][1] = __ldg(tp + 1);
            }
            int s = 0;
#pragma unroll
            for (int k = 0; k < NIN; k++) {
                if (MASK >= 0 && !streams(MASK, k)) continue;
                if constexpr (kRaw) {
                    ld_raw<kB16>(p.in[k], w.ioff[k] + col, raw[u][s]);
                } else if (MASK < 0 && !streams(mask, k)) {
#pragma unroll
                    for (int e = 0; e < V; e++) v[u][k][e] = w.bc[k];
                } else if (kVec) {
                    ld8(p.in[k], p.in_dtype[k], w.ioff[k] + col, v[u][MASK < 0 ? k : s]);
                } else {
                    v[u][MASK < 0 ? k : s][0] = ld_elem(p.in[k], p.in_dtype[k], w.ioff[k] + col * w.iinn[k]);
                }
                s++;
            }
        }
#pragma unroll
        for (int u = 0; u < U; u++) {
            const int c = c0 + u * lpr;
            if (c >= cpr) continue;
            const int col = c * V;
            auto val = [&](int s, int k, int e) -> float {
                if constexpr (kRaw) return raw_at<kB16>(raw[u][s], e);
                else return v[u][MASK < 0 ? k : s][e];
            };
            float o[V];
            if constexpr (MAP == EA_MAP_ROPE) {
                if constexpr (kVec) {
                    const float *tf = reinterpret_cast<const float *>(&tab[u][0]);
#pragma unroll
                    for (int e = 0; e < V; e += 2) {
                        const float2 cs = make_float2(tf[e], tf[e + 1]);
                        const float x0 = val(0, 0, e), x1 = val(0, 0, e + 1);
                        o[e] = x0 * cs.x - x1 * cs.y;
                        o[e + 1] = x0 * cs.y + x1 * cs.x;
                    }
                } else {
                    const int64_t g = 2 * w.pair0 + col;  // global index along the pair letter
                    const float2 cs = __ldg(w.tab + (g >> 1));
                    const float partner =
                        ld_elem(p.in[0], p.in_dtype[0], w.ioff[0] + (col + ((g & 1) ? -1 : 1)) * w.iinn[0]);
                    const float x = val(0, 0, 0);
                    o[0] = (g & 1) ? partner * cs.y + x * cs.x : x * cs.x - partner * cs.y;
                }
            } else {
#pragma unroll
                for (int e = 0; e < V; e++) {
                    float x[3] = {1.0f, 1.0f, 1.0f};
                    int s = 0;
#pragma unroll
                    for (int k = 0; k < NIN; k++) {
                        if constexpr (MASK < 0) x[k] = val(k, k, e);
                        else if (streams(MASK, k)) x[k] = val(s++, k, e);
                        else x[k] = w.bc[k];
                    }
                    o[e] = apply<MAP, NIN, MASK>(p, x[0], x[1], x[2]);
                }
            }
            if (masked) {
#pragma unroll
                for (int e = 0; e < V; e++)
                    if (col + e < w.cmin || col + e > w.cmax) o[e] = 0.0f;  // a removed cell holds 0
            }
            if (kVec) st8(p.out, p.out_dtype, w.ooff + col, o);
            else st_elem(p.out, p.out_dtype, w.ooff + (int64_t)col * out_inner, o[0]);
        }
    }
}

// The geometry of the current tile: every row of a tile is one step along
// the innermost row dimension (the host never lets a tile cross a run of
// it), so offsets, predicate values and the rope position are linear in
// the row index.
struct TileGeom {
    int64_t ooff, ostr, ostr2;     // output offset at the first row, change per row / per run
    int64_t ioff[kMaxIn], istr[kMaxIn], istr2[kMaxIn];
    int64_t iinn[kMaxIn];
    int32_t e1;                    // rows per run of the innermost row dim (0: the tile is one run)
    int32_t da2, db2, dpos2;       // change of the special values per run
    int64_t a0, b0, pos0;          // predicate letters and rope position at the first row
    int32_t da, db, dpos;          // their change per row (0 or 1)
    int32_t mode;                  // 0 none, 1 lo letter along the row, 2 hi letter along the row, 3 neither
    int64_t inner_lo;              // global coordinate of the tile's column 0 (predicate letter)
    int64_t pair0;                 // rope: global pair index of the tile's column 0
    int32_t vec, pad;
    int64_t out_inner;
};

template <int MAP, bool kVec, int NIN, int MASK, int DT>
__global__ void __launch_bounds__(kThreads, 3) ewise_kernel(const EwParams p) {
    constexpr int V = kVec ? 8 : 1;
    __shared__ TileGeom g;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int mask = MASK < 0 ? p.stream_mask : MASK;
    for (int64_t t = blockIdx.x; t < p.ntiles; t += gridDim.x) {
        const EwTile T = p.tiles[t];
        if constexpr (kBoundsCheck) {
            if (!view_in(p.items[T.item], p.n_in, p.in_elems, p.out_elems) || T.row0 < 0 ||
                T.row0 + T.nrows > p.items[T.item].rows || T.col0 < 0 || T.col0 + T.ncols > p.items[T.item].len) {
                if (threadIdx.x == 0) bounds_fail(p.err);
                continue;
            }
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            const EwItem &it = p.items[T.item];
            int64_t cd[kViewDims];
            decode_row(it, T.row0, cd);
            const int last = it.nd - 1, sec = it.nd - 2;
            // a tile spanning several runs starts at a run boundary and stays
            // inside one run of the second-innermost dim (the host cuts them so)
            g.e1 = (last >= 0 && T.nrows > it.ext[last] - cd[last]) ? (int32_t)it.ext[last] : 0;
            g.vec = it.vec;
            g.out_inner = it.out_inner;
            g.ooff = it.out_base + T.col0 * it.out_inner;
            g.ostr = last >= 0 ? it.ostr[last] : 0;
            g.ostr2 = sec >= 0 ? it.ostr[sec] : 0;
            for (int k = 0; k < kMaxIn; k++) {
                int64_t o = it.in_base[k] + T.col0 * it.in_inner[k];
                for (int d = 0; d < it.nd; d++) o += cd[d] * it.istr[k][d];
                g.ioff[k] = o;
                g.istr[k] = last >= 0 ? it.istr[k][last] : 0;
                g.istr2[k] = sec >= 0 ? it.istr[k][sec] : 0;
                g.iinn[k] = it.in_inner[k];
            }
            for (int d = 0; d < it.nd; d++) g.ooff += cd[d] * it.ostr[d];
            g.mode = 0;
            g.a0 = g.b0 = 0;
            g.da = g.db = 0;
            if (p.pred) {
                g.a0 = special_coord(it, 0, cd, 0);
                g.b0 = special_coord(it, 1, cd, 0);
                g.da = it.sdim[0] == last && last >= 0 ? 1 : 0;
                g.db = it.sdim[1] == last && last >= 0 ? 1 : 0;
                g.da2 = it.sdim[0] == sec && sec >= 0 ? 1 : 0;
                g.db2 = it.sdim[1] == sec && sec >= 0 ? 1 : 0;
                if (it.sdim[0] == kViewDims) {
                    g.mode = 1;
                    g.inner_lo = it.slo[0] + T.col0;
                } else if (it.sdim[1] == kViewDims) {
                    g.mode = 2;
                    g.inner_lo = it.slo[1] + T.col0;
                } else {
                    g.mode = 3;
                }
            }
            g.pos0 = 0;
            g.dpos = g.dpos2 = 0;
            g.pair0 = 0;
            if (MAP == EA_MAP_ROPE) {
                g.pos0 = special_coord(it, 2, cd, 0);
                g.dpos = it.sdim[2] == last && last >= 0 ? 1 : 0;
                g.dpos2 = it.sdim[2] == sec && sec >= 0 ? 1 : 0;
                g.pair0 = (it.inner_lo + T.col0) >> 1;
            }
        }
        __syncthreads();
        if ((g.vec != 0) != kVec) continue;
        const int cpr = (int)(T.ncols / V);  // chunks per row in this tile
        // lanes per row: a power of two giving each lane about U chunks of
        // the row, so short rows pack several to a warp and every lane keeps
        // several loads in flight
        constexpr int NSr = MASK < 0 ? NIN : ((MASK & 1) + ((MASK >> 1) & 1) + ((MASK >> 2) & 1));
        constexpr int Ur = Batch<kVec, NSr, DT, MAP>::U;
        int lpr = 32;
        while (lpr > 1 && lpr * Ur > cpr) lpr /= 2;
        const int rpw = 32 / lpr;             // rows per warp pass
        const int sub = lane / lpr, sl = lane % lpr;
        for (int64_t r = (int64_t)warp * rpw + sub; r < T.nrows; r += (int64_t)kWarps * rpw) {
            // row r of the tile: q whole runs of the innermost row dim, then rem rows
            const int64_t q = g.e1 ? (int)r / g.e1 : 0, rem = g.e1 ? r - q * g.e1 : r;
            Row<NIN> w;
            w.ooff = g.ooff + rem * g.ostr + q * g.ostr2;
#pragma unroll
            for (int k = 0; k < NIN; k++) {
                w.ioff[k] = g.ioff[k] + rem * g.istr[k] + q * g.istr2[k];
                w.iinn[k] = g.iinn[k];
                w.bc[k] = streams(mask, k) ? 1.0f : ld_elem(p.in[k], p.in_dtype[k], w.ioff[k]);
            }
            int64_t cmin = 0, cmax = T.ncols - 1;
            const int64_t av = g.a0 + g.da * rem + g.da2 * q, bv = g.b0 + g.db * rem + g.db2 * q;
            if (g.mode == 1) cmax = min64(cmax, bv - g.inner_lo);
            else if (g.mode == 2) cmin = max64(cmin, av - g.inner_lo);
            else if (g.mode == 3 && av > bv) cmin = T.ncols;
            const bool masked = cmin > 0 || cmax < T.ncols - 1;
            w.cmin = (int)max64(cmin, -1);
            w.cmax = (int)min64(cmax, T.ncols);
            w.tab = nullptr;
            w.pair0 = g.pair0;
            if (MAP == EA_MAP_ROPE)
                w.tab = reinterpret_cast<const float2 *>(p.rope_table) + (g.pos0 + g.dpos * rem + g.dpos2 * q) * p.rope_half;
            ew_row<MAP, kVec, NIN, MASK, DT>(p, w, cpr, sl, lpr, masked, g.out_inner);
        }
    }
}

// DT: the dtype every streamed input shares (1 bf16, 2 fp32), 0 if mixed.
template <int MAP, int NIN, int MASK>
cudaError_t go(const EwParams &p, int64_t grid, bool vec, cudaStream_t st) {
    int dt = -1;
    for (int k = 0; k < NIN; k++) {
        if (MASK >= 0 && !((MASK >> k) & 1)) continue;
        const int d = p.in_dtype[k] == EA_BF16 ? 1 : 2;
        dt = dt < 0 ? d : (dt == d ? dt : 0);
    }
    if (MASK < 0 || dt <= 0 || !vec) {
        if (vec) ewise_kernel<MAP, true, NIN, MASK, 0><<<(unsigned)grid, kThreads, 0, st>>>(p);
        else ewise_kernel<MAP, false, NIN, MASK, 0><<<(unsigned)grid, kThreads, 0, st>>>(p);
    } else if (dt == 1) {
        ewise_kernel<MAP, true, NIN, MASK, 1><<<(unsigned)grid, kThreads, 0, st>>>(p);
    } else {
        ewise_kernel<MAP, true, NIN, MASK, 2><<<(unsigned)grid, kThreads, 0, st>>>(p);
    }
    return cudaGetLastError();
}

// Specialised instances for the (map, inputs, streamed inputs) of the hot
// path; everything else runs the generic instance (map and mask read at
// run time).
cudaError_t dispatch(const EwParams &p, int64_t grid, bool vec, cudaStream_t st) {
    const int m = p.stream_mask, n = p.n_in;
    switch (p.map) {
    case EA_MAP_ROPE:
        if (n == 1 && m == 1) return go<EA_MAP_ROPE, 1, 1>(p, grid, vec, st);
        break;
    case EA_MAP_IDENTITY:
        if (n == 1 && m == 1) return go<EA_MAP_IDENTITY, 1, 1>(p, grid, vec, st);
        break;
    case EA_MAP_ADD:
        if (n == 2 && m == 3) return go<EA_MAP_ADD, 2, 3>(p, grid, vec, st);
        break;
    case EA_MAP_SILU_MUL:
        if (n == 2 && m == 3) return go<EA_MAP_SILU_MUL, 2, 3>(p, grid, vec, st);
        break;
    case EA_MAP_PRODUCT:
        if (n == 2 && m == 3) return go<EA_MAP_PRODUCT, 2, 3>(p, grid, vec, st);
        break;
    case EA_MAP_EXP_SUB:
        if (n == 2 && m == 1) return go<EA_MAP_EXP_SUB, 2, 1>(p, grid, vec, st);
        break;
    case EA_MAP_RMS_APPLY:
        if (n == 3 && m == 5) return go<EA_MAP_RMS_APPLY, 3, 5>(p, grid, vec, st);
        break;
    case EA_MAP_EXP_SUB_DIV:
        if (n == 3 && m == 1) return go<EA_MAP_EXP_SUB_DIV, 3, 1>(p, grid, vec, st);
        break;
    default:
        break;
    }
    if (p.map == EA_MAP_ROPE) return go<EA_MAP_ROPE, 1, -1>(p, grid, vec, st);
    if (n == 1) return go<-1, 1, -1>(p, grid, vec, st);
    if (n == 2) return go<-1, 2, -1>(p, grid, vec, st);
    return go<-1, 3, -1>(p, grid, vec, st);
}

}  // namespace

cudaError_t launch_ewise(const EwParams &p, int num_sms, cudaStream_t st) {
    int64_t grid = std::min<int64_t>(p.ntiles, (int64_t)num_sms * 8);
    cudaError_t e = cudaSuccess;
    if (p.has_vec) e = dispatch(p, grid, true, st);
    if (e == cudaSuccess && p.has_scalar) e = dispatch(p, grid, false, st);
    return e;
}

}  // namespace ea
