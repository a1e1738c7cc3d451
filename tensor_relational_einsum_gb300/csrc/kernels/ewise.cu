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
template <bool kVec, int NS, int DT>
struct Batch {
    static constexpr int V = kVec ? 8 : 1;
    static constexpr int BYTES = DT == 1 ? 16 : 32;  // one chunk of one input
    static constexpr int U = !kVec ? 4 : (NS <= 1 ? 128 / BYTES : (128 / BYTES) / NS > 0 ? (128 / BYTES) / NS : 1);
};

// Stream one row: chunks sl, sl + lpr, ... of V cells, U chunks per batch.
// DT: 1 = streamed inputs are bf16, 2 = fp32, 0 = read at run time.
template <int MAP, bool kVec, int NIN, int MASK, int DT>
__device__ __forceinline__ void ew_row(const EwParams &p, const Row<NIN> &w, int cpr, int sl, int lpr, bool masked,
                                       int64_t out_inner) {
    constexpr int V = kVec ? 8 : 1;
    constexpr int NS = MASK < 0 ? NIN : ((MASK & 1) + ((MASK >> 1) & 1) + ((MASK >> 2) & 1));
    constexpr int NSV = NS > 0 ? NS : 1;
    constexpr int U = Batch<kVec, NS, DT>::U;
    constexpr bool kRaw = kVec && DT != 0 && MASK >= 0;
    constexpr bool kB16 = DT == 1;
    const int mask = MASK < 0 ? p.stream_mask : MASK;
    for (int c0 = sl; c0 < cpr; c0 += lpr * U) {
        uint4 raw[kRaw ? U : 1][kRaw ? NSV : 1][kB16 ? 1 : 2];
        float v[kRaw ? 1 : U][kRaw ? 1 : NSV][kRaw ? 1 : V];
#pragma unroll
        for (int u = 0; u < U; u++) {
            const int c = c0 + u * lpr;
            if (c >= cpr) continue;
            const int64_t col = (int64_t)c * V;
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
#pragma unroll
                    for (int e = 0; e < V; e += 2) {
                        const float2 cs = __ldg(w.tab + w.pair0 + ((col + e) >> 1));
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

template <int MAP, bool kVec, int NIN, int MASK, int DT>
__global__ void __launch_bounds__(kThreads, 3) ewise_kernel(const EwParams p) {
    constexpr int V = kVec ? 8 : 1;
    __shared__ EwItem sit;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int mask = MASK < 0 ? p.stream_mask : MASK;
    for (int64_t t = blockIdx.x; t < p.ntiles; t += gridDim.x) {
        const EwTile T = p.tiles[t];
        __syncthreads();
        {
            const int64_t *src = reinterpret_cast<const int64_t *>(p.items + T.item);
            int64_t *dst = reinterpret_cast<int64_t *>(&sit);
            for (int i = threadIdx.x; i < (int)(sizeof(EwItem) / 8); i += kThreads) dst[i] = src[i];
        }
        __syncthreads();
        if ((sit.vec != 0) != kVec) continue;
        const int cpr = (int)(T.ncols / V);  // chunks per row in this tile
        // lanes per row: a power of two giving each lane about U chunks of
        // the row, so short rows pack several to a warp and every lane keeps
        // several loads in flight
        constexpr int NSr = MASK < 0 ? NIN : ((MASK & 1) + ((MASK >> 1) & 1) + ((MASK >> 2) & 1));
        constexpr int Ur = Batch<kVec, NSr, DT>::U;
        int lpr = 32;
        while (lpr > 1 && lpr * Ur > cpr) lpr /= 2;
        const int rpw = 32 / lpr;             // rows per warp pass
        const int sub = lane / lpr, sl = lane % lpr;
        const int nd = sit.nd;
        for (int64_t r = (int64_t)warp * rpw + sub; r < T.nrows; r += (int64_t)kWarps * rpw) {
            int64_t coord[kViewDims];
            decode_row(sit, T.row0 + r, coord);
            Row<NIN> w;
            w.ooff = sit.out_base + T.col0 * sit.out_inner;
#pragma unroll
            for (int k = 0; k < NIN; k++) {
                w.ioff[k] = sit.in_base[k] + T.col0 * sit.in_inner[k];
                w.iinn[k] = sit.in_inner[k];
            }
            for (int d = 0; d < nd; d++) {
                w.ooff += coord[d] * sit.ostr[d];
#pragma unroll
                for (int k = 0; k < NIN; k++) w.ioff[k] += coord[d] * sit.istr[k][d];
            }
#pragma unroll
            for (int k = 0; k < NIN; k++)
                w.bc[k] = streams(mask, k) ? 1.0f : ld_elem(p.in[k], p.in_dtype[k], w.ioff[k]);
            int64_t cmin = 0, cmax = T.ncols - 1;
            if (p.pred) {
                if (sit.sdim[0] == kViewDims)  // the predicate's lo letter runs along the row
                    cmax = min64(cmax, special_coord(sit, 1, coord, 0) - sit.slo[0] - T.col0);
                else if (sit.sdim[1] == kViewDims)
                    cmin = max64(cmin, special_coord(sit, 0, coord, 0) - sit.slo[1] - T.col0);
                else if (special_coord(sit, 0, coord, 0) > special_coord(sit, 1, coord, 0))
                    cmin = T.ncols;
            }
            const bool masked = cmin > 0 || cmax < T.ncols - 1;
            w.cmin = (int)max64(cmin, -1);
            w.cmax = (int)min64(cmax, T.ncols);
            w.tab = nullptr;
            w.pair0 = 0;
            if (MAP == EA_MAP_ROPE) {
                w.tab = reinterpret_cast<const float2 *>(p.rope_table) + special_coord(sit, 2, coord, 0) * p.rope_half;
                w.pair0 = (sit.inner_lo + T.col0) >> 1;
            }
            ew_row<MAP, kVec, NIN, MASK, DT>(p, w, cpr, sl, lpr, masked, sit.out_inner);
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
