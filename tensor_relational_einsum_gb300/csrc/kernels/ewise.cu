// ewise.cu -- elementwise join-agg kernel (aggregation NONE).
//
// "Every Kernel Is a Join", Section 1: elementwise operations (ReLU, SiLU,
// residual adds, normalisation steps) are joins of relations on equal keys
// -- or of a relation with a broadcast one, keyed by a subset of its
// letters -- followed by a map and no aggregation.  Each function
// specification of such a join-agg owns one output block; the host gives
// every block a strided view (EwItem) and cuts it into tiles of ~32K
// cells.  Each thread maps 8 consecutive cells of a row with 16-byte loads
// and stores (fp32 math), so the kernel streams HBM at full width.
// Broadcast inputs (stride 0 along the row) are read once per chunk.
#include <algorithm>

#include "dev_common.cuh"

namespace ea {

namespace {

constexpr int kThreads = 256;

template <bool kVec>
__global__ void __launch_bounds__(kThreads) ewise_kernel(const EwParams p) {
    constexpr int V = kVec ? 8 : 1;
    for (int64_t t = blockIdx.x; t < p.ntiles; t += gridDim.x) {
        const EwTile T = p.tiles[t];
        const EwItem &it = p.items[T.item];
        if ((it.vec != 0) != kVec) continue;
        const int64_t cpr = T.ncols / V;
        const int64_t n = T.nrows * cpr;
        for (int64_t c = threadIdx.x; c < n; c += kThreads) {
            int64_t rr = c / cpr;
            int64_t col = T.col0 + (c - rr * cpr) * V;
            int64_t coord[kViewDims];
            decode_row(it, T.row0 + rr, coord);
            int64_t ooff = it.out_base + col * it.out_inner;
            int64_t ioff[kMaxIn];
            for (int k = 0; k < p.n_in; k++) ioff[k] = it.in_base[k] + col * it.in_inner[k];
#pragma unroll
            for (int d = 0; d < kViewDims; d++) {
                if (d >= it.nd) break;
                ooff += coord[d] * it.ostr[d];
                for (int k = 0; k < p.n_in; k++) ioff[k] += coord[d] * it.istr[k][d];
            }
            float v[kMaxIn][V];
            for (int k = 0; k < kMaxIn; k++) {
                if (k >= p.n_in) {
#pragma unroll
                    for (int e = 0; e < V; e++) v[k][e] = 1.0f;
                } else if (kVec && it.in_inner[k] == 1) {
                    ld8(p.in[k], p.in_dtype[k], ioff[k], v[k]);
                } else if (it.in_inner[k] == 0) {
                    float s = ld_elem(p.in[k], p.in_dtype[k], ioff[k]);
#pragma unroll
                    for (int e = 0; e < V; e++) v[k][e] = s;
                } else {
#pragma unroll
                    for (int e = 0; e < V; e++) v[k][e] = ld_elem(p.in[k], p.in_dtype[k], ioff[k] + e * it.in_inner[k]);
                }
            }
            float o[V];
            if (p.map == EA_MAP_ROPE) {
                // Rotate interleaved pairs (2i, 2i+1) of the pair letter by the
                // angle of (position, i) in the (cos, sin) table.
                int64_t pos = special_coord(it, 2, coord, 0);
                const float2 *tab = reinterpret_cast<const float2 *>(p.rope_table) + pos * p.rope_half;
#pragma unroll
                for (int e = 0; e < V; e += 2) {
                    int64_t pi = (it.inner_lo + col + e) >> 1;
                    float2 cs = __ldg(tab + pi);
                    float x0 = v[0][e], x1 = (e + 1 < V) ? v[0][e + 1] : 0.0f;
                    o[e] = x0 * cs.x - x1 * cs.y;
                    if (e + 1 < V) o[e + 1] = x0 * cs.y + x1 * cs.x;
                }
                if (!kVec) {
                    // scalar path: rotate with the partner cell of the pair
                    int64_t g = it.inner_lo + col;
                    int64_t pi = g >> 1;
                    float2 cs = __ldg(tab + pi);
                    float partner = ld_elem(p.in[0], p.in_dtype[0], ioff[0] + ((g & 1) ? -1 : 1) * it.in_inner[0]);
                    o[0] = (g & 1) ? partner * cs.y + v[0][0] * cs.x : v[0][0] * cs.x - partner * cs.y;
                }
            } else {
#pragma unroll
                for (int e = 0; e < V; e++) o[e] = cell_map(p.map, v[0][e], v[1][e], v[2][e], p.scale, p.eps);
            }
            if (p.pred) {
#pragma unroll
                for (int e = 0; e < V; e++) {
                    int64_t a = special_coord(it, 0, coord, col + e), b = special_coord(it, 1, coord, col + e);
                    if (a > b) o[e] = 0.0f;  // a cell the predicate removes holds 0
                }
            }
            if (kVec) st8(p.out, p.out_dtype, ooff, o);
            else st_elem(p.out, p.out_dtype, ooff, o[0]);
        }
    }
}

}  // namespace

cudaError_t launch_ewise(const EwParams &p, int num_sms, cudaStream_t st) {
    int64_t grid = std::min<int64_t>(p.ntiles, (int64_t)num_sms * 8);
    cudaError_t e = cudaSuccess;
    if (p.has_vec) {
        ewise_kernel<true><<<(unsigned)grid, kThreads, 0, st>>>(p);
        e = cudaGetLastError();
    }
    if (e == cudaSuccess && p.has_scalar) {
        ewise_kernel<false><<<(unsigned)grid, kThreads, 0, st>>>(p);
        e = cudaGetLastError();
    }
    return e;
}

}  // namespace ea
