// rowreduce.cu -- row-reduction join-agg kernel (aggregation SUM or MAX
// over the trailing letters of input 0).
//
// "Every Kernel Is a Join", Section 1 and Definition 3.7: softmax and
// normalisation are a join (the scores, possibly with a broadcast row
// statistic) followed by an aggregation over the reduced letters.  When the
// reduced letters are split into blocks, every output block has one
// function specification per block of the reduced letters, and step (2)
// combines their outputs with the aggregation op.  Here one warp owns one
// output cell: it walks every function specification of the cell's group,
// maps the row segment 8 cells per lane (16-byte loads), accumulates in
// fp32, and combines lanes with warp shuffles -- the per-tuple results and
// their aggregation are fused, with no partial results in memory.
#include <algorithm>
#include <math.h>

#include "dev_common.cuh"

namespace ea {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

__device__ __forceinline__ float agg_op(int agg, float a, float b) { return agg == EA_AGG_MAX ? fmaxf(a, b) : a + b; }

__global__ void __launch_bounds__(kThreads) rowreduce_kernel(const RrParams p) {
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const float ident = p.agg == EA_AGG_MAX ? -INFINITY : 0.0f;
    for (int64_t t = blockIdx.x; t < p.ntiles; t += gridDim.x) {
        const RrTile T = p.tiles[t];
        const RrGroup G = p.groups[T.group];
        for (int64_t rr = warp; rr < T.nrows; rr += kWarps) {
            const int64_t r = T.row0 + rr;
            float acc = ident;
            int64_t coord[kViewDims];
            for (int i = G.i0; i < G.i1; i++) {
                const EwItem &it = p.items[i];
                decode_row(it, r, coord);
                int64_t ioff[kMaxIn];
                for (int k = 0; k < p.n_in; k++) {
                    ioff[k] = it.in_base[k];
                    for (int d = 0; d < it.nd; d++) ioff[k] += coord[d] * it.istr[k][d];
                }
                // broadcast operands: one value per row
                float bc[kMaxIn] = {1.0f, 1.0f, 1.0f};
                for (int k = 1; k < p.n_in; k++)
                    if (it.in_inner[k] == 0) bc[k] = ld_elem(p.in[k], p.in_dtype[k], ioff[k]);
                const int64_t len = it.len;
                if (it.vec) {
                    for (int64_t c0 = (int64_t)lane * 8; c0 < len; c0 += 32 * 8) {
                        float v[kMaxIn][8];
                        ld8(p.in[0], p.in_dtype[0], ioff[0] + c0, v[0]);
                        for (int k = 1; k < kMaxIn; k++) {
                            if (k < p.n_in && it.in_inner[k] == 1) ld8(p.in[k], p.in_dtype[k], ioff[k] + c0, v[k]);
                            else
#pragma unroll
                                for (int e = 0; e < 8; e++) v[k][e] = bc[k];
                        }
#pragma unroll
                        for (int e = 0; e < 8; e++) {
                            if (p.pred) {
                                int64_t a = special_coord(it, 0, coord, c0 + e), b = special_coord(it, 1, coord, c0 + e);
                                if (a > b) continue;
                            }
                            acc = agg_op(p.agg, acc, cell_map(p.map, v[0][e], v[1][e], v[2][e], p.scale, p.eps));
                        }
                    }
                } else {
                    for (int64_t c = lane; c < len; c += 32) {
                        if (p.pred) {
                            int64_t a = special_coord(it, 0, coord, c), b = special_coord(it, 1, coord, c);
                            if (a > b) continue;
                        }
                        float v0 = ld_elem(p.in[0], p.in_dtype[0], ioff[0] + c);
                        float v1 = p.n_in > 1 ? (it.in_inner[1] ? ld_elem(p.in[1], p.in_dtype[1], ioff[1] + c) : bc[1]) : 1.0f;
                        float v2 = p.n_in > 2 ? (it.in_inner[2] ? ld_elem(p.in[2], p.in_dtype[2], ioff[2] + c) : bc[2]) : 1.0f;
                        acc = agg_op(p.agg, acc, cell_map(p.map, v0, v1, v2, p.scale, p.eps));
                    }
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) acc = agg_op(p.agg, acc, __shfl_xor_sync(0xffffffffu, acc, o));
            if (lane == 0) {
                const EwItem &it0 = p.items[G.i0];
                decode_row(it0, r, coord);
                int64_t ooff = it0.out_base;
                for (int d = 0; d < it0.nd; d++) ooff += coord[d] * it0.ostr[d];
                st_elem(p.out, p.out_dtype, ooff, acc);
            }
        }
    }
}

}  // namespace

cudaError_t launch_rowreduce(const RrParams &p, int num_sms, cudaStream_t st) {
    int64_t grid = std::min<int64_t>(p.ntiles, (int64_t)num_sms * 8);
    rowreduce_kernel<<<(unsigned)grid, kThreads, 0, st>>>(p);
    return cudaGetLastError();
}

}  // namespace ea
