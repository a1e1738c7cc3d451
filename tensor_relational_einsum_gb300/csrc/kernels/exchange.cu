// exchange.cu -- the exchange (re-blocking) kernel.
//
// "Every Kernel Is a Join", Section 5.3: the overlay of the producer and
// consumer tilings cuts the tensor into atoms; every block of either tiling
// is a disjoint union of atoms, so the re-blocking is a set of atom copies
// (decompose from the source blocks, recompose into the destination
// blocks).  On one GPU both halves collapse into one pass: each atom is
// read once from its source block and written once into its destination
// block.  The host plans every atom as rows of a contiguous run (XSeg) cut
// into ~64 KiB tiles (XTile); the kernel is a persistent grid-stride loop
// over tiles: each tile's segment is staged in shared memory, a warp (or a
// slice of one) copies a row with eight 16-byte loads in flight per lane.
// The work is a pure HBM stream (no reuse), so the loads bypass L1 and the
// stores are marked streaming.
#include <algorithm>

#include "dev_common.cuh"

namespace ea {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kUnroll = 8;  // 16-byte chunks in flight per lane

__device__ __forceinline__ void seg_row(const XSeg &g, int64_t r, int64_t *so, int64_t *dof) {
    int64_t s = g.src_off, d = g.dst_off;
    for (int i = g.nd - 1; i >= 0; i--) {
        int64_t e = g.ext[i];
        int64_t c = (i == 0) ? r : r % e;
        if (i != 0) r /= e;
        s += c * g.sstr[i];
        d += c * g.dstr[i];
    }
    *so = s;
    *dof = d;
}

__global__ void __launch_bounds__(kThreads, 3) exchange_kernel(const XSeg *__restrict__ segs,
                                                            const XTile *__restrict__ tiles, int64_t ntiles,
                                                            const char *__restrict__ src, char *__restrict__ dst,
                                                            int esize, int64_t src_elems, int64_t dst_elems, int *err) {
    __shared__ XSeg sg;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
        const XTile T = tiles[t];
        __syncthreads();
        if (threadIdx.x < (int)(sizeof(XSeg) / 8))
            reinterpret_cast<int64_t *>(&sg)[threadIdx.x] = reinterpret_cast<const int64_t *>(segs + T.seg)[threadIdx.x];
        __syncthreads();
        if constexpr (kBoundsCheck) {
            if (!seg_in(sg, T, src_elems, dst_elems)) {
                if (threadIdx.x == 0) bounds_fail(err);
                continue;
            }
        }
        if (sg.vec) {
            // a warp (or a slice of one, for short rows) copies a row: each
            // lane keeps kUnroll 16-byte loads in flight before it stores
            const int cpr = (int)(T.ncols * esize / 16);
            int lpr = 32;
            while (lpr > 1 && lpr * kUnroll > cpr) lpr /= 2;
            const int rpw = 32 / lpr, sub = lane / lpr, sl = lane % lpr;
            const int64_t col_bytes = T.col0 * esize;
            for (int64_t r = (int64_t)warp * rpw + sub; r < T.nrows; r += (int64_t)kWarps * rpw) {
                int64_t so, dof;
                seg_row(sg, T.row0 + r, &so, &dof);
                const char *sp = src + so * esize + col_bytes;
                char *dp = dst + dof * esize + col_bytes;
                for (int c0 = sl; c0 < cpr; c0 += lpr * kUnroll) {
                    uint4 v[kUnroll];
#pragma unroll
                    for (int u = 0; u < kUnroll; u++) {
                        const int c = c0 + u * lpr;
                        if (c < cpr)
                            asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                                         : "=r"(v[u].x), "=r"(v[u].y), "=r"(v[u].z), "=r"(v[u].w)
                                         : "l"(sp + (int64_t)c * 16));
                    }
#pragma unroll
                    for (int u = 0; u < kUnroll; u++) {
                        const int c = c0 + u * lpr;
                        if (c < cpr) __stcs(reinterpret_cast<uint4 *>(dp + (int64_t)c * 16), v[u]);
                    }
                }
            }
        } else {
            const int64_t n = T.nrows * T.ncols;
            for (int64_t c = threadIdx.x; c < n; c += kThreads) {
                int64_t rr = c / T.ncols;
                int64_t q = c - rr * T.ncols + T.col0;
                int64_t so, dof;
                seg_row(sg, T.row0 + rr, &so, &dof);
                const char *sp = src + (so + q) * esize;
                char *dp = dst + (dof + q) * esize;
                if (esize == 4) *reinterpret_cast<uint32_t *>(dp) = *reinterpret_cast<const uint32_t *>(sp);
                else *reinterpret_cast<uint16_t *>(dp) = *reinterpret_cast<const uint16_t *>(sp);
            }
        }
    }
}

}  // namespace

cudaError_t launch_exchange(const XSeg *segs, const XTile *tiles, int64_t ntiles, const char *src, char *dst,
                            int esize, int num_sms, cudaStream_t st, int64_t src_elems, int64_t dst_elems, int *err) {
    // Eight resident CTAs of 256 threads per SM; persistent over the tiles.
    int64_t grid = std::min<int64_t>(ntiles, (int64_t)num_sms * 8);
    exchange_kernel<<<(unsigned)grid, kThreads, 0, st>>>(segs, tiles, ntiles, src, dst, esize, src_elems, dst_elems,
                                                         err);
    return cudaGetLastError();
}

}  // namespace ea
