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
// over tiles with four 16-byte loads in flight per thread.  The work is a
// pure HBM stream (no reuse), so the loads bypass L1 and the stores are
// marked streaming.
#include <algorithm>

#include "../ea_internal.h"

namespace ea {

namespace {

constexpr int kThreads = 512;
constexpr int kUnroll = 4;

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

__global__ void __launch_bounds__(kThreads) exchange_kernel(const XSeg *__restrict__ segs,
                                                            const XTile *__restrict__ tiles, int64_t ntiles,
                                                            const char *__restrict__ src, char *__restrict__ dst,
                                                            int esize) {
    for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
        const XTile T = tiles[t];
        const XSeg &g = segs[T.seg];
        if (g.vec) {
            // 16-byte chunks: cpr per row.
            const int64_t cpr = T.ncols * esize / 16;
            const int64_t n = T.nrows * cpr;
            const int64_t col_bytes = T.col0 * esize;
            for (int64_t base = threadIdx.x; base < n; base += (int64_t)kThreads * kUnroll) {
                uint4 v[kUnroll];
                int64_t dofs[kUnroll];
#pragma unroll
                for (int u = 0; u < kUnroll; u++) {
                    int64_t c = base + (int64_t)u * kThreads;
                    dofs[u] = -1;
                    if (c < n) {
                        int64_t rr = (cpr == 1) ? c : c / cpr;
                        int64_t q = c - rr * cpr;
                        int64_t so, dof;
                        seg_row(g, T.row0 + rr, &so, &dof);
                        const char *sp = src + so * esize + col_bytes + q * 16;
                        asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                                     : "=r"(v[u].x), "=r"(v[u].y), "=r"(v[u].z), "=r"(v[u].w)
                                     : "l"(sp));
                        dofs[u] = dof * esize + col_bytes + q * 16;
                    }
                }
#pragma unroll
                for (int u = 0; u < kUnroll; u++)
                    if (dofs[u] >= 0) __stcs(reinterpret_cast<uint4 *>(dst + dofs[u]), v[u]);
            }
        } else {
            const int64_t n = T.nrows * T.ncols;
            for (int64_t c = threadIdx.x; c < n; c += kThreads) {
                int64_t rr = c / T.ncols;
                int64_t q = c - rr * T.ncols + T.col0;
                int64_t so, dof;
                seg_row(g, T.row0 + rr, &so, &dof);
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
                            int esize, int num_sms, cudaStream_t st) {
    // Four resident CTAs of 512 threads per SM; persistent over the tiles.
    int64_t grid = std::min<int64_t>(ntiles, (int64_t)num_sms * 4);
    exchange_kernel<<<(unsigned)grid, kThreads, 0, st>>>(segs, tiles, ntiles, src, dst, esize);
    return cudaGetLastError();
}

}  // namespace ea
