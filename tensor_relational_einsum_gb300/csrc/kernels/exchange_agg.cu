// exchange_agg.cu -- the exchange with aggregation ("Every Kernel Is a
// Join", Section 5.3 and Example 5.4).
//
// The producer left m unaggregated copies of every block (one per function
// specification of its group); the consumer needs every block of another
// tiling, fully aggregated.  The overlay of the two tilings cuts the tensor
// into atoms; each destination atom is the (+)-aggregate of the m copies of
// the source atom at the same coordinates ("X1 + Y1" of the example).  On
// one GPU the decompose, the aggregation and the recompose are one pass:
// every atom row is read once from each copy, combined in copy order in fp32
// and written once.  The plan is the plain exchange's (atoms as rows of a
// contiguous run, ~64 KiB tiles); copy q lies copy_stride elements after
// copy 0 in the source arena.
#include <algorithm>

#include <cuda_bf16.h>

#include "dev_common.cuh"

namespace ea {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kUnroll = 4;  // 16-byte chunks per lane per copy in flight

__device__ __forceinline__ void seg_row_a(const XSeg &g, int64_t r, int64_t *so, int64_t *dof) {
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

template <bool kBf16, int AGG>
__device__ __forceinline__ void combine16(uint4 &acc_raw, float *acc, const uint4 &v, bool first) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    if constexpr (kBf16) {
#pragma unroll
        for (int e = 0; e < 4; e++) {
            const float lo = __uint_as_float(w[e] << 16), hi = __uint_as_float(w[e] & 0xFFFF0000u);
            if (first) {
                acc[2 * e] = lo;
                acc[2 * e + 1] = hi;
            } else if (AGG == EA_AGG_MAX) {
                acc[2 * e] = fmaxf(acc[2 * e], lo);
                acc[2 * e + 1] = fmaxf(acc[2 * e + 1], hi);
            } else {
                acc[2 * e] += lo;
                acc[2 * e + 1] += hi;
            }
        }
    } else {
#pragma unroll
        for (int e = 0; e < 4; e++) {
            const float x = __uint_as_float(w[e]);
            acc[e] = first ? x : AGG == EA_AGG_MAX ? fmaxf(acc[e], x) : acc[e] + x;
        }
    }
    (void)acc_raw;
}

template <bool kBf16>
__device__ __forceinline__ uint4 pack16(const float *acc) {
    uint4 o;
    if constexpr (kBf16) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; e++) {
            __nv_bfloat162 h = __floats2bfloat162_rn(acc[2 * e], acc[2 * e + 1]);
            w[e] = *reinterpret_cast<uint32_t *>(&h);
        }
        o = make_uint4(w[0], w[1], w[2], w[3]);
    } else {
        o = make_uint4(__float_as_uint(acc[0]), __float_as_uint(acc[1]), __float_as_uint(acc[2]),
                       __float_as_uint(acc[3]));
    }
    return o;
}

template <bool kBf16, int AGG>
__global__ void __launch_bounds__(kThreads, 3) exchange_agg_kernel(const XSeg *__restrict__ segs,
                                                                const XTile *__restrict__ tiles, int64_t ntiles,
                                                                const char *__restrict__ src, char *__restrict__ dst,
                                                                int ncopies, int64_t copy_stride, int64_t src_elems,
                                                                int64_t dst_elems, int *err) {
    constexpr int esize = kBf16 ? 2 : 4;
    constexpr int EPC = 16 / esize;  // elements per 16-byte chunk
    __shared__ XSeg sg;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int64_t cbytes = copy_stride * esize;
    for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
        const XTile T = tiles[t];
        __syncthreads();
        if (threadIdx.x < (int)(sizeof(XSeg) / 8))
            reinterpret_cast<int64_t *>(&sg)[threadIdx.x] = reinterpret_cast<const int64_t *>(segs + T.seg)[threadIdx.x];
        __syncthreads();
        if constexpr (kBoundsCheck) {
            if (!seg_in(sg, T, src_elems, dst_elems, ncopies, copy_stride)) {
                if (threadIdx.x == 0) bounds_fail(err);
                continue;
            }
        }
        if (sg.vec) {
            const int cpr = (int)(T.ncols * esize / 16);
            int lpr = 32;
            while (lpr > 1 && lpr * kUnroll > cpr) lpr /= 2;
            const int rpw = 32 / lpr, sub = lane / lpr, sl = lane % lpr;
            const int64_t col_bytes = T.col0 * esize;
            for (int64_t r = (int64_t)warp * rpw + sub; r < T.nrows; r += (int64_t)kWarps * rpw) {
                int64_t so, dof;
                seg_row_a(sg, T.row0 + r, &so, &dof);
                const char *sp = src + so * esize + col_bytes;
                char *dp = dst + dof * esize + col_bytes;
                for (int c0 = sl; c0 < cpr; c0 += lpr * kUnroll) {
                    float acc[kUnroll][EPC];
                    uint4 dummy;
                    for (int q = 0; q < ncopies; q++) {
                        uint4 v[kUnroll];
#pragma unroll
                        for (int u = 0; u < kUnroll; u++) {
                            const int c = c0 + u * lpr;
                            if (c < cpr)
                                asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                                             : "=r"(v[u].x), "=r"(v[u].y), "=r"(v[u].z), "=r"(v[u].w)
                                             : "l"(sp + q * cbytes + (int64_t)c * 16));
                        }
#pragma unroll
                        for (int u = 0; u < kUnroll; u++)
                            if (c0 + u * lpr < cpr) combine16<kBf16, AGG>(dummy, acc[u], v[u], q == 0);
                    }
#pragma unroll
                    for (int u = 0; u < kUnroll; u++) {
                        const int c = c0 + u * lpr;
                        if (c < cpr) __stcs(reinterpret_cast<uint4 *>(dp + (int64_t)c * 16), pack16<kBf16>(acc[u]));
                    }
                }
            }
        } else {
            const int64_t n = T.nrows * T.ncols;
            for (int64_t c = threadIdx.x; c < n; c += kThreads) {
                int64_t rr = c / T.ncols;
                int64_t col = c - rr * T.ncols + T.col0;
                int64_t so, dof;
                seg_row_a(sg, T.row0 + rr, &so, &dof);
                float a = 0.f;
                for (int q = 0; q < ncopies; q++) {
                    const int64_t e = so + col + q * copy_stride;
                    const float x = kBf16 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(src)[e])
                                          : reinterpret_cast<const float *>(src)[e];
                    a = q == 0 ? x : AGG == EA_AGG_MAX ? fmaxf(a, x) : a + x;
                }
                if (kBf16) reinterpret_cast<__nv_bfloat16 *>(dst)[dof + col] = __float2bfloat16_rn(a);
                else reinterpret_cast<float *>(dst)[dof + col] = a;
            }
        }
    }
}

}  // namespace

cudaError_t launch_exchange_agg(const XSeg *segs, const XTile *tiles, int64_t ntiles, const char *src, char *dst,
                                int dtype, int agg, int ncopies, int64_t copy_stride, int num_sms, cudaStream_t st,
                                int64_t src_elems, int64_t dst_elems, int *err) {
    const int64_t grid = std::min<int64_t>(ntiles, (int64_t)num_sms * 8);
    auto go = [&](auto kernel) {
        kernel<<<(unsigned)grid, kThreads, 0, st>>>(segs, tiles, ntiles, src, dst, ncopies, copy_stride, src_elems,
                                                    dst_elems, err);
    };
    if (dtype == EA_BF16) {
        if (agg == EA_AGG_MAX) go(exchange_agg_kernel<true, EA_AGG_MAX>);
        else go(exchange_agg_kernel<true, EA_AGG_SUM>);
    } else {
        if (agg == EA_AGG_MAX) go(exchange_agg_kernel<false, EA_AGG_MAX>);
        else go(exchange_agg_kernel<false, EA_AGG_SUM>);
    }
    return cudaGetLastError();
}

}  // namespace ea
