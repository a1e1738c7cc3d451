// rowreduce.cu -- row-reduction join-agg kernel (aggregation SUM, MAX, or
// the softmax statistics MAX + SUM of exp, over the trailing letters of
// input 0).
//
// "Every Kernel Is a Join", Section 1 and Definition 3.7: softmax and
// normalisation are a join (the scores, possibly with a broadcast row
// statistic) followed by an aggregation over the reduced letters.  When the
// reduced letters are split into blocks, every output block has one
// function specification per block of the reduced letters, and step (2)
// combines their outputs with the aggregation op.  One warp owns one output
// cell: it walks every function specification of the cell's group, streams
// the row segment with several 16-byte loads in flight per lane,
// accumulates in fp32 and combines lanes with warp shuffles -- the
// per-tuple results and their aggregation are fused, with no partial
// results in memory.  The row loop is instantiated per map, and rows the
// predicate leaves whole skip the per-cell test.
//
// The statistics variant computes m = MAX_t v and l = SUM_t exp(v - m) in
// one pass with the associative, commutative merge
//   (m1, l1) (+) (m2, l2) = (M, l1 exp(m1 - M) + l2 exp(m2 - M)),
//   M = max(m1, m2), identity (-inf, 0),
// so the scores are read once instead of twice.
#include <algorithm>
#include <math.h>

#include "dev_common.cuh"
#include "tc_common.cuh"

namespace ea {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

struct Stats {
    float m, l;
};

__device__ __forceinline__ Stats stats_merge(Stats a, Stats b) {
    const float M = fmaxf(a.m, b.m);
    if (M == -INFINITY) return Stats{-INFINITY, 0.0f};
    return Stats{M, a.l * __expf(a.m - M) + b.l * __expf(b.m - M)};
}

struct Acc {
    float a;   // SUM / MAX accumulator
    Stats st;  // statistics accumulator
};

template <int MAP>
__device__ __forceinline__ float rmap(const RrParams &p, float x0, float x1, float x2) {
    if constexpr (MAP >= 0) return fmap<MAP>(x0, x1, x2, p.scale, p.eps);
    else return cell_map(p.map, x0, x1, x2, p.scale, p.eps);
}

// Accumulate one row segment of one function specification.  MAP < 0 /
// MASK < 0: map / streamed inputs read at run time (generic instance).
// Chunks per batch: about 128 bytes of streamed inputs in flight per lane.
// DT: 1 = streamed inputs bf16, 2 = fp32, 0 = read at run time.
template <int NS, int DT>
struct RrBatch {
    static constexpr int BYTES = DT == 1 ? 16 : 32;
    static constexpr int U = (128 / BYTES) / (NS > 0 ? NS : 1) > 0 ? (128 / BYTES) / (NS > 0 ? NS : 1) : 1;
};

// Packed two-wide fp32 arithmetic (one instruction for two values).
__device__ __forceinline__ uint64_t pk2(uint32_t lo, uint32_t hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
    return r;
}
__device__ __forceinline__ float pk2_sum(uint64_t v) {
    float lo, hi;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
    return lo + hi;
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

template <int MAP, int AGG, int NIN, int MASK, int DT>
__device__ __forceinline__ void rr_seg(const RrParams &p, Acc &acc, const int64_t *ioff, const int64_t *iinn,
                                       const float *bc, int64_t len, int64_t cmin, int64_t cmax, bool vec, int sl,
                                       int lpr) {
    constexpr int NS = MASK < 0 ? NIN : ((MASK & 1) + ((MASK >> 1) & 1) + ((MASK >> 2) & 1));
    constexpr int U = RrBatch<NS, DT>::U;
    constexpr bool kRaw = DT != 0 && MASK >= 0;
    constexpr bool kB16 = DT == 1;
    const int mask = MASK < 0 ? (p.stream_mask | 1) : MASK;
    const bool whole = cmin <= 0 && cmax >= len - 1;
    const int64_t step = (int64_t)lpr * 8;  // cells between a lane's consecutive chunks
    if constexpr (AGG == EA_AGG_SUM && (MAP == EA_MAP_SQUARE || MAP == EA_MAP_IDENTITY) && kRaw && NS == 1) {
        // SUM of one streamed input (or of its squares) over whole rows: two
        // cells per packed f32x2 add or FMA, four running pair-sums, the
        // map's scale applied once to the row segment's sum
        if (vec && whole) {
            int k0 = 0;
#pragma unroll
            for (int k = 0; k < NIN; k++)
                if ((MASK >> k) & 1) k0 = k;
            uint64_t s2[4] = {0, 0, 0, 0};
            for (int64_t c0 = (int64_t)sl * 8; c0 < len; c0 += step * U) {
                uint4 raw[U][kB16 ? 1 : 2];
#pragma unroll
                for (int u = 0; u < U; u++) {
                    const int64_t c = c0 + (int64_t)u * step;
                    if (c < len) ld_raw<kB16>(p.in[k0], ioff[k0] + c, raw[u]);
                }
#pragma unroll
                for (int u = 0; u < U; u++) {
                    if (c0 + (int64_t)u * step >= len) continue;
                    const uint32_t *w = reinterpret_cast<const uint32_t *>(raw[u]);
#pragma unroll
                    for (int e = 0; e < 4; e++) {
                        const uint64_t x2 = kB16 ? pk2(w[e] << 16, w[e] & 0xFFFF0000u) : pk2(w[2 * e], w[2 * e + 1]);
                        if constexpr (MAP == EA_MAP_SQUARE) s2[e] = ffma2(x2, x2, s2[e]);
                        else s2[e] = fadd2(s2[e], x2);
                    }
                }
            }
            const float srow = pk2_sum(fadd2(fadd2(s2[0], s2[1]), fadd2(s2[2], s2[3])));
            acc.a += p.scale * srow;  // IDENTITY and SQUARE both carry the map's scale
            return;
        }
    }
    if (vec) {
        for (int64_t c0 = (int64_t)sl * 8; c0 < len; c0 += step * U) {
            uint4 raw[kRaw ? U : 1][kRaw ? NS : 1][kB16 ? 1 : 2];
            float v[kRaw ? 1 : U][kRaw ? 1 : NS][kRaw ? 1 : 8];
#pragma unroll
            for (int u = 0; u < U; u++) {
                const int64_t c = c0 + (int64_t)u * step;
                if (c >= len) continue;
                int s = 0;
#pragma unroll
                for (int k = 0; k < NIN; k++) {
                    if (MASK >= 0 && !((MASK >> k) & 1)) continue;
                    if constexpr (kRaw) {
                        ld_raw<kB16>(p.in[k], ioff[k] + c, raw[u][s]);
                    } else if (MASK < 0 && !((mask >> k) & 1)) {
#pragma unroll
                        for (int e = 0; e < 8; e++) v[u][k][e] = bc[k];
                    } else {
                        ld8(p.in[k], p.in_dtype[k], ioff[k] + c, v[u][MASK < 0 ? k : s]);
                    }
                    s++;
                }
            }
#pragma unroll
            for (int u = 0; u < U; u++) {
                const int64_t c = c0 + (int64_t)u * step;
                if (c >= len) continue;
                float f[8];
#pragma unroll
                for (int e = 0; e < 8; e++) {
                    float x[3] = {1.0f, 1.0f, 1.0f};
                    int s = 0;
#pragma unroll
                    for (int k = 0; k < NIN; k++) {
                        if constexpr (MASK < 0) {
                            x[k] = v[u][k][e];
                        } else if ((MASK >> k) & 1) {
                            if constexpr (kRaw) x[k] = raw_at<kB16>(raw[u][s], e);
                            else x[k] = v[u][s][e];
                            s++;
                        } else {
                            x[k] = bc[k];
                        }
                    }
                    f[e] = rmap<MAP>(p, x[0], x[1], x[2]);
                    if (!whole && (c + e < cmin || c + e > cmax)) f[e] = AGG == EA_AGG_SUM ? 0.0f : -INFINITY;
                }
                if constexpr (AGG == EA_AGG_MAX_SUMEXP) {
                    float mx = f[0];
#pragma unroll
                    for (int e = 1; e < 8; e++) mx = fmaxf(mx, f[e]);
                    if (mx > acc.st.m) {
                        acc.st.l *= __expf(acc.st.m - mx);  // exp(-inf) = 0 on the first chunk
                        acc.st.m = mx;
                    }
                    if (acc.st.m != -INFINITY) {
                        float s = 0.0f;
#pragma unroll
                        for (int e = 0; e < 8; e++) s += __expf(f[e] - acc.st.m);
                        acc.st.l += s;
                    }
                } else if constexpr (AGG == EA_AGG_MAX) {
#pragma unroll
                    for (int e = 0; e < 8; e++) acc.a = fmaxf(acc.a, f[e]);
                } else {
                    float s = 0.0f;
#pragma unroll
                    for (int e = 0; e < 8; e++) s += f[e];
                    acc.a += s;
                }
            }
        }
    } else {
        for (int64_t c = sl; c < len; c += lpr) {
            if (c < cmin || c > cmax) continue;
            float x[3] = {1.0f, 1.0f, 1.0f};
#pragma unroll
            for (int k = 0; k < NIN; k++)
                x[k] = ((mask >> k) & 1) ? ld_elem(p.in[k], p.in_dtype[k], ioff[k] + c * iinn[k]) : bc[k];
            const float f = rmap<MAP>(p, x[0], x[1], x[2]);
            if constexpr (AGG == EA_AGG_MAX_SUMEXP) acc.st = stats_merge(acc.st, Stats{f, 1.0f});
            else if constexpr (AGG == EA_AGG_MAX) acc.a = fmaxf(acc.a, f);
            else acc.a += f;
        }
    }
}

template <int AGG, int MAP, int MASK>
struct RrMinBlocks;

template <int AGG, int MAP, int NIN, int MASK, int DT>
__global__ void __launch_bounds__(kThreads, (RrMinBlocks<AGG, MAP, MASK>::value)) rowreduce_kernel(const RrParams p) {
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int mask = MASK < 0 ? (p.stream_mask | 1) : MASK;
    for (int64_t t = blockIdx.x; t < p.ntiles; t += gridDim.x) {
        const RrTile T = p.tiles[t];
        const RrGroup G = p.groups[T.group];
        if constexpr (kBoundsCheck) {
            bool in = true;
            for (int i = G.i0; i < G.i1 && in; i++)
                in = view_in(p.items[i], p.n_in, p.in_elems, p.out_elems) && T.row0 >= 0 &&
                     T.row0 + T.nrows <= p.items[i].rows;
            if (!in) {
                if (threadIdx.x == 0) bounds_fail(p.err);
                continue;
            }
        }
        // lanes per row: a power of two giving each lane about U chunks of
        // a row segment; short segments pack several rows to a warp
        constexpr int NSr = MASK < 0 ? NIN : ((MASK & 1) + ((MASK >> 1) & 1) + ((MASK >> 2) & 1));
        constexpr int Ur = RrBatch<NSr, DT>::U;
        const int64_t seg = p.items[G.i0].len;
        const int64_t chunks = p.items[G.i0].vec ? seg / 8 : seg;
        int lpr = 32;
        while (lpr > 1 && (int64_t)lpr * Ur > chunks) lpr /= 2;
        const int rpw = 32 / lpr;
        const int sub = lane / lpr, sl = lane % lpr;
        const int64_t nrows_pad = (T.nrows + rpw - 1) / rpw * rpw;
        for (int64_t rr0 = (int64_t)warp * rpw; rr0 < nrows_pad; rr0 += (int64_t)kWarps * rpw) {
            const int64_t rr = rr0 + sub;
            const bool live = rr < T.nrows;  // lanes past the tile still join the shuffles
            const int64_t r = T.row0 + (live ? rr : T.nrows - 1);
            Acc acc;
            acc.a = AGG == EA_AGG_SUM ? 0.0f : -INFINITY;
            acc.st = Stats{-INFINITY, 0.0f};
            int64_t coord[kViewDims];
            for (int i = G.i0; i < G.i1; i++) {
                const EwItem &it = p.items[i];
                decode_row(it, r, coord);
                const int nd = it.nd;
                int64_t ioff[NIN], iinn[NIN];
                float bc[NIN];
#pragma unroll
                for (int k = 0; k < NIN; k++) {
                    ioff[k] = it.in_base[k];
                    iinn[k] = it.in_inner[k];
                    for (int d = 0; d < nd; d++) ioff[k] += coord[d] * it.istr[k][d];
                }
#pragma unroll
                for (int k = 0; k < NIN; k++)
                    bc[k] = ((mask >> k) & 1) ? 1.0f : ld_elem(p.in[k], p.in_dtype[k], ioff[k]);
                const int64_t len = it.len;
                int64_t cmin = 0, cmax = len - 1;
                if (p.pred) {
                    if (it.sdim[0] == kViewDims) cmax = min64(cmax, special_coord(it, 1, coord, 0) - it.slo[0]);
                    else if (it.sdim[1] == kViewDims) cmin = max64(cmin, special_coord(it, 0, coord, 0) - it.slo[1]);
                    else if (special_coord(it, 0, coord, 0) > special_coord(it, 1, coord, 0)) cmax = -1;
                }
                if (!live) cmax = -1;
                rr_seg<MAP, AGG, NIN, MASK, DT>(p, acc, ioff, iinn, bc, len, cmin, cmax, it.vec != 0, sl, lpr);
            }
            // combine the lanes of each row (xor within aligned groups of lpr lanes)
            if constexpr (AGG == EA_AGG_MAX_SUMEXP) {
                for (int o = lpr / 2; o > 0; o >>= 1) {
                    Stats other{__shfl_xor_sync(0xffffffffu, acc.st.m, o), __shfl_xor_sync(0xffffffffu, acc.st.l, o)};
                    acc.st = stats_merge(acc.st, other);
                }
            } else {
                for (int o = lpr / 2; o > 0; o >>= 1) {
                    const float y = __shfl_xor_sync(0xffffffffu, acc.a, o);
                    acc.a = AGG == EA_AGG_MAX ? fmaxf(acc.a, y) : acc.a + y;
                }
            }
            if (sl == 0 && live) {
                const EwItem &it0 = p.items[G.i0];
                decode_row(it0, r, coord);
                int64_t ooff = it0.out_base;
                for (int d = 0; d < it0.nd; d++) ooff += coord[d] * it0.ostr[d];
                if constexpr (AGG == EA_AGG_MAX_SUMEXP) {
                    st_elem(p.out, p.out_dtype, ooff, acc.st.m);
                    st_elem(p.out2, p.out2_dtype, ooff, acc.st.l);
                } else {
                    st_elem(p.out, p.out_dtype, ooff, acc.a);
                }
            }
        }
    }
}

// DT: the dtype every streamed input shares (1 bf16, 2 fp32), 0 if mixed.
constexpr int kTileItems = 64;

// Per tuple, the geometry of the current tile: inside a tile every row is
// one step along the innermost row dimension, so offsets and predicate
// bounds are linear in the row index.
template <int NIN>
struct TileItem {
    int64_t off[NIN];   // input offsets at the tile's first row
    int64_t rstr[NIN];  // their change per row
    int64_t inn[NIN];   // strides along the reduced letters
    int64_t len;
    int64_t inner_lo;   // global coordinate of reduced index 0 (predicate)
    int64_t a0, b0;     // the predicate letters' global values at the first row
    int32_t da, db;     // their change per row (0 or 1)
    int32_t mode;       // 0 no predicate, 1 lo letter reduced, 2 hi letter reduced, 3 neither
    int32_t vec;
};

// Resident CTAs per SM the register budget is sized for: the packed SUM
// path (one streamed input, whole rows) keeps eight 16-byte chunks per lane
// in flight plus its pair-sums, which fits 128 registers but not 80.
template <int AGG, int MAP, int MASK>
struct RrMinBlocks {
    static constexpr int value =
        (AGG == EA_AGG_SUM && (MAP == EA_MAP_SQUARE || MAP == EA_MAP_IDENTITY) && MASK == 1) ? 2 : 3;
};

template <int AGG, int MAP, int NIN, int MASK, int DT>
__global__ void __launch_bounds__(kThreads, (RrMinBlocks<AGG, MAP, MASK>::value)) rowreduce_tile_kernel(const RrParams p) {
    __shared__ TileItem<NIN> ti[kTileItems];
    __shared__ int64_t s_out0, s_ostr;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int mask = MASK < 0 ? (p.stream_mask | 1) : MASK;
    constexpr int NSr = MASK < 0 ? NIN : ((MASK & 1) + ((MASK >> 1) & 1) + ((MASK >> 2) & 1));
    constexpr int Ur = RrBatch<NSr, DT>::U;
    for (int64_t t = blockIdx.x; t < p.ntiles; t += gridDim.x) {
        const RrTile T = p.tiles[t];
        const RrGroup G = p.groups[T.group];
        if constexpr (kBoundsCheck) {
            bool in = true;
            for (int i = G.i0; i < G.i1 && in; i++)
                in = view_in(p.items[i], p.n_in, p.in_elems, p.out_elems) && T.row0 >= 0 &&
                     T.row0 + T.nrows <= p.items[i].rows;
            if (!in) {
                if (threadIdx.x == 0) bounds_fail(p.err);
                continue;
            }
        }
        const int n = G.i1 - G.i0;
        __syncthreads();
        if (threadIdx.x < n) {
            const EwItem &it = p.items[G.i0 + threadIdx.x];
            int64_t cd[kViewDims];
            decode_row(it, T.row0, cd);
            const int last = it.nd - 1;
            TileItem<NIN> q;
#pragma unroll
            for (int k = 0; k < NIN; k++) {
                int64_t o = it.in_base[k];
                for (int d = 0; d < it.nd; d++) o += cd[d] * it.istr[k][d];
                q.off[k] = o;
                q.rstr[k] = last >= 0 ? it.istr[k][last] : 0;
                q.inn[k] = it.in_inner[k];
            }
            q.len = it.len;
            q.vec = it.vec;
            q.mode = 0;
            q.inner_lo = 0;
            q.a0 = q.b0 = 0;
            q.da = q.db = 0;
            if (p.pred) {
                q.a0 = special_coord(it, 0, cd, 0);
                q.b0 = special_coord(it, 1, cd, 0);
                q.da = it.sdim[0] == last && last >= 0 ? 1 : 0;
                q.db = it.sdim[1] == last && last >= 0 ? 1 : 0;
                if (it.sdim[0] == kViewDims) {
                    q.mode = 1;
                    q.inner_lo = it.slo[0];
                } else if (it.sdim[1] == kViewDims) {
                    q.mode = 2;
                    q.inner_lo = it.slo[1];
                } else {
                    q.mode = 3;
                }
            }
            ti[threadIdx.x] = q;
            if (threadIdx.x == 0) {
                int64_t o = it.out_base;
                for (int d = 0; d < it.nd; d++) o += cd[d] * it.ostr[d];
                s_out0 = o;
                s_ostr = last >= 0 ? it.ostr[last] : 0;
            }
        }
        __syncthreads();
        const int64_t chunks = ti[0].vec ? ti[0].len / 8 : ti[0].len;
        int lpr = 32;
        while (lpr > 1 && (int64_t)lpr * Ur > chunks) lpr /= 2;
        const int rpw = 32 / lpr;
        const int sub = lane / lpr, sl = lane % lpr;
        const int64_t nrows_pad = (T.nrows + rpw - 1) / rpw * rpw;
        for (int64_t rr0 = (int64_t)warp * rpw; rr0 < nrows_pad; rr0 += (int64_t)kWarps * rpw) {
            const int64_t rr = rr0 + sub;
            const bool live = rr < T.nrows;  // lanes past the tile still join the shuffles
            const int64_t dr = live ? rr : T.nrows - 1;
            Acc acc;
            acc.a = AGG == EA_AGG_SUM ? 0.0f : -INFINITY;
            acc.st = Stats{-INFINITY, 0.0f};
            for (int i = 0; i < n; i++) {
                const TileItem<NIN> &q = ti[i];
                int64_t ioff[NIN], iinn[NIN];
                float bc[NIN];
#pragma unroll
                for (int k = 0; k < NIN; k++) {
                    ioff[k] = q.off[k] + dr * q.rstr[k];
                    iinn[k] = q.inn[k];
                    bc[k] = ((mask >> k) & 1) ? 1.0f : ld_elem(p.in[k], p.in_dtype[k], ioff[k]);
                }
                const int64_t len = q.len;
                int64_t cmin = 0, cmax = len - 1;
                if (q.mode == 1) cmax = min64(cmax, q.b0 + q.db * dr - q.inner_lo);
                else if (q.mode == 2) cmin = max64(cmin, q.a0 + q.da * dr - q.inner_lo);
                else if (q.mode == 3 && q.a0 + q.da * dr > q.b0 + q.db * dr) cmax = -1;
                if (!live) cmax = -1;
                rr_seg<MAP, AGG, NIN, MASK, DT>(p, acc, ioff, iinn, bc, len, cmin, cmax, q.vec != 0, sl, lpr);
            }
            if constexpr (AGG == EA_AGG_MAX_SUMEXP) {
                for (int o = lpr / 2; o > 0; o >>= 1) {
                    Stats other{__shfl_xor_sync(0xffffffffu, acc.st.m, o), __shfl_xor_sync(0xffffffffu, acc.st.l, o)};
                    acc.st = stats_merge(acc.st, other);
                }
            } else {
                for (int o = lpr / 2; o > 0; o >>= 1) {
                    const float y = __shfl_xor_sync(0xffffffffu, acc.a, o);
                    acc.a = AGG == EA_AGG_MAX ? fmaxf(acc.a, y) : acc.a + y;
                }
            }
            if (sl == 0 && live) {
                const int64_t ooff = s_out0 + dr * s_ostr;
                if constexpr (AGG == EA_AGG_MAX_SUMEXP) {
                    st_elem(p.out, p.out_dtype, ooff, acc.st.m);
                    st_elem(p.out2, p.out2_dtype, ooff, acc.st.l);
                } else {
                    st_elem(p.out, p.out_dtype, ooff, acc.a);
                }
            }
        }
    }
}

// The row-batch kernels work in units of one warp pass over a tile (tile
// t, warp slot w: rows w * rpb + [0, rpb), then every kWarps * rpb further
// rows of the tile).  A CTA takes one contiguous range of tiles, so that
// its warps stream through neighbouring rows of each block; its warp w
// takes slot w of each, with no CTA barrier, and a tile's flat descriptor
// (kRbWords words, lane i holding word i) is loaded while the tile before
// it is still being reduced.
struct RbUnit {
    int64_t off[4], out0, len;
    int32_t rstr[4], ostr, nrows, n;  // the planner keeps the strides below 2^31
};

__device__ __forceinline__ int64_t rb_word(const RrParams &p, int64_t tile, int lane) {
    return lane < kRbWords ? __ldg(p.rb_desc + tile * kRbWords + lane) : 0;
}

__device__ __forceinline__ RbUnit rb_unpack(int64_t w) {
    RbUnit d;
#pragma unroll
    for (int i = 0; i < 4; i++) {
        d.off[i] = __shfl_sync(0xffffffffu, w, i);
        d.rstr[i] = __shfl_sync(0xffffffffu, (int32_t)w, 4 + i);
    }
    d.out0 = __shfl_sync(0xffffffffu, w, 8);
    d.ostr = __shfl_sync(0xffffffffu, (int32_t)w, 9);
    d.len = __shfl_sync(0xffffffffu, w, 10);
    d.nrows = __shfl_sync(0xffffffffu, (int32_t)w, 11);
    d.n = __shfl_sync(0xffffffffu, (int32_t)(w >> 32), 11);
    return d;
}

// A row-batch tile's rows inside the input and output arenas (its flat
// descriptor: first-row offset and row stride per block, output offset and
// stride, segment length, rows and blocks).
__device__ __forceinline__ bool rb_in(const RrParams &p, int64_t t) {
    const int64_t *w = p.rb_desc + t * kRbWords;
    const int64_t rows = (int64_t)(uint32_t)(w[11] & 0xFFFFFFFF), nb = w[11] >> 32, len = w[10];
    if (nb < 1 || nb > 4) return false;
    for (int64_t b = 0; b < nb; b++)
        if (!range_in(w[b], 1, &rows, &w[4 + b], len, 1, p.in_elems[0])) return false;
    return range_in(w[8], 1, &rows, &w[9], 1, 0, p.out_elems);
}

// SUM (or SUM of squares) of one input over rows whose segments lie in at
// most four blocks of one length (no predicate): a warp (or a slice of one)
// requests a row's segments in all its blocks together, 64 bytes per lane
// per segment, then sums them -- one memory round trip per batch instead of
// one per block.  Packed f32x2 sums; the map's scale on the row's sum.
template <int MAP, int DT>
__global__ void __launch_bounds__(kThreads, 2) rowreduce_rowbatch_kernel(const RrParams p) {
    constexpr bool kB16 = DT == 1;
    constexpr int kRowU = kB16 ? 4 : 2;  // 64 bytes per lane per segment in flight
    const int lane = threadIdx.x % 32;
    const int slot = threadIdx.x / 32;
    const int64_t t1 = ((int64_t)blockIdx.x + 1) * p.ntiles / gridDim.x;
    int64_t t = (int64_t)blockIdx.x * p.ntiles / gridDim.x;
    int64_t wnext = t < t1 ? rb_word(p, t, lane) : 0;
    for (; t < t1; t++) {
        const RbUnit d = rb_unpack(wnext);
        if (t + 1 < t1) wnext = rb_word(p, t + 1, lane);
        if constexpr (kBoundsCheck) {
            if (!rb_in(p, t)) {
                if (lane == 0) bounds_fail(p.err);
                continue;
            }
        }
        const int n = d.n;
        const int64_t len = d.len, chunks = len / 8;
        int lpb = 32;
        while (lpb > 1 && (int64_t)lpb * kRowU > chunks) lpb /= 2;
        const int rpb = 32 / lpb, subb = lane / lpb, slb = lane % lpb;
        const int64_t step = (int64_t)lpb * 8;
        const int64_t pad = (d.nrows + rpb - 1) / rpb * rpb;
        for (int64_t rr0 = (int64_t)slot * rpb; rr0 < pad; rr0 += (int64_t)kWarps * rpb) {
            const int64_t rr = rr0 + subb;
            const bool live = rr < d.nrows;  // lanes past the tile still join the shuffles
            const int64_t dr = live ? rr : d.nrows - 1;
            uint64_t s2[4] = {0, 0, 0, 0};
            for (int64_t c0 = (int64_t)slb * 8; c0 < len; c0 += step * kRowU) {
                uint4 raw[4][kRowU][kB16 ? 1 : 2];
#pragma unroll
                for (int i = 0; i < 4; i++) {
                    if (i >= n) continue;
                    const int64_t off = d.off[i] + dr * d.rstr[i];
#pragma unroll
                    for (int uu = 0; uu < kRowU; uu++) {
                        const int64_t c = c0 + (int64_t)uu * step;
                        if (c < len) ld_raw<kB16>(p.in[0], off + c, raw[i][uu]);
                    }
                }
#pragma unroll
                for (int i = 0; i < 4; i++) {
                    if (i >= n) continue;
#pragma unroll
                    for (int uu = 0; uu < kRowU; uu++) {
                        if (c0 + (int64_t)uu * step >= len) continue;
                        const uint32_t *w = reinterpret_cast<const uint32_t *>(raw[i][uu]);
#pragma unroll
                        for (int e = 0; e < 4; e++) {
                            const uint64_t x2 = kB16 ? pk2(w[e] << 16, w[e] & 0xFFFF0000u) : pk2(w[2 * e], w[2 * e + 1]);
                            if constexpr (MAP == EA_MAP_SQUARE) s2[e] = ffma2(x2, x2, s2[e]);
                            else s2[e] = fadd2(s2[e], x2);
                        }
                    }
                }
            }
            float a = pk2_sum(fadd2(fadd2(s2[0], s2[1]), fadd2(s2[2], s2[3])));
            a *= p.scale;  // the map's scale (IDENTITY: scale v, SQUARE: scale v^2)
            for (int o = lpb / 2; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
            if (slb == 0 && live) st_elem(p.out, p.out_dtype, d.out0 + dr * d.ostr, a);
        }
    }
}

// SUM (or SUM of squares) of one input over rows whose segments lie in at
// most four blocks, where the rows of each block are stored back to back
// (16-byte aligned, at most 2 KB a row segment): one thread streams chunks
// of 8 rows of one block (8 x the segment, at most 16 KB) into a ring of 8
// shared-memory stages with bulk copies that complete on the stage's
// mbarrier -- a tile's rows in groups of 8, each group's blocks in order --
// so up to 128 KB of each SM's input is in flight with no per-lane loads
// outstanding; eight warps reduce them, warp w row w of each chunk, keeping
// the row's packed f32x2 partial sums across its blocks.  Tile descriptors
// are loaded two tiles ahead.
constexpr int kBulkStages = 8;
constexpr int kBulkStage = kRbBulkBytes;  // bytes of one chunk at most
constexpr int kBulkRows = kRbBulkRows;    // rows of a chunk (= consumer warps)
constexpr int kBulkThreads = 32 * (kBulkRows + 1);  // the consumer warps + the producer warp

struct BulkCtl {
    uint64_t full[kBulkStages], empty[kBulkStages];
    int abort;
};

constexpr int kBulkSmem = 128 + kBulkStages * kBulkStage + (int)sizeof(BulkCtl);

__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(tc::smem_u32(bar))
                 : "memory");
}

template <int MAP, int DT>
__global__ void __launch_bounds__(kBulkThreads, 1) rowreduce_bulk_kernel(const RrParams p) {
    constexpr bool kB16 = DT == 1;
    constexpr int kEs = kB16 ? 2 : 4;
    extern __shared__ uint8_t bulk_raw[];
    uint8_t *ring = reinterpret_cast<uint8_t *>(((uintptr_t)bulk_raw + 127) & ~(uintptr_t)127);
    BulkCtl *ctl = reinterpret_cast<BulkCtl *>(ring + kBulkStages * kBulkStage);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int64_t t1 = ((int64_t)blockIdx.x + 1) * p.ntiles / gridDim.x;
    const int64_t tb = (int64_t)blockIdx.x * p.ntiles / gridDim.x;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kBulkStages; s++) {
            tc::mbar_init(&ctl->full[s], 1);
            tc::mbar_init(&ctl->empty[s], kBulkRows);
        }
        ctl->abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        tc::fence_proxy_async();
    }
    __syncthreads();
    volatile int *abort = &ctl->abort;
    // this CTA's tile descriptors, lane i holding word i, two tiles ahead
    int64_t wa = tb < t1 ? rb_word(p, tb, lane) : 0, wb = tb + 1 < t1 ? rb_word(p, tb + 1, lane) : 0;
    uint32_t k = 0;  // chunks so far
    if (warp == kBulkRows) {
        // ------------------------------------------------ producer (lane 0 issues)
        uint32_t armed = 0, par = 0;
        bool ok = true;
        for (int64_t t = tb; t < t1 && ok; t++) {
            const RbUnit d = rb_unpack(wa);
            wa = wb;
            if (t + 2 < t1) wb = rb_word(p, t + 2, lane);
            if constexpr (kBoundsCheck) {
                if (!rb_in(p, t)) continue;  // the consumers skip it too
            }
            for (int r0 = 0; r0 < d.nrows && ok; r0 += kBulkRows) {
                const int rows = min(kBulkRows, d.nrows - r0);
                const uint32_t bytes = (uint32_t)(rows * d.len * kEs);
                for (int i = 0; i < d.n && ok; i++, k++) {
                    const int s = (int)(k % kBulkStages);
                    if (lane == 0) {
                        if (k >= kBulkStages && !tc::mbar_wait(&ctl->empty[s], (k / kBulkStages - 1) & 1, abort, p.err,
                                                                kDevTimeoutProducer))
                            ok = false;
                        if (ok) {
                            tc::mbar_expect_tx(&ctl->full[s], bytes);
                            bulk_load(tc::smem_u32(ring + s * kBulkStage),
                                      p.in[0] + (d.off[i] + (int64_t)r0 * d.rstr[i]) * kEs, bytes, &ctl->full[s]);
                            armed |= 1u << s;
                            par = (par & ~(1u << s)) | (((k / kBulkStages) & 1) << s);
                        }
                    }
                    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
                }
            }
        }
        if (lane == 0 && *abort) {
            // let this CTA's copies land before it can exit
            for (int s = 0; s < kBulkStages; s++)
                if (armed & (1u << s)) tc::mbar_wait(&ctl->full[s], (par >> s) & 1, abort, p.err, 0, tc::kDrainNs, false);
        }
    } else {
        // ------------------------------------------------ consumers: warp w reduces row w of each chunk
        bool ok = true;
        for (int64_t t = tb; t < t1 && ok; t++) {
            const RbUnit d = rb_unpack(wa);
            wa = wb;
            if (t + 2 < t1) wb = rb_word(p, t + 2, lane);
            if constexpr (kBoundsCheck) {
                if (!rb_in(p, t)) {
                    if (warp == 0 && lane == 0) bounds_fail(p.err);
                    continue;
                }
            }
            const int units = (int)(d.len * kEs / 16);  // 16-byte units of a row segment
            for (int r0 = 0; r0 < d.nrows && ok; r0 += kBulkRows) {
                const bool live = r0 + warp < d.nrows;
                uint64_t s2[4] = {0, 0, 0, 0};
                for (int i = 0; i < d.n; i++, k++) {
                    const int s = (int)(k % kBulkStages);
                    if (!tc::warp_wait(&ctl->full[s], (k / kBulkStages) & 1, abort, p.err, kDevTimeoutReduce)) {
                        ok = false;
                        break;
                    }
                    if (live) {
                        const uint32_t row = tc::smem_u32(ring + s * kBulkStage) + (uint32_t)(warp * units * 16);
                        for (int u = lane; u < units; u += 32) {
                            uint32_t w[4];
                            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                                         : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                                         : "r"(row + (uint32_t)(u * 16)));
                            if constexpr (kB16) {
#pragma unroll
                                for (int e = 0; e < 4; e++) {
                                    const uint64_t x2 = pk2(w[e] << 16, w[e] & 0xFFFF0000u);
                                    if constexpr (MAP == EA_MAP_SQUARE) s2[e] = ffma2(x2, x2, s2[e]);
                                    else s2[e] = fadd2(s2[e], x2);
                                }
                            } else {
#pragma unroll
                                for (int e = 0; e < 2; e++) {
                                    const uint64_t x2 = pk2(w[2 * e], w[2 * e + 1]);
                                    if constexpr (MAP == EA_MAP_SQUARE) s2[e] = ffma2(x2, x2, s2[e]);
                                    else s2[e] = fadd2(s2[e], x2);
                                }
                            }
                        }
                    }
                    __syncwarp();
                    if (lane == 0) tc::mbar_arrive(&ctl->empty[s]);
                }
                if (!ok) break;
                float a = pk2_sum(fadd2(fadd2(s2[0], s2[1]), fadd2(s2[2], s2[3])));
                a *= p.scale;  // the map's scale (IDENTITY: scale v, SQUARE: scale v^2)
                for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
                if (lane == 0 && live) st_elem(p.out, p.out_dtype, d.out0 + (int64_t)(r0 + warp) * d.ostr, a);
            }
        }
        if (!ok) *abort = 1;
    }
}

// The softmax statistics (MAX and SUM of exp) of one input over rows whose
// segments lie in at most four blocks of one length, no predicate: a row's
// segments in all its blocks are requested together (64 bytes per lane per
// segment), the batch's maximum is merged into the running one once per
// batch, and the lanes' (m, l) pairs are merged by shuffles.
template <int DT>
__global__ void __launch_bounds__(kThreads, 2) rowreduce_rowbatch_stats_kernel(const RrParams p) {
    constexpr bool kB16 = DT == 1;
    constexpr int kRowU = kB16 ? 4 : 2;
    constexpr int EPC = 8;  // cells per chunk
    const int lane = threadIdx.x % 32;
    const int slot = threadIdx.x / 32;
    const int64_t t1 = ((int64_t)blockIdx.x + 1) * p.ntiles / gridDim.x;
    int64_t t = (int64_t)blockIdx.x * p.ntiles / gridDim.x;
    int64_t wnext = t < t1 ? rb_word(p, t, lane) : 0;
    for (; t < t1; t++) {
        const RbUnit d = rb_unpack(wnext);
        if (t + 1 < t1) wnext = rb_word(p, t + 1, lane);
        if constexpr (kBoundsCheck) {
            if (!rb_in(p, t)) {
                if (lane == 0) bounds_fail(p.err);
                continue;
            }
        }
        const int n = d.n;
        const int64_t len = d.len, chunks = len / EPC;
        int lpb = 32;
        while (lpb > 1 && (int64_t)lpb * kRowU > chunks) lpb /= 2;
        const int rpb = 32 / lpb, subb = lane / lpb, slb = lane % lpb;
        const int64_t step = (int64_t)lpb * EPC;
        const int64_t pad = (d.nrows + rpb - 1) / rpb * rpb;
        for (int64_t rr0 = (int64_t)slot * rpb; rr0 < pad; rr0 += (int64_t)kWarps * rpb) {
            const int64_t rr = rr0 + subb;
            const bool live = rr < d.nrows;
            const int64_t dr = live ? rr : d.nrows - 1;
            Stats st{-INFINITY, 0.0f};
            for (int64_t c0 = (int64_t)slb * EPC; c0 < len; c0 += step * kRowU) {
                uint4 raw[4][kRowU][kB16 ? 1 : 2];
#pragma unroll
                for (int i = 0; i < 4; i++) {
                    if (i >= n) continue;
                    const int64_t off = d.off[i] + dr * d.rstr[i];
#pragma unroll
                    for (int uu = 0; uu < kRowU; uu++) {
                        const int64_t c = c0 + (int64_t)uu * step;
                        if (c < len) ld_raw<kB16>(p.in[0], off + c, raw[i][uu]);
                    }
                }
                // the batch maximum, then its exponentials against the running maximum
                float bm = -INFINITY;
#pragma unroll
                for (int i = 0; i < 4; i++) {
                    if (i >= n) continue;
#pragma unroll
                    for (int uu = 0; uu < kRowU; uu++) {
                        if (c0 + (int64_t)uu * step >= len) continue;
#pragma unroll
                        for (int e = 0; e < EPC; e++) bm = fmaxf(bm, raw_at<kB16>(raw[i][uu], e));
                    }
                }
                if (bm > st.m) {
                    st.l *= __expf(st.m - bm);  // exp(-inf) = 0 on the first batch
                    st.m = bm;
                }
                if (st.m != -INFINITY) {
                    float sum = 0.0f;
#pragma unroll
                    for (int i = 0; i < 4; i++) {
                        if (i >= n) continue;
#pragma unroll
                        for (int uu = 0; uu < kRowU; uu++) {
                            if (c0 + (int64_t)uu * step >= len) continue;
#pragma unroll
                            for (int e = 0; e < EPC; e++) sum += __expf(raw_at<kB16>(raw[i][uu], e) - st.m);
                        }
                    }
                    st.l += sum;
                }
            }
            for (int o = lpb / 2; o > 0; o >>= 1) {
                Stats other{__shfl_xor_sync(0xffffffffu, st.m, o), __shfl_xor_sync(0xffffffffu, st.l, o)};
                st = stats_merge(st, other);
            }
            if (slb == 0 && live) {
                st_elem(p.out, p.out_dtype, d.out0 + dr * d.ostr, st.m);
                st_elem(p.out2, p.out2_dtype, d.out0 + dr * d.ostr, st.l);
            }
        }
    }
}

// The bulk kernel's shared memory is above the default 48 KB: raise the
// limit once per device.
template <int MAP, int DT>
cudaError_t bulk_configure() {
    static bool done[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64 && done[dev]) return cudaSuccess;
    e = cudaFuncSetAttribute(rowreduce_bulk_kernel<MAP, DT>, cudaFuncAttributeMaxDynamicSharedMemorySize, kBulkSmem);
    if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev] = true;
    return e;
}

template <int AGG, int MAP, int NIN, int MASK>
cudaError_t go(const RrParams &p, int64_t grid, cudaStream_t st, int num_sms) {
    int dt = -1;
    for (int k = 0; k < NIN; k++) {
        if (MASK >= 0 && !((MASK >> k) & 1)) continue;
        const int d = p.in_dtype[k] == EA_BF16 ? 1 : 2;
        dt = dt < 0 ? d : (dt == d ? dt : 0);
    }
    const bool tile = p.tile_linear && p.max_items <= kTileItems;
    if constexpr (AGG == EA_AGG_MAX_SUMEXP && MAP == EA_MAP_IDENTITY && NIN == 1 && MASK == 1) {
        if (tile && p.row_batch && p.rb_desc && dt > 0) {
            const unsigned g2 = (unsigned)std::min<int64_t>(p.ntiles, 2 * (int64_t)num_sms);
            if (dt == 1) rowreduce_rowbatch_stats_kernel<1><<<g2, kThreads, 0, st>>>(p);
            else rowreduce_rowbatch_stats_kernel<2><<<g2, kThreads, 0, st>>>(p);
            return cudaGetLastError();
        }
    }
    if constexpr (AGG == EA_AGG_SUM && (MAP == EA_MAP_SQUARE || MAP == EA_MAP_IDENTITY) && NIN == 1 && MASK == 1) {
        if (tile && p.row_batch && p.row_bulk && p.rb_desc && dt > 0) {
            // one CTA per SM (its 128 KB ring), each over a contiguous range of tiles
            const unsigned g1 = (unsigned)std::min<int64_t>(p.ntiles, (int64_t)num_sms);
            cudaError_t e = dt == 1 ? bulk_configure<MAP, 1>() : bulk_configure<MAP, 2>();
            if (e != cudaSuccess) return e;
            if (dt == 1) rowreduce_bulk_kernel<MAP, 1><<<g1, kBulkThreads, kBulkSmem, st>>>(p);
            else rowreduce_bulk_kernel<MAP, 2><<<g1, kBulkThreads, kBulkSmem, st>>>(p);
            return cudaGetLastError();
        }
        if (tile && p.row_batch && p.rb_desc && dt > 0) {
            // persistent: the CTAs that fit (two per SM) loop over the tiles
            const unsigned g2 = (unsigned)std::min<int64_t>(p.ntiles, 2 * (int64_t)num_sms);
            if (dt == 1) rowreduce_rowbatch_kernel<MAP, 1><<<g2, kThreads, 0, st>>>(p);
            else rowreduce_rowbatch_kernel<MAP, 2><<<g2, kThreads, 0, st>>>(p);
            return cudaGetLastError();
        }
    }
    if (tile) {
        if (MASK < 0 || dt <= 0) rowreduce_tile_kernel<AGG, MAP, NIN, MASK, 0><<<(unsigned)grid, kThreads, 0, st>>>(p);
        else if (dt == 1) rowreduce_tile_kernel<AGG, MAP, NIN, MASK, 1><<<(unsigned)grid, kThreads, 0, st>>>(p);
        else rowreduce_tile_kernel<AGG, MAP, NIN, MASK, 2><<<(unsigned)grid, kThreads, 0, st>>>(p);
    } else {
        if (MASK < 0 || dt <= 0) rowreduce_kernel<AGG, MAP, NIN, MASK, 0><<<(unsigned)grid, kThreads, 0, st>>>(p);
        else if (dt == 1) rowreduce_kernel<AGG, MAP, NIN, MASK, 1><<<(unsigned)grid, kThreads, 0, st>>>(p);
        else rowreduce_kernel<AGG, MAP, NIN, MASK, 2><<<(unsigned)grid, kThreads, 0, st>>>(p);
    }
    return cudaGetLastError();
}

template <int AGG>
cudaError_t generic(const RrParams &p, int64_t grid, cudaStream_t st, int num_sms) {
    if (p.n_in == 1) return go<AGG, -1, 1, -1>(p, grid, st, num_sms);
    if (p.n_in == 2) return go<AGG, -1, 2, -1>(p, grid, st, num_sms);
    return go<AGG, -1, 3, -1>(p, grid, st, num_sms);
}

}  // namespace

// Specialised instances for the row reductions of the hot path; the rest
// run the generic instances (map and streamed inputs read at run time).
cudaError_t launch_rowreduce(const RrParams &p, int num_sms, cudaStream_t st) {
    int64_t grid = std::min<int64_t>(p.ntiles, (int64_t)num_sms * 8);
    const int n = p.n_in, m = p.stream_mask | 1;
    switch (p.agg) {
    case EA_AGG_MAX_SUMEXP:
        if (n == 1 && p.map == EA_MAP_IDENTITY) return go<EA_AGG_MAX_SUMEXP, EA_MAP_IDENTITY, 1, 1>(p, grid, st, num_sms);
        return generic<EA_AGG_MAX_SUMEXP>(p, grid, st, num_sms);
    case EA_AGG_MAX:
        if (n == 1 && p.map == EA_MAP_IDENTITY) return go<EA_AGG_MAX, EA_MAP_IDENTITY, 1, 1>(p, grid, st, num_sms);
        return generic<EA_AGG_MAX>(p, grid, st, num_sms);
    default:
        if (n == 1 && p.map == EA_MAP_SQUARE) return go<EA_AGG_SUM, EA_MAP_SQUARE, 1, 1>(p, grid, st, num_sms);
        if (n == 1 && p.map == EA_MAP_IDENTITY) return go<EA_AGG_SUM, EA_MAP_IDENTITY, 1, 1>(p, grid, st, num_sms);
        if (n == 2 && m == 1 && p.map == EA_MAP_EXP_SUB) return go<EA_AGG_SUM, EA_MAP_EXP_SUB, 2, 1>(p, grid, st, num_sms);
        if (n == 2 && m == 3 && p.map == EA_MAP_PRODUCT) return go<EA_AGG_SUM, EA_MAP_PRODUCT, 2, 3>(p, grid, st, num_sms);
        return generic<EA_AGG_SUM>(p, grid, st, num_sms);
    }
}

}  // namespace ea
