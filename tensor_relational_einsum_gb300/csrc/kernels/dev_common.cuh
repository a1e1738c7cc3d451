// dev_common.cuh -- device helpers shared by the join-agg kernels:
// element loads/stores for fp32 and bf16, and the per-cell operators f of
// the join-agg maps (computed in fp32).
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "../ea_internal.h"

namespace ea {

__device__ __forceinline__ float ld_elem(const char *base, int dtype, int64_t i) {
    if (dtype == EA_F32) return __ldg(reinterpret_cast<const float *>(base) + i);
    return __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(base)[i]);
}

__device__ __forceinline__ void st_elem(char *base, int dtype, int64_t i, float v) {
    if (dtype == EA_F32) reinterpret_cast<float *>(base)[i] = v;
    else reinterpret_cast<__nv_bfloat16 *>(base)[i] = __float2bfloat16_rn(v);
}

// 8 consecutive elements starting at i (16-byte aligned for bf16, 32 for fp32).
__device__ __forceinline__ void ld8(const char *base, int dtype, int64_t i, float *v) {
    if (dtype == EA_F32) {
        const float4 *p = reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(base) + i);
        float4 a = __ldg(p), b = __ldg(p + 1);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    } else {
        uint4 u = __ldg(reinterpret_cast<const uint4 *>(reinterpret_cast<const __nv_bfloat16 *>(base) + i));
        const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
        for (int q = 0; q < 4; q++) {
            float2 f = __bfloat1622float2(h[q]);
            v[2 * q] = f.x;
            v[2 * q + 1] = f.y;
        }
    }
}

__device__ __forceinline__ void st8(char *base, int dtype, int64_t i, const float *v) {
    if (dtype == EA_F32) {
        float4 *p = reinterpret_cast<float4 *>(reinterpret_cast<float *>(base) + i);
        p[0] = make_float4(v[0], v[1], v[2], v[3]);
        p[1] = make_float4(v[4], v[5], v[6], v[7]);
    } else {
        uint4 u;
        __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(&u);
#pragma unroll
        for (int q = 0; q < 4; q++) h[q] = __floats2bfloat162_rn(v[2 * q], v[2 * q + 1]);
        *reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(base) + i) = u;
    }
}

// The per-cell operator f of a join (v2 = 1 when the join has two inputs).
__device__ __forceinline__ float cell_map(int map, float v0, float v1, float v2, float scale, float eps) {
    switch (map) {
    case EA_MAP_PRODUCT: return scale * v0 * v1 * v2;
    case EA_MAP_IDENTITY: return scale * v0;
    case EA_MAP_SILU_MUL: return v0 / (1.0f + expf(-v0)) * v1;
    case EA_MAP_ADD: return v0 + v1;
    case EA_MAP_EXP_SUB: return expf(v0 - v1);
    case EA_MAP_DIV: return v0 / v1;
    case EA_MAP_SQUARE: return scale * v0 * v0;
    case EA_MAP_RMS_APPLY: return v0 * rsqrtf(v1 + eps) * v2;
    case EA_MAP_EXP_SUB_DIV: return expf(v0 - v1) / v2;
    default: return v0;
    }
}

// Raw 16-byte chunk loads (kept packed in registers until used) and their
// conversion: a bf16 chunk of 8 cells is one uint4, an fp32 chunk two.
template <bool kBf16>
__device__ __forceinline__ void ld_raw(const char *base, int64_t i, uint4 *r) {
    if constexpr (kBf16) {
        r[0] = __ldg(reinterpret_cast<const uint4 *>(reinterpret_cast<const __nv_bfloat16 *>(base) + i));
    } else {
        const uint4 *p = reinterpret_cast<const uint4 *>(reinterpret_cast<const float *>(base) + i);
        r[0] = __ldg(p);
        r[1] = __ldg(p + 1);
    }
}

template <bool kBf16>
__device__ __forceinline__ float raw_at(const uint4 *r, int e) {
    const uint32_t *w = reinterpret_cast<const uint32_t *>(r);
    if constexpr (kBf16) {
        const uint32_t x = w[e >> 1];
        return __uint_as_float((e & 1) ? (x & 0xFFFF0000u) : (x << 16));
    } else {
        return __uint_as_float(w[e]);
    }
}

// The per-cell operator as a compile-time choice (the hot loops of the
// elementwise and row-reduction kernels are instantiated per map).  exp and
// division use the fast hardware approximations (a few ulp), well inside
// the fp32 and bf16 tolerances of the outputs.
template <int MAP>
__device__ __forceinline__ float fmap(float v0, float v1, float v2, float scale, float eps) {
    if constexpr (MAP == EA_MAP_PRODUCT) return scale * v0 * v1 * v2;
    else if constexpr (MAP == EA_MAP_IDENTITY) return scale * v0;
    else if constexpr (MAP == EA_MAP_SILU_MUL) return __fdividef(v0, 1.0f + __expf(-v0)) * v1;
    else if constexpr (MAP == EA_MAP_ADD) return v0 + v1;
    else if constexpr (MAP == EA_MAP_EXP_SUB) return __expf(v0 - v1);
    else if constexpr (MAP == EA_MAP_DIV) return __fdividef(v0, v1);
    else if constexpr (MAP == EA_MAP_SQUARE) return scale * v0 * v0;
    else if constexpr (MAP == EA_MAP_RMS_APPLY) return v0 * rsqrtf(v1 + eps) * v2;
    else if constexpr (MAP == EA_MAP_EXP_SUB_DIV) return __fdividef(__expf(v0 - v1), v2);
    else return v0;
}

// ---- bounds checks of a library built with EA_DEBUG_BOUNDS: before a tile
// (or segment, view, operand block) is touched, its element range is
// checked against its arena; outside it, the kernel raises the device error
// word (kDevBounds) and skips the access.  Compiled out otherwise.
#ifdef EA_DEBUG_BOUNDS
constexpr bool kBoundsCheck = true;
#else
constexpr bool kBoundsCheck = false;
#endif

// base + sum_i c_i str_i (0 <= c_i < ext_i) + c len_str (0 <= c < len)
// inside [0, elems); an empty range always is.
__device__ __forceinline__ bool range_in(int64_t base, int n, const int64_t *ext, const int64_t *str, int64_t len,
                                         int64_t len_str, int64_t elems) {
    if (len <= 0) return true;
    int64_t lo = base, hi = base;
    for (int i = 0; i < n; i++) {
        if (ext[i] <= 0) return true;
        const int64_t span = (ext[i] - 1) * str[i];
        if (span < 0) lo += span;
        else hi += span;
    }
    const int64_t span = (len - 1) * len_str;
    if (span < 0) lo += span;
    else hi += span;
    return lo >= 0 && hi < elems;
}

__device__ __forceinline__ bool bounds_fail(int *err) {
    if (err) atomicCAS(err, 0, (int)kDevBounds);
    return false;
}

// A view (elementwise join or row reduction) inside its output and input arenas.
__device__ __forceinline__ bool view_in(const EwItem &it, int n_in, const int64_t *in_elems, int64_t out_elems) {
    if (!range_in(it.out_base, it.nd, it.ext, it.ostr, it.len, it.out_inner, out_elems)) return false;
    for (int k = 0; k < n_in; k++)
        if (!range_in(it.in_base[k], it.nd, it.ext, it.istr[k], it.len, it.in_inner[k], in_elems[k])) return false;
    return true;
}

// An exchange segment's rows inside both arenas (copies: copy q read at
// q * copy_stride further on).
__device__ __forceinline__ bool seg_in(const XSeg &g, const XTile &T, int64_t src_elems, int64_t dst_elems,
                                       int copies = 1, int64_t copy_stride = 0) {
    if (T.row0 < 0 || T.row0 + T.nrows > g.rows || T.col0 < 0 || T.col0 + T.ncols > g.inner) return false;
    const int64_t s_hi = (copies - 1) * copy_stride;
    return range_in(g.src_off, g.nd, g.ext, g.sstr, g.inner, 1, src_elems - s_hi) &&
           range_in(g.dst_off, g.nd, g.ext, g.dstr, g.inner, 1, dst_elems);
}

__device__ __forceinline__ int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }
__device__ __forceinline__ int64_t max64(int64_t a, int64_t b) { return a > b ? a : b; }

// Decode a row index over the first nd outer dims (innermost last).
__device__ __forceinline__ void decode_row(const EwItem &it, int64_t r, int64_t *coord) {
#pragma unroll
    for (int d = kViewDims - 1; d >= 0; d--) {
        if (d >= it.nd) {
            coord[d] = 0;
            continue;
        }
        if (d == 0) {
            coord[0] = r;
        } else {
            int64_t e = it.ext[d];
            coord[d] = r % e;
            r /= e;
        }
    }
}

// Global coordinate of special letter `slot` at row coordinates `coord`
// and inner index `col`.
__device__ __forceinline__ int64_t special_coord(const EwItem &it, int slot, const int64_t *coord, int64_t col) {
    int sd = it.sdim[slot];
    if (sd < 0) return it.slo[slot];
    if (sd == kViewDims) return it.slo[slot] + col;
    return it.slo[slot] + coord[sd];
}

}  // namespace ea
