// attn_common.cuh -- helpers shared by the attention join-agg kernels:
// packed two-wide fp32 arithmetic, the base-2 exponential and bf16 packing.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "tc_common.cuh"

namespace ea {
namespace attn {

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Packed two-wide fp32 arithmetic (one instruction for two values).
__device__ __forceinline__ uint64_t pack_f32x2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ uint64_t pack_u32x2(uint32_t lo, uint32_t hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
    return r;
}
__device__ __forceinline__ float lo_f32(uint64_t v) { return __uint_as_float((uint32_t)v); }
__device__ __forceinline__ float hi_f32(uint64_t v) { return __uint_as_float((uint32_t)(v >> 32)); }
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t add_f32x2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t mul_f32x2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// Maximum of three (the inputs hold no NaN).
__device__ __forceinline__ float max3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

// Masked softmax over 32-key chunks of a row's scores (one row per thread,
// the scores in u as raw f32 bits).

// Drop the keys of a chunk (columns [q0, q0 + 32) of the row) outside the
// row's visible columns [jlo, jhi]; returns the maximum of the rest.
__device__ __forceinline__ float mask_chunk(uint32_t *u, int q0, int jlo, int jhi) {
#pragma unroll
    for (int q = 0; q < 32; q++)
        if (q0 + q < jlo || q0 + q > jhi) u[q] = __float_as_uint(-INFINITY);
    float m0 = -INFINITY, m1 = -INFINITY, m2 = -INFINITY, m3 = -INFINITY;
#pragma unroll
    for (int q = 0; q < 32; q += 8) {
        m0 = max3(m0, __uint_as_float(u[q]), __uint_as_float(u[q + 1]));
        m1 = max3(m1, __uint_as_float(u[q + 2]), __uint_as_float(u[q + 3]));
        m2 = max3(m2, __uint_as_float(u[q + 4]), __uint_as_float(u[q + 5]));
        m3 = max3(m3, __uint_as_float(u[q + 6]), __uint_as_float(u[q + 7]));
    }
    return fmaxf(max3(m0, m1, m2), m3);
}

// Exponentials of chunk Q0 / 16 (scores u[2 Q0, 2 Q0 + 32)), 2^(c s - base),
// packed two per word into u[Q0, Q0 + 16) (P's bf16 pairs), the pair-sums
// added into ls.  In place: a row's chunks are taken in increasing order.
template <int Q0>
__device__ __forceinline__ void exp_chunk(uint32_t *u, uint64_t c2, uint64_t nb2, uint64_t *ls) {
#pragma unroll
    for (int q = Q0; q < Q0 + 16; q++) {
        const uint64_t y = fma_f32x2(pack_u32x2(u[2 * q], u[2 * q + 1]), c2, nb2);
        const float e0 = ex2(lo_f32(y)), e1 = ex2(hi_f32(y));
        ls[q & 3] = add_f32x2(ls[q & 3], pack_f32x2(e0, e1));
        u[q] = pack_bf16(e0, e1);
    }
}

// P of a chunk with no visible key: zero.
template <int Q0>
__device__ __forceinline__ void zero_chunk(uint32_t *u) {
#pragma unroll
    for (int q = Q0; q < Q0 + 16; q++) u[q] = 0u;
}

}  // namespace attn
}  // namespace ea
