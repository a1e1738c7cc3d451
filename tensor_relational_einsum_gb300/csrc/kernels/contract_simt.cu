// contract_simt.cu -- grouped contraction on the CUDA cores (FFMA, fp32
// accumulate).  Used for fp32 relations (plain TF32 tensor-core math would
// not meet an fp32 tolerance) and for any layout the TMA path cannot tile.
//
// "Every Kernel Is a Join", Examples 3.8/3.9 and Definition 3.7: a matrix
// multiply is a join on the shared inner index followed by a SUM; every
// function specification multiplies one pair of blocks, and the
// specifications with the same output block are summed.  One CTA owns a
// 64x64 tile of one output block and runs every function specification of
// that block's group in canonical order, keeping the SUM in registers --
// the aggregation is fused, no partial block is written.
#include <algorithm>
#include <math.h>

#include "dev_common.cuh"

namespace ea {

namespace {

constexpr int kK = 64;  // k chunk

// One CTA per TT x TT output tile, MT x MT outputs per thread; the next k
// chunk is read into registers while the current one is multiplied from
// shared memory, so each chunk costs one global round trip overlapped with
// math.
// A CTA's output tile, and every operand block its group's tuples read,
// inside the arenas (checked by a library built with EA_DEBUG_BOUNDS).
__device__ __forceinline__ bool ct_in(const CtParams &p, const CtGroup &G) {
    const int64_t ce[3] = {G.M, G.N, G.nb}, cs[3] = {G.c_sm, G.c_sn, G.c_sb};
    if (!range_in(G.c_base, 3, ce, cs, 1, 0, p.c_elems)) return false;
    for (int t = G.t0; t < G.t1; t++) {
        const CtTuple U = p.tuples[t];
        const int64_t ae[3] = {G.M, U.K, G.nb}, as[3] = {U.a_sm, U.a_sk, U.a_sb};
        const int64_t be[3] = {U.K, G.N, G.nb}, bs[3] = {U.b_sk, U.b_sn, U.b_sb};
        if (!range_in(U.a_base, 3, ae, as, 1, 0, p.a_elems) || !range_in(U.b_base, 3, be, bs, 1, 0, p.b_elems))
            return false;
    }
    return true;
}

template <int TT, int MT>
__global__ void __launch_bounds__((TT / MT) * (TT / MT)) simt_contract_kernel(const CtParams p) {
    constexpr int NT = (TT / MT) * (TT / MT);
    constexpr int PER = kK * TT / NT;  // elements of each operand a thread stages per chunk
    __shared__ float As[kK][TT + 4];
    __shared__ float Bs[kK][TT + 4];
    const CtTile tile = p.tiles[blockIdx.x];
    const CtGroup G = p.groups[tile.group];
    if constexpr (kBoundsCheck) {
        if (!ct_in(p, G)) {
            if (threadIdx.x == 0) bounds_fail(p.err);
            return;
        }
    }
    const int tx = threadIdx.x % (TT / MT), ty = threadIdx.x / (TT / MT);
    float acc[MT][MT];
#pragma unroll
    for (int i = 0; i < MT; i++)
#pragma unroll
        for (int j = 0; j < MT; j++) acc[i][j] = 0.0f;
    const int64_t m0 = tile.m0, n0 = tile.n0, bb = tile.batch;
    float ra[PER], rb[PER];
    // stage chunk (t, k0) of both operands into registers
    auto fetch = [&](const CtTuple &U, int64_t k0) {
        const bool a_m_fast = U.a_sk != 1 && U.a_sm == 1;
        const bool b_n_fast = !(U.b_sk == 1 && U.b_sn != 1);
#pragma unroll
        for (int q = 0; q < PER; q++) {
            const int i = threadIdx.x + q * NT;
            const int m = a_m_fast ? i % TT : i / kK, k = a_m_fast ? i / TT : i % kK;
            const int64_t gm = m0 + m, gk = k0 + k;
            ra[q] = (gm < G.M && gk < U.K) ? ld_elem(p.a, p.a_dtype, U.a_base + gm * U.a_sm + gk * U.a_sk + bb * U.a_sb)
                                           : 0.0f;
            const int n = b_n_fast ? i % TT : i / kK, k2 = b_n_fast ? i / TT : i % kK;
            const int64_t gn = n0 + n, gk2 = k0 + k2;
            rb[q] = (gn < G.N && gk2 < U.K) ? ld_elem(p.b, p.b_dtype, U.b_base + gk2 * U.b_sk + gn * U.b_sn + bb * U.b_sb)
                                            : 0.0f;
        }
    };
    auto stash = [&](const CtTuple &U) {
        const bool a_m_fast = U.a_sk != 1 && U.a_sm == 1;
        const bool b_n_fast = !(U.b_sk == 1 && U.b_sn != 1);
#pragma unroll
        for (int q = 0; q < PER; q++) {
            const int i = threadIdx.x + q * NT;
            const int m = a_m_fast ? i % TT : i / kK, k = a_m_fast ? i / TT : i % kK;
            As[k][m] = ra[q];
            const int n = b_n_fast ? i % TT : i / kK, k2 = b_n_fast ? i / TT : i % kK;
            Bs[k2][n] = rb[q];
        }
    };
    int t = G.t0;
    int64_t k0 = 0;
    if (t < G.t1) fetch(p.tuples[t], 0);
    while (t < G.t1) {
        const CtTuple U = p.tuples[t];
        stash(U);
        __syncthreads();
        // the next chunk: the rest of this tuple, else the next tuple's first
        int tn = t;
        int64_t kn = k0 + kK;
        if (kn >= U.K) {
            tn = t + 1;
            kn = 0;
        }
        if (tn < G.t1) fetch(p.tuples[tn], kn);
#pragma unroll
        for (int k = 0; k < kK; k++) {
            float a[MT], b[MT];
#pragma unroll
            for (int i = 0; i < MT; i++) a[i] = As[k][ty * MT + i];
#pragma unroll
            for (int j = 0; j < MT; j++) b[j] = Bs[k][tx * MT + j];
#pragma unroll
            for (int i = 0; i < MT; i++)
#pragma unroll
                for (int j = 0; j < MT; j++) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
        t = tn;
        k0 = kn;
    }
#pragma unroll
    for (int i = 0; i < MT; i++) {
        int64_t gm = m0 + ty * MT + i;
        if (gm >= G.M) continue;
#pragma unroll
        for (int j = 0; j < MT; j++) {
            int64_t gn = n0 + tx * MT + j;
            if (gn >= G.N) continue;
            float v = acc[i][j] * p.scale;
            if (p.pred_mode == 1 && G.n_lo + gn > G.m_lo + gm) v = -INFINITY;
            if (p.pred_mode == 2 && G.m_lo + gm > G.n_lo + gn) v = -INFINITY;
            st_elem(p.c, p.c_dtype, G.c_base + gm * G.c_sm + gn * G.c_sn + bb * G.c_sb, v);
        }
    }
}

// fp32 operands: the k chunks of a group stream through a ring of S shared-
// memory stages with cp.async (4-byte copies, any operand layout, zeros past
// the block edges), S - 1 chunks in flight ahead of the one being
// multiplied -- so a small group's chunks (C1: four tuples of 64) are all
// requested at once instead of one global round trip after another.  The
// chunks are still multiplied, and summed, in canonical tuple order.
__device__ __forceinline__ void cp_async4(float *dst, const float *src, bool valid) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)), "l"(src),
                 "r"(valid ? 4 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

template <int TT, int MT, int S>
struct MsCfg {
    static constexpr int LD = TT + 4;                      // padded row of a stage
    static constexpr int STAGE = 2 * kK * LD;              // floats of one stage (A and B)
    static constexpr int SMEM = S * STAGE * (int)sizeof(float);
};

template <int TT, int MT, int S>
__global__ void __launch_bounds__((TT / MT) * (TT / MT)) simt_ms_kernel(const CtParams p) {
    using C = MsCfg<TT, MT, S>;
    constexpr int NT = (TT / MT) * (TT / MT);
    constexpr int PER = kK * TT / NT;
    extern __shared__ float sm[];
    const CtTile tile = p.tiles[blockIdx.x];
    const CtGroup G = p.groups[tile.group];
    if constexpr (kBoundsCheck) {
        if (!ct_in(p, G)) {
            if (threadIdx.x == 0) bounds_fail(p.err);
            return;
        }
    }
    const int tx = threadIdx.x % (TT / MT), ty = threadIdx.x / (TT / MT);
    const int64_t m0 = tile.m0, n0 = tile.n0, bb = tile.batch;
    const float *A = reinterpret_cast<const float *>(p.a), *B = reinterpret_cast<const float *>(p.b);
    float acc[MT][MT];
#pragma unroll
    for (int i = 0; i < MT; i++)
#pragma unroll
        for (int j = 0; j < MT; j++) acc[i][j] = 0.0f;
    // issue cursor: the next chunk to request (tuple ti, offset ki)
    int ti = G.t0;
    int64_t ki = 0;
    CtTuple Ui;
    while (ti < G.t1 && p.tuples[ti].K <= 0) ti++;  // (tilings have no empty blocks; kept for safety)
    if (ti < G.t1) Ui = p.tuples[ti];
    auto issue = [&](int stage) {
        if (ti < G.t1) {
            float *As = sm + stage * C::STAGE, *Bs = As + kK * C::LD;
            const bool a_m_fast = Ui.a_sk != 1 && Ui.a_sm == 1;
            const bool b_n_fast = !(Ui.b_sk == 1 && Ui.b_sn != 1);
#pragma unroll
            for (int q = 0; q < PER; q++) {
                const int i = threadIdx.x + q * NT;
                const int m = a_m_fast ? i % TT : i / kK, k = a_m_fast ? i / TT : i % kK;
                const int64_t gm = m0 + m, gk = ki + k;
                const bool va = gm < G.M && gk < Ui.K;
                cp_async4(As + k * C::LD + m, va ? A + Ui.a_base + gm * Ui.a_sm + gk * Ui.a_sk + bb * Ui.a_sb : A, va);
                const int n = b_n_fast ? i % TT : i / kK, k2 = b_n_fast ? i / TT : i % kK;
                const int64_t gn = n0 + n, gk2 = ki + k2;
                const bool vb = gn < G.N && gk2 < Ui.K;
                cp_async4(Bs + k2 * C::LD + n, vb ? B + Ui.b_base + gk2 * Ui.b_sk + gn * Ui.b_sn + bb * Ui.b_sb : B, vb);
            }
            ki += kK;
            if (ki >= Ui.K) {
                ki = 0;
                ++ti;
                while (ti < G.t1 && p.tuples[ti].K <= 0) ti++;
                if (ti < G.t1) Ui = p.tuples[ti];
            }
        }
        cp_async_commit();  // an empty group past the last chunk keeps the counting uniform
    };
    int64_t nchunks = 0;
    for (int t = G.t0; t < G.t1; t++)
        if (p.tuples[t].K > 0) nchunks += (p.tuples[t].K + kK - 1) / kK;
#pragma unroll
    for (int s = 0; s < S - 1; s++) issue(s);
    for (int64_t c = 0; c < nchunks; c++) {
        cp_async_wait<S - 2>();  // this thread's copies of chunk c have landed
        __syncthreads();         // ... and everyone's; stage (c - 1) % S is free again
        issue((int)((c + S - 1) % S));
        const float *As = sm + (c % S) * C::STAGE, *Bs = As + kK * C::LD;
#pragma unroll 8
        for (int k = 0; k < kK; k++) {
            float a[MT], b[MT];
#pragma unroll
            for (int i = 0; i < MT; i++) a[i] = As[k * C::LD + ty * MT + i];
#pragma unroll
            for (int j = 0; j < MT; j++) b[j] = Bs[k * C::LD + tx * MT + j];
#pragma unroll
            for (int i = 0; i < MT; i++)
#pragma unroll
                for (int j = 0; j < MT; j++) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
    }
    cp_async_wait<0>();
#pragma unroll
    for (int i = 0; i < MT; i++) {
        int64_t gm = m0 + ty * MT + i;
        if (gm >= G.M) continue;
#pragma unroll
        for (int j = 0; j < MT; j++) {
            int64_t gn = n0 + tx * MT + j;
            if (gn >= G.N) continue;
            float v = acc[i][j] * p.scale;
            if (p.pred_mode == 1 && G.n_lo + gn > G.m_lo + gm) v = -INFINITY;
            if (p.pred_mode == 2 && G.m_lo + gm > G.n_lo + gn) v = -INFINITY;
            st_elem(p.c, p.c_dtype, G.c_base + gm * G.c_sm + gn * G.c_sn + bb * G.c_sb, v);
        }
    }
}

// Small groups (fp32, 32x32 output tiles, at most four tuples of one k chunk
// each): warp group g (64 threads, 4x4 outputs each) multiplies tuple t0 + g
// on its own pair of staged chunks, all tuples' copies in flight at once;
// the per-tuple products -- the function specifications' outputs of
// Definition 3.7 -- are then summed in canonical order (t0, t0 + 1, ...).
constexpr int kSplitLD = 32 + 4;
constexpr int kSplitSmem = 4 * 2 * kK * kSplitLD * (int)sizeof(float);

__global__ void __launch_bounds__(256) simt_split_kernel(const CtParams p) {
    extern __shared__ float sm[];
    const CtTile tile = p.tiles[blockIdx.x];
    const CtGroup G = p.groups[tile.group];
    if constexpr (kBoundsCheck) {
        if (!ct_in(p, G)) {
            if (threadIdx.x == 0) bounds_fail(p.err);
            return;
        }
    }
    const int g = threadIdx.x / 64, lt = threadIdx.x % 64;
    const int tx = lt % 8, ty = lt / 8;
    const int64_t m0 = tile.m0, n0 = tile.n0, bb = tile.batch;
    const float *A = reinterpret_cast<const float *>(p.a), *B = reinterpret_cast<const float *>(p.b);
    float *As = sm + g * 2 * kK * kSplitLD, *Bs = As + kK * kSplitLD;
    const int nt = G.t1 - G.t0;
    if (g < nt) {
        const CtTuple U = p.tuples[G.t0 + g];
        const bool a_m_fast = U.a_sk != 1 && U.a_sm == 1;
        const bool b_n_fast = !(U.b_sk == 1 && U.b_sn != 1);
#pragma unroll
        for (int q = 0; q < kK * 32 / 64; q++) {
            const int i = lt + q * 64;
            const int m = a_m_fast ? i % 32 : i / kK, k = a_m_fast ? i / 32 : i % kK;
            const int64_t gm = m0 + m;
            const bool va = gm < G.M && k < U.K;
            cp_async4(As + k * kSplitLD + m, va ? A + U.a_base + gm * U.a_sm + k * U.a_sk + bb * U.a_sb : A, va);
            const int n = b_n_fast ? i % 32 : i / kK, k2 = b_n_fast ? i / 32 : i % kK;
            const int64_t gn = n0 + n;
            const bool vb = gn < G.N && k2 < U.K;
            cp_async4(Bs + k2 * kSplitLD + n, vb ? B + U.b_base + k2 * U.b_sk + gn * U.b_sn + bb * U.b_sb : B, vb);
        }
    }
    cp_async_commit();
    cp_async_wait<0>();
    __syncthreads();
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; i++)
#pragma unroll
        for (int j = 0; j < 4; j++) acc[i][j] = 0.0f;
    if (g < nt) {
#pragma unroll 8
        for (int k = 0; k < kK; k++) {
            float a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; i++) a[i] = As[k * kSplitLD + ty * 4 + i];
#pragma unroll
            for (int j = 0; j < 4; j++) b[j] = Bs[k * kSplitLD + tx * 4 + j];
#pragma unroll
            for (int i = 0; i < 4; i++)
#pragma unroll
                for (int j = 0; j < 4; j++) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
    }
    __syncthreads();  // every group is done with its chunks: reuse them for the partial tiles
    float *part = sm + g * 32 * 32;
#pragma unroll
    for (int i = 0; i < 4; i++)
#pragma unroll
        for (int j = 0; j < 4; j++) part[(ty * 4 + i) * 32 + tx * 4 + j] = acc[i][j];
    __syncthreads();
    // output cells r of the tile, four per thread: the tuples' products in order
#pragma unroll
    for (int q = 0; q < 4; q++) {
        const int r = threadIdx.x + q * 256;
        const int mi = r / 32, nj = r % 32;
        const int64_t gm = m0 + mi, gn = n0 + nj;
        if (gm >= G.M || gn >= G.N) continue;
        float v = sm[r];
        for (int t = 1; t < nt; t++) v += sm[t * 32 * 32 + r];
        v *= p.scale;
        if (p.pred_mode == 1 && G.n_lo + gn > G.m_lo + gm) v = -INFINITY;
        if (p.pred_mode == 2 && G.m_lo + gm > G.n_lo + gn) v = -INFINITY;
        st_elem(p.c, p.c_dtype, G.c_base + gm * G.c_sm + gn * G.c_sn + bb * G.c_sb, v);
    }
}

cudaError_t launch_split(const CtParams &p, cudaStream_t st) {
    static bool configured[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64 && !configured[dev]) {
        e = cudaFuncSetAttribute(simt_split_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSplitSmem);
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    simt_split_kernel<<<(unsigned)p.ntiles, 256, kSplitSmem, st>>>(p);
    return cudaGetLastError();
}

template <int TT, int MT, int S>
cudaError_t launch_ms(const CtParams &p, cudaStream_t st) {
    using C = MsCfg<TT, MT, S>;
    static bool configured[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64 && !configured[dev]) {
        e = cudaFuncSetAttribute(simt_ms_kernel<TT, MT, S>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    simt_ms_kernel<TT, MT, S><<<(unsigned)p.ntiles, (TT / MT) * (TT / MT), C::SMEM, st>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_contract_simt(const CtParams &p, cudaStream_t st) {
    const bool f32 = p.a_dtype == EA_F32 && p.b_dtype == EA_F32;
    if (f32 && p.split) return launch_split(p, st);
    if (f32) return p.tile == 32 ? launch_ms<32, 2, 4>(p, st) : launch_ms<64, 4, 3>(p, st);
    if (p.tile == 32) simt_contract_kernel<32, 2><<<(unsigned)p.ntiles, 256, 0, st>>>(p);
    else simt_contract_kernel<64, 4><<<(unsigned)p.ntiles, 256, 0, st>>>(p);
    return cudaGetLastError();
}

}  // namespace ea
