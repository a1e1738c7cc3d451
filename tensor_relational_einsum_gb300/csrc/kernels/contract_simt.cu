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
template <int TT, int MT>
__global__ void __launch_bounds__((TT / MT) * (TT / MT)) simt_contract_kernel(const CtParams p) {
    constexpr int NT = (TT / MT) * (TT / MT);
    constexpr int PER = kK * TT / NT;  // elements of each operand a thread stages per chunk
    __shared__ float As[kK][TT + 4];
    __shared__ float Bs[kK][TT + 4];
    const CtTile tile = p.tiles[blockIdx.x];
    const CtGroup G = p.groups[tile.group];
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

}  // namespace

cudaError_t launch_contract_simt(const CtParams &p, cudaStream_t st) {
    if (p.tile == 32) simt_contract_kernel<32, 2><<<(unsigned)p.ntiles, 256, 0, st>>>(p);
    else simt_contract_kernel<64, 4><<<(unsigned)p.ntiles, 256, 0, st>>>(p);
    return cudaGetLastError();
}

}  // namespace ea
