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

constexpr int kT = 64;   // output tile
constexpr int kK = 16;   // k chunk
constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads) simt_contract_kernel(const CtParams p) {
    __shared__ float As[kK][kT + 4];
    __shared__ float Bs[kK][kT + 4];
    const CtTile tile = p.tiles[blockIdx.x];
    const CtGroup G = p.groups[tile.group];
    const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; i++)
#pragma unroll
        for (int j = 0; j < 4; j++) acc[i][j] = 0.0f;
    const int64_t m0 = tile.m0, n0 = tile.n0, bb = tile.batch;
    for (int t = G.t0; t < G.t1; t++) {
        const CtTuple U = p.tuples[t];
        const bool a_m_fast = U.a_sk != 1 && U.a_sm == 1;
        const bool b_n_fast = !(U.b_sk == 1 && U.b_sn != 1);
        for (int64_t k0 = 0; k0 < U.K; k0 += kK) {
            for (int i = threadIdx.x; i < kK * kT; i += kThreads) {
                int m, k;
                if (a_m_fast) {
                    m = i % kT;
                    k = i / kT;
                } else {
                    m = i / kK;
                    k = i % kK;
                }
                int64_t gm = m0 + m, gk = k0 + k;
                As[k][m] = (gm < G.M && gk < U.K)
                               ? ld_elem(p.a, p.a_dtype, U.a_base + gm * U.a_sm + gk * U.a_sk + bb * U.a_sb)
                               : 0.0f;
                int n, k2;
                if (b_n_fast) {
                    n = i % kT;
                    k2 = i / kT;
                } else {
                    n = i / kK;
                    k2 = i % kK;
                }
                int64_t gn = n0 + n, gk2 = k0 + k2;
                Bs[k2][n] = (gn < G.N && gk2 < U.K)
                                ? ld_elem(p.b, p.b_dtype, U.b_base + gk2 * U.b_sk + gn * U.b_sn + bb * U.b_sb)
                                : 0.0f;
            }
            __syncthreads();
#pragma unroll
            for (int k = 0; k < kK; k++) {
                float a[4], b[4];
#pragma unroll
                for (int i = 0; i < 4; i++) a[i] = As[k][ty * 4 + i];
#pragma unroll
                for (int j = 0; j < 4; j++) b[j] = Bs[k][tx * 4 + j];
#pragma unroll
                for (int i = 0; i < 4; i++)
#pragma unroll
                    for (int j = 0; j < 4; j++) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
            }
            __syncthreads();
        }
    }
#pragma unroll
    for (int i = 0; i < 4; i++) {
        int64_t gm = m0 + ty * 4 + i;
        if (gm >= G.M) continue;
#pragma unroll
        for (int j = 0; j < 4; j++) {
            int64_t gn = n0 + tx * 4 + j;
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
    simt_contract_kernel<<<(unsigned)p.ntiles, kThreads, 0, st>>>(p);
    return cudaGetLastError();
}

}  // namespace ea
