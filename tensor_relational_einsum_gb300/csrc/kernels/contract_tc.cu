// contract_tc.cu -- grouped bf16 contraction on the sm_103a tensor cores
// (tcgen05.mma with the accumulator in TMEM, operands staged by TMA).
//
// "Every Kernel Is a Join", Examples 3.8/3.9 and Definition 3.7: every
// function specification of a contraction multiplies one block of each
// input, and the specifications that share an output block are combined by
// SUM.  One output tile (128 x BN of one output block) accumulates, in the
// same TMEM accumulator, every k-chunk of every function specification of
// its group: the SUM aggregation is the MMA's own accumulate, with no
// partial block in memory and no separate reduction pass.
//
// Warp roles (256 threads, one CTA per SM, persistent over tiles):
//   warp 0   TMA producer: for each tile, each tuple of the group, each
//            64-wide k-chunk: A tile [128 x 64] and B tile [BN x 64] into a
//            stage of the smem ring (128-byte swizzle), one mbarrier with
//            the byte count per stage.
//   warp 1   MMA issuer (one thread): 4 x tcgen05.mma (K = 16 each) per
//            stage into the tile's TMEM accumulator; tcgen05.commit frees
//            the stage; after the last stage of a tile, commit signals the
//            epilogue.  Two accumulators (2 x BN TMEM columns) let the MMA
//            of tile i+1 run while the epilogue drains tile i.
//   warp 2   allocates and frees TMEM.
//   warps 4-7 epilogue: tcgen05.ld of its 32 rows, scale, predicate mask
//            (-inf), convert, write 128-byte swizzled rows into a staging
//            buffer, TMA store (double-buffered).
// Every mbarrier wait is bounded (2 s of %globaltimer); on time-out the
// kernel raises the device error word, the other roles leave their loops,
// the MMA issuer waits for its own MMAs, TMEM is freed and the CTA exits.
#include <algorithm>

#include "dev_common.cuh"
#include "tc_common.cuh"

namespace ea {

namespace {

using namespace tc;

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int kThreads = 256;

template <int BN>
struct Cfg {
    static constexpr int A_BYTES = BM * BK * 2;
    static constexpr int B_BYTES = BN * BK * 2;
    static constexpr int STAGE = A_BYTES + B_BYTES;
    static constexpr int STAGES = BN == 256 ? 4 : 6;
    static constexpr int STAGING = 2 * 16384;
    static constexpr int CTL = 256;
    static constexpr int SMEM = 1024 + STAGES * STAGE + STAGING + CTL;
    static constexpr uint32_t TMEM_COLS = 2 * BN;
};

struct SmemCtl {
    uint64_t full[8];
    uint64_t empty[8];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t mma_done;
    uint32_t tmem_base;
    int abort;
    int ep_ok;
};

// ------------------------------------------------------------------ kernel

template <int BN, int CL>
__global__ void __launch_bounds__(kThreads, 1) tc_contract_kernel(const TcParams p) {
    using C = Cfg<BN>;
    // CL CTAs of a cluster run tiles that share their B tile: each loads
    // 1/CL of it and multicasts it to all, so L2 serves each B byte once
    // per cluster; a stage is refilled only when every CTA's MMAs are done
    // with it (their commits arrive on every CTA's `empty`).
    constexpr uint16_t kMask = (uint16_t)((1u << CL) - 1);
    const int rank = CL > 1 ? (int)cluster_rank() : 0;
    const int nunits = (p.ntiles + CL - 1) / CL, unit0 = blockIdx.x / CL, ustep = gridDim.x / CL;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t *stages = smem;
    uint8_t *staging = smem + C::STAGES * C::STAGE;
    SmemCtl *ctl = reinterpret_cast<SmemCtl *>(staging + C::STAGING);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const CUtensorMap *maps = reinterpret_cast<const CUtensorMap *>(p.tmaps);
    volatile int *abort = &ctl->abort;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; s++) {
            mbar_init(&ctl->full[s], 1);
            mbar_init(&ctl->empty[s], CL);
        }
        for (int a = 0; a < 2; a++) {
            mbar_init(&ctl->tfull[a], 1);
            mbar_init(&ctl->tempty[a], 1);
        }
        mbar_init(&ctl->mma_done, 1);
        ctl->abort = 0;
        ctl->ep_ok = 1;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        fence_proxy_async();
    }
    if (warp == 2) tmem_alloc(smem_u32(&ctl->tmem_base), C::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    if (CL > 1) cluster_sync();  // every CTA's barriers are initialised before any multicast
    tc_fence_after();
    const uint32_t tmem = ctl->tmem_base;

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------ TMA producer
        int stage = 0;
        uint32_t ph = 0;
        uint32_t armed = 0, armed_par = 0;  // per stage: a load issued, and its phase parity
        for (int unit = unit0; unit < nunits; unit += ustep) {
            const TcTile T = p.tiles[unit * CL + rank];
            const TcGroup G = p.groups[T.group];
            bool ok = true;
            for (int t = G.t0; t < G.t1 && ok; t++) {
                const TcTuple U = p.tuples[t];
                const CUtensorMap *am = maps + U.a_map;
                const CUtensorMap *bm = maps + U.b_map;
                for (int kc = 0; kc < U.kchunks; kc++) {
                    if (!mbar_wait(&ctl->empty[stage], ph ^ 1, abort, p.err, kDevTimeoutProducer)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sa = smem_u32(stages + stage * C::STAGE), sb = sa + C::A_BYTES;
                    uint64_t *fb = &ctl->full[stage];
                    mbar_expect_tx(fb, C::STAGE);
                    if (!p.a_mn_major) {
                        tma_load_3d(sa, am, fb, kc * BK, T.m0, T.batch);
                    } else {
                        tma_load_3d(sa, am, fb, T.m0, kc * BK, T.batch);
                        tma_load_3d(sa + 8192, am, fb, T.m0 + 64, kc * BK, T.batch);
                    }
                    if (CL == 1) {
                        if (!p.b_mn_major) {
                            tma_load_3d(sb, bm, fb, kc * BK, T.n0, T.batch);
                        } else {
#pragma unroll
                            for (int j = 0; j < BN / 64; j++)
                                tma_load_3d(sb + j * 8192, bm, fb, T.n0 + 64 * j, kc * BK, T.batch);
                        }
                    } else {
                        // this CTA's 1/CL of the B tile, to every CTA of the cluster
                        constexpr int ROWS = BN / CL;
                        if (!p.b_mn_major) {
                            tma_load_3d_mc(sb + rank * ROWS * 128, bm, fb, kc * BK, T.n0 + rank * ROWS, T.batch, kMask);
                        } else {
#pragma unroll
                            for (int j = 0; j < ROWS / 64; j++) {
                                const int jj = rank * (ROWS / 64) + j;
                                tma_load_3d_mc(sb + jj * 8192, bm, fb, T.n0 + 64 * jj, kc * BK, T.batch, kMask);
                            }
                        }
                    }
                    armed |= 1u << stage;
                    armed_par = (armed_par & ~(1u << stage)) | (ph << stage);
                    if (++stage == C::STAGES) {
                        stage = 0;
                        ph ^= 1;
                    }
                }
            }
            if (!ok) break;
        }
        if (*abort) {
            // Let our own copies land before the CTA can exit.
            for (int s = 0; s < C::STAGES; s++)
                if (armed & (1u << s)) mbar_wait(&ctl->full[s], (armed_par >> s) & 1, abort, p.err, 0, kDrainNs, false);
        }
    } else if (warp == 1 && lane == 0) {
        // ------------------------------------------------ MMA issuer
        const uint32_t idesc = make_idesc(BM, BN, p.a_mn_major, p.b_mn_major);
        int stage = 0, acc = 0;
        uint32_t ph = 0, acc_ph = 0;
        bool ok = true;
        for (int unit = unit0; unit < nunits && ok; unit += ustep) {
            const TcTile T = p.tiles[unit * CL + rank];
            const TcGroup G = p.groups[T.group];
            if (!mbar_wait(&ctl->tempty[acc], acc_ph ^ 1, abort, p.err, kDevTimeoutMma)) break;
            tc_fence_after();
            const uint32_t d = tmem + (uint32_t)(acc * BN);
            uint32_t accumulate = 0;
            for (int t = G.t0; t < G.t1 && ok; t++) {
                const TcTuple U = p.tuples[t];
                for (int kc = 0; kc < U.kchunks; kc++) {
                    if (!mbar_wait(&ctl->full[stage], ph, abort, p.err, kDevTimeoutMma)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(stages + stage * C::STAGE), sb = sa + C::A_BYTES;
#pragma unroll
                    for (int kk = 0; kk < BK / 16; kk++) {
                        const uint64_t ad = p.a_mn_major ? sdesc(sa + kk * 2048, 8192, 1024) : sdesc(sa + kk * 32, 16, 1024);
                        const uint64_t bd = p.b_mn_major ? sdesc(sb + kk * 2048, 8192, 1024) : sdesc(sb + kk * 32, 16, 1024);
                        umma_bf16(d, ad, bd, idesc, accumulate);
                        accumulate = 1;
                    }
                    if (CL == 1) umma_commit(&ctl->empty[stage]);
                    else umma_commit_mc(&ctl->empty[stage], kMask);
                    if (++stage == C::STAGES) {
                        stage = 0;
                        ph ^= 1;
                    }
                }
            }
            if (!ok) break;
            umma_commit(&ctl->tfull[acc]);
            acc ^= 1;
            if (acc == 0) acc_ph ^= 1;
        }
        // Every MMA this thread issued has completed once mma_done flips.
        umma_commit(&ctl->mma_done);
        mbar_wait(&ctl->mma_done, 0, abort, p.err, kDevTimeoutMma, kTimeoutNs, false);
    } else if (warp >= 4) {
        // ------------------------------------------------ epilogue
        const int ep = threadIdx.x - 128;  // = TMEM lane = row of the tile
        const int wq = warp & 3;
        const int CW = p.out_f32 ? 32 : 64;  // columns per 128-byte row chunk
        int acc = 0, buf = 0;
        uint32_t acc_ph = 0;
        for (int unit = unit0; unit < nunits; unit += ustep) {
            const TcTile T = p.tiles[unit * CL + rank];
            const TcGroup G = p.groups[T.group];
            const CUtensorMap *om = maps + G.out_map;
            const bool store = T.m0 < G.m_ext;  // a padding tile of a cluster is computed, not stored
            if (ep == 0) ctl->ep_ok = mbar_wait(&ctl->tfull[acc], acc_ph, abort, p.err, kDevTimeoutEpilogue) ? 1 : 0;
            named_bar(1, 128);
            if (!ctl->ep_ok) break;
            tc_fence_after();
            const uint32_t tb = tmem + ((uint32_t)(wq * 32) << 16) + (uint32_t)(acc * BN);
            const int64_t m_g = G.m_lo + T.m0 + ep;
            // the row's scale: scale, times rsqrt(row_rms + eps) for a fused RMSNorm apply
            const float sc = (p.row_rms && T.m0 + ep < G.m_ext)
                                 ? p.scale * rsqrtf(__ldg(p.row_rms + G.r_lo + T.m0 + ep) + p.eps)
                                 : p.scale;
            // epilogue join SiLU(g) * u over column pairs: 128 planned columns -> 64 stored
            for (int c0 = 0; p.epi == 2 && c0 < BN; c0 += 128) {
                if (T.n0 + c0 >= G.n_ext || !store) break;
                uint8_t *sbuf = staging + buf * 16384;
                const uint32_t rowbase = smem_u32(sbuf) + ep * 128;
#pragma unroll
                for (int hh = 0; hh < 2; hh++) {
                    uint32_t r[64];
                    tmem_ld32(tb + c0 + 64 * hh, r);
                    tmem_ld32(tb + c0 + 64 * hh + 32, r + 32);
                    tmem_wait_ld();
#pragma unroll
                    for (int q = 0; q < 4; q++) {
                        uint32_t w[4];
#pragma unroll
                        for (int e = 0; e < 4; e++) {
                            float o2[2];
#pragma unroll
                            for (int z = 0; z < 2; z++) {
                                const int jj = 8 * q + 2 * e + z;  // stored column inside the half
                                const float g = __uint_as_float(r[2 * jj]) * sc;
                                const float u = __uint_as_float(r[2 * jj + 1]) * sc;
                                o2[z] = __fdividef(g, 1.0f + __expf(-g)) * u;
                            }
                            __nv_bfloat162 hv = __floats2bfloat162_rn(o2[0], o2[1]);
                            w[e] = *reinterpret_cast<uint32_t *>(&hv);
                        }
                        const uint32_t addr = rowbase + ((uint32_t)((4 * hh + q) ^ (ep & 7)) << 4);
                        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(w[0]), "r"(w[1]),
                                     "r"(w[2]), "r"(w[3])
                                     : "memory");
                    }
                }
                fence_proxy_async();
                named_bar(1, 128);
                if (ep == 0) {
                    tma_store_3d(om, smem_u32(sbuf), (T.n0 + c0) / 2, T.m0, T.batch);
                    bulk_commit();
                    bulk_wait_read1();
                }
                buf ^= 1;
                named_bar(1, 128);
            }
            for (int c0 = 0; p.epi != 2 && c0 < BN; c0 += CW) {
                if (T.n0 + c0 >= G.n_ext || !store) break;  // whole chunk past the block edge
                uint32_t r[64];
                tmem_ld32(tb + c0, r);
                if (!p.out_f32) tmem_ld32(tb + c0 + 32, r + 32);
                tmem_wait_ld();
                float v[64];
#pragma unroll
                for (int j = 0; j < 64; j++) {
                    if (j < CW) {
                        float x = __uint_as_float(r[j]) * sc;
                        if (p.pred_mode) {
                            int64_t n_g = G.n_lo + T.n0 + c0 + j;
                            if ((p.pred_mode == 1 && n_g > m_g) || (p.pred_mode == 2 && m_g > n_g)) x = -INFINITY;
                        }
                        v[j] = x;
                    }
                }
                if (p.epi == 3 && T.m0 + ep < G.m_ext) {
                    // epilogue join ROPE: rotate the interleaved column pairs of this row
                    // by the angles of its position (rows = positions, packed sequences)
                    // (a pair-major table puts the warp's 32 consecutive positions
                    // of one pair side by side: one 256-byte read per pair)
                    const int64_t pos = (G.r_lo + T.m0 + ep) % p.rope_npos;
                    const float2 *tab = reinterpret_cast<const float2 *>(p.rope_table) +
                                        (p.rope_pm ? pos : pos * p.rope_half);
                    const int64_t pstride = p.rope_pm ? p.rope_npos : 1;
                    int ip = (int)(((G.c_lo + T.n0 + c0) >> 1) % p.rope_half);
#pragma unroll
                    for (int q = 0; q < 32; q++) {
                        if (2 * q < CW) {
                            const float2 cs = __ldg(tab + ip * pstride);
                            const float x0 = v[2 * q], x1 = v[2 * q + 1];
                            v[2 * q] = x0 * cs.x - x1 * cs.y;
                            v[2 * q + 1] = x0 * cs.y + x1 * cs.x;
                            if (++ip == p.rope_half) ip = 0;
                        }
                    }
                }
                if (p.epi == 1 && T.m0 + ep < G.m_ext) {
                    // epilogue join ADD: the joined relation's cells of this row segment
                    const int64_t e0 = G.e_base + (int64_t)T.batch * G.e_sb + (int64_t)(T.m0 + ep) * G.e_sm + T.n0 + c0;
                    const int nvalid = (int)min64((int64_t)CW, (int64_t)G.n_ext - (T.n0 + c0));
                    if (nvalid == CW) {
                        const uint4 *src = reinterpret_cast<const uint4 *>(p.epi_in + e0 * (p.out_f32 ? 4 : 2));
#pragma unroll
                        for (int q = 0; q < 8; q++) {
                            const uint4 w = __ldg(src + q);
                            const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                            for (int e = 0; e < 4; e++) {
                                if (p.out_f32) {
                                    v[4 * q + e] += __uint_as_float(ww[e]);
                                } else {
                                    v[8 * q + 2 * e] += __uint_as_float(ww[e] << 16);
                                    v[8 * q + 2 * e + 1] += __uint_as_float(ww[e] & 0xFFFF0000u);
                                }
                            }
                        }
                    } else {
#pragma unroll
                        for (int jj = 0; jj < 64; jj++)
                            if (jj < nvalid) {
                                if (p.out_f32) v[jj] += reinterpret_cast<const float *>(p.epi_in)[e0 + jj];
                                else v[jj] += __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(p.epi_in)[e0 + jj]);
                            }
                    }
                }
                uint8_t *sbuf = staging + buf * 16384;
                const uint32_t rowbase = smem_u32(sbuf) + ep * 128;
#pragma unroll
                for (int q = 0; q < 8; q++) {
                    uint32_t w0, w1, w2, w3;
                    if (p.out_f32) {
                        w0 = __float_as_uint(v[4 * q + 0]);
                        w1 = __float_as_uint(v[4 * q + 1]);
                        w2 = __float_as_uint(v[4 * q + 2]);
                        w3 = __float_as_uint(v[4 * q + 3]);
                    } else {
                        __nv_bfloat162 h0 = __floats2bfloat162_rn(v[8 * q + 0], v[8 * q + 1]);
                        __nv_bfloat162 h1 = __floats2bfloat162_rn(v[8 * q + 2], v[8 * q + 3]);
                        __nv_bfloat162 h2 = __floats2bfloat162_rn(v[8 * q + 4], v[8 * q + 5]);
                        __nv_bfloat162 h3 = __floats2bfloat162_rn(v[8 * q + 6], v[8 * q + 7]);
                        w0 = *reinterpret_cast<uint32_t *>(&h0);
                        w1 = *reinterpret_cast<uint32_t *>(&h1);
                        w2 = *reinterpret_cast<uint32_t *>(&h2);
                        w3 = *reinterpret_cast<uint32_t *>(&h3);
                    }
                    const uint32_t addr = rowbase + ((uint32_t)(q ^ (ep & 7)) << 4);
                    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(w0), "r"(w1), "r"(w2),
                                 "r"(w3)
                                 : "memory");
                }
                fence_proxy_async();
                named_bar(1, 128);
                if (ep == 0) {
                    tma_store_3d(om, smem_u32(sbuf), T.n0 + c0, T.m0, T.batch);
                    bulk_commit();
                    bulk_wait_read1();
                }
                buf ^= 1;
                named_bar(1, 128);
            }
            tc_fence_before();
            named_bar(1, 128);
            if (ep == 0) mbar_arrive(&ctl->tempty[acc]);
            acc ^= 1;
            if (acc == 0) acc_ph ^= 1;
        }
        if (ep == 0) bulk_wait_all();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
    if (CL > 1) cluster_sync();  // no CTA leaves while a peer may still signal or fill its shared memory
}

template <int BN, int CL>
cudaError_t launch_bn(const TcParams &p, int num_sms, cudaStream_t st) {
    using C = Cfg<BN>;
    static bool configured[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64 && !configured[dev]) {
        e = cudaFuncSetAttribute(tc_contract_kernel<BN, CL>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    const int units = (p.ntiles + CL - 1) / CL;
    if (CL == 1) {
        tc_contract_kernel<BN, CL><<<std::min<int>(units, num_sms), kThreads, C::SMEM, st>>>(p);
        return cudaGetLastError();
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(CL * std::min<int>(units, num_sms / CL), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // a persistent grid of no more clusters than can be resident at once
    static int resident[64] = {};
    const int di = (dev >= 0 && dev < 64) ? dev : 0;
    if (resident[di] == 0) {
        int n = 0;
        e = cudaOccupancyMaxActiveClusters(&n, tc_contract_kernel<BN, CL>, &cfg);
        if (e != cudaSuccess) return e;
        resident[di] = n > 0 ? n : std::max(1, num_sms / CL);
    }
    cfg.gridDim = dim3(CL * std::max(1, std::min(units, resident[di])), 1, 1);
    return cudaLaunchKernelEx(&cfg, tc_contract_kernel<BN, CL>, p);
}

}  // namespace

int tc_smem_bytes(int bn) { return bn == 256 ? Cfg<256>::SMEM : Cfg<128>::SMEM; }

cudaError_t launch_contract_tc(const TcParams &p, int num_sms, cudaStream_t st) {
    if (p.cluster == 2) {
        if (p.bn == 256) return launch_bn<256, 2>(p, num_sms, st);
        return launch_bn<128, 2>(p, num_sms, st);
    }
    if (p.bn == 256) return launch_bn<256, 1>(p, num_sms, st);
    return launch_bn<128, 1>(p, num_sms, st);
}

}  // namespace ea
