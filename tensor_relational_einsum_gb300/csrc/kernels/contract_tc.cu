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
// With enough tiles the CTAs run in pairs (clusters of two, tcgen05
// cta_group::2): a pair computes two M-adjacent tiles of the same output
// columns as one 256 x BN tile.  Each CTA loads its own 128 A rows and its
// own half of the B tile (plain TMA loads; the byte counts of both CTAs
// complete on the even CTA's stage barrier), and the even CTA's MMA thread
// issues M = 256 MMAs that read both CTAs' shared memory and write both
// CTAs' TMEM.  L2 and each SM's shared memory serve every B byte once per
// pair.  The MMA thread's commits signal the stage and accumulator barriers
// of both CTAs (the odd CTA's through its shared::cluster address), and the
// odd CTA's epilogue hands an accumulator back by a remote arrive.
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

template <int BN, bool PAIR>
struct Cfg {
    static constexpr int A_BYTES = BM * BK * 2;
    static constexpr int B_ROWS = PAIR ? BN / 2 : BN;  // this CTA's rows of the B tile
    static constexpr int B_BYTES = B_ROWS * BK * 2;
    static constexpr int STAGE = A_BYTES + B_BYTES;
    static constexpr int STAGES = (192 * 1024) / STAGE;  // 4 or 6 alone, 6 or 8 in a pair
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

template <int BN, bool PAIR>
__global__ void __launch_bounds__(kThreads, 1) tc_contract_kernel(const TcParams p) {
    using C = Cfg<BN, PAIR>;
    static_assert(C::STAGES <= 8, "stage barriers");
    constexpr int CL = PAIR ? 2 : 1;
    // In a pair, CTA rank 0 issues the MMAs; tiles 2u and 2u + 1 are rank 0's
    // and rank 1's rows of unit u.
    const int rank = PAIR ? (int)cluster_rank() : 0;
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
            mbar_init(&ctl->empty[s], 1);
        }
        for (int a = 0; a < 2; a++) {
            mbar_init(&ctl->tfull[a], 1);
            mbar_init(&ctl->tempty[a], CL);  // a pair's accumulator is free once both epilogues are done
        }
        mbar_init(&ctl->mma_done, 1);
        ctl->abort = 0;
        ctl->ep_ok = 1;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        fence_proxy_async();
    }
    if (warp == 2) {
        if (PAIR) tmem_alloc_pair(smem_u32(&ctl->tmem_base), C::TMEM_COLS);
        else tmem_alloc(smem_u32(&ctl->tmem_base), C::TMEM_COLS);
    }
    tc_fence_before();
    __syncthreads();
    if (PAIR) cluster_sync();  // both CTAs' barriers are initialised before either signals the other
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
                    if (!PAIR) {
                        mbar_expect_tx(fb, C::STAGE);
                        if (!p.a_mn_major) {
                            tma_load_3d(sa, am, fb, kc * BK, T.m0, T.batch);
                        } else {
                            tma_load_3d(sa, am, fb, T.m0, kc * BK, T.batch);
                            tma_load_3d(sa + 8192, am, fb, T.m0 + 64, kc * BK, T.batch);
                        }
                        if (!p.b_mn_major) {
                            tma_load_3d(sb, bm, fb, kc * BK, T.n0, T.batch);
                        } else {
#pragma unroll
                            for (int j = 0; j < BN / 64; j++)
                                tma_load_3d(sb + j * 8192, bm, fb, T.n0 + 64 * j, kc * BK, T.batch);
                        }
                    } else {
                        // this CTA's A rows and its half of the B tile, counted on rank 0's barrier
                        const uint32_t fc = mapa_u32(smem_u32(fb), 0);
                        if (rank == 0) mbar_expect_tx(fb, 2 * C::STAGE);
                        if (!p.a_mn_major) {
                            tma_load_3d_pair(sa, am, fc, kc * BK, T.m0, T.batch);
                        } else {
                            tma_load_3d_pair(sa, am, fc, T.m0, kc * BK, T.batch);
                            tma_load_3d_pair(sa + 8192, am, fc, T.m0 + 64, kc * BK, T.batch);
                        }
                        const int n_half = T.n0 + rank * C::B_ROWS;
                        if (!p.b_mn_major) {
                            tma_load_3d_pair(sb, bm, fc, kc * BK, n_half, T.batch);
                        } else {
#pragma unroll
                            for (int j = 0; j < C::B_ROWS / 64; j++)
                                tma_load_3d_pair(sb + j * 8192, bm, fc, n_half + 64 * j, kc * BK, T.batch);
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
            if (!PAIR || rank == 0) {
                for (int s = 0; s < C::STAGES; s++)
                    if (armed & (1u << s))
                        mbar_wait(&ctl->full[s], (armed_par >> s) & 1, abort, p.err, 0, kDrainNs, false);
            } else if (armed) {
                // rank 1's copies complete on rank 0's barriers: give them the drain time
                const uint64_t t0 = gtime();
                while (gtime() - t0 < kDrainNs) {
                }
            }
        }
    } else if (warp == 1 && rank == 0) {
        // ------------------------------------------------ MMA warp
        // The whole warp runs the issue loop (warp-uniform waits, cursors
        // and descriptors); one elected lane issues each stage's MMAs and
        // commits.
        const uint32_t idesc = make_idesc(CL * BM, BN, p.a_mn_major, p.b_mn_major);
        // descriptor layout and the address step of one K = 16 slice: a
        // K-major operand advances 32 bytes inside its 128-byte rows, an
        // MN-major one 16 rows of 128 bytes
        const uint32_t a_lbo = p.a_mn_major ? 8192 : 16, b_lbo = p.b_mn_major ? 8192 : 16;
        const uint64_t a_step = sdesc_off(p.a_mn_major ? 2048 : 32), b_step = sdesc_off(p.b_mn_major ? 2048 : 32);
        int stage = 0, acc = 0;
        uint32_t ph = 0, acc_ph = 0;
        bool ok = true;
        for (int unit = unit0; unit < nunits && ok; unit += ustep) {
            const TcTile T = p.tiles[unit * CL + rank];
            const TcGroup G = p.groups[T.group];
            if (!warp_wait(&ctl->tempty[acc], acc_ph ^ 1, abort, p.err, kDevTimeoutMma)) break;
            tc_fence_after();
            const uint32_t d = tmem + (uint32_t)(acc * BN);
            uint32_t accumulate = 0;
            for (int t = G.t0; t < G.t1 && ok; t++) {
                const TcTuple U = p.tuples[t];
                for (int kc = 0; kc < U.kchunks; kc++) {
                    if (!warp_wait(&ctl->full[stage], ph, abort, p.err, kDevTimeoutMma)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // the stage's descriptors once; each MMA adds a constant step
                    const uint32_t sa = smem_u32(stages + stage * C::STAGE), sb = sa + C::A_BYTES;
                    const uint64_t ad = sdesc(sa, a_lbo, 1024), bd = sdesc(sb, b_lbo, 1024);
                    if (elect_one()) {
#pragma unroll
                        for (int kk = 0; kk < BK / 16; kk++) {
                            const uint32_t acc_in = (accumulate | (uint32_t)kk) ? 1u : 0u;
                            if (PAIR) umma_bf16_pair(d, ad + kk * a_step, bd + kk * b_step, idesc, acc_in);
                            else umma_bf16(d, ad + kk * a_step, bd + kk * b_step, idesc, acc_in);
                        }
                        if (!PAIR) {
                            umma_commit(&ctl->empty[stage]);
                        } else {
                            umma_commit_pair(smem_u32(&ctl->empty[stage]));
                            umma_commit_pair(mapa_u32(smem_u32(&ctl->empty[stage]), 1));  // rank 1's
                        }
                    }
                    __syncwarp();
                    accumulate = 1;
                    if (++stage == C::STAGES) {
                        stage = 0;
                        ph ^= 1;
                    }
                }
            }
            if (!ok) break;
            if (elect_one()) {
                if (!PAIR) {
                    umma_commit(&ctl->tfull[acc]);
                } else {
                    umma_commit_pair(smem_u32(&ctl->tfull[acc]));
                    umma_commit_pair(mapa_u32(smem_u32(&ctl->tfull[acc]), 1));
                }
            }
            __syncwarp();
            acc ^= 1;
            if (acc == 0) acc_ph ^= 1;
        }
        // Every MMA this warp issued has completed once mma_done flips.
        if (elect_one()) {
            if (PAIR) umma_commit_pair(smem_u32(&ctl->mma_done));
            else umma_commit(&ctl->mma_done);
        }
        __syncwarp();
        if (lane == 0) mbar_wait(&ctl->mma_done, 0, abort, p.err, kDevTimeoutMma, kTimeoutNs, false);
        __syncwarp();
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
            bool store = T.m0 < G.m_ext;  // a padding tile of a CTA pair is computed, not stored
            if constexpr (kBoundsCheck) {
                // the rows of the tile the epilogue reads: the residual block
                // and the row scale (the output goes through its tensor map)
                const int64_t rows = min64(128, (int64_t)G.m_ext - T.m0), cols = min64(BN, (int64_t)G.n_ext - T.n0);
                bool in = true;
                if (store && p.epi == 1)
                    in = range_in(G.e_base + (int64_t)T.batch * G.e_sb + (int64_t)T.m0 * G.e_sm + T.n0, 1, &rows,
                                  &G.e_sm, cols, 1, p.epi_elems);
                const int64_t one = 1;
                if (store && p.row_rms) in = in && range_in(G.r_lo + T.m0, 1, &rows, &one, 1, 0, p.rms_elems);
                if (!in) {
                    if (ep == 0) bounds_fail(p.err);
                    store = false;
                }
            }
            if (ep == 0) ctl->ep_ok = mbar_wait(&ctl->tfull[acc], acc_ph, abort, p.err, kDevTimeoutEpilogue) ? 1 : 0;
            named_bar(1, 128);
            if (!ctl->ep_ok) break;
            tc_fence_after();
            const uint32_t tb = tmem + ((uint32_t)(wq * 32) << 16) + (uint32_t)(acc * BN);
            const int64_t m_g = G.m_lo + T.m0 + ep;
            // the row's scale: scale, times rsqrt(row_rms + eps) for a fused RMSNorm apply
            const float sc = (p.row_rms && store && T.m0 + ep < G.m_ext)
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
            if (ep == 0) {
                if (rank == 0) mbar_arrive(&ctl->tempty[acc]);
                else mbar_arrive_cluster(mapa_u32(smem_u32(&ctl->tempty[acc]), 0));
            }
            acc ^= 1;
            if (acc == 0) acc_ph ^= 1;
        }
        if (ep == 0) bulk_wait_all();
    }

    tc_fence_before();
    __syncthreads();
    // No CTA of a pair frees TMEM or leaves while the other may still signal
    // it, or the pair's MMAs may still read its shared memory.
    if (PAIR) cluster_sync();
    if (warp == 2) {
        tc_fence_after();
        if (PAIR) tmem_dealloc_pair(tmem, C::TMEM_COLS);
        else tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

template <int BN, bool PAIR>
cudaError_t launch_bn(const TcParams &p, int num_sms, cudaStream_t st) {
    using C = Cfg<BN, PAIR>;
    constexpr int CL = PAIR ? 2 : 1;
    static bool configured[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64 && !configured[dev]) {
        e = cudaFuncSetAttribute(tc_contract_kernel<BN, PAIR>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    const int units = (p.ntiles + CL - 1) / CL;
    if (!PAIR) {
        tc_contract_kernel<BN, PAIR><<<std::min<int>(units, num_sms), kThreads, C::SMEM, st>>>(p);
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
        e = cudaOccupancyMaxActiveClusters(&n, tc_contract_kernel<BN, PAIR>, &cfg);
        if (e != cudaSuccess) return e;
        resident[di] = n > 0 ? n : std::max(1, num_sms / CL);
    }
    cfg.gridDim = dim3(CL * std::max(1, std::min(units, resident[di])), 1, 1);
    return cudaLaunchKernelEx(&cfg, tc_contract_kernel<BN, PAIR>, p);
}

}  // namespace

cudaError_t launch_contract_tc(const TcParams &p, int num_sms, cudaStream_t st) {
    if (p.cluster == 2) {
        if (p.bn == 256) return launch_bn<256, true>(p, num_sms, st);
        return launch_bn<128, true>(p, num_sms, st);
    }
    if (p.bn == 256) return launch_bn<256, false>(p, num_sms, st);
    return launch_bn<128, false>(p, num_sms, st);
}

}  // namespace ea
