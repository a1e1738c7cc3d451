// attention.cu -- flash attention as one join-agg on the sm_103a tensor
// cores ("Every Kernel Is a Join", Example 3.10).
//
// The join-agg: an aggregation group is one tile of 128 query positions of
// one query head; its tuples are the key tiles (128 keys of a K/V block
// pair) the predicate keeps.  Each tuple's kernel computes the scores
// S = scale Q K^T of the tile, their row maximum m, p = exp(S - m), the
// row sum l of p and the partial output A = p V.  The group's tuples are
// aggregated with the merge of (m, l, A) triples
//     (m1, l1, A1) + (m2, l2, A2) = (M, l1 a1 + l2 a2, A1 a1 + A2 a2),
//     M = max(m1, m2), a_i = exp(m_i - M),
// which is associative and commutative; the output block is A / l.  The
// merge runs on chip, one key tile at a time: A accumulates in TMEM (the
// MMA's own accumulate), l and m in registers, so no score, probability or
// partial output ever reaches memory.
//
// The reference maximum of a row is only moved when a tile's maximum
// exceeds it by more than 2^kLazy in exp: until then the exponentials are
// taken against the older, smaller maximum, and A and l stay consistent
// with it, so A / l is unchanged.  With kLazy = 64 the exponentials stay
// below 2^64; fp32 and bf16 both have 8 exponent bits, so P, l and A (a sum
// of fewer than 2^31 keys' products with |v| < 2^32) stay far below the
// overflow at 2^128, and their relative rounding does not depend on the
// magnitude.  Moving the maximum rescales the row of A in TMEM; with a
// threshold this wide it happens on a row's first tile and almost never
// after, even where the scores spread over tens of units (unscaled scores
// of 128-wide heads).
//
// A work item is one or two groups that share their key tiles: two query
// tiles of the same head, X = 0 and X = 1, each with its own softmax
// warpgroup, score buffer S_X and output accumulator O_X in TMEM (columns
// S_0 [0, 128), S_1 [128, 256), O_0 [256, 256 + d), O_1 [256 + d, 256 + 2d)).
// Each K and V tile is loaded once for both, and while one warpgroup works
// on its scores the tensor cores run the other's products.
//
// Roles (384 threads, one CTA per SM, persistent over its list of items;
// warps 10 and 11 only complete the third warpgroup of the register split):
//   warp 8     TMA: Q tiles (one buffer per X), K and V of a key tile into
//              one stage of a two-stage ring with one barrier (128-byte
//              swizzle, one [128 x 64] box per 64 head-dim columns).
//   warp 9     TMEM owner and MMA issuer (the whole warp runs the loop with
//              warp-wide waits; one elected lane issues).  Per X and key tile
//              j (the first nt[X] tiles of the item: X stops after the last
//              tile it keeps): S_X = Q_X K_j^T; after the softmax of X has written P_X,
//              O_X (+)= P_X V_j with P_X read from TMEM, then at once
//              S_X = Q_X K_{j+1}^T (in order on the tensor pipe, so the
//              next scores land after P_X has been read).
//   warps 0-3 (X = 0), 4-7 (X = 1): one query row per thread (TMEM lane =
//              row): load the row of S_X, mask (causal, sequence ends,
//              ragged block ends), the row maximum, p = 2^(S c - m c) with
//              c = scale log2(e), the row sum, P_X as bf16 into the first 64
//              columns of S_X, the rescale of the row of O_X when the
//              reference maximum moves; at the end of the item O_X / l as
//              bf16 to global memory.
// Every mbarrier wait is bounded (2 s); on time-out the kernel raises the
// device error word, all roles leave their loops, the copies and MMAs in
// flight are waited for and TMEM is freed before the CTA exits.
#include <algorithm>

#include "attn_common.cuh"
#include "dev_common.cuh"
#include "tc_common.cuh"

namespace ea {

namespace {

using namespace tc;
using namespace attn;

constexpr int kRows = 128;  // query rows of a tile (= TMEM lanes)
constexpr int kKeys = 128;  // keys of a key tile
constexpr int kAtThreads = 384;  // three warpgroups: softmax X = 0, softmax X = 1, TMA + MMA (+2 idle warps)
// Register split (setmaxnreg): the block is launched with 168 registers a
// thread (384 x 168 = 64512); the TMA/MMA warpgroup gives up 80 a thread
// and the two softmax warpgroups take 40 each, so that a softmax thread keeps
// its row of 128 scores in registers.  The split uses exactly the launch's
// registers: 2 x 128 x 208 + 128 x 88 = 64512.
constexpr int kLaunchRegs = 168;
constexpr int kCtlRegs = 88;
constexpr int kSoftmaxRegs = 208;
static_assert(2 * 128 * kSoftmaxRegs + 128 * kCtlRegs <= kAtThreads * kLaunchRegs, "register split");
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kOCol = 256;  // first TMEM column of the output accumulators
constexpr float kLazy = 64.0f;   // log2 of the largest exponential taken against a stale maximum
constexpr int kKvStages = 2;     // K/V ring depth: stage s holds K and V of one key tile

struct AtCtl {
    uint64_t q_full[2], q_empty[2];
    uint64_t kv_full[kKvStages], kv_empty[kKvStages];
    uint64_t s_full[2], p_full[2], o_fin[2];
    uint64_t mma_done;
    uint32_t tmem_base;
    int abort;
};

template <int D>
struct AtCfg {
    static constexpr int CH = D / 64;            // 64-column (128-byte) chunks of the head dimension
    static constexpr int TILE = kRows * D * 2;   // one [128 x D] bf16 tile
    static constexpr int Q_OFF = 0;              // Q_0, Q_1
    static constexpr int K_OFF = 2 * TILE;       // K of each K/V stage
    static constexpr int V_OFF = 2 * TILE + kKvStages * TILE;  // V of each K/V stage
    static constexpr int CTL_OFF = 2 * TILE + 2 * kKvStages * TILE;
    static constexpr int SMEM = 1024 + CTL_OFF + (int)sizeof(AtCtl);
};

template <int D>
__global__ void __launch_bounds__(kAtThreads, 1) attention_kernel(const AtParams p) {
    using C = AtCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    AtCtl *ctl = reinterpret_cast<AtCtl *>(smem + C::CTL_OFF);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const CUtensorMap *maps = reinterpret_cast<const CUtensorMap *>(p.tmaps);
    volatile int *abort = &ctl->abort;
    const int i0 = p.cta_ptr[blockIdx.x], i1 = p.cta_ptr[blockIdx.x + 1];

    if (threadIdx.x == 0) {
        for (int b = 0; b < 2; b++) {
            mbar_init(&ctl->q_full[b], 1);
            mbar_init(&ctl->q_empty[b], 1);
            mbar_init(&ctl->s_full[b], 1);
            mbar_init(&ctl->p_full[b], 4);
            mbar_init(&ctl->o_fin[b], 1);
        }
        for (int b = 0; b < kKvStages; b++) {
            mbar_init(&ctl->kv_full[b], 1);
            mbar_init(&ctl->kv_empty[b], 1);
        }
        mbar_init(&ctl->mma_done, 1);
        ctl->abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        fence_proxy_async();
    }
    if (warp == 9) tmem_alloc(smem_u32(&ctl->tmem_base), kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl->tmem_base;

    if (warp >= 8) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kCtlRegs));
    if (warp == 8) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            // K and V of key tile t into stage t % kKvStages, one barrier for
            // both: the stage is released once O += P V of tile t is done.
            uint32_t ct = 0, qx0 = 0, qx1 = 0;  // key tiles; items per query slot
            uint32_t q_armed = 0, q_par = 0, kv_armed = 0, kv_par = 0;
            bool ok = true;
            for (int ii = i0; ii < i1 && ok; ii++) {
                const AtItem &it = p.items[ii];
                const int ntiles = it.ntiles, nq = it.nq;
                if (ntiles == 0) continue;
                for (int x = 0; x < nq && ok; x++) {
                    const uint32_t qn = x == 0 ? qx0 : qx1;
                    if (!mbar_wait(&ctl->q_empty[x], (qn & 1) ^ 1, abort, p.err, kDevTimeoutProducer)) {
                        ok = false;
                        break;
                    }
                    const AtQTile &Q = it.q[x];
                    const CUtensorMap *qm = maps + Q.q_map;
                    const uint32_t qs = smem_u32(smem + C::Q_OFF + x * C::TILE);
                    mbar_expect_tx(&ctl->q_full[x], C::TILE);
#pragma unroll
                    for (int c = 0; c < C::CH; c++)
                        tma_load_4d(qs + c * (kRows * 128), qm, &ctl->q_full[x], 64 * c, Q.q_c[0], Q.q_c[1], Q.q_c[2]);
                    q_armed |= 1u << x;
                    q_par = (q_par & ~(1u << x)) | ((qn & 1) << x);
                    if (x == 0) qx0++;
                    else qx1++;
                }
                for (int r = it.r0; r < it.r1 && ok; r++) {
                    const AtRun R = p.runs[r];
                    const CUtensorMap *km = maps + R.k_map, *vm = maps + R.k_map + p.n_kv;
                    for (int k = 0; k < R.ntiles; k++) {
                        const int st = ct % kKvStages;
                        const uint32_t ph = (ct / kKvStages) & 1;
                        if (!mbar_wait(&ctl->kv_empty[st], ph ^ 1, abort, p.err, kDevTimeoutProducer)) {
                            ok = false;
                            break;
                        }
                        const int step = kKeys * k;
                        const int c1 = R.k_c[0] + (R.pos_slot == 0 ? step : 0);
                        const int c2 = R.k_c[1] + (R.pos_slot == 1 ? step : 0);
                        const int c3 = R.k_c[2] + (R.pos_slot == 2 ? step : 0);
                        const uint32_t ks = smem_u32(smem + C::K_OFF + st * C::TILE);
                        const uint32_t vs = smem_u32(smem + C::V_OFF + st * C::TILE);
                        mbar_expect_tx(&ctl->kv_full[st], 2 * C::TILE);
#pragma unroll
                        for (int c = 0; c < C::CH; c++)
                            tma_load_4d(ks + c * (kKeys * 128), km, &ctl->kv_full[st], 64 * c, c1, c2, c3);
#pragma unroll
                        for (int c = 0; c < C::CH; c++)
                            tma_load_4d(vs + c * (kKeys * 128), vm, &ctl->kv_full[st], 64 * c, c1, c2, c3);
                        kv_armed |= 1u << st;
                        kv_par = (kv_par & ~(1u << st)) | (ph << st);
                        ct++;
                    }
                }
            }
            if (*abort) {
                // Let our own copies land before the CTA can exit.
                for (int s = 0; s < 2; s++)
                    if (q_armed & (1u << s)) mbar_wait(&ctl->q_full[s], (q_par >> s) & 1, abort, p.err, 0, kDrainNs, false);
                for (int s = 0; s < kKvStages; s++)
                    if (kv_armed & (1u << s)) mbar_wait(&ctl->kv_full[s], (kv_par >> s) & 1, abort, p.err, 0, kDrainNs, false);
            }
        }
    } else if (warp == 9) {
        {
            // ------------------------------------------------ MMA issuer (the whole warp; one elected lane issues)
            const uint32_t idesc_s = make_idesc(kRows, kKeys, 0, 0);  // Q (K-major) x K (K-major)
            const uint32_t idesc_o = make_idesc(kRows, D, 0, 1);      // P (TMEM) x V (MN-major)
            // key tiles; items and tiles per query slot (scalars: no local-memory arrays)
            uint32_t ct = 0, qx0 = 0, qx1 = 0, tx0 = 0, tx1 = 0;
            bool ok = true;
            // S_x = Q_x K_t^T
            auto mma_s = [&](int x, uint32_t t) {
                // the operands' descriptors once; each MMA adds a constant offset
                const uint64_t qd = sdesc(smem_u32(smem + C::Q_OFF + x * C::TILE), 16, 1024);
                const uint64_t kd = sdesc(smem_u32(smem + C::K_OFF + (t % kKvStages) * C::TILE), 16, 1024);
                const uint32_t d = tmem + (uint32_t)(x * kKeys);
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < D / 16; kk++)
                        umma_bf16(d, qd + (uint64_t)sdesc_off((kk >> 2) * (kRows * 128) + (kk & 3) * 32),
                                  kd + (uint64_t)sdesc_off((kk >> 2) * (kKeys * 128) + (kk & 3) * 32), idesc_s,
                                  kk > 0 ? 1u : 0u);
                    umma_commit(&ctl->s_full[x]);
                }
                __syncwarp();
            };
            // O_x (+)= P_x V_t, P_x in the first 64 columns of S_x
            auto mma_o = [&](int x, uint32_t t, bool first) {
                const uint64_t vd = sdesc(smem_u32(smem + C::V_OFF + (t % kKvStages) * C::TILE), kKeys * 128, 1024);
                const uint32_t pa = tmem + (uint32_t)(x * kKeys);
                const uint32_t d = tmem + kOCol + (uint32_t)(x * D);
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < kKeys / 16; kk++)
                        umma_bf16_ts(d, pa + kk * 8, vd + (uint64_t)sdesc_off(kk * 2048), idesc_o,
                                     (!first || kk > 0) ? 1u : 0u);
                }
                __syncwarp();
            };
            auto commit1 = [&](uint64_t *b) {
                if (elect_one()) umma_commit(b);
                __syncwarp();
            };
            for (int ii = i0; ii < i1 && ok; ii++) {
                const AtItem &it = p.items[ii];
                const int n = it.ntiles, nq = it.nq;
                if (n == 0) continue;
                const int nt0 = it.nt[0], nt1 = nq > 1 ? it.nt[1] : 0;  // scalars: no local-memory array
                // first scores of the item
                if (!warp_wait(&ctl->kv_full[ct % kKvStages], (ct / kKvStages) & 1, abort, p.err, kDevTimeoutMma)) {
                    ok = false;
                    break;
                }
                for (int x = 0; x < nq && ok; x++) {
                    if (!warp_wait(&ctl->q_full[x], (x == 0 ? qx0 : qx1) & 1, abort, p.err, kDevTimeoutMma)) {
                        ok = false;
                        break;
                    }
                    if (x == 0) qx0++;
                    else qx1++;
                    tc_fence_after();
                    mma_s(x, ct);
                    if ((x == 0 ? nt0 : nt1) == 1) commit1(&ctl->q_empty[x]);
                }
                if (!ok) break;
                for (int j = 0; j < n && ok; j++) {
                    const uint32_t t = ct + j;
                    bool kv_next = false;  // K and V of tile t + 1 have landed
                    for (int x = 0; x < nq; x++) {
                        const int ntx = x == 0 ? nt0 : nt1;
                        if (j >= ntx) continue;  // the rest of the item is masked for x
                        // V of tile t arrived with its K (waited for before S of tile t)
                        if (!warp_wait(&ctl->p_full[x], ((x == 0 ? tx0 : tx1) + j) & 1, abort, p.err, kDevTimeoutMma)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        mma_o(x, t, j == 0);
                        if (j == ntx - 1) commit1(&ctl->o_fin[x]);
                        if (j + 1 < ntx) {
                            if (!kv_next) {
                                if (!warp_wait(&ctl->kv_full[(t + 1) % kKvStages], ((t + 1) / kKvStages) & 1, abort,
                                               p.err, kDevTimeoutMma)) {
                                    ok = false;
                                    break;
                                }
                                kv_next = true;
                            }
                            mma_s(x, t + 1);
                            if (j + 1 == ntx - 1) commit1(&ctl->q_empty[x]);
                        }
                    }
                    if (!ok) break;
                    commit1(&ctl->kv_empty[t % kKvStages]);  // K and V of tile t are done
                }
                ct += n;
                tx0 += nt0;
                tx1 += nt1;
            }
            // Every MMA this thread issued has completed once mma_done flips.
            commit1(&ctl->mma_done);
            if (lane == 0) mbar_wait(&ctl->mma_done, 0, abort, p.err, kDevTimeoutMma, kTimeoutNs, false);
            __syncwarp();
        }
    } else if (warp < 8) {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kSoftmaxRegs));
        // ------------------------------------------------ softmax and output (warps 0-7)
        const int x = warp >> 2;
        const int row = threadIdx.x & (kRows - 1);
        const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        const uint32_t srow = lane_base + (uint32_t)(x * kKeys);
        const uint32_t orow = lane_base + kOCol + (uint32_t)(x * D);
        const float c = p.scale_log2;
        uint32_t ci = 0, ct = 0;  // items and key tiles of this query slot
        bool ok = true;
        for (int ii = i0; ii < i1 && ok; ii++) {
            const AtItem &it = p.items[ii];
            if (x >= it.nq) continue;
            const int n = it.nt[x];  // key tiles of this query slot: a prefix of the item's
            const AtQTile &Q = it.q[x];
            const int nrows = Q.nrows;
            const int64_t s_g = Q.s_glob0 + row;
            // keys this row may see: [lo_t, hi_t] (global positions)
            int64_t lo_t = 0, hi_t = INT64_MAX;
            if (p.nseq > 0) {
                int a = 0, b = p.nseq - 1;
                while (a < b) {
                    const int mid = (a + b) >> 1;
                    if (p.seq_ends[mid] > s_g) b = mid;
                    else a = mid + 1;
                }
                lo_t = a > 0 ? p.seq_ends[a - 1] : 0;
                hi_t = p.seq_ends[a] - 1;
            }
            if (p.causal) hi_t = s_g < hi_t ? s_g : hi_t;
            float m_ref = -INFINITY, m_max = -INFINITY, l = 0.f;  // raw score units
            int j = 0;
            for (int r = it.r0; r < it.r1 && ok && j < n; r++) {
                const AtRun R = p.runs[r];
                for (int k = 0; k < R.ntiles && j < n; k++, j++) {
                    const uint32_t t = ct + j;
                    if (!warp_wait(&ctl->s_full[x], t & 1, abort, p.err, kDevTimeoutSoftmax)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // the scores, with the maximum of each 32 of them from the load
                    uint32_t u[kKeys];
                    float hm0, hm1, hm2, hm3;
                    tmem_ld32_max(srow, u, hm0);
                    tmem_ld32_max(srow + 32, u + 32, hm1);
                    tmem_ld32_max(srow + 64, u + 64, hm2);
                    tmem_ld32_max(srow + 96, u + 96, hm3);
                    tmem_wait_ld();

                    const int64_t t0 = R.t_glob0 + (int64_t)kKeys * k;
                    const int nv = min(kKeys, R.nkeys - kKeys * k);
                    const int jlo = (int)max64(0, min64(kKeys, lo_t - t0));
                    const int jhi = (int)max64(-1, min64(nv - 1, hi_t - t0));
                    float mx = fmaxf(max3(hm0, hm1, hm2), hm3);
                    if (jlo > 0 || jhi < kKeys - 1) {
                        // a masked tile: drop the removed keys and take the maximum again
#pragma unroll
                        for (int q = 0; q < kKeys; q++)
                            if (q < jlo || q > jhi) u[q] = __float_as_uint(-INFINITY);
                        float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
                        for (int q = 0; q < kKeys; q += 8) {
                            mx0 = max3(mx0, __uint_as_float(u[q]), __uint_as_float(u[q + 1]));
                            mx1 = max3(mx1, __uint_as_float(u[q + 2]), __uint_as_float(u[q + 3]));
                            mx2 = max3(mx2, __uint_as_float(u[q + 4]), __uint_as_float(u[q + 5]));
                            mx3 = max3(mx3, __uint_as_float(u[q + 6]), __uint_as_float(u[q + 7]));
                        }
                        mx = fmaxf(max3(mx0, mx1, mx2), mx3);
                    }
                    m_max = fmaxf(m_max, mx);
                    // move the reference maximum only when exponentials would pass 2^kLazy
                    float alpha = 1.f;
                    if (mx != -INFINITY && (m_ref == -INFINITY || (mx - m_ref) * c > kLazy)) {
                        alpha = m_ref == -INFINITY ? 0.f : ex2((m_ref - mx) * c);
                        m_ref = mx;
                    }
                    const float base = m_ref == -INFINITY ? 0.f : m_ref * c;
                    // two scores per packed f32x2 FMA and add; four running pair-sums
                    const uint64_t c2 = pack_f32x2(c, c), nb2 = pack_f32x2(-base, -base);
                    uint64_t ls[4] = {0, 0, 0, 0};
#pragma unroll
                    for (int q = 0; q < kKeys / 2; q++) {
                        const uint64_t y = fma_f32x2(pack_u32x2(u[2 * q], u[2 * q + 1]), c2, nb2);
                        const float e0 = ex2(lo_f32(y)), e1 = ex2(hi_f32(y));
                        ls[q & 3] = add_f32x2(ls[q & 3], pack_f32x2(e0, e1));
                        u[q] = pack_bf16(e0, e1);
                    }
                    const uint64_t s01 = add_f32x2(add_f32x2(ls[0], ls[1]), add_f32x2(ls[2], ls[3]));
                    l = fmaf(l, alpha, lo_f32(s01) + hi_f32(s01));
                    // P over the scores just read (the A operand of O += P V)
                    tmem_st32(srow, u);
                    tmem_st32(srow + 32, u + 32);
                    // The previous O += P V of this query tile has completed: the
                    // scores of this tile were computed after it, in order.
                    if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
                        for (int cc = 0; cc < D / 32; cc++) {
                            uint32_t o[32];
                            tmem_ld32(orow + 32 * cc, o);
                            tmem_wait_ld();
#pragma unroll
                            for (int i = 0; i < 32; i++) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                            tmem_st32(orow + 32 * cc, o);
                        }
                    }
                    tmem_wait_st();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&ctl->p_full[x]);
                }
            }
            if (!ok) break;
            // The item's aggregate is complete once its last O += P V is done.
            if (n > 0) {
                if (!warp_wait(&ctl->o_fin[x], ci & 1, abort, p.err, kDevTimeoutSoftmax)) {
                    ok = false;
                    break;
                }
                ct += n;
                ci++;
            }
            tc_fence_after();
            bool in = true;
            if constexpr (kBoundsCheck) {
                // the query tile's output rows (and statistics rows) inside their arenas
                const int64_t nr = nrows;
                in = range_in(Q.o_off, 1, &nr, &Q.o_rstr, D, 1, p.o_elems) &&
                     (!p.m_out || range_in(Q.ml_off, 1, &nr, &Q.ml_rstr, 1, 0, p.ml_elems));
                if (!in && row == 0) bounds_fail(p.err);
            }
            const float inv = l > 0.f ? 1.f / l : 0.f;
            uint4 *dst = reinterpret_cast<uint4 *>(p.o + (Q.o_off + (int64_t)(row < nrows ? row : 0) * Q.o_rstr) * 2);
#pragma unroll
            for (int cc = 0; cc < D / 32; cc++) {
                uint32_t o[32];
                if (n > 0) {
                    tmem_ld32(orow + 32 * cc, o);
                    tmem_wait_ld();
                } else {
#pragma unroll
                    for (int i = 0; i < 32; i++) o[i] = 0u;
                }
                if (row < nrows && in) {
#pragma unroll
                    for (int q = 0; q < 4; q++) {
                        const float *f = reinterpret_cast<const float *>(o + 8 * q);
                        uint4 w;
                        w.x = pack_bf16(f[0] * inv, f[1] * inv);
                        w.y = pack_bf16(f[2] * inv, f[3] * inv);
                        w.z = pack_bf16(f[4] * inv, f[5] * inv);
                        w.w = pack_bf16(f[6] * inv, f[7] * inv);
                        dst[4 * cc + q] = w;
                    }
                }
            }
            tc_fence_before();
            if (p.m_out && row < nrows && in) {
                const int64_t o = Q.ml_off + (int64_t)row * Q.ml_rstr;
                p.m_out[o] = m_max * p.scale;
                p.l_out[o] = m_max == -INFINITY ? 0.f : l * ex2((m_ref - m_max) * c);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <int D>
cudaError_t launch_d(const AtParams &p, cudaStream_t st) {
    using C = AtCfg<D>;
    static bool configured[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64 && !configured[dev]) {
        // The register split assumes the block starts with kLaunchRegs a
        // thread: with fewer, setmaxnreg.inc would wait for registers that
        // never come, so such a build is refused before it can launch.
        cudaFuncAttributes fa;
        e = cudaFuncGetAttributes(&fa, attention_kernel<D>);
        if (e != cudaSuccess) return e;
        if (fa.numRegs != kLaunchRegs) return cudaErrorInvalidConfiguration;
        e = cudaFuncSetAttribute(attention_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    attention_kernel<D><<<p.ncta, kAtThreads, C::SMEM, st>>>(p);
    return cudaGetLastError();
}

}  // namespace

int attention_smem_bytes(int d) { return d == 64 ? AtCfg<64>::SMEM : AtCfg<128>::SMEM; }

cudaError_t launch_attention(const AtParams &p, cudaStream_t st) {
    if (p.ncta <= 0) return cudaSuccess;
    if (p.pair) return launch_attention_pair(p, st);
    if (p.d == 64) return launch_d<64>(p, st);
    return launch_d<128>(p, st);
}

}  // namespace ea
