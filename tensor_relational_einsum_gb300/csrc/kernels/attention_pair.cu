// attention_pair.cu -- the attention join-agg ("Every Kernel Is a Join",
// Example 3.10) on CTA pairs: tcgen05 cta_group::2, head dimension 128.
//
// The join-agg is the one of attention.cu: an aggregation group is one tile
// of 128 query positions of one query head, its tuples are the key tiles
// (128 keys) the predicate keeps, and the tuples are aggregated with the
// merge of (m, l, A) triples
//     (m1, l1, A1) + (m2, l2, A2) = (M, l1 a1 + l2 a2, A1 a1 + A2 a2),
//     M = max(m1, m2), a_i = exp(m_i - M),
// which is associative and commutative; the output block is A / l.
//
// Two CTAs of a cluster run two groups of the same head side by side (two
// query tiles that share their key tiles): CTA r holds query tile r.  One
// thread of CTA 0 issues every MMA for both, 256 rows at a time
// (cta_group::2): the scores S = Q K^T of the pair's 256 query rows against
// a key tile, each CTA loading only its half of the tile's keys (64 keys x
// 128 head dims), and the accumulations A (+)= P V, each CTA loading only
// its half of the head dims of V (128 keys x 64 head dims).  So every SM
// loads half of each K and V tile, and every MMA instruction does the work
// of two SMs.
//
// Each key tile is cut into two halves of 64 keys, and each group's tuples
// are aggregated in two chains, chain h over the h-th halves of its key
// tiles, each with its own (m, l, A); the two results are merged once, with
// the same (+), when the group is complete (the merge is associative and
// commutative, so this is the same aggregate).  The reference maximum of a
// chain's row moves only when a half tile's maximum exceeds it by more than
// 2^kLazy in exp (its A row is then rescaled in TMEM); kLazy = 64, as in
// the single-CTA kernel, for which attention.cu gives the range argument.
// On a tile the predicate cuts (the causal diagonal, a sequence boundary,
// the ragged last tile of a run) each 32-key chunk of a warp's scores is,
// for the warp's 32 rows, all dropped (its P is zero, no exponentials),
// all kept, or mixed (masked key by key): the diagonal costs little more
// than a full tile.
//
// TMEM of each CTA (512 columns): two score buffers S_0 [0, 128) and
// S_1 [128, 256) (key tile g's scores go to S_(g mod 2), so the scores of
// tile g + 1 are computed while the softmax of tile g runs) and the two
// chains' accumulators A_0 [256, 384), A_1 [384, 512).  The probabilities
// of half h are written as bf16 over the first 32 columns of that half's
// scores and read from there by the MMA.
//
// Roles (384 threads per CTA, both CTAs persistent over the pair's list of
// query-tile pairs; key tiles numbered g = 0, 1, ... over the list):
//   warp 8     TMA: this CTA's query tile (two buffers), its half of K of
//              tile g (stage g mod 3); warp 10: its half of V (stage
//              g mod 3).  The byte counts of both CTAs' loads complete on
//              CTA 0's barriers.
//   warp 9     TMEM (both CTAs); in CTA 0, the MMA warp: the whole warp
//              runs the issue loop (warp-uniform waits, cursors and
//              descriptors; one elected lane issues), in the order S(0),
//              S(1), A(0), S(2), A(1), S(3), ...; each A(g), S(g + 2) pair
//              goes out back to back once P of tile g is written, all its
//              other waits taken before.  Its commits signal both CTAs'
//              barriers (CTA 1's through shared::cluster addresses).
//   warps 0-7  softmax of chain h = warp / 4 for this CTA's query rows (one
//              row per thread); CTA 1's warps report to CTA 0's barriers by
//              remote arrives.  At the end of a group the two chains'
//              (m, l) are exchanged through shared memory, each thread
//              stages its 64 values of O = (A_0 a_0 + A_1 a_1) /
//              (l_0 a_0 + l_1 a_1) in its warp's slice of a staging tile,
//              and each warp stores its slice (32 rows x 64 head dims) with
//              one asynchronous TMA tensor store.  The query-tile and run
//              descriptors they read sit in shared memory (copied at the
//              start), so no group start or end waits on a global load.
// Every mbarrier wait is bounded (2 s); on time-out the kernel raises the
// device error word and every role leaves its loop; no CTA frees TMEM or
// leaves before the other has finished with it.
#include <algorithm>

#include "attn_common.cuh"
#include "dev_common.cuh"
#include "tc_common.cuh"

namespace ea {

namespace {

using namespace tc;
using namespace attn;

constexpr int kRows = 128;   // query rows of a tile (= TMEM lanes)
constexpr int kKeys = 128;   // keys of a key tile
constexpr int kHalf = 64;    // keys of a half tile (one chain); also this CTA's keys of K, head dims of V
constexpr int kD = 128;      // head dimension
constexpr int kThreads = 384;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kOCol = 256;
constexpr float kLazy = 64.0f;
constexpr int kItemCache = 256;  // key-tile counts of the pair's first query-tile pairs, in shared memory

constexpr int kQBytes = kRows * kD * 2;    // this CTA's query tile (32 KB)
constexpr int kKBytes = kHalf * kD * 2;    // its half of a K tile (16 KB)
constexpr int kVBytes = kKeys * kHalf * 2; // its half of a V tile (16 KB)
constexpr int Q_OFF = 0;                   // two Q buffers
constexpr int kStages = 3;                 // K and V ring depth
constexpr int kEBytes = kRows * kD * 2;    // output staging (32 KB)
constexpr int K_OFF = 2 * kQBytes;         // K stages
constexpr int V_OFF = K_OFF + kStages * kKBytes; // V stages
constexpr int E_OFF = V_OFF + kStages * kVBytes; // output staging: warp w owns [4 KB w, 4 KB (w + 1))
constexpr int CTL_OFF = E_OFF + kEBytes;

// Key tile g uses score buffer S_(g mod 2), K stage g mod 3 and V stage
// g mod 3; its score commit frees the K stage, its accumulation commit the
// V stage (a load waits for the products of the tile three back: the loads
// of the next tiles are in flight while the tensor cores and the softmax
// work on this one).  Barriers that a thread signals once
// per tile are split by tile parity (or by stage), so that every wait is
// within one phase of its barrier.  The barriers CTA 0's MMA thread waits
// on live in CTA 0.
// What the softmax warps read of a query tile and of a run, cached in
// shared memory for the first kDescItems items of the pair and the first
// kDescRuns runs of their (contiguous) run range: a descriptor load from
// global memory at a group's start or end would stall all softmax warps.
constexpr int kDescItems = 64;
constexpr int kDescRuns = 256;
struct DescQ {
    int64_t s_glob0, o_off, o_rstr, ml_off, ml_rstr;
    int32_t nrows, r0, r1, q_map;
    int32_t q_c[3], pos_slot;  // the tile's map coordinates; which of them is the position
};
struct DescRun {
    int64_t t_glob0;
    int32_t ntiles, nkeys;
};

struct PairCtl {
    uint64_t q_full[2], q_empty[2];
    uint64_t k_full[kStages], v_full[kStages];    // CTA 0: both CTAs' halves landed
    uint64_t k_empty[kStages], v_empty[kStages];  // the stage's products are done (each CTA)
    uint64_t s_full[2];   // scores of tile g computed (each CTA)
    uint64_t p_full[2];   // CTA 0: both chains' probabilities of tile g written in both CTAs (16 warps)
    uint64_t o_done[2];   // accumulation of tile g done (each CTA)
    uint64_t ml_ready[2]; // both chains' (m, l) of a group written (this CTA, two slots)
    uint64_t e_done;      // CTA 0: all 16 softmax warps have read their accumulators
    uint64_t mma_done;
    uint32_t tmem_base;
    int abort;
    float4 ml[2][2][kRows];  // end of a group: [slot][chain][row] (m_ref, l, m_max)
    int32_t item_n[kItemCache];
    DescQ dq[kDescItems];    // this CTA's query tile of items i0, i0 + 1, ...
    DescQ dqx[8];            // softmax warp w: its copy of an item past the cache
    DescRun dr[kDescRuns];   // runs r_base, r_base + 1, ...
};

constexpr int kSmem = 1024 + CTL_OFF + (int)sizeof(PairCtl);

__device__ __forceinline__ void tma_load_4d_pair(uint32_t dst, const void *map, uint32_t bar_cl, int c0, int c1,
                                                 int c2, int c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, "
        "{%3, %4, %5, %6}], [%2];" ::"r"(dst),
        "l"(map), "r"(bar_cl), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
        : "memory");
}

// This warp's staged output rows (a 32-row x 64-column box, 128-byte
// swizzle) to global memory through the tensor map of the O block.
__device__ __forceinline__ void tma_store_4d(const void *map, uint32_t src, int c0, int c1, int c2, int c3) {
    asm volatile("cp.async.bulk.tensor.4d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4, %5}], [%1];" ::"l"(map),
                 "r"(src), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
                 : "memory");
}
__device__ __forceinline__ void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }

__device__ __forceinline__ void st_shared_v4(uint32_t a, uint32_t x, uint32_t y, uint32_t z, uint32_t w) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(x), "r"(y), "r"(z), "r"(w) : "memory");
}

// 16-byte unit q of row `row` of a staging tile with 128-byte rows: units
// are permuted by row mod 8 -- the 128-byte swizzle the output's tensor map
// reads, with 1024-byte-aligned 8-row atoms -- so a warp writing one row
// per lane touches every bank once per 128 bytes.
__device__ __forceinline__ uint32_t sw128_unit(uint32_t tile, int row, int q) {
    return tile + (uint32_t)(row * 128) + (uint32_t)((q ^ (row & 7)) << 4);
}

// Arrive on CTA 0's copy of barrier `b` (a local arrive in CTA 0).
__device__ __forceinline__ void arrive_on_rank0(uint64_t *b, int rank) {
    if (rank == 0) mbar_arrive(b);
    else mbar_arrive_cluster(mapa_u32(smem_u32(b), 0));
}

// Commit the pair MMAs issued so far to barrier `b` of both CTAs.
__device__ __forceinline__ void commit_both(uint64_t *b) {
    umma_commit_pair(smem_u32(b));
    umma_commit_pair(mapa_u32(smem_u32(b), 1));
}

__global__ void __launch_bounds__(kThreads, 1) attention_pair_kernel(const AtParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    PairCtl *ctl = reinterpret_cast<PairCtl *>(smem + CTL_OFF);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int rank = (int)cluster_rank();
    const CUtensorMap *maps = reinterpret_cast<const CUtensorMap *>(p.tmaps);
    volatile int *abort = &ctl->abort;
    const int pr = blockIdx.x >> 1;  // the pair
    const int i0 = p.cta_ptr[pr], i1 = p.cta_ptr[pr + 1];

    if (threadIdx.x == 0) {
        for (int b = 0; b < kStages; b++) {
            mbar_init(&ctl->k_full[b], 1);
            mbar_init(&ctl->v_full[b], 1);
            mbar_init(&ctl->k_empty[b], 1);
            mbar_init(&ctl->v_empty[b], 1);
        }
        for (int b = 0; b < 2; b++) {
            mbar_init(&ctl->q_full[b], 1);
            mbar_init(&ctl->q_empty[b], 1);
            mbar_init(&ctl->s_full[b], 1);
            mbar_init(&ctl->p_full[b], 16);
            mbar_init(&ctl->o_done[b], 1);
            mbar_init(&ctl->ml_ready[b], 8);
        }
        mbar_init(&ctl->e_done, 16);
        mbar_init(&ctl->mma_done, 1);
        ctl->abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        fence_proxy_async();
    }
    for (int ii = i0 + (int)threadIdx.x; ii < i1 && ii - i0 < kItemCache; ii += kThreads)
        ctl->item_n[ii - i0] = p.items[ii].ntiles;
    if (warp == 9) tmem_alloc_pair(smem_u32(&ctl->tmem_base), kTmemCols);
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // both CTAs' barriers are initialised before either signals the other
    tc_fence_after();
    const uint32_t tmem = ctl->tmem_base;
    auto item_n = [&](int ii) -> int { return ii - i0 < kItemCache ? ctl->item_n[ii - i0] : p.items[ii].ntiles; };

    if ((warp == 8 || warp == 10) && lane == 0) {
        // ------------------------------------------------ TMA producers
        // warp 8: this CTA's query tile and its 64 keys of each K tile;
        // warp 10: its 64 head dims of each V tile.  K stage g mod 4 is free
        // once the scores of tile g - 4 are done, V stage g mod 4 once the
        // accumulation of tile g - 4 is; CTA 0 expects both CTAs' bytes.
        const bool is_k = warp == 8;
        uint64_t *full = is_k ? ctl->k_full : ctl->v_full;
        uint64_t *freed = is_k ? ctl->k_empty : ctl->v_empty;
        const int off = is_k ? K_OFF : V_OFF;
        const int bytes = is_k ? kKBytes : kVBytes;
        uint32_t g = 0, qi = 0;
        uint32_t armed = 0, par = 0, q_armed = 0, q_par = 0;
        bool ok = true;
        for (int ii = i0; ii < i1 && ok; ii++) {
            const int n = item_n(ii);
            if (n == 0) continue;
            const AtItem &it = p.items[ii];
            if (is_k) {
                const int qb = qi & 1;
                if (!mbar_wait(&ctl->q_empty[qb], ((qi >> 1) & 1) ^ 1, abort, p.err, kDevTimeoutProducer)) break;
                const AtQTile &Q = it.q[rank];
                const CUtensorMap *qm = maps + Q.q_map;
                const uint32_t qs = smem_u32(smem + Q_OFF + qb * kQBytes);
                if (rank == 0) mbar_expect_tx(&ctl->q_full[qb], 2 * kQBytes);
                const uint32_t qf = mapa_u32(smem_u32(&ctl->q_full[qb]), 0);
#pragma unroll
                for (int c = 0; c < kD / 64; c++)
                    tma_load_4d_pair(qs + c * (kRows * 128), qm, qf, 64 * c, Q.q_c[0], Q.q_c[1], Q.q_c[2]);
                q_armed |= 1u << qb;
                q_par = (q_par & ~(1u << qb)) | (((qi >> 1) & 1) << qb);
            }
            qi++;
            int j = 0;
            for (int r = it.r0; r < it.r1 && ok && j < n; r++) {
                const AtRun R = p.runs[r];
                // K: this CTA's 64 keys (maps with 64-key boxes); V: its 64 head dims
                const CUtensorMap *m = maps + (is_k ? R.k_map : R.k_map + p.n_kv);
                for (int k = 0; k < R.ntiles && j < n; k++, j++, g++) {
                    const int st = g % kStages;
                    const int step = kKeys * k + (is_k ? kHalf * rank : 0);
                    const int c1 = R.k_c[0] + (R.pos_slot == 0 ? step : 0);
                    const int c2 = R.k_c[1] + (R.pos_slot == 1 ? step : 0);
                    const int c3 = R.k_c[2] + (R.pos_slot == 2 ? step : 0);
                    if (g >= kStages &&
                        !mbar_wait(&freed[st], (g / kStages - 1) & 1, abort, p.err, kDevTimeoutProducer)) {
                        ok = false;
                        break;
                    }
                    const uint32_t ds = smem_u32(smem + off + st * bytes);
                    if (rank == 0) mbar_expect_tx(&full[st], 2 * bytes);
                    const uint32_t fc = mapa_u32(smem_u32(&full[st]), 0);
                    if (is_k) {
#pragma unroll
                        for (int c = 0; c < kD / 64; c++)
                            tma_load_4d_pair(ds + c * (kHalf * 128), m, fc, 64 * c, c1, c2, c3);
                    } else {
                        tma_load_4d_pair(ds, m, fc, kHalf * rank, c1, c2, c3);
                    }
                    armed |= 1u << st;
                    par = (par & ~(1u << st)) | (((g / kStages) & 1) << st);
                }
            }
        }
        if (*abort) {
            // Let our own copies land before the CTA can exit: CTA 0 waits for
            // its barriers; CTA 1's copies complete there, so it gives them time.
            if (rank == 0) {
                for (int s = 0; s < 2; s++)
                    if (q_armed & (1u << s)) mbar_wait(&ctl->q_full[s], (q_par >> s) & 1, abort, p.err, 0, kDrainNs, false);
                for (int s = 0; s < kStages; s++)
                    if (armed & (1u << s)) mbar_wait(&full[s], (par >> s) & 1, abort, p.err, 0, kDrainNs, false);
            } else if (armed | q_armed) {
                const uint64_t t0 = gtime();
                while (gtime() - t0 < kDrainNs) {
                }
            }
        }
    } else if (warp == 9 && rank == 0) {
        // ------------------------------------------------ MMA issuer (CTA 0's warp 9)
        // The whole warp runs the issue loop: its waits (lane 0's, shared
        // by shuffle), cursors and descriptors are warp-uniform, and one
        // elected lane issues each batch of MMAs and their commits.
        const uint32_t idesc_s = make_idesc(2 * kRows, kKeys, 0, 0);  // Q (K-major) x K (K-major), 256 rows
        const uint32_t idesc_o = make_idesc(2 * kRows, kD, 0, 1);     // P (TMEM) x V (MN-major), 256 rows
        bool ok = true;
        // Two cursors over the key tiles: `s` issues the scores two tiles
        // ahead, `a` the accumulations.  Each step first waits for all that
        // the accumulation of tile g and the scores of tile g + 2 need except
        // P of tile g (none of it waits on an MMA not yet issued), then,
        // once P is written, issues both back to back: the scores of g + 2
        // (into the buffer P of g leaves) are then on the tensor pipe right
        // behind the products that free it.
        auto next_nonempty = [&](int ii) {
            while (ii < i1 && item_n(ii) == 0) ii++;
            return ii;
        };
        int s_item = next_nonempty(i0), a_item = next_nonempty(i0), s_j = 0, a_j = 0;
        int s_n = s_item < i1 ? item_n(s_item) : 0, a_n = a_item < i1 ? item_n(a_item) : 0;
        uint32_t s_g = 0, a_g = 0, s_qi = 0, a_qi = 0;
        auto wait_s = [&]() -> bool {
            if (s_j == 0 && !warp_wait(&ctl->q_full[s_qi & 1], (s_qi >> 1) & 1, abort, p.err, kDevTimeoutMma))
                return false;
            return warp_wait(&ctl->k_full[s_g % kStages], (s_g / kStages) & 1, abort, p.err, kDevTimeoutMma);
        };
        auto issue_s = [&]() {
            const int qb = s_qi & 1;
            const int st = s_g & 1, ks = s_g % kStages;
            const uint64_t qd = sdesc(smem_u32(smem + Q_OFF + qb * kQBytes), 16, 1024);
            const uint64_t kd = sdesc(smem_u32(smem + K_OFF + ks * kKBytes), 16, 1024);
            const uint32_t d = tmem + (uint32_t)(st * kKeys);
            if (elect_one()) {
#pragma unroll
                for (int kk = 0; kk < kD / 16; kk++)
                    umma_bf16_pair(d, qd + (uint64_t)sdesc_off((kk >> 2) * (kRows * 128) + (kk & 3) * 32),
                                   kd + (uint64_t)sdesc_off((kk >> 2) * (kHalf * 128) + (kk & 3) * 32), idesc_s,
                                   kk > 0 ? 1u : 0u);
                commit_both(&ctl->s_full[st]);    // the scores of tile s_g, in both CTAs
                commit_both(&ctl->k_empty[ks]);   // K stage ks free, in both CTAs
                if (s_j == s_n - 1) commit_both(&ctl->q_empty[qb]);
            }
            __syncwarp();
            s_g++;
            if (++s_j == s_n) {
                s_j = 0;
                s_qi++;
                s_item = next_nonempty(s_item + 1);
                s_n = s_item < i1 ? item_n(s_item) : 0;
            }
        };
        auto wait_a = [&]() -> bool {  // all but P of tile a_g
            // a group's first accumulation overwrites A_0 and A_1 in both CTAs:
            // all 16 softmax warps must have read the previous group's output
            if (a_j == 0 && a_qi > 0 && !warp_wait(&ctl->e_done, (a_qi - 1) & 1, abort, p.err, kDevTimeoutMma))
                return false;
            return warp_wait(&ctl->v_full[a_g % kStages], (a_g / kStages) & 1, abort, p.err, kDevTimeoutMma);
        };
        auto issue_a = [&]() {
            const int st = a_g & 1, vs = a_g % kStages;
            const uint32_t pb = tmem + (uint32_t)(st * kKeys);
            const uint64_t vd = sdesc(smem_u32(smem + V_OFF + vs * kVBytes), kKeys * 128, 1024);
            if (elect_one()) {
#pragma unroll
                for (int h = 0; h < 2; h++) {
                    const uint32_t d = tmem + kOCol + (uint32_t)(h * kD);
#pragma unroll
                    for (int kk = 0; kk < kHalf / 16; kk++)
                        umma_bf16_ts_pair(d, pb + (uint32_t)(h * kHalf) + kk * 8,
                                          vd + (uint64_t)sdesc_off((h * (kHalf / 16) + kk) * 2048), idesc_o,
                                          (a_j > 0 || kk > 0) ? 1u : 0u);
                }
                commit_both(&ctl->o_done[st]);    // the accumulation of tile a_g, in both CTAs
                commit_both(&ctl->v_empty[vs]);   // V stage vs free, in both CTAs
            }
            __syncwarp();
            a_g++;
            if (++a_j == a_n) {
                a_j = 0;
                a_qi++;
                a_item = next_nonempty(a_item + 1);
                a_n = a_item < i1 ? item_n(a_item) : 0;
            }
        };
        for (int w = 0; w < 2 && ok && s_item < i1; w++) {
            ok = wait_s();
            if (ok) {
                tc_fence_after();
                issue_s();
            }
        }
        while (ok && a_item < i1) {
            const bool more_s = s_item < i1;
            ok = wait_a() && (!more_s || wait_s()) &&
                 warp_wait(&ctl->p_full[a_g & 1], (a_g >> 1) & 1, abort, p.err, kDevTimeoutMma);
            if (!ok) break;
            tc_fence_after();
            issue_a();
            if (more_s) issue_s();
        }
        // Every MMA this warp issued has completed once mma_done flips.
        if (elect_one()) umma_commit_pair(smem_u32(&ctl->mma_done));
        __syncwarp();
        if (lane == 0) mbar_wait(&ctl->mma_done, 0, abort, p.err, kDevTimeoutMma, kTimeoutNs, false);
        __syncwarp();
    } else if (warp < 8) {
        // ------------------------------------------------ softmax chains and output (warps 0-7)
        const int h = warp >> 2;  // chain: keys [64 h, 64 h + 64) of every tile
        const int row = threadIdx.x & (kRows - 1);
        const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        const uint32_t arow = lane_base + kOCol + (uint32_t)(h * kD);
        const float c = p.scale_log2;
        // the descriptor caches (the 256 softmax threads fill them; every one
        // of them reaches the named barrier)
        const int n_dq = min(i1 - i0, kDescItems);
        const int r_base = i1 > i0 ? p.items[i0].r0 : 0;
        const int n_dr = i1 > i0 ? min(p.items[i0 + n_dq - 1].r1 - r_base, kDescRuns) : 0;
        for (int t = (int)threadIdx.x; t < n_dq; t += 256) {
            const AtItem &it = p.items[i0 + t];
            const AtQTile &Q = it.q[rank];
            DescQ d;
            d.s_glob0 = Q.s_glob0;
            d.o_off = Q.o_off;
            d.o_rstr = Q.o_rstr;
            d.ml_off = Q.ml_off;
            d.ml_rstr = Q.ml_rstr;
            d.nrows = Q.nrows;
            d.r0 = it.r0;
            d.r1 = it.r1;
            d.q_map = Q.q_map;
            for (int i = 0; i < 3; i++) d.q_c[i] = Q.q_c[i];
            d.pos_slot = Q.pos_slot;
            ctl->dq[t] = d;
        }
        for (int t = (int)threadIdx.x; t < n_dr; t += 256) {
            const AtRun R = p.runs[r_base + t];
            ctl->dr[t] = DescRun{R.t_glob0, R.ntiles, R.nkeys};
        }
        named_bar(1, 256);
        uint32_t g = 0, qi = 0;  // key tiles and non-empty groups so far
        bool ok = true;
        for (int ii = i0; ii < i1 && ok; ii++) {
            const int n = item_n(ii);
            const DescQ *Qp = &ctl->dq[ii - i0];
            if (ii - i0 >= n_dq) {
                const AtItem &it = p.items[ii];
                const AtQTile &G = it.q[rank];
                if (lane == 0)
                    ctl->dqx[warp] = DescQ{G.s_glob0, G.o_off, G.o_rstr, G.ml_off, G.ml_rstr, G.nrows, it.r0, it.r1,
                                           G.q_map, {G.q_c[0], G.q_c[1], G.q_c[2]}, G.pos_slot};
                __syncwarp();
                Qp = &ctl->dqx[warp];
            }
            const DescQ &Q = *Qp;
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
            if (row >= nrows) hi_t = -1;  // rows past the tile (or a padding tile) keep no key
            float m_ref = -INFINITY, m_max = -INFINITY, l = 0.f;  // raw score units
            int j = 0;
            for (int r = Q.r0; r < Q.r1 && ok && j < n; r++) {
                DescRun R;
                if ((unsigned)(r - r_base) < (unsigned)n_dr) {
                    R = ctl->dr[r - r_base];
                } else {
                    const AtRun G = p.runs[r];
                    R = DescRun{G.t_glob0, G.ntiles, G.nkeys};
                }
                for (int k = 0; k < R.ntiles && j < n; k++, j++, g++) {
                    if (!warp_wait(&ctl->s_full[g & 1], (g >> 1) & 1, abort, p.err, kDevTimeoutSoftmax)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t srow = lane_base + (uint32_t)((g & 1) * kKeys + h * kHalf);
                    // this chain's 64 scores, with the maximum of each 32 from the load
                    uint32_t u[kHalf];
                    float hm0, hm1;
                    tmem_ld32_max(srow, u, hm0);
                    tmem_ld32_max(srow + 32, u + 32, hm1);
                    tmem_wait_ld();
                    const int64_t t0 = R.t_glob0 + (int64_t)kKeys * k + h * kHalf;
                    const int nv = min(kHalf, R.nkeys - kKeys * k - h * kHalf);
                    const int jlo = (int)max64(0, min64(kHalf, lo_t - t0));
                    const int jhi = (int)max64(-1, min64(nv - 1, hi_t - t0));
                    // Each 32-key chunk is, for the whole warp, all dropped (no exponentials: P is
                    // zero there), all kept (the maximum comes from the load) or mixed (masked key
                    // by key and its maximum taken again).  Rows are consecutive positions, so on
                    // a diagonal tile at most one chunk of a warp is mixed.
                    bool live0 = true, live1 = true;
                    const bool masked = __any_sync(0xffffffffu, jlo > 0 || jhi < kHalf - 1);
                    if (masked) {
                        live0 = __any_sync(0xffffffffu, jlo < 32 && jhi >= 0);
                        live1 = __any_sync(0xffffffffu, jlo < kHalf && jhi >= 32);
                        const bool mix0 = __any_sync(0xffffffffu, jlo > 0 || jhi < 31);
                        const bool mix1 = __any_sync(0xffffffffu, jlo > 32 || jhi < kHalf - 1);
                        if (!live0) hm0 = -INFINITY;
                        else if (mix0) hm0 = mask_chunk(u, 0, jlo, jhi);
                        if (!live1) hm1 = -INFINITY;
                        else if (mix1) hm1 = mask_chunk(u + 32, 32, jlo, jhi);
                    }
                    const float mx = fmaxf(hm0, hm1);
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
                    if (!masked) {
                        // one straight run of 32 pairs: the common case, scheduled as a whole
                        exp_chunk<0>(u, c2, nb2, ls);
                        exp_chunk<16>(u, c2, nb2, ls);
                    } else {
                        if (live0) exp_chunk<0>(u, c2, nb2, ls);
                        else zero_chunk<0>(u);
                        if (live1) exp_chunk<16>(u, c2, nb2, ls);
                        else zero_chunk<16>(u);
                    }
                    const uint64_t s01 = add_f32x2(add_f32x2(ls[0], ls[1]), add_f32x2(ls[2], ls[3]));
                    l = fmaf(l, alpha, lo_f32(s01) + hi_f32(s01));
                    // P over the first 32 columns of this chain's scores (the A operand of A_h += P V)
                    tmem_st32(srow, u);
                    if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
                        // rescale this chain's row of A once the previous accumulation is done
                        if (!warp_wait(&ctl->o_done[(g - 1) & 1], ((g - 1) >> 1) & 1, abort, p.err,
                                       kDevTimeoutSoftmax)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
#pragma unroll
                        for (int cc = 0; cc < kD / 32; cc++) {
                            uint32_t o[32];
                            tmem_ld32(arow + 32 * cc, o);
                            tmem_wait_ld();
#pragma unroll
                            for (int i = 0; i < 32; i++) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                            tmem_st32(arow + 32 * cc, o);
                        }
                    }
                    tmem_wait_st();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) arrive_on_rank0(&ctl->p_full[g & 1], rank);
                }
            }
            if (!ok) break;
            // this warpgroup's half of the head-dim columns of the output rows
            uint4 *dst = reinterpret_cast<uint4 *>(p.o + (Q.o_off + (int64_t)(row < nrows ? row : 0) * Q.o_rstr) * 2) +
                         h * (kD / 16);
            bool in = true;
            if constexpr (kBoundsCheck) {
                const int64_t nr = nrows;
                in = range_in(Q.o_off, 1, &nr, &Q.o_rstr, kD, 1, p.o_elems) &&
                     (!p.m_out || range_in(Q.ml_off, 1, &nr, &Q.ml_rstr, 1, 0, p.ml_elems));
                if (!in && row == 0 && h == 0) bounds_fail(p.err);
            }
            if (n == 0) {
                // no key kept: O = 0, m = -inf, l = 0
                if (row < nrows && in) {
#pragma unroll
                    for (int q = 0; q < kD / 16; q++) dst[q] = make_uint4(0u, 0u, 0u, 0u);
                    if (h == 0 && p.m_out) {
                        const int64_t o = Q.ml_off + (int64_t)row * Q.ml_rstr;
                        p.m_out[o] = -INFINITY;
                        p.l_out[o] = 0.f;
                    }
                }
                continue;
            }
            // Merge the two chains: exchange (m_ref, l, m_max) through shared memory.
            const int slot = qi & 1;
            ctl->ml[slot][h][row] = make_float4(m_ref, l, m_max, 0.f);
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl->ml_ready[slot]);
            // Both chains' accumulations of the group are complete once the
            // accumulation of its last key tile g - 1 is.
            ok = warp_wait(&ctl->o_done[(g - 1) & 1], ((g - 1) >> 1) & 1, abort, p.err, kDevTimeoutSoftmax);
            if (ok) ok = warp_wait(&ctl->ml_ready[slot], (qi >> 1) & 1, abort, p.err, kDevTimeoutSoftmax);
            if (!ok) break;
            tc_fence_after();
            const float4 mine = ctl->ml[slot][h][row], other = ctl->ml[slot][h ^ 1][row];
            const float4 c0 = h == 0 ? mine : other, c1 = h == 0 ? other : mine;
            const float M = fmaxf(c0.x, c1.x);
            const float a0 = c0.x == -INFINITY ? 0.f : ex2((c0.x - M) * c);
            const float a1 = c1.x == -INFINITY ? 0.f : ex2((c1.x - M) * c);
            const float L = c0.y * a0 + c1.y * a1;
            const float inv = L > 0.f ? 1.f / L : 0.f;
            const float w0 = a0 * inv, w1 = a1 * inv;
            const uint64_t w0x2 = pack_f32x2(w0, w0), w1x2 = pack_f32x2(w1, w1);
            // This thread's 64 output values, staged in its own row of this
            // warp's slice of the staging tile, then written by one tensor
            // store per warp (asynchronous: the warp moves on to the next
            // group while the store drains).
            const uint32_t c0row = lane_base + kOCol + (uint32_t)(h * (kD / 2));
            const uint32_t stage = smem_u32(smem + E_OFF + h * (kRows * 128));
            if (lane == 0) bulk_wait_read0();  // this warp's previous store has read its slice
            __syncwarp();
#pragma unroll
            for (int cc = 0; cc < kD / 64; cc++) {
                uint32_t o0[32], o1[32];
                tmem_ld32(c0row + 32 * cc, o0);
                tmem_ld32(c0row + kD + 32 * cc, o1);
                tmem_wait_ld();
#pragma unroll
                for (int q = 0; q < 4; q++) {
                    uint32_t b[4];  // A_0 a_0 + A_1 a_1, two columns per packed multiply and FMA
#pragma unroll
                    for (int e = 0; e < 4; e++) {
                        const int i = 8 * q + 2 * e;
                        const uint64_t y = fma_f32x2(pack_u32x2(o1[i], o1[i + 1]), w1x2,
                                                     mul_f32x2(pack_u32x2(o0[i], o0[i + 1]), w0x2));
                        b[e] = pack_bf16(lo_f32(y), hi_f32(y));
                    }
                    st_shared_v4(sw128_unit(stage, row, 4 * cc + q), b[0], b[1], b[2], b[3]);
                }
            }
            fence_proxy_async();  // each lane's staged row, visible to the bulk store
            __syncwarp();
            {
                // one store per warp; rows past the tile are past the O block
                // (TMA clips them), a warp whose rows all are stores nothing
                const int r0 = (warp & 3) * 32;
                if (lane == 0 && r0 < nrows && in) {
                    int32_t cc[3] = {Q.q_c[0], Q.q_c[1], Q.q_c[2]};
                    cc[Q.pos_slot] += r0;
                    tma_store_4d(maps + p.o_map0 + Q.q_map, stage + (uint32_t)(r0 * 128), h * (kD / 2), cc[0], cc[1],
                                 cc[2]);
                    bulk_commit();
                }
            }
            if (h == 0 && p.m_out && row < nrows && in) {
                const int64_t o = Q.ml_off + (int64_t)row * Q.ml_rstr;
                const float mm = fmaxf(c0.z, c1.z);
                const float b0 = c0.x == -INFINITY ? 0.f : ex2((c0.x - mm) * c);
                const float b1 = c1.x == -INFINITY ? 0.f : ex2((c1.x - mm) * c);
                p.m_out[o] = mm * p.scale;
                p.l_out[o] = mm == -INFINITY ? 0.f : c0.y * b0 + c1.y * b1;
            }
            // This warp has read both accumulators: the next group's first
            // accumulation may overwrite them once all 16 warps of the pair have.
            tc_fence_before();
            __syncwarp();
            if (lane == 0) arrive_on_rank0(&ctl->e_done, rank);
            qi++;
        }
        if (lane == 0) bulk_wait_all();  // this warp's output stores are complete
        __syncwarp();
        if (!ok) *abort = 1;
    }

    tc_fence_before();
    __syncthreads();
    // Neither CTA frees TMEM or leaves while the other may still signal it or
    // the pair's MMAs may still use its shared memory and TMEM.
    cluster_sync();
    if (warp == 9) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, kTmemCols);
    }
}

cudaLaunchConfig_t pair_config(int grid, cudaStream_t st, cudaLaunchAttribute *attr) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmem;
    cfg.stream = st;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cfg;
}

cudaError_t configure_pair(int dev) {
    static bool configured[64] = {};
    if (dev >= 0 && dev < 64 && configured[dev]) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(attention_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e == cudaSuccess && dev >= 0 && dev < 64) configured[dev] = true;
    return e;
}

}  // namespace

int attention_pair_clusters(int num_sms) {
    static int resident[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return std::max(1, num_sms / 2);
    if (resident[dev] == 0) {
        int n = 0;
        cudaLaunchAttribute attr[1];
        cudaLaunchConfig_t cfg = pair_config(2 * std::max(1, num_sms / 2), nullptr, attr);
        if (configure_pair(dev) != cudaSuccess ||
            cudaOccupancyMaxActiveClusters(&n, attention_pair_kernel, &cfg) != cudaSuccess || n <= 0) {
            cudaGetLastError();
            n = std::max(1, num_sms / 2);
        }
        resident[dev] = n;
    }
    return resident[dev];
}

cudaError_t launch_attention_pair(const AtParams &p, cudaStream_t st) {
    if (p.ncta <= 0) return cudaSuccess;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = configure_pair(dev);
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = pair_config(p.ncta, st, attr);
    return cudaLaunchKernelEx(&cfg, attention_pair_kernel, p);
}

}  // namespace ea
