// ea_internal.h -- types shared by the host planner (host.cpp) and the CUDA
// kernels of libea.so.  Not part of the public ABI (include/ea.h is).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "ea.h"

namespace ea {

constexpr int kMaxRank = 8;
constexpr int kMaxIn = 3;
constexpr int kViewDims = 6;  // outer (row) dimensions of an elementwise / row-reduction view

// Error flag codes written by kernels into the device error word.
enum DeviceErr : int {
    kDevOk = 0,
    kDevTimeoutProducer = 1,
    kDevTimeoutMma = 2,
    kDevTimeoutEpilogue = 3,
    kDevBounds = 4,
    kDevTimeoutSoftmax = 5,
    kDevTimeoutCorrection = 6,
    kDevTimeoutSelftest = 7,
    kDevTimeoutReduce = 8,
};

// ---------------------------------------------------------------- exchange
// One overlay atom (Section 5.3) copied as rows of a contiguous inner run.
struct XSeg {
    int64_t src_off;       // element offset of the atom origin in the source arena
    int64_t dst_off;       // ... in the destination arena
    int64_t inner;         // contiguous elements per row (merged trailing dims)
    int64_t rows;          // product of ext[]
    int64_t ext[4];        // outer extents, outermost first (unused = 1)
    int64_t sstr[4];       // source strides of the outer dims (elements)
    int64_t dstr[4];       // destination strides
    int32_t nd;            // number of outer dims used
    int32_t vec;           // 1: every row start and length is 16-byte aligned
};

struct XTile {
    int32_t seg;
    int32_t pad;
    int64_t row0;   // rows [row0, row0 + nrows) of the segment ...
    int64_t nrows;
    int64_t col0;   // ... and inner elements [col0, col0 + ncols) of each row
    int64_t ncols;
};

// ------------------------------------------------- elementwise / row reduce
// A strided view of one tuple's blocks: output cells are addressed as
// (row coordinates over `nd` outer dims) x (inner index < len).
struct EwItem {
    int64_t out_base;                  // element offsets into the arenas
    int64_t in_base[kMaxIn];
    int64_t len;                       // inner extent
    int64_t rows;                      // product of ext[]
    int64_t out_inner;                 // output stride along the inner dim (1 for elementwise)
    int64_t in_inner[kMaxIn];          // input strides along the inner dim (0 = broadcast)
    int64_t ext[kViewDims];
    int64_t ostr[kViewDims];
    int64_t istr[kMaxIn][kViewDims];
    // Global coordinates of special letters (predicate lo, predicate hi, rope
    // position): sdim = index of the outer dim holding it, kViewDims = the
    // inner dim, -1 = constant (block extent 1); slo = global value at 0.
    int32_t sdim[3];
    int16_t vec;                       // 1: vectorised (16-byte) path is safe
    int16_t nd;                        // outer dims in use
    int64_t slo[3];
    int64_t inner_lo;                  // global coordinate of inner index 0
};

struct EwTile {
    int32_t item;
    int32_t pad;
    int64_t row0;   // rows [row0, row0 + nrows) ...
    int64_t nrows;
    int64_t col0;   // ... inner elements [col0, col0 + ncols)
    int64_t ncols;
};

// Row reduction: items grouped per output block (CSR over items).
struct RrGroup {
    int32_t i0, i1;                    // items [i0, i1) of this output block
    int32_t pad0, pad1;
};

struct RrTile {
    int32_t group;
    int32_t pad;
    int64_t row0;
    int64_t nrows;
};

// Flat tile descriptor of the row-batch reductions, kRbWords int64 words:
// [0, 4) element offset of the tile's first row in each block, [4, 8) row
// stride in each block, 8 output offset of the first row, 9 output row
// stride, 10 segment length, 11 rows (low 32 bits) | blocks per row << 32.
constexpr int kRbWords = 12;
// The row-batch reductions' bulk-copy path: a tile has at most kRbBulkRows
// rows, and its rows of one block (one contiguous range) at most
// kRbBulkBytes bytes.
constexpr int kRbBulkRows = 8;
constexpr int kRbBulkBytes = 16384;

// ------------------------------------------------------------ contraction
// Generic (SIMT) grouped contraction: C[b][m][n] (+)= A[b][m][k] * B[b][k][n].
struct CtGroup {
    int64_t c_base;
    int64_t M, N, nb;                  // extents; nb = batch extent
    int64_t c_sm, c_sn, c_sb;          // output strides (elements)
    int64_t m_lo, n_lo;                // global coordinates of m = 0, n = 0 (predicate)
    int32_t t0, t1;                    // tuples [t0, t1)
};

struct CtTuple {
    int64_t a_base, b_base;
    int64_t K;
    int64_t a_sm, a_sk, a_sb;
    int64_t b_sk, b_sn, b_sb;
};

struct CtTile {
    int32_t group;
    int32_t batch;
    int32_t m0;
    int32_t n0;
};

// tcgen05 grouped contraction: operands are described by TMA tensor maps.
struct TcGroup {
    int32_t t0, t1;                    // tuples [t0, t1)
    int32_t out_map;                   // tensor map index of the output block
    int32_t n_ext;                     // N extent of the output block
    int32_t m_ext;                     // M extent (tiles at m0 >= m_ext are padding: computed, not stored)
    int32_t pad;
    int64_t m_lo, n_lo;                // predicate coordinates
    int64_t e_base, e_sm, e_sb;        // epilogue ADD: element offset of the block in epi_in, row and
                                       // batch strides (the output's: same extents and tiling)
    int64_t r_lo, c_lo;                // global row index of row 0 (ROPE position, row scale), global column 0
};

struct TcTuple {
    int32_t a_map, b_map;              // tensor map indices
    int32_t kchunks;                   // ceil(K / 64)
    int32_t pad;
};

struct TcTile {
    int32_t group;
    int32_t batch;
    int32_t m0;
    int32_t n0;
};

// ------------------------------------------------------------ launchers
// Each returns cudaSuccess or the launch error.  All take a device error
// word (int*) for bounded-wait / bounds failures.

// src_elems, dst_elems: arena sizes in elements (checked per tile by a
// library built with EA_DEBUG_BOUNDS, which raises `err` on a violation).
cudaError_t launch_exchange(const XSeg *segs, const XTile *tiles, int64_t ntiles, const char *src, char *dst,
                            int esize, int num_sms, cudaStream_t st, int64_t src_elems, int64_t dst_elems, int *err);

struct EwParams {
    const EwItem *items;
    const EwTile *tiles;
    int64_t ntiles;
    const char *in[kMaxIn];
    int in_dtype[kMaxIn];
    char *out;
    int out_dtype;
    int n_in;
    int map;
    float scale, eps;
    int pred;                          // 1: predicate active
    const float *rope_table;
    int64_t rope_npos;
    int64_t rope_half;                 // pairs per position in rope_table
    int has_vec, has_scalar;           // which kernel variants have tiles
    int stream_mask;                   // bit k: input k runs along the row (else broadcast)
    int *err;
    int64_t in_elems[kMaxIn], out_elems;  // arena sizes (elements), for EA_DEBUG_BOUNDS checks
};
cudaError_t launch_ewise(const EwParams &p, int num_sms, cudaStream_t st);

struct RrParams {
    const EwItem *items;               // one per (group, tuple)
    const RrGroup *groups;
    const RrTile *tiles;
    int64_t ntiles;
    const char *in[kMaxIn];
    int in_dtype[kMaxIn];
    char *out;
    int out_dtype;
    char *out2;                        // MAX_SUMEXP: the SUM of exp
    int out2_dtype;
    int n_in;
    int map;
    int agg;
    float scale, eps;
    int pred;
    int stream_mask;                   // bit k: input k runs along the row (else broadcast)
    int max_items;                     // most tuples in one group
    int tile_linear;                   // 1: no tile crosses a run of the innermost row dim
    int row_batch;                     // 1: the row-batch kernels (rb_desc) serve this plan
    int row_bulk;                      // 1: ... through bulk copies (every tile's block segment one contiguous,
                                       //    16-byte aligned range of at most 8 rows and 16 KB)
    const int64_t *rb_desc;            // kRbWords per tile when row_batch
    int *err;
    int64_t in_elems[kMaxIn], out_elems;  // arena sizes (elements), for EA_DEBUG_BOUNDS checks
};
cudaError_t launch_rowreduce(const RrParams &p, int num_sms, cudaStream_t st);

struct CtParams {
    const CtGroup *groups;
    const CtTuple *tuples;
    const CtTile *tiles;
    int64_t ntiles;
    const char *a, *b;
    char *c;
    int a_dtype, b_dtype, c_dtype;
    float scale;
    int pred_mode;                     // 0 none; 1 mask n > m; 2 mask m > n
    int tile;                          // output tile edge: 64, or 32 when 64-wide tiles would leave SMs idle
    int split;                         // fp32, 32-wide tiles, <= 4 tuples of K <= 64 per group: one warp
                                       // group per tuple, the tuples' products summed in canonical order
    int64_t a_elems, b_elems, c_elems;  // arena sizes (elements), for EA_DEBUG_BOUNDS checks
    int *err;
};
cudaError_t launch_contract_simt(const CtParams &p, cudaStream_t st);

struct TcParams {
    const void *tmaps;                 // device array of CUtensorMap (64-byte aligned)
    const TcGroup *groups;
    const TcTuple *tuples;
    const TcTile *tiles;
    int32_t ntiles;
    int32_t a_mn_major, b_mn_major;
    int32_t out_f32;
    float scale;
    int32_t pred_mode;
    int32_t bn;                        // 128 or 256
    int32_t cluster;                   // 1, or 2: CTA pairs (cta_group::2); tiles 2 p and 2 p + 1
                                       // have the same group, batch and n0, and m0 128 apart
    int32_t epi;                       // epilogue join: 0 none, 1 ADD epi_in, 2 SiLU(g) * u of column pairs,
                                       // 3 ROPE rotation of column pairs
    const char *epi_in;                // epi 1: the joined relation's arena (output dtype)
    const float *row_rms;              // row scale rsqrt(row_rms[global row] + eps), or null
    float eps;
    const float *rope_table;           // epi 3: [rope_npos][rope_half][2] = (cos, sin), or pair-major
    int64_t rope_npos;
    int32_t rope_half;                 // pairs per period along the columns
    int32_t rope_pm;                   // table pair-major: [rope_half][rope_npos][2]
    int *err;
    int64_t epi_elems, rms_elems;      // arena sizes of epi_in and row_rms (elements), for EA_DEBUG_BOUNDS
};
cudaError_t launch_contract_tc(const TcParams &p, int num_sms, cudaStream_t st);

// --------------------------------------------------------------- attention
// Flash attention as one join-agg: an aggregation group is one tile of 128
// query positions of one query head; its tuples are the key tiles (128 keys
// of one K/V block pair) that the predicate keeps, taken in runs.  A work
// item holds one or two groups that share their key tiles (two query tiles
// of the same head), run side by side by the two softmax warpgroups.
struct AtQTile {
    int64_t s_glob0;   // global query position of row 0
    int64_t o_off;     // element offset in the O arena of row 0, head-dim index 0
    int64_t o_rstr;    // O element stride between consecutive query positions
    int64_t ml_off;    // element offset of row 0 in the m and l arenas
    int64_t ml_rstr;   // their stride between consecutive query positions
    int32_t q_map;     // tensor map of the Q block
    int32_t q_c[3];    // map coordinates (dims 1..3) of row 0
    int32_t nrows;     // valid query rows (<= 128)
    int32_t pos_slot;  // which of q_c is the query position
};

struct AtItem {
    AtQTile q[2];      // q[1] unused when nq == 1
    int32_t nq;        // query tiles of the item: 1 or 2
    int32_t r0, r1;    // key-tile runs [r0, r1), shared by the query tiles
    int32_t ntiles;    // key tiles over all runs
    int32_t nt[2];     // query slot x runs the first nt[x] key tiles (its later ones are all masked)
    int32_t pad;
};

struct AtRun {
    int64_t t_glob0;   // global key position of the run's first key
    int32_t k_map;     // tensor map of the K block (the V block's is k_map + n_kv)
    int32_t k_c[3];    // map coordinates (dims 1..3) of the run's first key
    int32_t pos_slot;  // which of k_c steps by 128 from one key tile to the next
    int32_t ntiles;
    int32_t nkeys;     // keys in the run (its last tile may be partial)
    int32_t pad;
};

struct AtParams {
    const void *tmaps;       // Q maps, then K maps, then V maps (CUtensorMap, 64-byte aligned)
    const AtItem *items;     // in the order each CTA runs them
    const int32_t *cta_ptr;  // CTA x runs items [cta_ptr[x], cta_ptr[x + 1])
    const AtRun *runs;
    const int64_t *seq_ends; // packed sequences: end positions (nseq of them), or null
    char *o;                 // O arena (bf16)
    float *m_out, *l_out;    // optional row statistics (f32 arenas) or null
    int32_t ncta;
    int32_t n_kv;            // number of K (and of V) maps
    int32_t o_map0;          // CTA pairs: first of the O maps (one per Q block, 32-row boxes), in Q block order
    int32_t nseq;
    int32_t causal;
    float scale;             // score scale (> 0)
    float scale_log2;        // scale * log2(e)
    int32_t d;               // head dimension: 64 or 128
    int32_t pair;            // 1: CTA pairs (head dim 128): cta_ptr indexes pairs, ncta = 2 x pairs, items hold
                             // two query tiles (q[1] a padding tile of no rows when the head has an odd count),
                             // K maps have 64-key boxes
    int *err;
    int64_t o_elems, ml_elems;  // arena sizes of O and of m / l (elements), for EA_DEBUG_BOUNDS
};
cudaError_t launch_attention(const AtParams &p, cudaStream_t st);
cudaError_t launch_attention_pair(const AtParams &p, cudaStream_t st);
int attention_pair_clusters(int num_sms);  // CTA pairs of the attention kernel resident at once
cudaError_t launch_wait_timeout(int *err, uint64_t limit_ns, cudaStream_t st);
cudaError_t launch_exchange_agg(const XSeg *segs, const XTile *tiles, int64_t ntiles, const char *src, char *dst,
                                int dtype, int agg, int ncopies, int64_t copy_stride, int num_sms, cudaStream_t st,
                                int64_t src_elems, int64_t dst_elems, int *err);
int attention_smem_bytes(int d);

}  // namespace ea
