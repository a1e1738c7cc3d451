/*
 * ea.h -- C ABI of the GB300 (sm_103a) join-agg library (libea.so).
 *
 * The library executes the data-parallel hot path of Einsummable ("Every
 * Kernel Is a Join: Automatic Multi-GPU Parallelism for AI Computations in
 * Einsummable") on one GPU:
 *   - tensor relations: sets of (sub-tensor key, sub-tensor) blocks
 *     (Section 1; Definitions 3.1, 3.2);
 *   - one join-agg: join the blocks of the inputs on shared index letters,
 *     run a per-tuple kernel f, aggregate the outputs that share an output
 *     block with SUM or MAX, recompose (Definitions 3.5-3.7, Section 3.3);
 *   - the exchange: re-block a relation from one tiling to another through
 *     the overlay of the two tilings (Section 5.3).
 *
 * Conventions shared by every call
 * --------------------------------
 * - Plain C types only.  Pointers named dev_* / arena are device pointers;
 *   all others are host pointers that the call reads (or writes, where
 *   stated) before it returns and does not keep.
 * - Every call returns an ea_status; EA_OK is 0.  On failure nothing is
 *   launched, no output is written, and ea_last_error() returns a message
 *   for the calling host thread.
 * - GPU work is enqueued on the caller's CUDA stream (a cudaStream_t passed
 *   as void*; NULL = the legacy default stream).  No call blocks the host
 *   except ea_check().
 * - A relation of rank r over dims[0..r-1] is tiled per dimension d into
 *   nblocks[d] intervals [b_i, b_{i+1}) with 0 = b_0 <= ... <= b_n = dims[d]
 *   (Definition 3.2: the blocks cover the tensor and are pairwise disjoint).
 *   Blocks are numbered row-major over the block grid.  Each block is stored
 *   row-major (its last dimension contiguous), and the blocks follow one
 *   another in block-id order in one arena with no padding.  A block's key
 *   is its tensor type: lower bounds lo[] (inclusive), upper bounds hi[]
 *   (exclusive) (Definition 3.1).
 * - Near-equal split (bounds == NULL): b_i = floor(i * n / k).
 */
#ifndef EA_H
#define EA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define EA_ABI_VERSION 5

typedef int ea_status;
#define EA_OK 0
#define EA_ERR_SPEC 1        /* malformed spec string or unsupported letter use    */
#define EA_ERR_SHAPE 2       /* extents disagree between inputs / output           */
#define EA_ERR_PARTITION 3   /* bounds do not tile, or partitions of a letter differ */
#define EA_ERR_DTYPE 4       /* dtype not supported for this join-agg              */
#define EA_ERR_ALLOC 5       /* device or host allocation failed                   */
#define EA_ERR_CUDA 6        /* a CUDA runtime call failed (message has the name)  */
#define EA_ERR_ARG 7         /* NULL pointer, bad count, bad enum value            */
#define EA_ERR_UNSUPPORTED 8 /* valid join-agg the library has no kernel for      */
#define EA_ERR_DEVICE 9      /* a kernel raised the device error flag (ea_check)   */
#define EA_ERR_BOUNDS 10     /* a plan descriptor addresses memory outside its arena */

typedef struct ea_relation_s *ea_relation; /* opaque handle */

typedef enum { EA_F32 = 0, EA_BF16 = 1 } ea_dtype;

/* Aggregation op (+) of Definition 3.7 step (2).  NONE: every output block
 * receives exactly one tuple (elementwise joins).  MAX_SUMEXP: the softmax
 * statistics as one aggregation with two results -- out = MAX of the
 * mapped values over the aggregated letters, opts->out2 = SUM over them of
 * exp(value - max); the same as a MAX join-agg followed by a SUM join-agg
 * with the EXP_SUB map, computed in one pass with the associative,
 * commutative merge (m1,l1)+(m2,l2) = (M, l1 e^(m1-M) + l2 e^(m2-M)). */
typedef enum { EA_AGG_NONE = 0, EA_AGG_SUM = 1, EA_AGG_MAX = 2, EA_AGG_MAX_SUMEXP = 3 } ea_agg;

/* The per-tuple concrete operator f, applied cell by cell to the joined
 * values v0, v1, v2 (inputs in spec order), computed in fp32:
 *   PRODUCT     scale * v0 * v1 (* v2)          (SUM of PRODUCT = contraction)
 *   IDENTITY    scale * v0
 *   SILU_MUL    v0 / (1 + exp(-v0)) * v1
 *   ADD         v0 + v1
 *   EXP_SUB     exp(v0 - v1)
 *   DIV         v0 / v1
 *   SQUARE      scale * v0 * v0
 *   RMS_APPLY   v0 * rsqrt(v1 + eps) * v2
 *   EXP_SUB_DIV exp(v0 - v1) / v2              (softmax normalisation)
 *   ROPE        rotation of interleaved pairs (2i, 2i+1) of the last letter
 *               by the angle from rope_table at the position letter.       */
typedef enum {
    EA_MAP_PRODUCT = 0,
    EA_MAP_IDENTITY = 1,
    EA_MAP_SILU_MUL = 2,
    EA_MAP_ADD = 3,
    EA_MAP_EXP_SUB = 4,
    EA_MAP_DIV = 5,
    EA_MAP_SQUARE = 6,
    EA_MAP_RMS_APPLY = 7,
    EA_MAP_EXP_SUB_DIV = 8,
    EA_MAP_ROPE = 9
} ea_map;

/* Tiling of one tensor dimension.  bounds: nblocks + 1 values, or NULL for
 * the near-equal split.  Every interval must be non-empty unless the
 * dimension's extent is 0 (then nblocks must be 1). */
typedef struct {
    int32_t nblocks;
    int32_t reserved;
    const int64_t *bounds;
} ea_dim_part;

/* Tiling of one index letter of a spec (Section 3.3: the intervals of a
 * shardable index).  Same rules as ea_dim_part. */
typedef struct {
    char index; /* 'a'..'z' */
    char reserved[3];
    int32_t nblocks;
    const int64_t *bounds;
} ea_index_part;

/* Options of ea_joinagg_run.  Zero-initialise, then set what is needed.
 *   out_dtype  dtype of an output the call creates: 0 = the dtype of
 *              input 0, otherwise 1 + ea_dtype (1 = fp32, 2 = bf16).
 *   scale, eps map parameters (scale 0 is read as 1).
 *   pred_lo, pred_hi  cell predicate: a joined tuple is kept only if the
 *              value of letter pred_lo is <= the value of letter pred_hi
 *              (causal attention: pred_lo='t', pred_hi='s').  0 = none.
 *              Tuples of blocks that hold no such cell are dropped from the
 *              work list.  Output cells the predicate removes are absent:
 *              a contraction stores -inf in them, an elementwise join 0.
 *              A contraction whose predicate names a contracted letter
 *              relies on the operand holding 0 in removed cells.
 *   rope_pos   ROPE: the position letter.  The position of a cell is the
 *              value of that letter modulo rope_npos (sequences of rope_npos
 *              positions packed end to end); the elementwise join requires
 *              values below rope_npos.
 *   rope_table ROPE: device pointer, fp32 [rope_npos][d/2][2] = (cos, sin)
 *              of angle pos * theta^(-2i/d) (rope_layout 0), or
 *              [d/2][rope_npos][2] (rope_layout 1, pair-major: consecutive
 *              positions of one pair are adjacent, which a contraction's
 *              epilogue, one row per thread, reads coalesced).  Not owned.
 *   rope_layout ROPE: 0 or 1 as above; the elementwise ROPE join takes 0
 *              only (EA_ERR_UNSUPPORTED otherwise), any other value is
 *              EA_ERR_ARG.
 *   rope_dim   ROPE: d, the period of the pairs along the last letter (the
 *              head dimension when that letter merges heads and head dims);
 *              0 = the last letter's extent.
 *   out2       EA_AGG_MAX_SUMEXP: the relation receiving the SUM of exp;
 *              same extents and tiling as the output, created by the
 *              caller.  Ignored otherwise.
 *   epi_map, epi_in, epi_pair  an elementwise join fused into a
 *              contraction (SUM of PRODUCT over two bf16 inputs), applied to
 *              every aggregated output cell v (after scale) before it is
 *              stored ("Every Kernel Is a Join", Definition 3.7: the
 *              contraction's output relation is consumed by the join
 *              without ever being written):
 *                EA_MAP_ADD       out = v + epi_in at the same output cell;
 *                                 epi_in has the output's extents, tiling
 *                                 and dtype (the residual join "o,o->o").
 *                EA_MAP_ROPE      the rotation of the ROPE map applied to
 *                                 the output's interleaved column pairs
 *                                 (rope_pos: the output's row letter;
 *                                 pairs along its last letter, period
 *                                 rope_dim).
 *                EA_MAP_SILU_MUL  epi_pair names a letter of the second
 *                                 input only, extent 2, one block, absent
 *                                 from the output term.  The contraction
 *                                 is computed as if epi_pair were the
 *                                 output's innermost letter, and each pair
 *                                 of cells g (epi_pair = 0), u (= 1) is
 *                                 stored as SiLU(g) * u (the join
 *                                 "of,of->of" of the two slices).  bf16
 *                                 output only.
 *              0 = no epilogue.  A join-agg that does not run on the
 *              tcgen05 contraction kernel returns EA_ERR_UNSUPPORTED.
 *   row_rms    a contraction's row scale (with or without epi_map): an f32
 *              relation over one letter, the output's row letter (its
 *              only letter of input 0 kept in the output, other than
 *              batch letters of extent 1 per block), tiled as that letter;
 *              every aggregated cell of row r is multiplied by
 *              rsqrt(row_rms[r] + eps) before the epilogue join.  This is
 *              RMSNorm's apply join pushed through the SUM over the
 *              contracted letter (sum_d x[r,d] s[r] W[d,e] = s[r] sum_d
 *              x[r,d] W[d,e]); a gain over d belongs in the weight.
 *   partials   a contraction run without its aggregation ("Every Kernel Is
 *              a Join", Definition 3.7 before step (2); Section 5.3): the
 *              output relation has one more, leading dimension of extent m,
 *              tiled into m unit blocks, and copy q receives the output block
 *              of the q-th function specification of each group (canonical
 *              order); every group must have m specifications.  The copies
 *              are aggregated later, e.g. by ea_exchange_agg.
 *   simt_bf16  a bf16 contraction that the tcgen05 kernel cannot take (an
 *              operand or output whose rows are not 16-byte aligned for
 *              TMA, an operand with neither its row nor its contracted
 *              dimension contiguous, a block edge or a predicate it does
 *              not handle) returns EA_ERR_UNSUPPORTED unless this is
 *              nonzero; nonzero lets it run on the SIMT contraction kernel
 *              (fp32 FMA, a small fraction of the tensor-core rate).
 *              fp32 contractions always run on the SIMT kernel.             */
typedef struct {
    int32_t out_dtype;
    float scale;
    float eps;
    char pred_lo;
    char pred_hi;
    char rope_pos;
    char epi_pair;
    const float *rope_table;
    int64_t rope_npos;
    ea_relation out2;
    ea_relation epi_in;
    int32_t epi_map;
    int32_t rope_dim;
    ea_relation row_rms;
    int32_t partials;
    int32_t rope_layout;
    int32_t simt_bf16;
} ea_opts;

/* ------------------------------------------------------------ basics */

int ea_abi_version(void);

/* Last error message of the calling host thread ("" if none). */
const char *ea_last_error(void);

/* Synchronise `stream`, then report (and clear) any asynchronous CUDA error
 * and the device error flag that kernels raise when a bounded wait runs out
 * or a bounds check fails.  Returns EA_ERR_CUDA or EA_ERR_DEVICE on error. */
ea_status ea_check(void *stream);

/* Failure-detection self-test: launch a one-CTA kernel whose thread waits
 * on an mbarrier phase that nothing completes, through the same bounded
 * wait the tcgen05 kernels use; after `limit_us` microseconds (1 ..
 * 1000000) the wait gives up, raises the device error word and the kernel
 * returns.  The next ea_check on `stream` then reports EA_ERR_DEVICE
 * ("bounded wait ran out in the wait self-test") and clears the word; the
 * context stays usable.  Errors: EA_ERR_ARG (limit), EA_ERR_CUDA. */
ea_status ea_selftest_wait_timeout(int64_t limit_us, void *stream);

/* Free every cached plan (work lists, tensor maps).  Synchronises the
 * device first.  Plans are otherwise kept for the life of the process. */
ea_status ea_plan_cache_clear(void);

/* Device memory the library takes for itself: the arenas of relations
 * created with dev_ptr == NULL and the device copies of cached plans (work
 * lists, tensor maps, exchange segments).  By default cudaMalloc/cudaFree;
 * ea_set_allocator(alloc, free, ctx) routes later allocations through
 * alloc(bytes, ctx) and their release through free(ptr, ctx) (for instance
 * a framework's caching allocator).  alloc must return device memory of
 * the current device, 16-byte aligned, or NULL (the call that needed it
 * then fails with EA_ERR_ALLOC).  Memory is released through the pair that
 * allocated it, even after the allocator has been changed.  Both NULL:
 * back to cudaMalloc/cudaFree.  Exactly one NULL: EA_ERR_ARG.  Not called
 * concurrently with other ea_* calls that allocate.  This is the library's
 * own memory only; ea_exchange_noalloc never allocates. */
typedef void *(*ea_alloc_fn)(size_t bytes, void *ctx);
typedef void (*ea_free_fn)(void *ptr, void *ctx);
ea_status ea_set_allocator(ea_alloc_fn alloc, ea_free_fn free_fn, void *ctx);

/* ------------------------------------------------------------ relations */

/* Create a relation: a tensor of `dtype` and extents dims[0..rank-1]
 * (1 <= rank <= 8) tiled by parts[0..rank-1] (Definitions 3.1, 3.2).
 * dev_ptr: an existing device arena of at least prod(dims) * elemsize bytes
 * in the layout described above, borrowed (the caller keeps it alive and
 * frees it); NULL: the library allocates the arena (cudaMalloc, or the
 * allocator given to ea_set_allocator) and frees it in ea_relation_destroy.  The arena must be 16-byte aligned.
 * *out receives the handle. */
ea_status ea_relation_create(ea_dtype dtype, int rank, const int64_t *dims, const ea_dim_part *parts, void *dev_ptr,
                             ea_relation *out);

ea_status ea_relation_destroy(ea_relation rel);

/* dtype, rank, extents (dims: room for 8) and block count. */
ea_status ea_relation_info(ea_relation rel, int32_t *dtype, int32_t *rank, int64_t *dims, int64_t *nblocks);

/* Block `block_id`: device pointer to its first element and its key
 * (lo, hi: room for rank values each; either may be NULL). */
ea_status ea_relation_block(ea_relation rel, int64_t block_id, void **dev_ptr, int64_t *lo, int64_t *hi);

/* Arena pointer and size in bytes. */
ea_status ea_relation_data(ea_relation rel, void **arena, size_t *bytes);

/* Bounds of dimension `dim` (room for nblocks + 1 values). */
ea_status ea_relation_bounds(ea_relation rel, int dim, int32_t *nblocks, int64_t *bounds);

/* Load a relation from, or offload it to, a dense row-major tensor in host
 * memory (the pages' "load NumPy inputs ... offload"): `host` holds the
 * relation's prod(dims) elements of its dtype in row-major order.
 * direction EA_TO_DEVICE copies host -> the relation's blocks,
 * EA_TO_HOST the blocks -> host.  Every block is moved with strided copies
 * on `stream` (cudaMemcpy2DAsync, one per block and per index of its dims
 * outside the two innermost non-merged ones), so no device-side re-blocking
 * is needed; asynchronous with respect to the host only when `host` is
 * pinned.  The caller keeps `host` alive until the stream has passed the
 * copies.  Errors: EA_ERR_ARG (NULL, direction), EA_ERR_CUDA. */
#define EA_TO_HOST 0
#define EA_TO_DEVICE 1
ea_status ea_relation_copy_host(ea_relation rel, void *host, int direction, void *stream);

/* ------------------------------------------------------------ join-agg */

/* Run one join-agg (Definition 3.7) on the GPU.
 *   spec      einsum-style "ij,jk->ik": one term per input, letters a-z, no
 *             letter twice in a term, every output letter in some input.
 *             Letters in inputs but not in the output are aggregated.
 *   inputs    n_inputs relations (1..3); term k's letters name the
 *             dimensions of inputs[k] in order.
 *   parts     optional per-letter tilings (may be NULL / 0).  A letter
 *             without an entry takes the tiling of the inputs that hold it;
 *             all inputs holding a letter must agree with each other and
 *             with parts (else EA_ERR_PARTITION: re-block with ea_exchange).
 *   agg, map  the aggregation op and the per-tuple operator.
 *   opts      may be NULL (defaults).
 *   out       in/out.  *out == NULL: the call creates the output relation
 *             (extents from the letters, tiling from the letter tilings,
 *             arena from cudaMalloc) and stores its handle; otherwise *out
 *             must have the output's extents and tiling and is overwritten.
 * Kernel classes, chosen from the spec, map and agg:
 *   contraction  SUM of PRODUCT over two inputs with >= 1 aggregated letter:
 *                grouped contraction, the SUM over a group's tuples fused in
 *                the accumulator (bf16: tcgen05/TMEM/TMA; fp32: FFMA);
 *   row reduction  SUM/MAX/MAX_SUMEXP whose aggregated letters are the trailing
 *                letters of input 0: one warp per output cell, warp-shuffle
 *                (+) across the row and across the group's tuples;
 *   elementwise  agg NONE: one output block per tuple, vectorised. */
ea_status ea_joinagg_run(const char *spec, const ea_relation *inputs, int n_inputs, const ea_index_part *parts,
                         int n_parts, ea_agg agg, ea_map map, const ea_opts *opts, void *stream, ea_relation *out);

/* ------------------------------------------------- attention join-agg */

/* Options of ea_attention_run; zero-initialise, every field is optional. */
typedef struct {
    float scale;             /* score scale, > 0; 0 = 1/sqrt(head dim)                      */
    int32_t causal;          /* nonzero: a query at position s keeps only keys t <= s        */
    int32_t n_seq_ends;      /* packed sequences: entries of seq_ends (0: none)              */
    int32_t reserved0;
    const int64_t *seq_ends; /* host; increasing end positions, the last = the s extent     */
    ea_relation m_out;       /* optional f32 relation: row maximum of the scaled scores      */
    ea_relation l_out;       /* optional f32 relation: row sum of exp(score - maximum)       */
    int64_t reserved[4];
} ea_attn_opts;

/* Flash attention as one join-agg ("Every Kernel Is a Join", Example 3.10:
 * grouped-query heads, packed sequences).
 *   spec   "bshd,bthd,bthd->bshd" (Q, K, V -> O) or any other letters and
 *          order with these roles: the last letter of every term is the
 *          head dimension d (extent 64 or 128, one block); the letter in Q
 *          but not in K is the query position s, the letter in K but not in
 *          Q the key position t; the other one or two letters are shared by
 *          all terms.  K and V have the same term; O has Q's term.  A shared
 *          letter may have g times as many values in Q as in K (the query
 *          heads): query head h then reads key-value head floor(h / g), so
 *          heads g m .. g m + g - 1 share head m.
 *   q, k, v  bf16 relations.  Tilings: d whole; each shared letter tiled the
 *          same in all four relations (the grouped letter's Q bounds are g
 *          times its K bounds); s tiled the same in Q and O, t the same in K
 *          and V.  Else EA_ERR_PARTITION (re-block with ea_exchange).
 *   out    *out == NULL: the call creates O (bf16, Q's extents and tiling);
 *          otherwise *out must match and is overwritten.
 * Result, per query row (b, s, h):
 *   O = SUM_t softmax_t(scale Q.K_t) V_t over the kept keys t: those of the
 *   same packed sequence as s (opts->seq_ends; all keys when none) and, if
 *   causal, t <= s.  A row that keeps no key gets O = 0 (m = -inf, l = 0).
 *   m_out / l_out (optional, both or neither): f32 relations over Q's term
 *   without d, tiled as Q, receiving m = max_t scale Q.K_t and
 *   l = SUM_t exp(scale Q.K_t - m) over the kept keys.
 * How it runs: a group is one tile of 128 query positions of one query head,
 * its tuples the key tiles of 128 keys that the predicate keeps; the
 * aggregation over t merges (m, l, A) triples, A = SUM exp(S - m) V,
 * (m1,l1,A1) + (m2,l2,A2) = (M, l1 e^(m1-M) + l2 e^(m2-M), A1 e^(m1-M) +
 * A2 e^(m2-M)) with M = max(m1, m2), in registers; O = A / l.  Scores are
 * fp32 from bf16 inputs; the probabilities enter the second product as bf16.
 * Errors: EA_ERR_SPEC (roles above), EA_ERR_SHAPE, EA_ERR_PARTITION,
 * EA_ERR_DTYPE (not bf16 / stats not f32), EA_ERR_UNSUPPORTED (head dim not
 * 64 or 128, a block not 16-byte aligned, no tensor-map encoder),
 * EA_ERR_ARG (bad seq_ends, scale < 0, one of m_out/l_out). */
ea_status ea_attention_run(const char *spec, ea_relation q, ea_relation k, ea_relation v, const ea_attn_opts *opts,
                           void *stream, ea_relation *out);

/* ------------------------------------------------------------ exchange */

/* Re-block `in` into the tiling new_parts[0..rank-1] (Section 5.3: the
 * overlay of the two tilings gives the atoms; each atom is copied from its
 * source block into its destination block; every element keeps its global
 * coordinates).  The copy is bit-exact.  *out == NULL: the call creates the
 * output relation; otherwise *out must have the same dtype and extents and
 * the tiling new_parts (new_parts may then be NULL), and must not share
 * memory with `in`. */
ea_status ea_exchange(ea_relation in, const ea_dim_part *new_parts, void *stream, ea_relation *out);

/* The exchange with aggregation ("Every Kernel Is a Join", Section 5.3 and
 * Example 5.4): `in` holds m unaggregated copies of a relation along its
 * first dimension (extent m, tiled into m unit blocks, copy q = in[q, ...],
 * e.g. the partials of a join-agg); every cell x of `out` receives the
 * aggregate (+)_q in[q, x] of its m copies, re-blocked into out's tiling
 * through the overlay of the two tilings (each atom's copies are read and
 * combined once, in copy order, in fp32, and written once).  agg:
 * EA_AGG_SUM or EA_AGG_MAX.  *out == NULL: the call creates the output with
 * in's dtype, extents in->dims[1..] and tiling new_parts (rank in->rank - 1);
 * otherwise *out must have them (new_parts may then be NULL).  Errors:
 * EA_ERR_SHAPE (extents or rank), EA_ERR_PARTITION (in's first dimension not
 * in unit blocks, out's tiling unlike new_parts), EA_ERR_ARG (agg, overlap). */
ea_status ea_exchange_agg(ea_relation in, ea_agg agg, const ea_dim_part *new_parts, void *stream, ea_relation *out);

/* What the last ea_joinagg_run / ea_exchange of the calling host thread
 * launched: kernel class (0 exchange, 1 elementwise, 2 row reduction,
 * 3 SIMT contraction, 4 tcgen05 contraction, 5 attention, 6 exchange with
 * aggregation), kernel launches, work tiles,
 * aggregation groups and function specifications (tuples).  Any pointer
 * may be NULL. */
ea_status ea_last_plan(int32_t *kernel_class, int32_t *launches, int64_t *tiles, int64_t *groups, int64_t *tuples);

/* How many CTAs shared one MMA tile in that launch: 1, or 2 when the
 * tcgen05 contraction ran as CTA pairs (tcgen05 cta_group::2: one 256-row
 * tile over two SMs, each SM loading its own A rows and half of the B tile;
 * chosen when the work has at least two tiles per SM).  1 for every other
 * kernel.  Errors: EA_ERR_ARG (NULL). */
ea_status ea_last_plan_cluster(int32_t *ctas);

/* The exchange for callers that must not allocate device memory.  This
 * call has no counterpart in the paper.  ea_exchange and ea_joinagg_run
 * upload their plans into memory they take from cudaMalloc; a process
 * whose device memory is handed out by its own pool, a latency-sensitive
 * path that cannot afford cudaMalloc's implicit device-wide
 * synchronisation, or an embedding that forbids the library from owning
 * device memory cannot accept that.  ea_exchange_noalloc re-blocks `in`
 * into the tiling of `out` (same dtype and extents, arenas not
 * overlapping; create both with ea_relation_create over your own memory)
 * and calls no cudaMalloc, cudaFree or other allocating routine: its plan
 * goes into one static device array of 1 MiB inside libea.so, which every
 * GPU that loads the library holds until the process exits.  A plan larger
 * than that (about 6000 overlay atoms, or more than 2048 split points in
 * one dimension) is rejected with EA_ERR_UNSUPPORTED before anything is
 * launched.  The first call on each device looks up the array's device
 * address (cudaGetSymbolAddress) with that device current.  The plan is
 * staged in a static host buffer and copied into the array with
 * cudaMemcpyAsync on `stream`, then the kernel runs on `stream`.  A call on
 * a stream that is being captured into a CUDA graph returns
 * EA_ERR_UNSUPPORTED (a replayed copy would read whatever plan a later call
 * left in the host buffer).  Every call shares the one array, so calls
 * whose work overlaps on the GPU (different streams with no ordering
 * between them) race on it. */
ea_status ea_exchange_noalloc(ea_relation in, ea_relation out, void *stream);

/* ------------------------------------------------ host-only planning hooks */

/* The work list of a join-agg, computed on the host exactly as
 * ea_joinagg_run plans it (no GPU needed).  shapes: the extents of every
 * input term, concatenated; parts: one entry per letter that is not whole.
 * pred_lo/pred_hi: the cell predicate letters or 0.
 * Outputs (each may be NULL to ask only for the counts):
 *   groups[n_groups]      output block id of each aggregation group
 *   grp_ptr[n_groups+1]   CSR offsets into tuples
 *   tuples[n_tuples*n_in] input block ids of each function specification
 * Order: groups by increasing output block id (row-major over the output
 * block grid); inside a group, by the interval indices of the aggregated
 * letters in order of first appearance in the spec.
 * join_volume: sum over tuples of the cells of their input blocks;
 * agg_volume: sum over groups of (m - 1) * cells of the output block
 * (the sub-costs (2) and (3) of Section 4.3).  Capacities cap_groups and
 * cap_tuples bound what is written; EA_ERR_ARG if too small. */
ea_status ea_plan_worklist(const char *spec, const int64_t *shapes, const ea_index_part *parts, int n_parts,
                           char pred_lo, char pred_hi, int64_t cap_groups, int64_t cap_tuples, int64_t *groups,
                           int64_t *grp_ptr, int64_t *tuples, int64_t *n_groups, int64_t *n_tuples,
                           int64_t *join_volume, int64_t *agg_volume);

/* The exchange as a permutation (no GPU needed): perm[i] = position in the
 * source arena of the element at position i of the destination arena. */
ea_status ea_exchange_permutation(int rank, const int64_t *dims, const ea_dim_part *src_parts,
                                  const ea_dim_part *dst_parts, int64_t *perm);

/* The plan check on hand-made exchange descriptors (no GPU needed).  Every
 * plan the library builds passes the same check before it is uploaded; a
 * plan with a descriptor outside its arenas is rejected with EA_ERR_BOUNDS
 * and nothing is launched.  An exchange plan is a list of segments, each
 * rows of a contiguous run (16 int64 words per segment: source offset,
 * destination offset, run length, number of outer dimensions nd <= 4,
 * ext[4], source strides[4], destination strides[4]; elements, outermost
 * first, only the first nd of each group used), and tiles that cut the
 * segments (5 words per tile: segment index, first row, rows, first
 * element of the run, elements).  Returns EA_OK if every segment's source
 * and destination elements lie in [0, src_elems) and [0, dst_elems) and
 * every tile inside its segment, else EA_ERR_BOUNDS (message names the
 * first offending descriptor); EA_ERR_ARG for bad counts or pointers. */
ea_status ea_plan_check_exchange(const int64_t *seg_words, int64_t nseg, const int64_t *tile_words, int64_t ntiles,
                                 int64_t src_elems, int64_t dst_elems);

/* 1 if this library was built with EA_DEBUG_BOUNDS, else 0.  In that build
 * every kernel also checks, before it touches a tile (an exchange segment's
 * rows, an elementwise or row-reduction view, a contraction's operand and
 * output blocks, the residual and row-scale rows of a contraction's
 * epilogue, an attention query tile's output rows), that the tile's element
 * range lies inside its arena; if not it raises the device error word,
 * which ea_check reports as EA_ERR_DEVICE, and skips the tile (the
 * allocation-free exchange, which has no error word, only skips it).  The
 * default build leaves these checks out; both builds check every plan on
 * the host before upload (EA_ERR_BOUNDS). */
int ea_debug_bounds(void);

/* Number of atoms of the overlay of two tilings (Section 5.3). */
ea_status ea_overlay_atoms(int rank, const int64_t *dims, const ea_dim_part *src_parts, const ea_dim_part *dst_parts,
                           int64_t *n_atoms);

#ifdef __cplusplus
}
#endif

#endif /* EA_H */
