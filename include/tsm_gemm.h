/*
 * tsm_gemm.h -- C ABI of the GB300 (sm_103a) K-tiled, operand-staged GEMM.
 *
 *   C = A . B      A: M x K f16, B: K x N f16, C: M x N f32, f32 accumulation
 *
 * What the operation is, and where it is defined:
 *
 * - One output cell is the K-long dot product sum_k A[i][k] * B[k][j]
 *   ("The PTSS Cliff: A Kernel That Won't Build", section "The Arithmetic of
 *   'Fully Unrolled K'").  The library computes it the way that page's fix
 *   does: operands staged in fast on-chip memory (here TMA into a
 *   shared-memory ring), the K dimension walked in K_TILE chunks with the
 *   accumulator carried across them (here 64-deep k-blocks into a TMEM
 *   accumulator) -- sections "The Idea: Stage in SLM, Tile K" and "The Pass,
 *   Step by Step".
 * - The accumulator is f32 even though the operands are 16-bit ("A Dumb
 *   Triton Runtime Error", section "Step 1": the chunk is converted to
 *   float32 before it is summed, because 16-bit sums overflow or lose
 *   precision).
 * - Edge tiles read zeros past the matrix ("Intel XPU Backend for Triton",
 *   section "Use Tensor Descriptors to load tl.dot arguments and save
 *   results": the descriptor's shape masks out-of-bounds values to zero;
 *   "A Dumb Triton Runtime Error", section "Step 2": masked lanes take
 *   other=0, the additive identity).  No divisibility of M, N or K by any
 *   tile size is required.  Stores are clipped to i < M, j < N.
 * - Operands are row-major with strides in elements and a unit last stride
 *   ("Intel XPU Backend for Triton", sections "Set last stride to 1" and
 *   "Use Proper Type Annotations", whose GEMM signature takes M, N, K and a
 *   row stride per matrix).  Offsets are computed in 64 bits (same page,
 *   section "Avoid int32 Overflow").
 * - C is overwritten (beta = 0): its previous contents are never read.  The
 *   pages show that accumulating into an output left over from a previous
 *   allocation gives wrong answers ("A Dumb Triton Runtime Error", section
 *   "1. Atomics accumulate onto whatever is already in out"); the split-K
 *   path below therefore uses no atomics on C and sums its partial products
 *   in a fixed order.
 *
 * Memory and ownership.  A, B and C are DEVICE pointers on the current CUDA
 * device, owned by the caller (for example torch tensors), and must stay
 * valid until the work queued on `stream` has finished.  The library owns
 * only its scratch -- the split-K workspace, and packed copies of operands
 * the tensor-memory accelerator cannot address (below) -- taken from a
 * private stream-ordered memory pool on `stream` and returned to it on the
 * same stream, and a small per-device status word.
 *
 * Layout.  The fast path loads A and B and stores C with the tensor-memory
 * accelerator, which needs 16-byte aligned bases and row (and batch)
 * pitches that are multiples of 16 bytes: lda, ldb (and strideA, strideB)
 * multiples of 8 elements, ldc (strideC) a multiple of 4.  Any other pitch
 * or an otherwise aligned base is accepted too: that operand is first copied
 * into a packed, aligned scratch layout (C is computed there and copied
 * out), which costs one extra read and write of it through HBM.
 *
 * Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 * default stream).  Argument errors are found on the host, before anything
 * is queued, and return at once; nothing aborts, traps or prints.  Every
 * device-side wait is bounded in time: if one runs out the kernel records
 * GEMM_ERR_DEVICE_TIMEOUT in the status word and returns, and
 * gemm_get_device_status() reports it.
 *
 * Requirements, each checked (the status returned is in brackets):
 *   M, N, K >= 0 and < 2^31                          [INVALID_VALUE]
 *   lda >= K, ldb >= N, ldc >= N (elements)          [INVALID_VALUE]
 *   A, B 2-byte and C 4-byte aligned (elements at
 *   their natural alignment)                         [MISALIGNED]
 *   A, B, C device memory of the current device,
 *   each spanning the rows it is said to have        [INVALID_VALUE]
 *   C's bytes overlap neither A's nor B's            [ALIAS]
 *   a compute-capability 10.3 GPU (GB300)            [UNSUPPORTED_DEVICE]
 * M == 0 or N == 0 (or batch == 0) queues nothing and returns GEMM_OK;
 * K == 0 writes zeros into C (the empty sum).
 */
#ifndef TSM_GEMM_H
#define TSM_GEMM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* The same type as cudaStream_t, declared here so that this header needs no
 * CUDA header. */
typedef struct CUstream_st *gemm_stream_t;

typedef enum gemm_status {
    GEMM_OK = 0,
    GEMM_ERR_INVALID_VALUE = 1,      /* null pointer, bad size or stride, not device memory */
    GEMM_ERR_MISALIGNED = 2,         /* an element not at its natural alignment (any call), or a
                                        layout the no-allocation entry point cannot address */
    GEMM_ERR_ALIAS = 3,              /* C overlaps A or B, or two batches of C overlap */
    GEMM_ERR_UNSUPPORTED_DEVICE = 4, /* not a compute-capability 10.3 device */
    GEMM_ERR_CUDA = 5,               /* a CUDA runtime or driver call failed; see gemm_last_error_string */
    GEMM_ERR_DEVICE_TIMEOUT = 6      /* a bounded device-side wait ran out (reported by gemm_get_device_status) */
} gemm_status_t;

/* Tuning and test options.  Zero in every field means "the planner
 * chooses"; a NULL pointer means the same. */
typedef struct gemm_options {
    int32_t split_k;    /* 0: planner's choice; S >= 1: split K into S contiguous ranges
                           (clamped to the number of 64-deep k-blocks) */
    int32_t tile_n;     /* 0: planner's choice; else 64, 128, 256 or 512 output columns per
                           tile.  512 is a CTA pair's tile (tile_m 0 or 256) holding one
                           256 x 512 accumulator (all of TMEM) and issuing two 256-column
                           MMAs per k-step on one A tile: whole tiles only, so split_k must
                           be 0 or 1 and there is no tail; the planner takes it by itself
                           only for ungrouped calls where no split or tail is requested.
                           Its sums are bitwise those of 256-wide whole tiles. */
    int32_t timeout_ms; /* 0: default; else the limit of every device-side wait, in ms */
    int32_t inject_stall; /* test hook, 0 in normal use; 1 makes the epilogue wait on a
                             barrier that nothing signals, so that its bounded wait runs
                             out and the call reports GEMM_ERR_DEVICE_TIMEOUT */
    int32_t tile_m;     /* 0: planner's choice; 128: one CTA per tile; 256: a CTA pair per
                           tile (a 2-CTA cluster issuing tcgen05 cta_group::2 MMAs; needs
                           tile_n 128, 256 or 512) */
    int32_t splitk_reduce; /* 0 or 2: sum split-K partials inside the GEMM kernel when the
                              plan allows it (every cluster owns one unit), else in a second
                              kernel; 1: always the second kernel, and no split tail.  Both
                              sum the splits in ascending order, so the results of one split
                              count are bitwise the same. */
    int32_t l2_prefetch; /* 0 or 1: off; 2: on -- each unit first asks L2 for its whole K
                            range of A and B (measured slower on GB300, kept for study) */
    int32_t split_tail; /* when there are more tiles than slots and the last wave is at most half
                           full, spread that wave's tiles over every slot: either split each into
                           K ranges summed in the kernel, or cut it into column slices (halves or
                           quarters, at least 64 columns of B per CTA) each computed over all of K,
                           with no partial sums.  0: the planner decides, comparing the time each
                           takes off the last wave with its cost -- about 6 us for storing and
                           summing K-range partials, the narrower tile's lower efficiency for
                           slices; 1: K ranges whenever they apply (never for batches or with
                           splitk_reduce = 1); 2: never; 3: column slices whenever they apply.
                           Never for grouped calls. */
    uint64_t *trace;    /* NULL, or a device buffer of grid x 8 uint64 (grid from gemm_plan):
                           per CTA, %globaltimer stamps (ns) of kernel entry, setup done,
                           first k-block landed, last MMA issued, last accumulator ready,
                           output written, in-kernel split-K sum written, exit (0 where a
                           stage does not apply to the CTA's role).  For profiling only:
                           the timer ticks in steps of about a quarter microsecond and
                           stamps of different warps are not ordered within a step. */
    int32_t red_cluster; /* split-K summed inside the kernel with one CTA per tile: 0 or 1:
                            off (measured slower on GB300, so never the planner's choice); 2
                            or 4, when the plan allows it: the grid runs in clusters of that
                            many CTAs holding consecutive K ranges of one tile, which add their
                            partials on chip (distributed shared memory) before one partial
                            per cluster goes through the workspace.  The sum is then taken in
                            a fixed two-level order -- the cluster's ranges in ascending
                            order, then the clusters in ascending order -- so a given plan is
                            bitwise reproducible and integer-valued inputs are exact, but
                            random inputs may differ in the last bits from a plan that sums
                            the ranges one by one. */
} gemm_options_t;

/* What the planner chose for a problem (see gemm_plan). */
typedef struct gemm_plan_info {
    int32_t tile_m;       /* rows of C per tile: 128 (one CTA) or 256 (a CTA pair) */
    int32_t tile_n;       /* columns of C per tile */
    int32_t tile_k;       /* K depth of one staged k-block (64) */
    int32_t stages;       /* k-blocks in flight in the shared-memory ring */
    int32_t split_k;      /* number of K ranges (1 = no split) */
    int32_t tiles_m;      /* ceil(M / tile_m) */
    int32_t tiles_n;      /* ceil(N / tile_n) */
    int32_t k_blocks;     /* ceil(K / tile_k) */
    int64_t units;        /* batch * split_k * tiles_m * tiles_n work units */
    int32_t grid;         /* persistent CTAs launched: min(units, SMs) for one CTA per
                             tile, 2 x min(units, SMs / 2) for CTA pairs */
    int32_t group_m;      /* tiles of M walked together in the raster order */
    int64_t stage_bytes;  /* shared memory of one k-block: A tile + B tile */
    int64_t smem_bytes;   /* dynamic shared memory of one CTA */
    int64_t workspace_bytes; /* split-K partials, plus arrival counters and a launch tag
                                when summed in-kernel (0 when split_k == 1) */
    int32_t fused_reduce; /* 1: split partials are summed inside the GEMM kernel */
    int32_t tail_tiles;   /* with a split tail: the tiles of the partial last wave, each split
                             into tail_split pieces; 0: none */
    int32_t tail_split;
    int32_t tail_narrow;  /* 1: the pieces are column slices of tile_n / tail_split columns over
                             all of K; 0: K ranges summed in the kernel */
    int32_t red_cluster;  /* > 1: split-K partials are first added on chip in clusters of this
                             many CTAs (see gemm_options_t.red_cluster); 1: not */
} gemm_plan_info_t;

/* C = A . B for one matrix.
 *   A    device, M rows of K f16 values (IEEE binary16 bit patterns), row stride lda
 *   B    device, K rows of N f16 values, row stride ldb
 *   C    device, M rows of N f32 values, row stride ldc; written, never read;
 *        elements of a row past N (up to ldc) are left untouched
 * Returns GEMM_OK once the work is queued on `stream`. */
gemm_status_t gemm_f16_f32acc(const uint16_t *A, const uint16_t *B, float *C,
                              int64_t M, int64_t N, int64_t K,
                              int64_t lda, int64_t ldb, int64_t ldc,
                              gemm_stream_t stream);

/* C[b] = A[b] . B[b] for b < batch, the matrices of a batch `strideA`,
 * `strideB` and `strideC` elements apart (int64; the pages' MoE example
 * indexes a 3-D [E, M, K] tensor by expert with such a stride -- "Intel XPU
 * Backend for Triton", section "Use Tensor Descriptors ...", the A[E, :M, :]
 * slice, and section "Avoid int32 Overflow").  With batch > 1 the strides
 * must be positive and the batches of C must not overlap; strides that are
 * not multiples of 8 (A, B) or 4 (C) elements take the repacking path. */
gemm_status_t gemm_f16_f32acc_batched(const uint16_t *A, const uint16_t *B, float *C,
                                      int64_t M, int64_t N, int64_t K,
                                      int64_t lda, int64_t ldb, int64_t ldc,
                                      int64_t strideA, int64_t strideB, int64_t strideC,
                                      int64_t batch, gemm_stream_t stream);

/* The batched call with explicit options (NULL = all defaults). */
gemm_status_t gemm_f16_f32acc_opts(const uint16_t *A, const uint16_t *B, float *C,
                                   int64_t M, int64_t N, int64_t K,
                                   int64_t lda, int64_t ldb, int64_t ldc,
                                   int64_t strideA, int64_t strideB, int64_t strideC,
                                   int64_t batch, const gemm_options_t *opts,
                                   gemm_stream_t stream);

/* Grouped (Mixture-of-Experts) GEMM: for each group g < groups,
 *     C[g][i][:] = A[g][i][:] . B[g]   for the rows i < group_rows[g],
 * the group's matrices strideA, strideB and strideC elements apart like the
 * batched call.  This is the pages' Mixture-of-Experts example ("Intel XPU
 * Backend for Triton", section "Use Tensor Descriptors to load tl.dot
 * arguments and save results": A is [E experts, M tokens, K features],
 * expert e works on A[e, :e_num_tokens, :], an expert with no tokens does
 * nothing and rows past its count are masked out).
 *   group_rows  device memory, `groups` int32 row counts (4-byte aligned),
 *               read by the kernel when it runs, so a preceding kernel on
 *               `stream` may write them; each must lie in [0, M] -- a count
 *               outside is clamped to that range and the next
 *               gemm_get_device_status reports GEMM_ERR_INVALID_VALUE (with
 *               K == 0 the counts only limit the rows zeroed)
 *   A, B        device, as the batched call with batch = groups; rows of A[g]
 *               at or past group_rows[g] must be readable (they are loaded
 *               with the tile that crosses the count) but never reach C
 *   C           device; rows at or past group_rows[g] of C[g] are left
 *               untouched, as are elements past N
 * M is the rows every group has room for.  No split-K (the work is known
 * only on the device); groups of 256 go to one launch each, in stream
 * order.  groups == 0, M == 0 or N == 0 queue nothing. */
gemm_status_t gemm_f16_f32acc_grouped(const uint16_t *A, const uint16_t *B, float *C,
                                      const int32_t *group_rows, int64_t groups,
                                      int64_t M, int64_t N, int64_t K,
                                      int64_t lda, int64_t ldb, int64_t ldc,
                                      int64_t strideA, int64_t strideB, int64_t strideC,
                                      gemm_stream_t stream);

/* The grouped call with explicit options (NULL = all defaults; split_k and
 * split_tail are ignored). */
gemm_status_t gemm_f16_f32acc_grouped_opts(const uint16_t *A, const uint16_t *B, float *C,
                                           const int32_t *group_rows, int64_t groups,
                                           int64_t M, int64_t N, int64_t K,
                                           int64_t lda, int64_t ldb, int64_t ldc,
                                           int64_t strideA, int64_t strideB, int64_t strideC,
                                           const gemm_options_t *opts, gemm_stream_t stream);

/* Fused epilogue.  The pages' GEMM kernel takes an ACTIVATION meta-parameter
 * ("Intel XPU Backend for Triton", section "Use Proper Type Annotations")
 * without fixing the set; these are the activations offered, each applied in
 * f32 to alpha * (A.B)[i][j] + bias[j] before the value is rounded (to
 * nearest even) to the output type and stored. */
typedef enum gemm_activation {
    GEMM_ACT_NONE = 0,
    GEMM_ACT_RELU = 1,        /* x > 0 ? x : 0 */
    GEMM_ACT_LEAKY_RELU = 2,  /* x > 0 ? x : slope * x */
    GEMM_ACT_GELU = 3,        /* x/2 * (1 + erf(x / sqrt 2)) */
    GEMM_ACT_GELU_TANH = 4,   /* x/2 * (1 + tanh(sqrt(2/pi) * (x + 0.044715 x^3))) */
    GEMM_ACT_SILU = 5         /* x / (1 + exp(-x)) */
} gemm_activation_t;

typedef enum gemm_out_type {
    GEMM_OUT_F32 = 0,
    GEMM_OUT_F16 = 1,   /* IEEE binary16 */
    GEMM_OUT_BF16 = 2   /* bfloat16: the upper half of a binary32 */
} gemm_out_type_t;

typedef struct gemm_epilogue {
    float alpha;          /* scale of A.B (1: none) */
    const float *bias;    /* device, N f32 values per matrix (bias_stride apart), or NULL; 4-byte
                             aligned; must not overlap C */
    int64_t bias_stride;  /* elements between the bias vectors of consecutive batches or groups;
                             0: one vector for all */
    int32_t activation;   /* gemm_activation_t */
    float slope;          /* GEMM_ACT_LEAKY_RELU: the slope for x <= 0 */
    int32_t out_type;     /* gemm_out_type_t: the element type of C; ldc and strideC count
                             these elements, and C must sit at their natural alignment */
} gemm_epilogue_t;

/* C = act(alpha * A.B + bias), stored as epi->out_type: the batched call with
 * a fused epilogue (NULL epi: the plain f32 GEMM).  Everything else --
 * layouts, repacking, split-K (the split partials stay f32, the epilogue is
 * applied to their sum), errors -- is as gemm_f16_f32acc_opts.  K == 0 gives
 * act(bias[j]) in every cell (the epilogue of the empty sum). */
gemm_status_t gemm_f16_fused(const uint16_t *A, const uint16_t *B, void *C,
                             int64_t M, int64_t N, int64_t K,
                             int64_t lda, int64_t ldb, int64_t ldc,
                             int64_t strideA, int64_t strideB, int64_t strideC,
                             int64_t batch, const gemm_epilogue_t *epi,
                             const gemm_options_t *opts, gemm_stream_t stream);

/* The grouped (Mixture-of-Experts) call with a fused epilogue: rows below
 * each group's count get act(alpha * A.B + bias), bias_stride apart per group;
 * the other rows stay untouched.  Otherwise as gemm_f16_f32acc_grouped_opts. */
gemm_status_t gemm_f16_grouped_fused(const uint16_t *A, const uint16_t *B, void *C,
                                     const int32_t *group_rows, int64_t groups,
                                     int64_t M, int64_t N, int64_t K,
                                     int64_t lda, int64_t ldb, int64_t ldc,
                                     int64_t strideA, int64_t strideB, int64_t strideC,
                                     const gemm_epilogue_t *epi, const gemm_options_t *opts,
                                     gemm_stream_t stream);

/* The tiled row sum of "A Dumb Triton Runtime Error" (section "The kernel
 * itself"): for r < R,
 *     out[r] = sum over c < C of X[r * row_stride + c * col_stride],
 * every element widened to f32 and the sum accumulated in f32.
 *   X      device, elements of type elem_type (GEMM_OUT_F32, GEMM_OUT_F16 or
 *          GEMM_OUT_BF16 -- the page's input may be any of the three) at
 *          their natural alignment; strides in elements, row_stride >= 0,
 *          col_stride >= 1 (any view of a tensor: no copy is made)
 *   out    device, R f32 values, written, never read; must not overlap X
 * Lanes past the end of a row contribute 0, the additive identity (the
 * page's "Step 2" and its -inf padding trap), and the lanes' partial sums
 * are combined by a fixed-order tree on the chip, not by atomics onto out
 * (the page's closing argument), so a call is bitwise reproducible.  C == 0
 * writes zeros; R == 0 queues nothing.  Errors as for gemm_f16_f32acc. */
gemm_status_t rowsum_f32acc(const void *X, int32_t elem_type, float *out, int64_t R, int64_t C,
                            int64_t row_stride, int64_t col_stride, gemm_stream_t stream);

/* y = A . x, the product with N = 1, by the row-sum kernels (each element of
 * a row of A times the matching element of x):
 *   A  device, M rows of K f16 values, row stride lda >= K
 *   x  device, K f16 values incx >= 1 apart
 *   y  device, M f32 values, written; must not overlap A or x
 * f32 accumulation, fixed-order reduce as rowsum_f32acc.  K == 0 writes
 * zeros. */
gemm_status_t gemv_f16_f32acc(const uint16_t *A, const uint16_t *x, float *y, int64_t M, int64_t K,
                              int64_t lda, int64_t incx, gemm_stream_t stream);

/* The plan the library would use, computed on the host only (no GPU is
 * touched).  num_sms is the SM count to plan for (0 = the current device's).
 * It is the plan of an ungrouped call; a grouped call plans with split_k 1
 * and no tail (gemm_plan_grouped).
 * This is the analogue of the pages' footprint check and K_TILE choice
 * ("The PTSS Cliff ...", sections "The SLM Footprint" and "Choosing
 * K_TILE"): the ring holds as many A+B k-block stages as fit the shared
 * memory budget, and at least two must fit. */
gemm_status_t gemm_plan(int64_t M, int64_t N, int64_t K, int64_t batch,
                        const gemm_options_t *opts, int32_t num_sms,
                        gemm_plan_info_t *plan);

/* The plan of each launch of a grouped call (gemm_f16_f32acc_grouped and its
 * fused and optioned forms run their groups in launches of at most 256),
 * computed on the host only like gemm_plan: `groups` is the number of groups
 * (clamped to 1..256, the groups of one launch), M the rows allotted to each
 * group.  Whole tiles only: split_k 1 and no tail, whatever opts asks; the
 * 512-column tile only when opts asks for it. */
gemm_status_t gemm_plan_grouped(int64_t M, int64_t N, int64_t K, int64_t groups,
                                const gemm_options_t *opts, int32_t num_sms,
                                gemm_plan_info_t *plan);

/* C = A . B like gemm_f16_f32acc, for callers that cannot allocate device
 * memory while they run: allocators or memory managers that call into this
 * library and may not re-enter themselves, and hosts that reserved all of
 * the GPU's memory in advance.  The paper has no counterpart to this entry
 * point; it exists for those callers only.
 *
 * It allocates nothing.  When the plan splits K (split_k: 0 = the planner's
 * choice, lowered if needed until the partials fit; S >= 1 = exactly S
 * ranges, clamped to the k-blocks), the f32 partial sums go to one fixed 16 MiB
 * array compiled into the library (a file-scope __device__ array, so every
 * GPU that loads the library holds those 16 MiB until the process exits),
 * instead of the stream-ordered pool.  A plan whose partials need more than
 * 16 MiB (S x M x round_up(N, 4) x 4 bytes) is rejected with
 * GEMM_ERR_INVALID_VALUE and a message naming the size.  K == 0 is rejected
 * too; use gemm_f16_f32acc for it.  Having no scratch to repack into, it
 * also rejects any layout the tensor-memory accelerator cannot address
 * (GEMM_ERR_MISALIGNED: A, B, C need 16-byte aligned bases, lda and ldb
 * multiples of 8, ldc a multiple of 4).
 *
 * The first call on a device resolves the array's device address and
 * queries the device (no allocation).  Every call on a device shares the one array and
 * it keeps the last call's partials: calls whose work overlaps on the GPU
 * (for example on two streams at once) race on it and must be ordered by the
 * caller.  Nothing in it needs to start at zero -- every partial the reduce
 * reads is written earlier in the same call.  Arguments, layout, ownership
 * and errors are otherwise those of gemm_f16_f32acc (single matrix). */
gemm_status_t gemm_f16_f32acc_splitk_noalloc(const uint16_t *A, const uint16_t *B, float *C,
                                             int64_t M, int64_t N, int64_t K,
                                             int64_t lda, int64_t ldb, int64_t ldc,
                                             int32_t split_k, gemm_stream_t stream);

/* Waits for `stream`, then reports and clears the current device's status
 * word: GEMM_OK, or GEMM_ERR_DEVICE_TIMEOUT if a bounded wait of an earlier
 * call ran out (that call's output is then incomplete), GEMM_ERR_INVALID_VALUE
 * if a grouped call met a row count outside [0, M] (it was clamped), or
 * GEMM_ERR_CUDA if the stream reported an error. */
gemm_status_t gemm_get_device_status(gemm_stream_t stream);

/* The message of the last failed call on this host thread ("" if none). */
const char *gemm_last_error_string(void);

/* A fixed name for a status code. */
const char *gemm_status_string(gemm_status_t status);

/* Library version, major * 10000 + minor * 100 + patch. */
int32_t gemm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* TSM_GEMM_H */
