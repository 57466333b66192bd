/*
 * bil.h -- batch-invariant selected-token log-probability, C ABI.
 *
 * The operator ("Batch-Invariant LogP" operator page, opening paragraph and
 * section "Reference Semantics"):
 *
 *     logp[r] = logits[r, target_ids[r]] - logsumexp(logits[r, :])   (float32)
 *     logp[r] = 0.0 and d logits[r, :] = 0.0   when target_ids[r] == ignore_index
 *
 * Optionally (the linear-logp operator of "[RFC][ROCm] End-to-end
 * optimization of bitwise VIME R/R beyond native P/P", section "Workstream 3:
 * fused ROCm LM-head and linear logp": temperature at one fixed point, and the
 * full-vocabulary entropy) the softmax sees z = x * rcp with rcp = 1/T
 * rounded once to float32, and the entropy H = -sum_c p_c log p_c is returned
 * from the same pass.
 *
 * The row's logsumexp is built the way the same page's section "Tensor
 * Parallel" (steps 1-6) builds it: the vocabulary is cut into fixed tiles of
 * tile_v columns; each tile gets a float32 (max m_t, sum-exp s_t) partial;
 * all tiles are merged in one fixed order,
 *     M = max_t m_t,   LSE = M + log(sum_{t = 0 .. T-1} s_t * exp(m_t - M)),
 * and the target logit is copied from the tile that owns it.  Every row's
 * result depends only on that row's logits, its target and tile_v -- never on
 * the number of rows, the row's position, its neighbours, the row stride,
 * the launch geometry, or on how the tiles are split between calls
 * (section "Batch-Invariance").  The backward recomputes the softmax from
 * the saved per-row LSE (section "Batch-Invariance", backward bullet):
 *     dlogits[r, c] = g[r] * ([c == target_ids[r]] - exp(logits[r, c] - lse[r])).
 *
 * Conventions shared by every call:
 *  - All array pointers are DEVICE pointers owned by the caller.  The library
 *    allocates no memory and keeps no per-call state.
 *  - Matrices are row-major.  `ld` is the row stride in elements (ld >= the
 *    columns read).  Columns at or beyond `vocab` are never read.
 *  - Work is queued on `stream` and the call returns without waiting, except
 *    where `validate` is set (it then synchronises, see below).
 *  - Every call returns a status code (BIL_OK on success).  Arguments are
 *    checked on the host before anything is queued; a failed check queues
 *    nothing and writes nothing.  There is no fallback path.
 *  - Element types: BIL_F32, BIL_BF16, BIL_F16.  Targets are int64.
 *  - The forward and the tile partials read logits with bulk asynchronous
 *    copies in whole 16-byte aligned units: from the unit that holds a tile's
 *    first element to the unit that holds its last.  Where rows start on
 *    16-byte boundaries (base address and stride) nothing outside the row's
 *    ld columns is read; elsewhere a read may take up to 15 bytes before a
 *    row's column 0 or past its column vocab-1, always within a 16-byte unit
 *    that holds an element of the row.  Those bytes never reach a result.
 *    The backward reads and writes by 16-byte units where the input and the
 *    output rows are both aligned, or from the first column where both are
 *    (rows of an input and an output that share their offsets, such as two
 *    contiguous [N, V] buffers), and element by element otherwise; it never
 *    touches bytes outside the rows' elements.  The results are bit-identical
 *    for every alignment.
 *  - bil_logp_fwd on at most 128 rows of a 16-bit type (16 rows when rows
 *    do not start on 16-byte boundaries; tiles of at most 4096) shares each
 *    row among a cluster of 8 blocks instead of streaming it through one
 *    block; the results are bit-identical to the streaming path.
 *
 * Results are bitwise reproducible for a given tile_v, element type and
 * library build (the arithmetic is fixed in bil_contract_id()).
 */
#ifndef BIL_H
#define BIL_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* An opaque CUDA stream handle (cudaStream_t); NULL is the legacy default stream. */
typedef struct CUstream_st *bil_stream_t;

/* ---- status codes ----------------------------------------------------- */
#define BIL_OK 0
#define BIL_E_INVALID_ARG 1   /* a size, pointer or range is out of its domain */
#define BIL_E_DTYPE 2         /* unknown element type */
#define BIL_E_ALIGN 3         /* a pointer is not aligned to its element size */
#define BIL_E_TARGET_RANGE 4  /* validate=1 found an active target outside [0, vocab) */
#define BIL_E_CUDA 5          /* a CUDA runtime call failed (launch, copy, device query) */
#define BIL_E_UNSUPPORTED 6   /* well-formed but beyond this library's limits (see below) */

/* ---- element types ---------------------------------------------------- */
#define BIL_F32 0
#define BIL_BF16 1
#define BIL_F16 2

/* Limits of the library: tile_v is a positive multiple of 8 with
 * tile_v * element_size <= BIL_MAX_TILE_BYTES; the fused forward handles at
 * most BIL_MAX_FUSED_TILES tiles per row (bil_logp_tile_partials and
 * bil_logp_merge have no such limit). */
#define BIL_MAX_TILE_BYTES (64 * 1024)
#define BIL_MAX_FUSED_TILES 2048

/* Every strided buffer a call reads or writes (logits, dlogits, the partials
 * and, for the LM-head calls, each operand and result) must span at most
 * BIL_MAX_EXTENT_BYTES: rows x row pitch x element size, 2^48 bytes, more than
 * any device holds.  A larger extent, or a vocabulary above it, returns
 * BIL_E_UNSUPPORTED before any CUDA call, so that no offset a kernel forms
 * can overflow 64 bits. */
#define BIL_MAX_EXTENT_BYTES ((int64_t)1 << 48)

/* The library's arithmetic contract as a printable string: the in-tile
 * lane layout and reduction tree, the exp/log primitives, the merge order.
 * Two builds with the same string give the same bits.  Static storage. */
const char *bil_contract_id(void);

/* Human-readable name of a status code.  Static storage. */
const char *bil_status_string(int status);

/*
 * bil_logp_fwd -- fused forward: tile partials, fixed-order merge, target
 * gather and combine in one pass over the logits ("Tensor Parallel", steps
 * 1-6, with every tile on this device).
 *
 *  logits        [n_rows, ld] elements of type `dtype`; columns [0, vocab) are read.
 *  dtype         BIL_F32 | BIL_BF16 | BIL_F16.
 *  n_rows        >= 0 (0 queues nothing).
 *  vocab         >= 1 real vocabulary columns; ld >= vocab.
 *  target_ids    [n_rows] int64.  A row with target == ignore_index is inactive:
 *                its logits are not read and logp = lse = +0.0.  An active row
 *                whose target lies outside [0, vocab) gets logp = NaN (lse is
 *                still its LSE) and nothing outside the row is read.
 *  tile_v        vocabulary tile width (columns), see the limits above.
 *  temperature   finite and > 0; 1 leaves the logits as they are (bit for bit).
 *  logp          [n_rows] float32 output: z_t - LSE(z).
 *  lse           [n_rows] float32 output (the per-row LSE the backward needs),
 *                or NULL when not wanted.
 *  entropy       [n_rows] float32 output (-sum p log p; +0.0 for inactive
 *                rows), or NULL.  Computing it does not change logp or lse.
 *  validate      0: no host synchronisation.  1: before queuing the kernel the
 *                call copies target_ids to the host (synchronising `stream`)
 *                and returns BIL_E_TARGET_RANGE, queuing nothing, if an active
 *                target is outside [0, vocab) (section "Reference Semantics":
 *                validate trades a synchronisation for a checked range).
 */
int bil_logp_fwd(const void *logits, int dtype, int64_t n_rows, int64_t vocab, int64_t ld,
                 const int64_t *target_ids, int64_t ignore_index, int32_t tile_v, float temperature,
                 float *logp, float *lse, float *entropy, int validate, bil_stream_t stream);

/*
 * bil_logp_tile_partials -- one vocabulary shard's tile partials
 * ("Tensor Parallel", steps 1, 2 and 5).
 *
 * The shard is the tile range [tile_begin, tile_end) of a vocabulary of
 * `vocab` columns cut into tiles of tile_v columns (num_tiles =
 * ceil(vocab / tile_v); 0 <= tile_begin < tile_end <= num_tiles).
 *
 *  logits        [n_rows, ld] elements whose column 0 is GLOBAL column
 *                tile_begin * tile_v.  For a full-vocabulary buffer, pass its
 *                base plus tile_begin * tile_v elements; for a rank's own
 *                shard, pass the shard.  Global columns >= vocab are not read.
 *  target_ids    [n_rows] int64 GLOBAL target columns; ignored rows as above.
 *  temperature   as for bil_logp_fwd.
 *  part_max,
 *  part_sum      [n_rows, ld_part] float32 (ld_part >= num_tiles).  For every row
 *                and every tile t of the range, column t receives the tile's
 *                max m_t of z and sum of exp(z - m_t).  Inactive rows receive
 *                (-inf, 0).  Other columns are not touched, so several calls
 *                (ranks) can fill one buffer.
 *  part_ent      [n_rows, ld_part] float32 (same row stride) receiving
 *                sum exp(z - m_t) * (z - m_t) per tile (0 for inactive rows),
 *                or NULL when the entropy is not wanted.
 *  target_logit  [n_rows] float32: written (the stored logit widened exactly,
 *                times rcp) only for active rows whose target lies in the range.
 */
int bil_logp_tile_partials(const void *logits, int dtype, int64_t n_rows, int64_t vocab,
                           int64_t ld, int32_t tile_v, int32_t tile_begin, int32_t tile_end,
                           float temperature, const int64_t *target_ids, int64_t ignore_index,
                           float *part_max, float *part_sum, float *part_ent, int64_t ld_part,
                           float *target_logit, bil_stream_t stream);

/*
 * bil_logp_merge -- the fixed-order merge and the combine ("Tensor Parallel",
 * steps 4 and 6).  Bit-identical to bil_logp_fwd when the partials come from
 * bil_logp_tile_partials with the same tile_v, however the tiles were split.
 *
 *  part_max, part_sum  [n_rows, ld_part] float32, columns [0, num_tiles) read.
 *  part_ent, entropy   both NULL, or the entropy partials [n_rows, ld_part] and
 *                      an [n_rows] float32 entropy output.
 *  target_logit        [n_rows] float32 (read for active rows with a valid target).
 *  target_ids, ignore_index, vocab   as for bil_logp_fwd (vocab only decides
 *                      which targets are valid).
 *  logp, lse           [n_rows] float32 outputs (lse may be NULL).
 *  validate            as for bil_logp_fwd.
 */
int bil_logp_merge(const float *part_max, const float *part_sum, const float *part_ent,
                   int64_t n_rows, int32_t num_tiles, int64_t ld_part, const float *target_logit,
                   const int64_t *target_ids, int64_t ignore_index, int64_t vocab, float *logp,
                   float *lse, float *entropy, int validate, bil_stream_t stream);

/*
 * bil_logp_bwd -- fused backward from the saved LSE ("Batch-Invariance":
 * one row tile per work unit, no cross-row reduction, no atomics; "Reference
 * Semantics": ignored rows receive a zero gradient).  The gradient of
 * g * logp + gh * H with respect to the stored logits x:
 *     a = z - lse,  p = exp(a),  d = g * (onehot - p) [- gh * (p * (a + H))] [* rcp]
 *
 *  logits, dtype, n_rows, vocab, ld, target_ids, ignore_index, temperature
 *                as for the forward.
 *  lse           [n_rows] float32, the forward's lse output.
 *  grad_logp     [n_rows] float32 upstream gradient g of logp.
 *  entropy,
 *  grad_entropy  both NULL, or the forward's entropy output and the upstream
 *                gradient gh of the entropy ([n_rows] float32 each).
 *  dlogits       [n_rows, ld_out] elements of type dlogits_dtype (BIL_F32 |
 *                BIL_BF16 | BIL_F16, rounded to nearest even).  Columns
 *                [0, vocab) receive g * (onehot - p); columns [vocab, out_cols)
 *                receive +0.0; columns >= out_cols are not touched.
 *                vocab <= out_cols <= ld_out.  Inactive rows are +0.0 throughout
 *                [0, out_cols) and their logits are not read; active rows with
 *                an out-of-range target are NaN over [0, vocab).
 */
int bil_logp_bwd(const void *logits, int dtype, int64_t n_rows, int64_t vocab, int64_t ld,
                 const int64_t *target_ids, int64_t ignore_index, float temperature,
                 const float *lse, const float *grad_logp, const float *entropy,
                 const float *grad_entropy, void *dlogits, int dlogits_dtype, int64_t ld_out,
                 int64_t out_cols, bil_stream_t stream);

/*
 * bil_stream_shape -- the pipeline shape the forward and tile-partials kernels
 * use for a tile of tile_v elements of `dtype` (fused != 0: the fused forward
 * with num_tiles tiles per row; entropy != 0: with the entropy output): the
 * number of shared-memory stages in each
 * block's ring, the number of consumer warps, and the block's dynamic shared
 * memory in bytes, for rows whose tiles start on 16-byte boundaries (when
 * they do not, each stage holds 128 bytes more).  Host arithmetic only;
 * touches no device.  The stage count is always a multiple of the consumer
 * count (each consumer warp owns its stages and meets them in fill order).
 */
int bil_stream_shape(int dtype, int32_t tile_v, int64_t num_tiles, int fused, int entropy,
                     int *stages, int *consumers, int64_t *smem_bytes);

/* Vocabulary tile width of the fused LM-head + logp (its GEMM's N tile). */
#define BIL_LINEAR_TILE_V 256

/*
 * bil_linear_logp_partials -- tile partials of the fused LM-head + logp
 * ("[RFC][ROCm] End-to-end optimization of bitwise VIME R/R beyond native
 * P/P", section "Workstream 3: fused ROCm LM-head and linear logp": the
 * projection and the vocabulary statistics are one operation, and no
 * [rows, vocabulary] logits are stored unless asked for; the statistics are
 * those of "Tensor Parallel", steps 1, 2 and 5).
 *
 * The logits are the projection z[r, c] = sum_k hidden[r, k] * weight[c, k]
 * (float32 accumulation on the tensor cores, K in increasing blocks of 64,
 * the same order for every row and tile), times rcp as in bil_logp_fwd.  The
 * vocabulary is cut into tiles of BIL_LINEAR_TILE_V columns (num_tiles =
 * ceil(vocab / BIL_LINEAR_TILE_V)); this call fills tiles [tile_begin,
 * tile_end), 0 <= tile_begin < tile_end <= num_tiles.
 *
 *  hidden        [n_rows, ld_hidden] hidden states, hidden_size <= ld_hidden.
 *  weight        the LM-head rows of the shard: [shard, ld_weight] with row j
 *                the weight of GLOBAL vocabulary column
 *                tile_begin * BIL_LINEAR_TILE_V + j, for the shard's columns
 *                (those below min(tile_end * BIL_LINEAR_TILE_V, vocab)).
 *                hidden_size <= ld_weight.
 *  dtype         BIL_BF16 or BIL_F16, for both hidden and weight.  Both base
 *                addresses 16-byte aligned; ld_hidden and ld_weight multiples
 *                of 8 (BIL_E_ALIGN otherwise).
 *  vocab         the full vocabulary size (decides the tiles and which
 *                targets are valid).
 *  temperature, target_ids, ignore_index, part_max, part_sum, part_ent,
 *  ld_part, target_logit
 *                as for bil_logp_tile_partials, with tile_v = BIL_LINEAR_TILE_V.
 *                Each tile's partial is taken by one thread over its 256
 *                columns: eight slot sums over columns 8g + j, g in increasing
 *                order, combined as ((a0+a1)+(a2+a3))+((a4+a5)+(a6+a7)).
 *  logits        NULL, or [n_rows, ld_logits] elements of logits_dtype
 *                (BIL_F32, or BIL_BF16 rounded to nearest even) receiving the
 *                shard's projection before the temperature is applied (column
 *                0 = global column tile_begin * BIL_LINEAR_TILE_V); 16-byte
 *                aligned base and row stride.  The partials are the same bits
 *                whether or not the logits are stored.
 * The hidden rows of ignored rows are read (the projection is computed per
 * 128-row tile) but their partials are (-inf, 0, 0) as in
 * bil_logp_tile_partials.
 */
int bil_linear_logp_partials(const void *hidden, const void *weight, int dtype, int64_t n_rows,
                             int64_t hidden_size, int64_t ld_hidden, int64_t vocab, int64_t ld_weight,
                             int32_t tile_begin, int32_t tile_end, float temperature,
                             const int64_t *target_ids, int64_t ignore_index, float *part_max,
                             float *part_sum, float *part_ent, int64_t ld_part, float *target_logit,
                             void *logits, int logits_dtype, int64_t ld_logits, bil_stream_t stream);

/*
 * bil_linear_logp_workspace_bytes -- bytes of device workspace that
 * bil_linear_logp_fwd needs for n_rows rows over a vocabulary of `vocab`
 * (entropy != 0: with the entropy output).  Host arithmetic only.
 */
int bil_linear_logp_workspace_bytes(int64_t n_rows, int64_t vocab, int entropy, int64_t *bytes);

/*
 * bil_linear_logp_fwd -- the fused LM-head + logp over the whole vocabulary:
 * bil_linear_logp_partials over every tile into the caller's workspace, then
 * bil_logp_merge.  logp, lse and entropy are as for bil_logp_fwd (of the
 * projection, with BIL_LINEAR_TILE_V tiles).
 *
 *  workspace        device memory of at least
 *                   bil_linear_logp_workspace_bytes(n_rows, vocab,
 *                   entropy != NULL) bytes, 256-byte aligned, owned by the
 *                   caller; its contents on entry do not matter and are
 *                   scratch afterwards.  Two calls in flight at once need two
 *                   workspaces.
 *  validate         as for bil_logp_fwd (checked before anything is queued).
 * Other arguments as for bil_linear_logp_partials.
 */
int bil_linear_logp_fwd(const void *hidden, const void *weight, int dtype, int64_t n_rows,
                        int64_t hidden_size, int64_t ld_hidden, int64_t vocab, int64_t ld_weight,
                        float temperature, const int64_t *target_ids, int64_t ignore_index,
                        float *logp, float *lse, float *entropy, void *logits, int logits_dtype,
                        int64_t ld_logits, void *workspace, int64_t workspace_bytes, int validate,
                        bil_stream_t stream);

/*
 * bil_linear_logp_bwd -- backward of the fused LM-head + logp ("[RFC][ROCm]
 * End-to-end optimization of bitwise VIME R/R beyond native P/P", section
 * "Workstream 3": the autograd actor path; the backward recomputes the
 * projection tiles from the saved LSE instead of keeping the logits).
 *
 * With z = hidden . weight^T (recomputed exactly as the forward computes it)
 * and the library's backward formula per element,
 *     dZ = (g (onehot - p) [- gh p (a + H)]) [* rcp],  a = z*rcp - lse, p = exp(a)
 * (the bits bil_logp_bwd gives for float32 logits z), rounded to dtype:
 *     dhidden = dZ . weight        [n_rows, hidden_size]
 *     dweight = dZ^T . hidden      [vocab, hidden_size]
 * both accumulated in float32 on the tensor cores in K blocks of 64 in
 * increasing order (K = vocab for dhidden, n_rows for dweight), so a row's
 * dhidden never depends on the other rows.  Three launches: dZ into `dz`, then
 * the two products, which read dz, weight and hidden where they lie (no
 * transposed copies).
 *
 *  hidden, weight, dtype, n_rows, hidden_size, ld_hidden, vocab, ld_weight,
 *  tile_begin, tile_end, temperature, target_ids, ignore_index
 *                as for bil_linear_logp_partials: `weight` holds the shard's
 *                rows, the global vocabulary columns [tile_begin * 256,
 *                min(tile_end * 256, vocab)) -- "cols" below; the whole
 *                vocabulary is tile_begin = 0, tile_end = ceil(vocab / 256).
 *                With a shard, dhidden is the shard's part of the sum over
 *                the vocabulary (the ranks' parts add up to it; see
 *                bil_sum_f32) and dweight holds the shard's rows.
 *  lse           [n_rows] float32, the forward's lse.
 *  grad_logp     [n_rows] float32 upstream gradient of logp.
 *  entropy, grad_entropy   both NULL, or the forward's entropy and its
 *                upstream gradient ([n_rows] float32 each).
 *  dz            [n_rows, ld_dz] (ld_dz >= cols) of dtype: receives dZ (the
 *                backward's scratch, owned by the caller, readable afterwards).
 *  dhidden       [n_rows, ld_dhidden] of dhidden_dtype (BIL_F32, or dtype
 *                rounded to nearest even).
 *  dweight       [cols, ld_dweight] of dweight_dtype (the same choice).
 * Every matrix argument needs a 16-byte aligned base and a row stride of a
 * multiple of 16 bytes (BIL_E_ALIGN otherwise).  Inactive rows contribute
 * zero; an active row with a target outside [0, vocab) makes its dZ row NaN
 * (and so its dhidden row and every dweight entry it touches).  n_rows = 0
 * sets dweight to zero.
 */
int bil_linear_logp_bwd(const void *hidden, const void *weight, int dtype, int64_t n_rows,
                        int64_t hidden_size, int64_t ld_hidden, int64_t vocab, int64_t ld_weight,
                        int32_t tile_begin, int32_t tile_end, float temperature,
                        const int64_t *target_ids, int64_t ignore_index, const float *lse,
                        const float *grad_logp, const float *entropy, const float *grad_entropy,
                        void *dz, int64_t ld_dz, void *dhidden, int dhidden_dtype, int64_t ld_dhidden,
                        void *dweight, int dweight_dtype, int64_t ld_dweight, bil_stream_t stream);

/*
 * bil_linear_logp_grad -- the first step of bil_linear_logp_bwd alone: dZ of
 * the shard's columns from the recomputed projection, written to dz
 * [n_rows, ld_dz] (the same bits as there).  Arguments, layouts and errors as
 * for bil_linear_logp_bwd; nothing else is written.  Together with
 * bil_linear_gemm it lets a caller queue (and time) the backward's steps one
 * by one: dhidden = bil_linear_gemm(dz K-major, weight MN-major), dweight =
 * bil_linear_gemm(dz MN-major, hidden MN-major).
 */
int bil_linear_logp_grad(const void *hidden, const void *weight, int dtype, int64_t n_rows,
                         int64_t hidden_size, int64_t ld_hidden, int64_t vocab, int64_t ld_weight,
                         int32_t tile_begin, int32_t tile_end, float temperature,
                         const int64_t *target_ids, int64_t ignore_index, const float *lse,
                         const float *grad_logp, const float *entropy, const float *grad_entropy,
                         void *dz, int64_t ld_dz, bil_stream_t stream);

/* How bil_linear_gemm finds an operand with `rows` rows over K: */
#define BIL_LAYOUT_K_MAJOR 0  /* stored [rows, K] row-major: element (i, k) at p[i * ld + k] */
#define BIL_LAYOUT_MN_MAJOR 1 /* stored [K, rows] row-major: element (i, k) at p[k * ld + i] */

/*
 * bil_linear_gemm -- C = A . B^T on the tensor cores, the contraction
 * bil_linear_logp_bwd uses for dhidden (A = dZ, B = weight read as [K, n])
 * and dweight (A = dZ read as [K, m], B = hidden read as [K, n]).  A has m
 * rows and B n rows over K = k, each stored as its layout says (row strides
 * lda, ldb >= the stored row length: k for K-major, m or n for MN-major), of
 * dtype (BIL_BF16 or BIL_F16).  C [m, ldc] (ldc >= n) receives
 * C[i, j] = sum_k A(i, k) B(j, k) accumulated in float32 in K blocks of 64 in
 * increasing order (the same bits for either layout), stored as c_dtype
 * (BIL_F32, or dtype rounded to nearest even).  Row i of C depends on row i
 * of A and on B only.  16-byte aligned bases and row strides of a multiple of
 * 16 bytes (BIL_E_ALIGN otherwise); k >= 1; a layout other than the two
 * above is BIL_E_INVALID_ARG; m = 0 or n = 0 queue nothing.  Device pointers
 * owned by the caller; asynchronous on `stream`.
 */
int bil_linear_gemm(const void *a, int a_layout, const void *b, int b_layout, int dtype, int64_t m,
                    int64_t n, int64_t k, int64_t lda, int64_t ldb, void *c, int c_dtype, int64_t ldc,
                    bil_stream_t stream);

/*
 * bil_sum_f32 -- dst[i] = ((srcs[0][i] + srcs[1][i]) + srcs[2][i]) + ... for
 * i < n: float32 sums in the order of `srcs` (1 <= count <= 16; `srcs` is a
 * host array of device pointers; dst may be one of the sources).  Adds the
 * tensor-parallel ranks' parts of dhidden in rank order, so that every rank
 * holds the same bits.
 */
int bil_sum_f32(const float *const *srcs, int count, int64_t n, float *dst, bil_stream_t stream);

/* Size of the device array that bil_linear_logp_fwd_static uses as its scratch. */
#define BIL_LINEAR_STATIC_SCRATCH_BYTES (8u * 1024u * 1024u)

/*
 * bil_linear_logp_fwd_static -- bil_linear_logp_fwd without a caller
 * workspace.  The pages have no counterpart of this entry point: it exists
 * for callers that cannot allocate device memory per call (a C or C++ host
 * driving this ABI directly, without a device memory pool, would otherwise
 * pay a cudaMalloc / cudaFree pair on every call, and those synchronise the
 * device).
 *
 * The scratch (tile partials and target logits) is one file-scope device
 * array of BIL_LINEAR_STATIC_SCRATCH_BYTES bytes (8 MiB) in the library's
 * device image; nothing is allocated or freed.  Sizes whose scratch,
 * bil_linear_logp_workspace_bytes(n_rows, vocab, entropy != NULL), exceeds
 * that return BIL_E_UNSUPPORTED and queue nothing (at vocab = 151936: up to
 * 1763 rows, or 1176 with the entropy).
 *
 *  First call on each device: the call looks up the array's device address
 *  (cudaGetSymbolAddress, with that device current) and keeps it together
 *  with the context it was found in; make that first call before any stream
 *  capture on the device.  A later call under another context on the same
 *  device (after cudaDeviceReset, or a context the caller made current with
 *  the driver API) looks the address up again, so it is a first call too.
 *  Nothing in the scratch has to start at zero: every entry the merge reads
 *  is written earlier in the same call.
 *  The array is shared by every call on the device: two calls whose work
 *  overlaps in time (different streams, or different host threads without
 *  ordering between their streams) race on it and give wrong results; order
 *  them (one stream, or events).
 *  The logits are not stored (use bil_linear_logp_fwd for that).
 * Other arguments, results and errors as for bil_linear_logp_fwd.
 */
int bil_linear_logp_fwd_static(const void *hidden, const void *weight, int dtype, int64_t n_rows,
                               int64_t hidden_size, int64_t ld_hidden, int64_t vocab, int64_t ld_weight,
                               float temperature, const int64_t *target_ids, int64_t ignore_index,
                               float *logp, float *lse, float *entropy, int validate,
                               bil_stream_t stream);

/*
 * bil_watchdog_status -- every wait inside this library's kernels is
 * bounded.  A wait that runs out sets a bit in a per-device word, and the
 * kernel stops instead of hanging (its outputs are then incomplete).  This
 * call reads that word for the current device into *flags (0 = no wait ever
 * ran out) and clears it when `clear` is non-zero.  It synchronises the device.
 * Bits: 1 a consumer's wait for a tile, 2 the producer's wait for a free
 * stage, 4 its wait for a free row slot, 8 its wait for its own copies to
 * land, 16 a consumer met a unit outside the launch's ranges (then stopped
 * before using it).  The LM-head kernel: 32 the epilogue's wait for an
 * accumulator, 64 the copy thread's wait for a free stage, 128 the MMA
 * thread's wait for a stage or a free accumulator, 256 a wait of either for
 * its own copies or MMAs to finish.  512: bil_watchdog_selftest.
 */
int bil_watchdog_status(unsigned int *flags, int clear);

/*
 * bil_watchdog_selftest -- queues one warp that waits, with the kernels'
 * bounded wait, on a barrier that nothing ever arrives at.  After the wait
 * limit (2 s) it sets bit 512 of the watchdog word and returns: the device
 * stays usable and bil_watchdog_status reports the bit.  For tests of the
 * failure detection; it takes the wait limit to run.
 */
int bil_watchdog_selftest(bil_stream_t stream);

/*
 * bil_probe_exp_rate -- a measurement helper, not part of the operator: it
 * measures the exponential unit, the second bound of the logits path after
 * HBM bandwidth ("Batch-Invariant LogP", "Batch-Invariance": one exponential
 * per element in every pass).  Queues `blocks` blocks of 256 threads; every
 * thread evaluates 8 independent chains of `iters` ex2.approx.ftz.f32 (the
 * instruction of the contract's exp).  Block b writes records[3b] = the SM it
 * ran on, records[3b+1] and records[3b+2] = that SM's clock64 counter before
 * and after its loop; so ex2 results per clock on an SM are its blocks' 2048 *
 * iters results over the span of its counters.  `sink` (one float) and
 * `records` (3 * blocks int64) are device memory owned by the caller; the
 * float is written only if a result were negative, which cannot happen.
 * Asynchronous on `stream`.
 */
int bil_probe_exp_rate(int32_t blocks, int32_t iters, float *sink, int64_t *records, bil_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* BIL_H */
