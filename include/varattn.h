/*
 * varattn -- the attention hot path of next-scale visual autoregressive (VAR)
 * generation on NVIDIA B300 (sm_103a), as a C ABI.
 *
 * At scale step k the queries of the current s_k x s_k token grid attend over
 * a KV cache that holds every token of scales 1..k ("SparVAR: Exploring
 * Sparsity in Visual AutoRegressive Modeling", abstract: each step attends to
 * all tokens across historical scales; "ARVAR", Background & Motivation: KV
 * caching).  Tokens of one scale are stored row-major (flat index r*s + c) and
 * the scales are concatenated in schedule order.
 *
 * Conventions shared by every entry point:
 *  - Tensors are bf16, dense row-major, no padding unless a field says so:
 *      Q, O            [B][H][N][D]             N = side[step]^2
 *      K, V            [B][H][kv_capacity][D]   first L rows used,
 *                                               L = sum_{i<=step} side[i]^2
 *  - Pointers to tensors are DEVICE pointers owned by the caller; the library
 *    never allocates, frees or retains them.  Pointers must be 16-byte aligned.
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *    default stream).  No call synchronises the device except
 *    var_device_status().
 *  - Return value: a var_status code.  Arguments are checked on the host before
 *    any launch; a failing check launches nothing.  Faults detected on the
 *    device (a pipeline wait that timed out, a malformed block mask, an input
 *    outside the exactly handled range) are recorded in the call's status
 *    word: the caller's own device word named by var_problem.status, read with
 *    var_check_status(), or, when that is NULL, the library's per-device word
 *    read with var_device_status().
 *  - No C++ exception crosses this interface.
 */
#ifndef VARATTN_H
#define VARATTN_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define VAR_API __attribute__((visibility("default")))
#else
#define VAR_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    VAR_OK = 0,
    VAR_ERR_INVALID_ARG = 1,  /* a null pointer, a size out of range, bad indices */
    VAR_ERR_UNSUPPORTED = 2,  /* head_dim not 64/128, misaligned pointer, shape limit */
    VAR_ERR_CUDA = 3,         /* a CUDA runtime call failed (launch, attribute, ...) */
    VAR_ERR_TIMEOUT = 4,      /* a device pipeline wait gave up (device status word) */
    VAR_ERR_NUMERIC = 5,      /* input outside the exactly-handled range (pivot select) */
    VAR_ERR_WORKSPACE = 6     /* workspace missing or smaller than required */
} var_status;

#define VAR_MAX_SCALES 32

/* The problem statement: the scale schedule, heads, head_dim, CFG batch. */
typedef struct {
    int32_t batch;        /* B: 2 for a classifier-free-guidance (cond, uncond) pair */
    int32_t heads;        /* H */
    int32_t head_dim;     /* D: 64 or 128 */
    int32_t n_scales;     /* number of entries of side[] in use, 1..VAR_MAX_SCALES */
    int32_t side[VAR_MAX_SCALES]; /* s_1..s_n: side lengths of the token grids */
    int32_t kv_capacity;  /* rows per (b,h) in the K/V buffers; 0 = exactly L(step) */
    float softmax_scale;  /* 0 = 1/sqrt(head_dim) */
    /* Optional DEVICE pointer to a caller-owned int32 status word (4-byte
     * aligned, zero before the first call).  The kernels of every call made
     * with this problem record there the first fault they detect (compare-and-
     * swap from 0), so a fault is tied to the calls that share the word, not
     * to the device.  NULL: the library's per-device word (var_device_status). */
    int32_t* status;
} var_problem;

/*
 * Dense cross-scale attention at scale index `step` (0-based):
 *   O[b,h,i,:] = sum_{j<L} softmax_j(Q[b,h,i,:] . K[b,h,j,:] * scale) V[b,h,j,:]
 * for every query i < N of the current grid, over all L cached tokens of scales
 * 0..step with no mask inside the step (SparVAR abstract).  fp32 accumulation
 * and online softmax, bf16 output.
 * q: [B][H][N][D]; k, v: [B][H][kv_capacity][D]; o: [B][H][N][D].
 * Errors: VAR_ERR_INVALID_ARG (null pointer, step out of range, kv_capacity < L),
 * VAR_ERR_UNSUPPORTED (head_dim, alignment), VAR_ERR_CUDA (launch failure).
 */
VAR_API int var_attn_dense(const var_problem* p, int32_t step, const void* q, const void* k,
                   const void* v, void* o, void* stream);

/*
 * Bytes of device workspace var_pivot_select needs for this step and channel
 * count (0 on invalid arguments).
 */
VAR_API size_t var_pivot_workspace_bytes(const var_problem* p, int32_t step, int32_t channels);

/*
 * Device workspace bytes the dense -> pivot -> pruned -> restore path needs at
 * `step` with `channels` hidden channels and keep_k kept queries.  Of those
 * calls only pivot selection takes scratch, so this equals
 * var_pivot_workspace_bytes; keep_k is checked (0 for keep_k outside [0, N] or
 * other invalid arguments) but does not change the size.  The attention-guided
 * pivots and the dynamic sparse pattern size their own scratch with
 * var_guided_pivot_workspace_bytes and var_sparvar_workspace_bytes.
 */
VAR_API size_t var_workspace_bytes(const var_problem* p, int32_t step, int32_t channels, int32_t keep_k);

/*
 * Pivot selection for cached token pruning ("FastVAR: Linear Visual
 * Autoregressive Modeling via Cached Token Pruning", abstract: only pivotal
 * tokens are forwarded; "ARVAR" Key Design 2: Top-K indices gather the tokens).
 * Per batch element b, with m_b the mean of x[b] over the N grid tokens:
 *   score[b,i] = ||x[b,i,:] - m_b||_2^2
 * keeps the keep_k largest scores (equal scores: the lower flat index first)
 * and writes their indices in ascending order.  The ranking is that of the
 * fp64 evaluation (exact channel sums, fp64 mean, squared differences summed
 * as a pairwise-halving tree over channels): fp32 scores with a certified
 * error bound decide every token outside a narrow band around the K-th score;
 * band tokens are decided by count or re-scored in fp64 on the device.
 * Three kernels on `stream`: the channel sums, then the scores and the
 * selection, each launched as a programmatic dependent of its predecessor.
 * x: [B][N][channels] bf16, channels a positive multiple of 32, |x| < 2^20.
 * idx: [B][keep_k] int32 (device).  scores: optional [B][N] fp32 (device) or NULL.
 * workspace: device memory of var_pivot_workspace_bytes() bytes, 256-byte
 * aligned; its contents on entry do not matter.
 * Errors: VAR_ERR_INVALID_ARG (keep_k < 0 or > N, null pointers, channels),
 * VAR_ERR_WORKSPACE, VAR_ERR_NUMERIC is reported through the device status
 * word when an input exceeds the exactly-summed range.
 */
VAR_API int var_pivot_select(const var_problem* p, int32_t step, const void* x, int32_t channels,
                     int32_t keep_k, int32_t* idx, float* scores, void* workspace,
                     size_t workspace_bytes, void* stream);

/*
 * var_pivot_select without a caller-supplied workspace.  The pages have no
 * counterpart to this entry point; it exists for callers that cannot allocate
 * device memory where they select pivots -- an engine that owns all device
 * memory and gives a plug-in no workspace, or a latency-critical stream on
 * which cudaMalloc (which may synchronise the device) is not allowed after
 * start-up.  It allocates nothing: its scratch is a file-scope device array
 * of this library, sized for batch <= 4, N <= 16384 and channels <= 4096
 * (about 1.5 MB, held on every GPU that loads the library until the process
 * exits).  Larger problems return VAR_ERR_WORKSPACE and launch nothing.
 * The first call on a device looks up the array's device address (once per
 * device, with that device current); make that first call before any stream
 * capture.  All calls share the one array and it keeps the last call's
 * contents (nothing in it needs clearing: each call writes every word it
 * reads before reading it): calls whose work overlaps on the GPU -- on
 * different streams, or from different host threads -- race and must be
 * serialised by the caller.
 * Arguments, results and other errors are those of var_pivot_select (the same
 * checks, in the same order), then VAR_ERR_WORKSPACE beyond the array's limits.
 */
VAR_API int var_pivot_select_noalloc(const var_problem* p, int32_t step, const void* x,
                                     int32_t channels, int32_t keep_k, int32_t* idx,
                                     float* scores, void* stream);

/*
 * Pruned attention: dense attention for the kept query rows only, against the
 * full L-token cache ("FastVAR" abstract; "ARVAR" Key Design 2: only the
 * gathered positions undergo attention).
 *   O_c[b,h,j,:] = attention(Q[b,h,idx[b,j],:], K[b,h,:L], V[b,h,:L]),  j < keep_k
 * q: [B][H][N][D]; idx: [B][keep_k] int32 device, each in [0, N);
 * o_compact: [B][H][keep_k][D].  keep_k = 0 is a no-op.
 * Errors: as var_attn_dense; indices are not checked on the device beyond
 * clamping reads into the (b,h) query block.
 */
VAR_API int var_attn_pruned(const var_problem* p, int32_t step, const void* q, const void* k,
                    const void* v, const int32_t* idx, int32_t keep_k, void* o_compact,
                    void* stream);

/*
 * Pruned attention with the outputs written in place ("ARVAR" Key Design 3,
 * Eq. (8)-(9): the sparse outputs are scattered back to their retained
 * positions): as var_attn_pruned, but the row for query idx[b, j] goes to
 * out[b, h, idx[b, j], :] of the full-grid output instead of a compact buffer.
 * Together with var_restore_fill, which writes every other row, this computes
 * the same out as var_attn_pruned followed by var_restore_scatter without the
 * compact buffer's write and read.  Rows not in idx are not touched.
 * q: [B][H][N][D]; idx: [B][keep_k] int32 device, distinct, each in [0, N);
 * out: [B][H][N][D].  keep_k = 0 is a no-op.
 * Errors: as var_attn_pruned.
 */
VAR_API int var_attn_pruned_scatter(const var_problem* p, int32_t step, const void* q, const void* k,
                                    const void* v, const int32_t* idx, int32_t keep_k, void* out,
                                    void* stream);

/*
 * The reconstruction's upsampled part alone ("ARVAR" Eq. (8)-(9)): writes
 * Up(prev; s, s) to every row of out whose token is NOT in idx[b, :] and leaves
 * the rows in idx untouched (var_attn_pruned_scatter writes those).  The two
 * calls write disjoint rows, so they may run in either order or concurrently
 * (var_pruned_in_place runs both with the fill started beside the attention).
 * prev: [B][H][s'^2][D]; idx: [B][keep_k] strictly ascending, in [0, s^2);
 * out: [B][H][s^2][D].  step >= 1.
 * Errors: as var_restore_scatter.
 */
VAR_API int var_restore_fill(const var_problem* p, int32_t step, const void* prev, const int32_t* idx,
                             int32_t keep_k, void* out, void* stream);

/*
 * The whole in-place pruned step ("ARVAR" Key Design 3, Eq. (8)-(9)): the
 * work of var_attn_pruned_scatter then var_restore_fill on `stream`, with the
 * fill's kernel started beside the attention's (a programmatic dependent
 * launch: its blocks take the SMs the attention leaves free; it reads and
 * writes none of the attention's rows) and completing after it.  out equals
 * var_attn_pruned followed by var_restore_scatter, with no compact buffer.
 * q, k, v, idx, keep_k: as var_attn_pruned_scatter (idx strictly ascending);
 * prev: as var_restore_fill; out: [B][H][N][D].  step >= 1; keep_k = 0
 * writes the upsampled grid alone (q, k, v, idx may then be NULL).
 * Errors: as var_attn_pruned_scatter and var_restore_fill.
 */
VAR_API int var_pruned_in_place(const var_problem* p, int32_t step, const void* q, const void* k,
                                const void* v, const void* prev, const int32_t* idx, int32_t keep_k,
                                void* out, void* stream);

/*
 * The whole pruned step in one call ("FastVAR", abstract: pivotal tokens
 * only; "ARVAR" Key Design 2 and Key Design 3, Eq. (8)-(9)): var_pivot_select
 * of x (writing idx), then var_pruned_in_place with those indices, on
 * `stream`.  The pruned attention is launched as a programmatic dependent of
 * the selection kernel: its blocks launch and set up beside the selection and
 * read their inputs once it has completed; the fill then starts beside the
 * attention.  idx and out equal those of var_pivot_select followed
 * by var_pruned_in_place (and so of the unfused chain).
 * x, channels, keep_k, idx, workspace: as var_pivot_select (no scores);
 * q, k, v, prev, out: as var_pruned_in_place.  keep_k = 0 writes the
 * upsampled grid alone (idx, q, k, v, workspace unused; they may be NULL).
 * Errors: as var_pivot_select and var_pruned_in_place.
 */
VAR_API int var_pruned_step(const var_problem* p, int32_t step, const void* x, int32_t channels,
                            int32_t keep_k, const void* q, const void* k, const void* v, const void* prev,
                            int32_t* idx, void* out, void* workspace, size_t workspace_bytes, void* stream);

/*
 * var_attn_dense that also writes each query row's log2-sum-exp of its scaled
 * scores, lse[b,h,i] = log2(sum_j 2^(s_ij)), s_ij = Q[b,h,i,:] . K[b,h,j,:] *
 * scale * log2(e) over the L keys, so that the attention probabilities are
 * P[i,j] = 2^(s_ij - lse_i).  A step whose attention guides a later step's
 * pivots ("ARVAR" Key Design 2) keeps these statistics for var_attn_saliency.
 * lse: [B][H][N] fp32 device (-inf for a row with no key).
 * Errors: as var_attn_dense.
 */
VAR_API int var_attn_dense_lse(const var_problem* p, int32_t step, const void* q, const void* k,
                               const void* v, void* o, float* lse, void* stream);

/*
 * Spatial saliency of the source step src_step ("ARVAR" Key Design 2:
 * attention retrospect -- the self-attention of an earlier, smaller step,
 * aggregated per position).  For each (b, h) and each token j of the source
 * grid (the self block: key rows L' - N' .. L' - 1 of the cache at src_step):
 *   sal[b,h,j] = sum_i P_h[i, L' - N' + j]
 * the attention probability it receives, summed over the N' source queries,
 * with the probabilities of var_attn_dense_lse's statistics (softmax over all
 * L' keys).  The head and query mean is taken by var_guided_pivot_select.
 * q_src: [B][H][N'][D] (the source step's queries); k: [B][H][kv_capacity][D];
 * lse: [B][H][N'] from var_attn_dense_lse at src_step; sal: [B][H][N'] fp32.
 * Errors: as var_attn_dense.
 */
VAR_API int var_attn_saliency(const var_problem* p, int32_t src_step, const void* q_src, const void* k,
                              const float* lse, float* sal, void* stream);

/* Bytes of device workspace var_guided_pivot_select needs (0 on invalid arguments). */
VAR_API size_t var_guided_pivot_workspace_bytes(const var_problem* p, int32_t step);

/*
 * Attention-guided pivot selection ("ARVAR" Key Design 2): the head and
 * query mean of var_attn_saliency's map, v[b, j'] = (1/(H N')) sum_h sal[b,h,j'],
 * is interpolated bilinearly from the side[src_step] grid to the side[step]
 * grid (half-pixel centres, edge clamp, as var_restore_scatter), and the
 * keep_k positions with the largest interpolated value are kept (equal values:
 * the lower flat index first), written in ascending order.  The values are
 * computed in fp32 and the ranking is exact on them.
 * sal: [B][H][side[src_step]^2] fp32; idx: [B][keep_k] int32; scores: optional
 * [B][side[step]^2] fp32 (the interpolated values) or NULL; workspace of
 * var_guided_pivot_workspace_bytes() bytes, 256-byte aligned.
 * Errors: VAR_ERR_INVALID_ARG (src_step >= step, keep_k out of range, null
 * pointers), VAR_ERR_UNSUPPORTED (more than 16384 tokens), VAR_ERR_WORKSPACE.
 */
VAR_API int var_guided_pivot_select(const var_problem* p, int32_t step, int32_t src_step, const float* sal,
                                    int32_t keep_k, int32_t* idx, float* scores, void* workspace,
                                    size_t workspace_bytes, void* stream);

/* Bytes of device workspace var_guided_pivot_select_exact needs (0 on invalid arguments). */
VAR_API size_t var_guided_pivot_exact_workspace_bytes(const var_problem* p, int32_t step, int32_t src_step);

/*
 * Attention-guided pivot selection ("ARVAR" Key Design 2) decided in fp64: the
 * same values as var_attn_saliency + var_guided_pivot_select describe, but
 * evaluated from the source step's queries and keys in fp64 on the device in
 * the definition's own order -- scores q.k summed over channels in order, the
 * softmax denominator over the L' keys added in key order, each token's
 * saliency added over the source queries in order, the head sum in head order,
 * divided by H N', the bilinear formula term by term -- and ranked exactly on
 * those values (equal values: lower flat index first).  Use it where the kept
 * set must equal the fp64 definition's; var_guided_pivot_select ranks fp32
 * values and is three orders of magnitude faster (fp64 runs at a small
 * fraction of the fp32 rate on B300).  Only two values closer than the last
 * bit of a double exp can still be ordered differently from a CPU evaluation.
 * q_src: [B][H][side[src_step]^2][D]; k: [B][H][kv_capacity][D] (the cache, at
 * least the source step's L' rows); idx: [B][keep_k] int32, ascending; values:
 * optional [B][side[step]^2] fp64 (the interpolated values) or NULL; workspace
 * of var_guided_pivot_exact_workspace_bytes() bytes, 256-byte aligned.
 * Errors: VAR_ERR_INVALID_ARG (src_step >= step, keep_k out of range, null
 * pointers), VAR_ERR_UNSUPPORTED (alignment, a target grid over ~20,000
 * tokens), VAR_ERR_WORKSPACE, VAR_ERR_CUDA.
 */
VAR_API int var_guided_pivot_select_exact(const var_problem* p, int32_t step, int32_t src_step, const void* q_src,
                                          const void* k, int32_t keep_k, int32_t* idx, double* values,
                                          void* workspace, size_t workspace_bytes, void* stream);

/*
 * Dense attention under Branch Halving ("ARVAR" Key Design 1: at a selected
 * step only the conditional branch goes through the block and its output is
 * repeated to restore the two-branch interface).  The batch is the two
 * classifier-free-guidance branches concatenated, the conditional half first:
 * batch elements [0, B/2) are computed as in var_attn_dense and each output
 * row is written to both o[b] and o[b + B/2].  The second half of q, k and v
 * is not read.  B must be even.
 * Errors: as var_attn_dense, plus VAR_ERR_INVALID_ARG for an odd batch.
 */
VAR_API int var_attn_dense_halved(const var_problem* p, int32_t step, const void* q, const void* k,
                                  const void* v, void* o, void* stream);

/*
 * Structural reconstruction ("ARVAR" Key Design 3, Eq. (8)-(9)):
 *   out = Scatter(Up(prev; s, s), idx, o_compact)
 * Up is bilinear interpolation of the previous step's s' x s' output grid
 * (s' = side[step-1], s = side[step]) with half-pixel centres and edge clamp;
 * Scatter overwrites rows idx[b, j] with o_compact[b, h, j] (no blending).
 * prev: [B][H][s'^2][D]; o_compact: [B][H][keep_k][D]; idx: [B][keep_k] strictly
 * ascending, in [0, s^2); out: [B][H][s^2][D].  step >= 1.  keep_k = 0 gives
 * the plain upsample; keep_k = N copies o_compact.
 * Errors: VAR_ERR_INVALID_ARG (step 0, keep_k out of range, null pointers).
 */
VAR_API int var_restore_scatter(const var_problem* p, int32_t step, const void* prev,
                        const void* o_compact, const int32_t* idx, int32_t keep_k, void* out,
                        void* stream);

/*
 * Block mask for cross-scale local sparse attention (SparVAR abstract:
 * attention sinks + cross-scale locality, evaluated block-wise).
 * The query grid (side s_q = side[step], a multiple of qblock_side) is cut into
 * qblock_side x qblock_side patches, numbered row-major.  For query block
 * (by, bx) and every key scale of side s:
 *   - s <= sink_max_side: every token of the scale is kept (the sink range,
 *     the first sink_len cache tokens when those scales lead the schedule);
 *   - otherwise the window of +-radius query blocks around (by, bx), clipped to
 *     the grid, is rescaled into the key scale (lo*s/s_q rounded down,
 *     hi*s/s_q rounded up) and every qblock_side x qblock_side key block of
 *     that scale meeting it is kept.
 * Entries are packed (scale << 24) | (u << 12) | v, u/v the key block row and
 * column inside the scale, ascending within a row.
 */
typedef struct {
    int32_t qblock_side;   /* query/key block side, e.g. 8 */
    int32_t n_qblocks;     /* (side[step] / qblock_side)^2 */
    int32_t sink_len;      /* tokens of the leading scales with side <= sink_max_side */
    int32_t nnz;           /* entries[] length */
    const int32_t* row_ptr;  /* device [n_qblocks + 1] */
    const int32_t* entries;  /* device [nnz] */
    /* Optional kernel plan (device copies of var_block_mask_plan's output), or
       n_squares = 0 and NULL pointers: the kernel then merges the lists itself. */
    int32_t n_squares;       /* ceil(side / qblock_side / 2)^2 */
    int32_t plan_units;      /* sq_ptr[n_squares]: units in sq_units */
    const int32_t* sq_ptr;   /* device [n_squares + 1] */
    const int32_t* sq_units; /* device [2 * sq_ptr[n_squares]] */
    const int32_t* sq_order; /* device [n_squares] */
} var_block_mask;

/*
 * Build the block mask on the HOST.  row_ptr must hold n_qblocks + 1 ints and
 * entries `entries_cap` ints (host memory).  Call once with entries = NULL to
 * get *nnz_out (and *n_qblocks_out, *sink_len_out) for sizing.
 * Errors: VAR_ERR_INVALID_ARG (sizes), VAR_ERR_UNSUPPORTED (side[step] not a
 * multiple of qblock_side, sink scales not leading the schedule).
 */
VAR_API int var_block_mask_build(const var_problem* p, int32_t step, int32_t qblock_side,
                         int32_t radius, int32_t sink_max_side, int32_t* row_ptr,
                         int32_t* entries, int32_t entries_cap, int32_t* nnz_out,
                         int32_t* n_qblocks_out, int32_t* sink_len_out);

/*
 * Build, on the HOST, the block-sparse kernel's plan for a mask: the kernel
 * runs one CTA per 2 x 2 square of query blocks over the union of the four
 * blocks' key lists.  The plan holds, per square, that union as the kernel's
 * 64-key units (the sink range in 64-token chunks, then the key blocks in
 * ascending order, each with the set of the square's blocks that keep it and
 * its extent at the scale edge; the encoding is the library's own), and the
 * order in which CTAs take the squares (most units first).  The mask depends
 * only on the schedule, so the plan is built once and reused; without it the
 * kernel merges the four lists in every CTA.
 * row_ptr / entries: var_block_mask_build's host output; sq_ptr: [n_squares+1];
 * sq_units: 2 * units_cap ints; sq_order: [n_squares] (host).  Call with
 * sq_units = NULL to get *n_squares_out and *n_units_out for sizing.
 * Errors: VAR_ERR_INVALID_ARG (sizes, malformed entries), VAR_ERR_UNSUPPORTED
 * (qblock_side other than 8, a square with more than 1024 units).
 */
VAR_API int var_block_mask_plan(const var_problem* p, int32_t step, int32_t qblock_side,
                                const int32_t* row_ptr, const int32_t* entries, int32_t sink_len,
                                int32_t* sq_ptr, int32_t* sq_units, int32_t units_cap, int32_t* sq_order,
                                int32_t* n_squares_out, int32_t* n_units_out);

/*
 * Block-sparse cross-scale attention: as var_attn_dense, but query i of block
 * qb attends only to the sink range plus the key blocks listed for qb in
 * `mask` (whose arrays are device copies of var_block_mask_build's output).
 * q, o: [B][H][N][D]; k, v: [B][H][kv_capacity][D].
 * Errors: as var_attn_dense, plus VAR_ERR_INVALID_ARG for a mask that does not
 * match the step (block counts).
 */
VAR_API int var_attn_blocksparse(const var_problem* p, int32_t step, const void* q, const void* k,
                         const void* v, const var_block_mask* mask, void* o, void* stream);

/*
 * Dynamic sparse pattern ("SparVAR" abstract: the sparse attention pattern of
 * later high-resolution scales is predicted from a sparse decision scale and
 * carried to them by an index-mapping mechanism, giving scale self-similar
 * sparse attention).  The pages fix no formula; this library's reading:
 *
 *   units   the decision step's keys in 64-key units: the sink range (the
 *           leading scales with side <= sink_max_side) in 64-token chunks
 *           (units [0, n_sink)), then every 8 x 8 key block of each later
 *           scale up to the decision scale, row-major, scale by scale;
 *   score   scores[qb][u]: the attention mass unit u receives (softmax over all
 *           the decision step's keys), averaged over the 64 queries of the
 *           decision step's 8 x 8 query block qb, the heads and the batch;
 *   select  per qb: the sinks, then the other units by decreasing score (equal
 *           scores: lower unit first) until the kept mass reaches tau of the
 *           row total (masses added in fp64 in that order);
 *   map     a query block of the target step takes the decision block under its
 *           centre; its kept blocks of scales below the decision scale are kept
 *           as they are, its kept blocks of the decision scale are kept and
 *           mapped into every later scale up to the target, to the blocks that
 *           meet the block rescaled (rounded outward).
 *
 * The result is a block mask in var_block_mask_build's format, for
 * var_block_mask_plan and var_attn_blocksparse.
 */

/* HOST: the decision step's unit count U and sink units n_sink.  Errors:
 * VAR_ERR_UNSUPPORTED (decision side not a multiple of 8 or a sink scale, sink
 * scales not leading), VAR_ERR_INVALID_ARG (problem). */
VAR_API int var_sparvar_units(const var_problem* p, int32_t decision_step, int32_t sink_max_side,
                              int32_t* n_units_out, int32_t* n_sink_units_out);

/* Device workspace bytes var_sparvar_scores and var_sparvar_scores_fast need
 * (0 for invalid arguments). */
VAR_API size_t var_sparvar_workspace_bytes(const var_problem* p, int32_t decision_step, int32_t sink_max_side);

/* var_sparvar_scores flag: re-score every block in fp64, not only the unsettled ones. */
#define VAR_SPARVAR_RESCORE_ALL 1

/*
 * Block scores of the decision step on the device: scores [n_qb][U] fp64
 * (n_qb = (side/8)^2, row-major query blocks; caller-owned device memory),
 * exact enough that the selection at this `tau` (var_sparvar_mask_build) keeps
 * the units the fp64 definition keeps.  Each score is first computed in fp32
 * with a rigorous error bound; a block whose selection the bounds do not settle
 * is re-scored in fp64 in the definition's own evaluation order (softmax
 * denominator and unit masses added key by key, the block sum over the batch,
 * heads and the block's queries in that order).  Only two fp64 values closer
 * than the last bits of a transcendental function's rounding can still be
 * ordered differently from a CPU evaluation.
 * q: the decision step's queries [B][H][N][D]; k: the cache [B][H][kv_capacity][D].
 * flags: 0 or VAR_SPARVAR_RESCORE_ALL.  rescored: optional device int32
 * [n_qb], 1 where the block was re-scored in fp64.  workspace:
 * var_sparvar_workspace_bytes bytes, 256-byte aligned.  At most 512 units.
 * Asynchronous on `stream`.
 * Errors: as var_attn_dense, VAR_ERR_INVALID_ARG (tau outside [0, 1], flags),
 * VAR_ERR_WORKSPACE (too small), VAR_ERR_UNSUPPORTED (more than 512 units,
 * alignment), and those of var_sparvar_units.
 */
VAR_API int var_sparvar_scores(const var_problem* p, int32_t decision_step, int32_t sink_max_side, double tau,
                               int32_t flags, const void* q, const void* k, void* workspace,
                               size_t workspace_bytes, double* scores, int32_t* rescored, void* stream);

/*
 * Block scores of the decision step on the tensor cores, from the row
 * log2-sum-exp its dense attention wrote (var_attn_dense_lse at
 * decision_step): p_ij = 2^(q_i.k_j * scale * log2 e - lse_i), summed per
 * (8x8 query block, unit) over the block's queries, the unit's keys, the heads
 * and the batch, / (B H 64).  fp32 products and masses, fp64 sums in a fixed
 * order: deterministic, but with no error bound -- the selection on these
 * scores can differ from the fp64 definition's where candidates lie within
 * the fp32 rounding of the cut (var_sparvar_scores decides those exactly).
 * q, k as var_sparvar_scores; lse: device fp32 [B][H][N] (N = side^2 of the
 * decision step).  scores: device fp64 [n_qb][U].  workspace:
 * var_sparvar_workspace_bytes bytes, 256-byte aligned.  The decision side is
 * at most 64 (64 query blocks).  Asynchronous on `stream`.
 * Errors: as var_sparvar_scores (no tau or flags), VAR_ERR_UNSUPPORTED
 * (decision side above 64, head_dim).
 */
VAR_API int var_sparvar_scores_fast(const var_problem* p, int32_t decision_step, int32_t sink_max_side,
                                    const void* q, const void* k, const float* lse, void* workspace,
                                    size_t workspace_bytes, double* scores, void* stream);

/*
 * HOST: the target step's block mask from the decision step's scores (host
 * copy, [n_qb_d][U] fp64): selection with fraction tau in [0, 1], then index
 * mapping, as described above.  Output as var_block_mask_build: row_ptr
 * [(side/8)^2 + 1], entries (sorted per row), sink_len; call with entries =
 * NULL to get *nnz_out for sizing.  step >= decision_step; the target side a
 * multiple of 8.  Errors: VAR_ERR_INVALID_ARG (arguments, entries_cap too
 * small), VAR_ERR_UNSUPPORTED (sides).
 */
VAR_API int var_sparvar_mask_build(const var_problem* p, int32_t decision_step, int32_t step,
                                   int32_t sink_max_side, const double* scores, double tau,
                                   int32_t* row_ptr, int32_t* entries, int32_t entries_cap,
                                   int32_t* nnz_out, int32_t* n_qblocks_out, int32_t* sink_len_out);

/*
 * Diagnostics: launch a one-thread kernel whose bounded wait on a barrier that
 * nothing arrives on gives up after limit_us microseconds (1 .. 10^7) and
 * records VAR_ERR_TIMEOUT in `status` (a device status word as in var_problem;
 * NULL = the per-device word), exactly as a pipeline wait of the kernels above
 * that gave up would.  It lets a caller check the failure path
 * (var_check_status, var_device_status) without a fault: the device stays
 * usable.  Asynchronous on `stream`.  Errors: VAR_ERR_INVALID_ARG, VAR_ERR_CUDA.
 */
VAR_API int var_selftest_wait_timeout(int32_t limit_us, int32_t* status, void* stream);

/* floor(n * num / den) in exact integer arithmetic (the kept-query count). */
VAR_API int32_t var_keep_count(int32_t n, int32_t num, int32_t den);

/* A static, human-readable name for a var_status code. */
VAR_API const char* var_status_string(int status);

/*
 * Read (and optionally clear) the library's per-device status word of the
 * current device -- the word of calls whose var_problem.status is NULL:
 * VAR_OK, or the first fault code a kernel recorded.  Synchronises the device.
 * Returns VAR_OK, VAR_ERR_INVALID_ARG (status_out NULL) or VAR_ERR_CUDA.
 */
VAR_API int var_device_status(int32_t* status_out, int32_t clear);

/*
 * Read (and optionally clear) a caller-owned device status word (see
 * var_problem.status; NULL = the per-device word) in stream order: the read
 * follows the work already queued on `stream`, and only `stream` is
 * synchronised.  *status_out = VAR_OK or the first fault code recorded there
 * (VAR_ERR_TIMEOUT, VAR_ERR_INVALID_ARG for a malformed block mask,
 * VAR_ERR_UNSUPPORTED for a mask beyond the kernel's limits, VAR_ERR_NUMERIC).
 * Returns VAR_OK, VAR_ERR_INVALID_ARG (status_out NULL, misaligned word) or
 * VAR_ERR_CUDA.
 */
VAR_API int var_check_status(const int32_t* status, int32_t* status_out, int32_t clear, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* VARATTN_H */
