/*
 * attnres.h -- C ABI of libattnres.so, the GB300 (sm_103a) hot path of
 * Attention Residuals: the depth-wise softmax aggregation of earlier layer
 * (or block) outputs, in its Full, Block and two-phase Block forms.
 *
 * The method (pages: "Attention Residual 深度残差", K3 course notes sec-09;
 * "Attention Residuals：当网络深度也拥有寻址能力"):
 *   A1  s_i   = w~^T RMS(v_i),  w~ = w (.) gamma (gain folded into the query),
 *             RMS(v) = v / sqrt(mean_d v^2 + eps)  (no gain)
 *   A2  alpha = softmax_i(s_i)  per token (b, t), over the source axis
 *   A3  h     = sum_i alpha_i v_i  over the RAW (un-normalised) sources
 *   OS1 (m, numer, denom) online-softmax state;  OS2 merge of two states.
 *
 * Conventions shared by every compute entry point:
 *   - Token rows: a source, output or partial is a row-major [B, T, D]
 *     tensor in device memory, rows contiguous with stride D.  Depth
 *     attention never mixes tokens, so the kernels treat it as B*T
 *     independent rows.
 *   - dtype: ATTNRES_F32 or ATTNRES_BF16 for every [B,T,D] tensor of one
 *     call.  Queries, gains, u and all statistics are fp32.  Arithmetic is
 *     fp32; outputs are rounded once (to nearest even) to the I/O dtype.
 *   - Alignment: every device pointer is 16-byte aligned and D is a
 *     multiple of 8 (bf16) or 4 (fp32), so rows move as 16-byte vectors.
 *   - gain == NULL means a gain of one.
 *   - Statistics: m is the max depth score of a token, lse = m + ln(sum_i
 *     exp(s_i - m)) (natural log).  Outputs named "optional" may be NULL.
 *   - Ownership: the caller allocates and owns every buffer.  The library
 *     allocates no device memory, keeps no state between calls and never
 *     synchronises: work is queued on `stream` (a cudaStream_t; NULL is
 *     the legacy default stream) and the call returns.
 *   - Stream order: the forward kernels are launched as programmatic
 *     dependents of the kernel before them on the stream (their launch may
 *     overlap its end), and each waits for that kernel to complete before
 *     it touches any memory, so results follow plain stream order, also
 *     under stream capture.
 *   - Errors: arguments are checked before anything is launched; a bad
 *     argument returns a negative attnres_status_t and launches nothing.
 *     A launch failure returns ATTNRES_ERR_CUDA.  Nothing aborts or prints.
 *   - Empty inputs (B*T == 0) are valid and launch nothing; their data
 *     pointers are not checked (an empty tensor's pointer may be NULL).
 */
#ifndef ATTNRES_H
#define ATTNRES_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { ATTNRES_F32 = 0, ATTNRES_BF16 = 1 } attnres_dtype_t;

typedef enum {
    ATTNRES_OK = 0,
    ATTNRES_ERR_NULL = -1,             /* a required pointer is NULL                 */
    ATTNRES_ERR_SHAPE = -2,            /* n, S, L, B, T or D out of range           */
    ATTNRES_ERR_DTYPE = -3,            /* dtype is not F32 / BF16                    */
    ATTNRES_ERR_ALIGNMENT = -4,        /* pointer not 16-B aligned, or D % vec != 0  */
    ATTNRES_ERR_TOO_MANY_SOURCES = -5, /* n > ATTNRES_MAX_SOURCES                    */
    ATTNRES_ERR_CUDA = -6,             /* a kernel launch failed                     */
    ATTNRES_ERR_CAPACITY = -7,         /* a host output buffer is too small          */
    ATTNRES_ERR_VALUE = -8,            /* eps negative / not finite, block size 0    */
    ATTNRES_ERR_TIMEOUT = -9,          /* a kernel wait gave up (see below)          */
    ATTNRES_ERR_SCRATCH = -10          /* request exceeds the library's fixed scratch */
} attnres_status_t;

/* Most sources one aggregation may read (Full stack: L + 1 <= this). */
#define ATTNRES_MAX_SOURCES 256
/* Most queries one phase-1 call may batch (S). */
#define ATTNRES_MAX_QUERIES 64

/*
 * Depth aggregation, eq. A1-A3 ("DepthResidual.forward"; the pages'
 * "block_attn_res" for the Block form, where the sources are the completed
 * block summaries followed by the running partial).
 *   sources  host array of n device pointers, each [B,T,D] of `dtype`
 *   n        1 .. ATTNRES_MAX_SOURCES
 *   query    device fp32 [D] (w); gain device fp32 [D] or NULL
 *   eps      >= 0, added to the mean square inside the square root
 *   out      device [B,T,D] of `dtype`: h = sum_i alpha_i v_i
 *   out_max, out_lse  device fp32 [B,T], optional
 * Sources are read once each, as an online softmax over the source axis.
 */
int attnres_depth_aggregate(const void *const *sources, int n, int64_t B, int64_t T, int64_t D,
                            int dtype, const float *query, const float *gain, float eps, void *out,
                            float *out_max, float *out_lse, void *stream);

/*
 * Phase 1 of the two-phase Block scheme ("两阶段算法（inter / intra）",
 * inter step; "attn_with_stats"): the S pseudo-queries of one block score
 * the same n completed block summaries in one pass.
 *   blocks   host array of n_blocks device pointers, each [B,T,D]
 *   n_blocks 1 .. 16 (ATTNRES_ERR_TOO_MANY_SOURCES above; the Full
 *            two-phase schedule runs phase 1 over more sources internally)
 *   queries  device fp32 [S,D]; gains device fp32 [S,D] or NULL
 *   S        1 .. ATTNRES_MAX_QUERIES
 *   out      device [S,B,T,D] of `dtype`: out[s] = normalised output o_s
 *   out_lse  device fp32 [S,B,T], required (phase 2 consumes it)
 *   out_max  device fp32 [S,B,T], optional
 * All S queries are served by one batched pass over the summaries: the
 * per-token-row kernel (few rows, fp32, more than ten summaries) reads each
 * summary once; the tensor-core kernels (bf16, at least 512 rows) read it
 * twice, once for the scores and once for the outputs.
 */
int attnres_block_phase1(const void *const *blocks, int n_blocks, int64_t B, int64_t T, int64_t D,
                         int dtype, const float *queries, const float *gains, int S, float eps,
                         void *out, float *out_max, float *out_lse, void *stream);

/*
 * Phase 2 of the two-phase Block scheme (intra step): merge the running
 * intra-block partial p, as a single source with state (s_p, p, 1)
 * ("single_source_stats"), into the phase-1 state of this sublayer's
 * query by eq. OS2, then normalise:
 *   M = max(lse, s_p),  h = (e^{lse-M} o + e^{s_p-M} p) / (e^{lse-M} + e^{s_p-M}).
 *   inter_out  device [B,T,D]: phase-1 output o of this sublayer's query
 *   inter_lse  device fp32 [B,T]: its lse
 *   partial    device [B,T,D], or NULL for the first sublayer of a block,
 *              in which case h = o (and out_lse = inter_lse)
 *   query, gain  as in attnres_depth_aggregate (the same query phase 1 used)
 *   h_out      device [B,T,D]; may not alias inter_out or partial
 *   out_lse    device fp32 [B,T], optional: the merged lse
 */
int attnres_block_phase2_merge(const void *inter_out, const float *inter_lse, const void *partial,
                               int64_t B, int64_t T, int64_t D, int dtype, const float *query,
                               const float *gain, float eps, void *h_out, float *out_lse,
                               void *stream);

/*
 * Backward of the depth aggregation (eq. A1-A3 of "Attention Residual 深度残差"
 * in reverse: the operator's forward/backward by recomputation that
 * "Attention Residuals：当网络深度也拥有寻址能力" describes in sections "Depth
 * attention 与 online merge reference" and "公开实现边界").  For the upstream
 * gradient dh of h = attnres_depth_aggregate(sources, query, gain, eps), per
 * token row, with r_i = (mean_d v_i^2 + eps)^(-1/2), s_i = r_i (w~ . v_i),
 * alpha = softmax(s) and ds_i = alpha_i (dh . v_i - sum_j alpha_j dh . v_j):
 *   grad_sources[i] (=, or += with accumulate = 1)
 *             alpha_i dh + ds_i r_i w~ - (ds_i s_i r_i^2 / D) v_i
 *   grad_query = dw~ (.) gain,  grad_gain = dw~ (.) query,
 *   dw~ = sum over all rows and sources of ds_i r_i v_i.
 * The softmax is recomputed from the sources; nothing from the forward is
 * needed.  fp32 arithmetic; grad_sources in the source dtype, rounded once.
 *   sources, n, B, T, D, dtype, query, gain, eps: as attnres_depth_aggregate
 *   grad_out     device [B,T,D] dh (source dtype)
 *   grad_sources host array of n device pointers [B,T,D]; must not alias the
 *                sources or grad_out
 *   accumulate   0: overwrite grad_sources; 1: add to them
 *   grad_query   device fp32 [D] or NULL;  grad_gain  device fp32 [D] or NULL
 *                (with gain == NULL the gain is one and grad_gain = dw~ (.) query)
 *   workspace    device fp32 [workspace_rows, D], caller-owned scratch for
 *                the per-CTA partial sums of dw~; required when grad_query or
 *                grad_gain is given, else unused (may be NULL).  Fewer rows than
 *                attnres_depth_aggregate_backward_workspace_rows() reports run
 *                fewer CTAs (at least 1 and 8 for narrow rows: ATTNRES_ERR_CAPACITY
 *                below that).  Its contents on entry do not matter.
 * The sum over rows runs in a fixed order: results are reproducible for
 * the same inputs and workspace_rows on the same device.
 * B*T == 0: grad_query / grad_gain are set to zero, nothing else is touched.
 * D limits: as attnres_depth_aggregate (up to 1024 16-byte vectors per row).
 */
int attnres_depth_aggregate_backward(const void *const *sources, int n, int64_t B, int64_t T, int64_t D,
                                     int dtype, const float *query, const float *gain, float eps,
                                     const void *grad_out, void *const *grad_sources, int accumulate,
                                     float *grad_query, float *grad_gain, float *workspace,
                                     int64_t workspace_rows, void *stream);

/*
 * attnres_depth_aggregate_backward without a workspace argument: the same
 * gradients (same arguments minus workspace / workspace_rows), for callers
 * that cannot allocate device memory -- for example a host program whose
 * device memory is all handed out by its own pool, or a real-time loop that
 * may not stall on the implicit synchronisation of cudaMalloc / cudaFree.
 * The pages have no counterpart of this call; it exists only for them.
 *   Scratch: the per-CTA partial sums of the query gradient live in one
 *   fixed 8 MiB device array inside this library (2^21 floats; every GPU
 *   that loads the library holds it until the process exits).  A call uses
 *   floor(2^21 / D) partial rows of it; a request whose D needs more rows
 *   than that (more than 2^18 features for rows owned by one CTA, 2^18 / 8
 *   for narrow rows) is refused with ATTNRES_ERR_SCRATCH.  Every supported
 *   D fits.  Nothing in the array has to start at zero: each partial row a
 *   call sums is written earlier in the same call.
 *   Set-up: the first call on a device that needs the scratch (token rows
 *   and a query or gain gradient) looks up the array's device address, with
 *   that device current, and caches it; make that first call before any
 *   stream capture.  A cudaDeviceReset unloads the library's device code:
 *   the cached address is then stale, so do not call this entry point on a
 *   device after resetting it.  All other arguments are checked before the
 *   lookup, as in attnres_depth_aggregate_backward.
 *   Calls share the array: two calls whose kernels overlap on the GPU (other
 *   streams, other host threads) race on it and give wrong query and gain
 *   gradients.  Calls in one stream are ordered and safe.
 * Nothing here allocates: no cudaMalloc, no cudaFree, no allocating library
 * routine.  Same status codes as attnres_depth_aggregate_backward, plus
 * ATTNRES_ERR_SCRATCH.
 */
int attnres_depth_aggregate_backward_noalloc(const void *const *sources, int n, int64_t B, int64_t T,
                                             int64_t D, int dtype, const float *query, const float *gain,
                                             float eps, const void *grad_out, void *const *grad_sources,
                                             int accumulate, float *grad_query, float *grad_gain,
                                             void *stream);

/*
 * Workspace rows with which attnres_depth_aggregate_backward fills the
 * current device (resident CTAs x SMs x rows per CTA) for this D and dtype;
 * a negative status on a bad argument or CUDA error.  Host-only query.
 */
int64_t attnres_depth_aggregate_backward_workspace_rows(int64_t D, int dtype);

/*
 * Running intra-block partial update ("forward_naive": partial = out, or
 * partial + out) with the benchmark recipes' synthetic sublayer
 * f(h) = 0.5 * tanh(u (.) h) standing in for the model's attention / FFN:
 *   partial_out = (partial_in ? partial_in : 0) + 0.5 * tanh(u (.) h)
 * computed in fp32 and rounded once.
 *   h          device [B,T,D] (the sublayer input)
 *   partial_in device [B,T,D] or NULL (first sublayer of a block)
 *   u          device fp32 [D]
 *   partial_out device [B,T,D]; may alias partial_in (in-place update)
 */
int attnres_partial_update(const void *h, const void *partial_in, const float *u, int64_t B,
                           int64_t T, int64_t D, int dtype, void *partial_out, void *stream);

/*
 * Fused intra-block step: the partial-sum update of sublayer k-1 and the
 * phase-2 merge of sublayer k in one pass (the decode-path fusion of
 * "intra-block merge + partial-sum update" described for K3 in
 * "Attention Residuals：当网络深度也拥有寻址能力", section "Kimi Linear 与 K3
 * 中的接入"):
 *   out_{k-1} = sub_out                        (u == NULL: the sublayer output)
 *             = 0.5 * tanh(u (.) sub_out)      (u != NULL: sub_out is h_{k-1},
 *                                               synthetic sublayer)
 *   p_{k-1}   = (partial_in ? partial_in : 0) + out_{k-1}, rounded once,
 *               written to partial_out
 *   h_k       = attnres_block_phase2_merge(inter_out, inter_lse, p_{k-1}, ...)
 * Per token it reads 3 rows and writes 2; the separate update and merge move 6.
 *   inter_out, inter_lse, query, gain, eps, out_lse: as attnres_block_phase2_merge
 *   partial_in  device [B,T,D] or NULL;  sub_out  device [B,T,D];  u  fp32 [D] or NULL
 *   partial_out device [B,T,D]: may alias partial_in
 *   h_out       device [B,T,D] or NULL (then normed_out is required): may
 *               alias sub_out (not inter_out)
 * Optional pre-norm of the next sublayer, fused ("Depth attention 与 online
 * merge reference": the optional fused output RMSNorm; the K3 decode path
 * fuses it with the merge and the partial update):
 *   normed_out = h_k / sqrt(mean_d h_k^2 + norm_eps) (.) norm_weight,
 * formed from the unrounded fp32 h_k and rounded once.
 *   norm_weight device fp32 [D] or NULL;  norm_eps finite, >= 0
 *   normed_out  device [B,T,D] or NULL; NULL exactly when norm_weight is NULL;
 *               may alias sub_out (not inter_out, not h_out)
 */
int attnres_block_merge_update(const void *inter_out, const float *inter_lse, const void *partial_in,
                               const void *sub_out, const float *u, int64_t B, int64_t T, int64_t D,
                               int dtype, const float *query, const float *gain, float eps,
                               void *partial_out, void *h_out, float *out_lse,
                               const float *norm_weight, float norm_eps, void *normed_out,
                               void *stream);

/*
 * The sublayer pre-norm as a pass of its own (for the first sublayer of a
 * block, whose input h_1 is the phase-1 output; same definition as the fused
 * form above):
 *   y = x / sqrt(mean_d x^2 + eps) (.) weight,   row by row, fp32, rounded once.
 *   x       device [B,T,D];  weight device fp32 [D];  eps finite, >= 0
 *   y       device [B,T,D]; may alias x
 * Same D limits as attnres_block_phase2_merge.
 */
int attnres_rms_norm(const void *x, int64_t B, int64_t T, int64_t D, int dtype, const float *weight,
                     float eps, void *y, void *stream);

/*
 * Full AttnRes stack forward ("FullAttnResStack", eq. A1-A4) with the
 * synthetic sublayer f_l(h) = 0.5 * tanh(u_l (.) h):
 *   for l = 1..L:  h_l = aggregate(v_0..v_{l-1}; query_l, gain_l)
 *                  v_l = f_l(h_l)            (written to sources[l])
 *   y = aggregate(v_0..v_L; query_L, gain_L)  (the final aggregate)
 * h_l never leaves the kernel: f_l is applied in its epilogue to the fp32
 * h_l, and only v_l is rounded and stored.
 *   sources  host array of L+1 device pointers [B,T,D]: sources[0] = v_0 is
 *            read, sources[1..L] are written
 *   L        1 .. ATTNRES_MAX_SOURCES - 1
 *   queries  device fp32 [L+1, D] (row l-1 for sublayer l, row L final)
 *   gains    device fp32 [L+1, D] or NULL;  u  device fp32 [L, D]
 *   y_out    device [B,T,D]
 */
int attnres_full_stack_forward(void *const *sources, int L, int64_t B, int64_t T, int64_t D,
                               int dtype, const float *queries, const float *gains, const float *u,
                               float eps, void *y_out, void *stream);

/*
 * The same Full stack with the two-phase schedule of block size S (Full
 * AttnRes run two-phase when a schedule block size is given: the remark
 * under "_run_block_two_phase" in "Attention Residual 深度残差", and the (S+N)d
 * residual I/O of "推理：block representations 像一份 depth KV cache" in
 * "Attention Residuals：当网络深度也拥有寻址能力").  For each block of
 * sublayers l = start+1 .. min(start+S, L):
 *   phase 1: the block's queries over v_0 .. v_start in one pass (the
 *            normalised output o_l and lse_l of every sublayer of the block);
 *   phase 2: in order, h_l = o_l's state merged online with the intra-block
 *            sources v_{start+1} .. v_{l-1}; v_l = f_l(h_l) (fused, as above).
 * Then y as above.  The same result as attnres_full_stack_forward up to
 * rounding: o_l is stored in the source dtype (lse fp32) in between.
 *   sources, L, B, T, D, dtype, queries, gains, u, eps, y_out: as above
 *   S          1 .. ATTNRES_MAX_QUERIES
 *   workspace  device, 256-byte aligned, at least
 *              attnres_full_stack_two_phase_workspace_bytes() bytes (the
 *              phase-1 outputs of one block and, for blocks past ten
 *              sources, their scores); contents on entry do not matter
 * Blocks with up to ten sources use the phase-1 kernels of
 * attnres_block_phase1; wider ones need bf16, D a multiple of 64 up to
 * 2048, and at least 48 phase-1 output rows (the block's sublayers x B x T
 * >= 48: the split queries are kept in the last 48 of them); else
 * ATTNRES_ERR_SHAPE, checked before anything runs.
 */
int attnres_full_stack_two_phase(void *const *sources, int L, int S, int64_t B, int64_t T, int64_t D,
                                 int dtype, const float *queries, const float *gains, const float *u,
                                 float eps, void *y_out, void *workspace, int64_t workspace_bytes,
                                 void *stream);

/* Workspace bytes attnres_full_stack_two_phase needs (negative status on bad shapes). */
int64_t attnres_full_stack_two_phase_workspace_bytes(int L, int S, int64_t B, int64_t T, int64_t D, int dtype);

/*
 * Host-only bookkeeping ("BlockAttnResStack.forward_naive"): the sources each
 * atomic sublayer attends over, for num_atomic sublayers in blocks of
 * block_size.  Block 0 is the embedding; a block boundary falls after
 * sublayer idx (1-based) when idx % block_size == 0 or idx == num_atomic,
 * and the partial sum then becomes a new block.  The first sublayer of a
 * block sees only the completed blocks; later ones also see the partial.
 *   n_sources_per_layer  host int [num_atomic + 1]; the last entry is the
 *                        final aggregate over all blocks
 *   source_ids           host int [capacity], flat: block id >= 0, or -1
 *                        for the running partial
 * Returns the number of ids written (>= 0), ATTNRES_ERR_CAPACITY if
 * `capacity` is too small, ATTNRES_ERR_SHAPE / _VALUE / _NULL on bad input.
 */
int attnres_block_schedule(int num_atomic, int block_size, int *n_sources_per_layer,
                           int *source_ids, int capacity);

/*
 * Config helper ("atomic_block_size"): the block size in DecoderBlocks of
 * the config, converted to atomic sublayers (x2: attention + FFN).
 * attnres_block_size < 0 means "unset": about eight blocks,
 * max(1, ceil(num_hidden_layers / 8)) DecoderBlocks each.  A block size of
 * 0 is invalid (ATTNRES_ERR_VALUE); num_hidden_layers < 1 is
 * ATTNRES_ERR_SHAPE.
 */
int attnres_atomic_block_size(int num_hidden_layers, int attnres_block_size);

/*
 * Kernels that wait on in-kernel events (bulk-copy and tensor-core
 * completion) bound every wait.  A wait that runs out records a device-side
 * flag; the part of the CTA that waited stops issuing work, every part
 * waits (bounded again) for the copies and tensor-core operations it still
 * has in flight, and the CTA ends: the kernel never hangs and leaves nothing
 * running, but its results are invalid.  While the flag is set, later
 * launches of those kernels skip their work, so every result of the calls
 * that use them stays invalid until the error is taken.
 * This call synchronises the current device, reads and clears those flags,
 * and returns ATTNRES_ERR_TIMEOUT if any was set since the previous call
 * (ATTNRES_ERR_CUDA if the device reports an error), else ATTNRES_OK.
 */
int attnres_take_device_error(void);

/*
 * Diagnostics: the limit of those in-kernel waits, in SM clock cycles, for
 * launches made after this call (process-wide; 0 restores the default of
 * 4e9 cycles, about 2 s).  A very short limit makes waits run out on
 * purpose, which exercises the give-up path above without a GPU fault.
 * The final drain of a CTA's own operations in flight always keeps the
 * default limit.  cycles < 0: ATTNRES_ERR_VALUE.
 */
int attnres_set_wait_limit(int64_t cycles);

/* Static, human-readable name of a status code. */
const char *attnres_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* ATTNRES_H */
