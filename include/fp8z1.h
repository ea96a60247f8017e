/*
 * fp8z1.h -- C ABI of libfp8z1.so: the ZeRO-1 optimizer step for
 * blockwise-FP8 weights, on one data-parallel rank's shard, on one GB300
 * (sm_103a).
 *
 * Method: "面向 Blockwise FP8 量化的 ZeRO 优化器设计" (A ZeRO Optimizer Design
 * for Blockwise FP8 Quantization):
 *   §Blockwise 量化         one FP32 scale per 128x128 block of a weight;
 *   §块粒度切分             pad each quantised dim to a multiple of 128, keep a
 *                           block lookup table, shard on block edges;
 *   §参数布局变换           fold / unfold between row-major [E,R,C] and a
 *                           128x128-block-contiguous 1-D buffer;
 *   §总结                   fold grads -> slice -> elementwise update ->
 *                           quantise FP8 + scales from the FP32 master -> unfold.
 * Step order, clipping and loss scaling: "DeepSpeed ZeRO 优化" §三 (global
 * norm -> loss-scale update -> unscale+clip -> update -> low-precision copy),
 * §六 Loss Scaling, §七 梯度裁剪.
 *
 * Conventions (all entry points):
 *   - A block is 128 x 128 = 16384 elements (FP8Z1_BLOCK_ELEMS).  Blocks are
 *     numbered over the params in the order given to fp8z1_build_layout, and
 *     inside a param [E,R,C] in (e, row block, col block) row-major order.
 *   - A shard is a block range [b0, b1).  Every *_shard pointer points at
 *     block b0 of its buffer and holds (b1 - b0) * 16384 elements
 *     (scale_shard: b1 - b0 floats).  Shard pointers must be 16-byte aligned.
 *   - The caller owns every device buffer it passes; the library owns only the
 *     layout (host tables; on the device the block lookup table, a table of
 *     16384-element runs of each param for the norm, and a small norm
 *     workspace).
 *   - Calls that take a `stream` (a cudaStream_t; NULL = legacy default
 *     stream) only enqueue work on it and never synchronise.  Asynchronous
 *     device faults surface at the caller's next synchronisation, as in CUDA.
 *   - Every call returns FP8Z1_OK (0) or a negative status; arguments are
 *     checked on the host before anything is enqueued, and a rejected call
 *     enqueues nothing.  No exception crosses the ABI; nothing aborts.
 *   - Floating point: IEEE FP32 for the update (explicit fused multiply-adds,
 *     correctly rounded division and square root), double for the norm scalars.
 */
#ifndef FP8Z1_H
#define FP8Z1_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define FP8Z1_TILE 128
#define FP8Z1_BLOCK_ELEMS 16384
#define FP8Z1_MX_GROUP 32

/* status codes */
#define FP8Z1_OK 0
#define FP8Z1_EINVAL (-1) /* bad argument: null, bad range/shape/elem_size, hp out of domain */
#define FP8Z1_EALIGN (-2) /* a pointer is not aligned as required */
#define FP8Z1_ENOMEM (-3) /* host or device allocation failed */
#define FP8Z1_ECUDA (-4)  /* a CUDA runtime call or kernel launch failed */
#define FP8Z1_ENODEV (-5) /* the layout was built host-only and has no device tables */

/* fp8z1_build_layout flags */
#define FP8Z1_LAYOUT_HOST_ONLY 1u /* build the tables on the host only (no CUDA call) */

typedef struct fp8z1_layout fp8z1_layout; /* opaque, owned by the library */

/* Shape of one quantised param: row-major [E, R, C]; a 2-D weight has E = 1.
 * E, R, C >= 1 and C < 2^31. */
typedef struct {
    int64_t E, R, C;
} fp8z1_shape;

/* One entry of the block lookup table (32 bytes):
 * §块粒度切分 -- the table that maps a flat block index to its param and its
 * real (unpadded) extent, so the 1-D buffers can be walked param by param. */
typedef struct {
    int64_t src_offset; /* element offset of the block's (0,0) element in its
                           param's row-major storage: (e*R + 128*rb)*C + 128*cb */
    int32_t param;      /* index into the shape list */
    int32_t expert;     /* e */
    int32_t row_block;  /* rb */
    int32_t col_block;  /* cb */
    int32_t ld;         /* row stride of the param in elements (= C) */
    int16_t rows_real;  /* min(128, R - 128*rb) */
    int16_t cols_real;  /* min(128, C - 128*cb) */
} fp8z1_block;

/* AdamW + clipping + loss-scale hyper-parameters of one step (read on the
 * host at call time).  The pages fix none of the AdamW details; the reading
 * is decoupled weight decay with bias correction:
 *   g = g_s / loss_scale, then g *= clip_coef when clip_coef < 1,
 *   clip_coef = max_norm / (||g_s|| / loss_scale + 1e-6)        (§七)
 *   m = beta1 m + (1-beta1) g;   v = beta2 v + (1-beta2) g^2
 *   p = p (1 - lr wd) - lr * (m / (1-beta1^t)) / (sqrt(v / (1-beta2^t)) + eps)
 * Domain: lr >= 0, 0 <= beta1, beta2 < 1, eps > 0, weight_decay >= 0,
 * max_norm > 0 (+inf disables clipping), loss_scale > 0 and finite (a power of
 * two makes g_s * (clip / loss_scale) bit-identical to unscale-then-clip),
 * step = t >= 1 (the 1-based index of the step being taken). */
typedef struct {
    float lr, beta1, beta2, eps, weight_decay, max_norm, loss_scale;
    int64_t step;
} fp8z1_adamw_hp;

/* Dynamic loss scaling state, updated on the host after each step (§六). */
typedef struct {
    float scale;             /* S, > 0 */
    int64_t step;            /* completed (not skipped) steps t */
    int32_t good_steps;      /* clean steps since S last changed */
    int32_t growth_interval; /* N >= 1: S doubles after N clean steps in a row */
} fp8z1_loss_scaler;

/* ---- layout (§块粒度切分, §参数布局变换) ------------------------------------ */

/* Build the block LUT and the shard ranges of `n_params` params for DP size
 * `dp_size`, and (unless FP8Z1_LAYOUT_HOST_ONLY) upload the LUT to the current
 * CUDA device with synchronous copies.  Shard of rank r: S = ceil(nblk / D)
 * blocks, [r*S, min((r+1)*S, nblk)) (the last ranks may be short or empty).
 * `shapes`: host array of n_params >= 1 shapes; dp_size >= 1.
 * On success *out receives a layout that fp8z1_destroy_layout frees.
 * Errors: EINVAL (null, n_params < 1, dp_size < 1, a dim < 1, C >= 2^31, an
 * element count that overflows int64), ENOMEM, ECUDA. */
int fp8z1_build_layout(const fp8z1_shape* shapes, int32_t n_params, int32_t dp_size,
                       uint32_t flags, fp8z1_layout** out);

/* Free a layout and its device tables (NULL is accepted).  Call only when no
 * work that uses it is still running on the device. */
int fp8z1_destroy_layout(fp8z1_layout* layout);

/* Totals: blocks, padded elements (= blocks * 16384) and real elements. */
int fp8z1_layout_info(const fp8z1_layout* layout, int64_t* n_blocks, int64_t* n_elems_padded,
                      int64_t* n_elems_real);

/* Block range [*b0, *b1) of DP rank `rank` (0 <= rank < dp_size). */
int fp8z1_shard_range(const fp8z1_layout* layout, int32_t rank, int64_t* b0, int64_t* b1);

/* Copy the LUT (n_blocks entries) to host memory; `capacity` is the number
 * of entries `host_dst` holds (EINVAL when too small). */
int fp8z1_copy_lut(const fp8z1_layout* layout, fp8z1_block* host_dst, int64_t capacity);

/* Where one param's blocks sit in the flat block order, and so where its
 * scales sit in the scale buffer (§总结: the 1-D blockwise scales unfolded
 * back into each param's 2-D / 3-D scales).  Block (e, rb, cb) of the param
 * is global block first_block + (e * row_blocks + rb) * col_blocks + cb, so
 * scales[first_block .. + experts * row_blocks * col_blocks) is the param's
 * [E, ceil(R/128), ceil(C/128)] scale tensor, row-major, with no copy. */
typedef struct {
    int64_t first_block; /* global index of block (0, 0, 0) of the param */
    int64_t experts;     /* E */
    int64_t row_blocks;  /* ceil(R / 128) */
    int64_t col_blocks;  /* ceil(C / 128) */
    int64_t e_begin;     /* experts [e_begin, e_end) have every block inside */
    int64_t e_end;       /* the range [b0, b1) asked about; equal when none */
} fp8z1_param_grid;

/* Fill *out for param `param` (0 <= param < n_params) and the block range
 * [b0, b1) (0 <= b0 <= b1 <= n_blocks), e.g. a rank's shard: a shard's scale
 * buffer, which starts at block b0, then holds experts [e_begin, e_end) of
 * the param as the [e_end - e_begin, row_blocks, col_blocks] stretch at
 * first_block + e_begin * row_blocks * col_blocks - b0.  Host only; works on
 * host-only layouts.  Errors: EINVAL (null, param or range out of bounds). */
int fp8z1_param_blocks(const fp8z1_layout* layout, int32_t param, int64_t b0, int64_t b1,
                       fp8z1_param_grid* out);

/* Read and clear the layout's device status word (synchronous; waits for the
 * copy).  Bit 1 (FP8Z1_DEVSTATUS_BADPTR): a fold, unfold, fused norm or
 * fused step met a param pointer in its device pointer array that was null or
 * not element aligned, and skipped the blocks of that param (the norm also
 * sets found_inf, so the step is skipped).  0 means no such event since the
 * last read.
 * Errors: EINVAL, ENODEV, ECUDA. */
#define FP8Z1_DEVSTATUS_BADPTR 1u
int fp8z1_device_status(const fp8z1_layout* layout, uint32_t* bits);

/* ---- fold / unfold (§参数布局变换) ----------------------------------------- */

/* fold: for every block k in [b0, b1) and (r, c) in 128 x 128,
 *   dst_shard[(k - b0)*16384 + r*128 + c] = param[e][128*rb + r][128*cb + c]
 * when the element is real, else 0 (the padding of §块粒度切分).
 * `d_src_params`: DEVICE array of n_params DEVICE pointers, each to a
 * row-major [E,R,C] param of `elem_size` bytes per element (1, 2 or 4), aligned
 * to elem_size.  The copy is bitwise.  `dst_shard`: device, 16-byte aligned.
 * An empty range (b0 == b1) enqueues nothing.
 * Errors: EINVAL (null, elem_size, b0 > b1, b1 > n_blocks), EALIGN, ENODEV, ECUDA. */
int fp8z1_fold(const fp8z1_layout* layout, const void* const* d_src_params, void* dst_shard,
               int32_t elem_size, int64_t b0, int64_t b1, void* stream);

/* unfold: the inverse of fold over the real elements of blocks [b0, b1):
 * param[e][128*rb + r][128*cb + c] = src_shard[(k - b0)*16384 + r*128 + c].
 * Padding is dropped; no element outside those blocks is written.
 * `d_dst_params`: DEVICE array of n_params DEVICE pointers. */
int fp8z1_unfold(const fp8z1_layout* layout, const void* src_shard, void* const* d_dst_params,
                 int32_t elem_size, int64_t b0, int64_t b1, void* stream);

/* ---- global grad norm ("DeepSpeed ZeRO 优化" §七, §六) --------------------- */

/* Add the sum of squares of the FP32 loss-scaled grads of blocks [b0, b1) to
 * *d_sumsq (device double; the caller zeroes it once per step and may then
 * call this for several ranges, which stands in for the all-reduce of the
 * per-rank partial sums), and OR 1 into *d_found_inf (device int32) when any
 * of those grads is inf or nan.  Squares are formed exactly and summed in
 * compensated single precision, then in double: the result is within about
 * 1e-13 relative of the exact sum.  With found_inf set the sum is not
 * meaningful.  Deterministic for a given device and range.
 * The reduction uses a workspace owned by the layout: calls that share a
 * layout must not overlap on the device (issue them on one stream).
 * Errors: EINVAL, EALIGN, ENODEV, ECUDA. */
int fp8z1_grad_norm(const fp8z1_layout* layout, const float* grad_shard, int64_t b0, int64_t b1,
                    double* d_sumsq, int32_t* d_found_inf, void* stream);

/* Clear a norm accumulator pair before a step: *d_sumsq = 0.0 and
 * *d_found_inf = 0, as two memsets enqueued on `stream` (no kernel; capturable).
 * Pointers: device; d_sumsq 8-byte aligned, d_found_inf 4-byte aligned.
 * Errors: EINVAL (null), EALIGN, ECUDA. */
int fp8z1_norm_reset(double* d_sumsq, int32_t* d_found_inf, void* stream);

/* ---- grad norm without any allocation ------------------------------------ */

/* The pages have no counterpart to this call: it serves callers that cannot
 * call cudaMalloc at all -- a framework whose caching allocator already owns
 * the device memory (a foreign cudaMalloc can fail or make the CUDA driver
 * synchronise the device), or a step loop that must never block on an
 * allocation.  It computes what fp8z1_grad_norm computes, for the
 * `n_blocks` blocks at `grad_shard` (pointing at block b0 of the grad buffer;
 * n_blocks = b1 - b0), with the same kernel and the same accuracy; the
 * summation is split differently, so the two results agree to about 1e-13
 * relative, not bit for bit.  It needs no layout and allocates nothing: its
 * workspace is a static device array of 4097 doubles (about 32 KB) that every
 * device loading the library holds until the process exits.  It runs the
 * same persistent grid as fp8z1_grad_norm (three CTAs per SM, at most one
 * per half block), one workspace slot per CTA.
 *   - At most FP8Z1_NOALLOC_MAX_BLOCKS blocks per call (EINVAL beyond that);
 *     split a larger range into several calls, which accumulate.
 *   - The first call on each device looks up the workspace address and the
 *     SM count on the host (cudaGetSymbolAddress, with that device current);
 *     make that first call before any stream capture.  The lookup is tied
 *     to the device's CUDA context: after a device reset (cudaDeviceReset)
 *     the next call looks the address up again, so it too must come before
 *     any capture.
 *   - Every call shares the one workspace, and a call leaves its contents
 *     behind; the call clears the part that must start at zero on its
 *     stream.  Calls that overlap on the device race: issue them on one
 *     stream or otherwise order them.
 * Errors: EINVAL (null, n_blocks < 0 or > FP8Z1_NOALLOC_MAX_BLOCKS), EALIGN,
 * ECUDA. */
#define FP8Z1_NOALLOC_MAX_BLOCKS 262144
int fp8z1_grad_norm_noalloc(const float* grad_shard, int64_t n_blocks, double* d_sumsq,
                            int32_t* d_found_inf, void* stream);

/* ---- fused step (§总结; "DeepSpeed ZeRO 优化" §三, §七) -------------------- */

/* One optimizer step over blocks [b0, b1) of the shard, in one HBM pass:
 * reads *d_sumsq (global) to form clip_coef on the device, unscales and clips
 * the grads, applies AdamW to master/m/v in place, and for every block writes
 * scale = amax|p_new| / 448 (1.0 when amax == 0) to scale_shard[k - b0] and
 * the E4M3 codes of p_new / scale (round to nearest even, finite overflow
 * saturates to +-448, sign kept) to fp8_shard.  When *d_found_inf != 0 the
 * kernel writes nothing (the skipped step of §六): every buffer stays
 * bit-identical.  `grad_shard` is not modified.
 * Padding: the elements of a block outside its real rows and columns must be
 * zero in grad_shard, master, m and v, as fp8z1_fold writes them.  The update
 * maps zero to zero there (g = 0 gives m = v = +0 and p = +0), so the step
 * neither reads nor writes the padding of those four buffers; fp8_shard gets
 * code 0x00 in its padding.
 * Pointers: device; grad/master/m/v/fp8 16-byte aligned, scale 4-byte aligned.
 * Errors: EINVAL (null, range, hp out of domain), EALIGN, ENODEV, ECUDA. */
int fp8z1_step(const fp8z1_layout* layout, const fp8z1_adamw_hp* hp, const float* grad_shard,
               float* master_shard, float* m_shard, float* v_shard, uint8_t* fp8_shard,
               float* scale_shard, int64_t b0, int64_t b1, const double* d_sumsq,
               const int32_t* d_found_inf, void* stream);

/* ---- fused forms: the same results in fewer HBM passes --------------------- */

/* Fold of the FP32 grads fused with the grad norm (§参数布局变换, §总结;
 * "DeepSpeed ZeRO 优化" §七): reads the real grads of blocks [b0, b1) from the
 * row-major params, adds their sum of squares to *d_sumsq and ORs inf/nan into
 * *d_found_inf -- as fp8z1_grad_norm does on the folded range -- and, when
 * `grad_shard` is not NULL, also stores the folded blocks there (as
 * fp8z1_fold with elem_size 4).  With grad_shard NULL nothing is folded: the
 * norm is taken straight from the row-major grads, for fp8z1_step_fused to
 * read them the same way.  `d_grad_params`: DEVICE array of n_params DEVICE
 * pointers to FP32 row-major params (4-byte aligned).  A null or misaligned
 * entry sets FP8Z1_DEVSTATUS_BADPTR and *d_found_inf (so the step is skipped).
 * Without the store the sum needs no block structure: the params the range
 * holds whole, and the whole row-block strips of a param it cuts, are read as
 * flat runs of their row-major elements; only partial strips go block by
 * block.  The call then enqueues one launch per piece (whole params, a span,
 * partial strips), each adding its total to *d_sumsq.  The result is
 * deterministic for a given device and range, and within about 1e-13 of the
 * exact sum (the summation order differs from fp8z1_grad_norm's, so the two
 * agree to that, not bit for bit).  It uses the layout's norm workspace, so
 * calls sharing a layout must not overlap on the device.
 * Errors: EINVAL, EALIGN, ENODEV, ECUDA, ENOMEM. */
int fp8z1_fold_norm(const fp8z1_layout* layout, const float* const* d_grad_params, float* grad_shard,
                    int64_t b0, int64_t b1, double* d_sumsq, int32_t* d_found_inf, void* stream);

/* fp8z1_step with the grad fold and the code unfold fused in (§总结: fold
 * grads ... update ... quantise ... unfold params).  Grads come from exactly
 * one of `grad_shard` (folded, as fp8z1_step) or `d_grad_params` (DEVICE
 * array of DEVICE pointers to the row-major FP32 grads, read through the
 * block lookup table).  Codes go to `fp8_shard` (folded, 16-byte aligned)
 * and/or `d_fp8_params` (DEVICE array of DEVICE pointers to the row-major
 * uint8 FP8 params, written on their real elements only: the fused unfold).
 * Master / m / v / scales and every numerical result are those of
 * fp8z1_step, and so is the padding contract (padding of master / m / v,
 * and of grad_shard when given, zero and neither read nor written).  A null
 * grad or FP8 param pointer (or a grad pointer that is not
 * 4-byte aligned) leaves that block untouched and sets
 * FP8Z1_DEVSTATUS_BADPTR.  The row-major grads may be read through the
 * read-only data path: nothing may write them while the step runs.
 * Quantisation monitors ("FP8训练技术与万亿参数模型优化实践" §1.2: underflow =
 * zeros / total, healthy below 0.5%; distortion = cosine(original,
 * dequantised), healthy above 0.995): when `block_cos` and
 * `block_underflow` (device, b1 - b0 entries each, both or neither) are given,
 * the kernel also writes per block the cosine between the new FP32 master
 * and its dequantised FP8 value (decode(code) * scale; 1 when both are all
 * zero) and the count of non-zero masters whose code decodes to 0 -- divide
 * by the block's real elements (rows_real * cols_real of the LUT) for the
 * fraction.  FP32 sums: a diagnostic, within about 1e-5 of exact.
 * Errors: EINVAL (both or neither grad source, no code destination, one of
 * the two monitor outputs, ...), EALIGN, ENODEV, ECUDA. */
int fp8z1_step_fused(const fp8z1_layout* layout, const fp8z1_adamw_hp* hp, const float* grad_shard,
                     const float* const* d_grad_params, float* master_shard, float* m_shard,
                     float* v_shard, uint8_t* fp8_shard, uint8_t* const* d_fp8_params,
                     float* scale_shard, float* block_cos, uint32_t* block_underflow, int64_t b0,
                     int64_t b1, const double* d_sumsq, const int32_t* d_found_inf, void* stream);

/* ---- re-targeting a captured step (CUDA graphs, scalars by value) ----------- */

/* The step kernels of this library that take their scalars by value
 * (those of fp8z1_step and fp8z1_step_fused) inside a captured CUDA graph `graph` (a cudaGraph_t): up to
 * `capacity` node handles (cudaGraphNode_t) go to `nodes`, their count to
 * *n_nodes.  Host only; EINVAL when there are more than `capacity` (n_nodes
 * then holds the count), ECUDA when the graph cannot be read. */
int fp8z1_graph_step_nodes(void* graph, void** nodes, int32_t capacity, int32_t* n_nodes);

/* Rewrite the per-step scalars (t, S and the rest, from *hp, formed as
 * fp8z1_step forms them) of those nodes in the instantiated graph
 * `graph_exec` (a cudaGraphExec_t of `graph`): the next launches of the
 * graph run the step with *hp, at the speed of the by-value kernel; launches
 * already made are unaffected.  Each node's other arguments stay as
 * captured.  Host only; EINVAL (a node is not one of this library's step
 * kernels, hp out of domain), ECUDA. */
int fp8z1_graph_set_step_hp(void* graph_exec, void* const* nodes, int32_t n_nodes, const fp8z1_adamw_hp* hp);

/* ---- the step with two candidate hyper-parameter sets ------------------------ */

/* fp8z1_step_fused (without monitors) taking two hyper-parameter sets, both by
 * value: the kernel uses `hp_if_clear` when *d_select == 0 and `hp_if_set`
 * otherwise, reading *d_select (device, 4-byte aligned) when it runs.  With
 * d_select = the previous step's found_inf, a caller can enqueue a step
 * before it knows whether the previous one was skipped ("DeepSpeed ZeRO 优化"
 * §六): hp_if_clear holds t+1 and the loss scale after a clean step,
 * hp_if_set the t and halved scale after a skipped one.  The host need not
 * wait for each step to finish before enqueuing the next, and the results
 * are those of fp8z1_step_fused with the set picked.  Both sets ride as kernel
 * parameters, so the pick costs no registers.
 * Errors: as fp8z1_step_fused; EINVAL when either set is out of domain. */
int fp8z1_step_fused_select(const fp8z1_layout* layout, const fp8z1_adamw_hp* hp_if_clear,
                            const fp8z1_adamw_hp* hp_if_set, const int32_t* d_select, const float* grad_shard,
                            const float* const* d_grad_params, float* master_shard, float* m_shard,
                            float* v_shard, uint8_t* fp8_shard, uint8_t* const* d_fp8_params, float* scale_shard,
                            int64_t b0, int64_t b1, const double* d_sumsq, const int32_t* d_found_inf,
                            void* stream);

/* ---- the step with its scalars in device memory (for CUDA graphs) --------- */

/* The FP32 scalars one step uses, derived on the host in double from
 * fp8z1_adamw_hp and rounded once: beta1, beta2, 1 - beta1, 1 - beta2, eps,
 * lr / (1 - beta1^t), 1 / sqrt(1 - beta2^t), 1 - lr * wd, max_norm, S. */
typedef struct {
    float beta1, beta2, omb1, omb2, eps, step_size, inv_sqrt_bc2, decay, max_norm, loss_scale;
} fp8z1_step_scalars;

/* Fill *out from *hp (host only; EINVAL when hp is out of its domain). */
int fp8z1_step_scalars_from_hp(const fp8z1_adamw_hp* hp, fp8z1_step_scalars* out);

/* fp8z1_step_fused with the per-step scalars read from DEVICE memory
 * (`d_scalars`, 4-byte aligned) when the kernel runs, instead of passed by
 * value at launch.  When `h_scalars` is not NULL, the call first enqueues on
 * `stream` a copy of *h_scalars into *d_scalars.  Under CUDA stream capture
 * that copy becomes a graph node which reads *h_scalars at every replay.
 * `h_scalars` must then be page-locked host memory (cudaHostAlloc or
 * cudaHostRegister), and the caller writes the next step's scalars there
 * (fp8z1_step_scalars_from_hp) before each replay, once the previous replay's
 * copy has run.  t and S change every step, so this is what lets a captured
 * step replay correctly.  The scalars are not checked on the device.  Every
 * result is that of fp8z1_step_fused with the hp they were made from.
 * Errors: as fp8z1_step_fused; ECUDA when the copy cannot be enqueued. */
int fp8z1_step_fused_dev(const fp8z1_layout* layout, const fp8z1_step_scalars* h_scalars,
                         fp8z1_step_scalars* d_scalars, const float* grad_shard,
                         const float* const* d_grad_params, float* master_shard, float* m_shard, float* v_shard,
                         uint8_t* fp8_shard, uint8_t* const* d_fp8_params, float* scale_shard, float* block_cos,
                         uint32_t* block_underflow, int64_t b0, int64_t b1, const double* d_sumsq,
                         const int32_t* d_found_inf, void* stream);

/* ---- tracing (host only) --------------------------------------------------- */

/* The number of kernels this library has enqueued in this process, on every
 * device and stream, since it was loaded: the difference across a region of
 * calls is the launch count of that region.  A launch made while a stream is
 * being captured counts once, at capture; graph replays do not count.
 * Errors: EINVAL (null). */
int fp8z1_kernel_launches(uint64_t* out);

/* ---- checked builds --------------------------------------------------------
 * libfp8z1_checked.so is this library compiled with -DFP8Z1_CHECKED=1: every
 * load and store a kernel makes to a row-major param (fold and unfold, the
 * fused norm's grad reads, the fused step's grad reads and code writes) is
 * first tested against that param's extent, E * R * C elements; an access
 * outside is skipped and counted instead of made.  It is a debug build, for
 * running the parity tests without a device memory checker: slower, and
 * equal to the release build in every result while the count stays 0. */
#define FP8Z1_BUILD_CHECKED 1u

/* FP8Z1_BUILD_CHECKED for a checked build, else 0. */
int fp8z1_build_flags(void);

/* The accesses the checked kernels have skipped on the current device since
 * the library was loaded (synchronous: waits for the device).  0 in a release
 * build.  Errors: EINVAL (null), ECUDA. */
int fp8z1_checked_misses(uint64_t* count);

/* Test hook of a checked build: overwrite the device copy of block `block`'s
 * LUT entry (the host copy is kept), e.g. with an entry that points past its
 * param, to see the checks skip and count those accesses.  The layout stays
 * broken until destroyed.  Errors: EINVAL (release build, null, block out of
 * range), ENODEV, ECUDA. */
int fp8z1_checked_set_lut_entry(fp8z1_layout* layout, int64_t block, const fp8z1_block* entry);

/* ---- param-wise split (§参数粒度切分; host only) ---------------------------- */

/* The page's alternative to the block-wise split, for comparing padding
 * waste: params sorted by size E*R*C, largest first (equal sizes keep their
 * order), each given to the DP bucket with the fewest elements so far (lowest
 * index on a tie); every bucket is then padded to the largest.  Writes
 * owner[n_params] (the bucket of each param), bucket_elems[dp_size] (real
 * elements per bucket) and, if not NULL, *padded_total = dp_size * largest
 * bucket.  Host only; no CUDA call.  Errors: EINVAL. */
int fp8z1_paramwise_split(const fp8z1_shape* shapes, int32_t n_params, int32_t dp_size,
                          int32_t* owner, int64_t* bucket_elems, int64_t* padded_total);

/* ---- MXFP8 variant (§Blockwise 量化: MXFP8; OCP MX specification v1.0) ----- */

/* MXFP8 gives every run of 32 consecutive elements its own power-of-two
 * (E8M0) scale, so a block never straddles rows of a weight whose C is a
 * multiple of 32 and no fold is needed: the ZeRO shard is a flat run of the
 * params' row-major elements, cut on group edges (the page's point that MXFP8
 * blocks are memory-contiguous).  The MX layout holds the group count, the
 * shard ranges and a small norm workspace.  Every C must be a multiple of 32
 * (EINVAL otherwise).  Shard of rank r: S = ceil(n_groups / D) groups,
 * [r*S, min((r+1)*S, n_groups)).  Flags as fp8z1_build_layout. */
typedef struct fp8z1_mx_layout fp8z1_mx_layout;
int fp8z1_mx_build_layout(const fp8z1_shape* shapes, int32_t n_params, int32_t dp_size,
                          uint32_t flags, fp8z1_mx_layout** out);
int fp8z1_mx_destroy_layout(fp8z1_mx_layout* layout);
int fp8z1_mx_layout_info(const fp8z1_mx_layout* layout, int64_t* n_groups, int64_t* n_elems);
int fp8z1_mx_shard_range(const fp8z1_mx_layout* layout, int32_t rank, int64_t* g0, int64_t* g1);

/* fp8z1_grad_norm for a flat MX shard: adds the sum of squares of the
 * (g1 - g0) * 32 FP32 grads at `grad_shard` (device, 16-byte aligned, at
 * group g0) to *d_sumsq and ORs inf/nan into *d_found_inf; same reduction,
 * accuracy and workspace rule.  Errors: EINVAL, EALIGN, ENODEV, ECUDA. */
int fp8z1_mx_grad_norm(const fp8z1_mx_layout* layout, const float* grad_shard, int64_t g0, int64_t g1,
                       double* d_sumsq, int32_t* d_found_inf, void* stream);

/* The fused step on groups [g0, g1) of a flat MX shard: the unscale + clip +
 * AdamW of fp8z1_step (same FP32 operations, same skip on found_inf), then per
 * group of 32 the scale X = 2^(floor(log2 amax) - 8) clamped to
 * 2^-127 .. 2^127 (X = 1 when amax == 0), written to scale_shard[g - g0] as
 * the E8M0 code log2(X) + 127, and the codes E4M3(p / X), round to nearest
 * even, saturating at 448, written to fp8_shard.  Pointers at group g0;
 * grad/master/m/v/fp8 16-byte aligned.  Errors: EINVAL, EALIGN, ENODEV, ECUDA. */
int fp8z1_mx_step(const fp8z1_mx_layout* layout, const fp8z1_adamw_hp* hp, const float* grad_shard,
                  float* master_shard, float* m_shard, float* v_shard, uint8_t* fp8_shard,
                  uint8_t* scale_shard, int64_t g0, int64_t g1, const double* d_sumsq,
                  const int32_t* d_found_inf, void* stream);

/* fp8z1_mx_step with two candidate hyper-parameter sets, as
 * fp8z1_step_fused_select: `hp_if_clear` when *d_select == 0 (device, 4-byte
 * aligned, read when the kernel runs), `hp_if_set` otherwise.
 * Errors: as fp8z1_mx_step. */
int fp8z1_mx_step_select(const fp8z1_mx_layout* layout, const fp8z1_adamw_hp* hp_if_clear,
                         const fp8z1_adamw_hp* hp_if_set, const int32_t* d_select, const float* grad_shard,
                         float* master_shard, float* m_shard, float* v_shard, uint8_t* fp8_shard,
                         uint8_t* scale_shard, int64_t g0, int64_t g1, const double* d_sumsq,
                         const int32_t* d_found_inf, void* stream);

/* ---- loss scaling (host; "DeepSpeed ZeRO 优化" §六, §九 Q6) ---------------- */

/* After a step whose found_inf flag the host has read: found_inf != 0 halves
 * S, resets good_steps and leaves t unchanged (the step was skipped);
 * otherwise t += 1 and, after growth_interval clean steps in a row, S doubles.
 * Host only.  Errors: EINVAL (null, scale <= 0, growth_interval < 1). */
int fp8z1_scaler_update(fp8z1_loss_scaler* scaler, int32_t found_inf);

/* The clip arithmetic the step kernels perform on the device ("DeepSpeed ZeRO
 * 优化" §七), on the host, for logging a step: global_norm = sqrt(sumsq) /
 * loss_scale and clip_coef = max_norm / (global_norm + 1e-6), in double; the
 * step applies clip_coef when it is < 1.  Host only.  Errors: EINVAL (null
 * outputs, sumsq < 0 or nan, loss_scale or max_norm <= 0). */
int fp8z1_clip_coef(double sumsq, float max_norm, float loss_scale, double* global_norm,
                    double* clip_coef);

/* Static text for a status code. */
const char* fp8z1_strerror(int status);

#ifdef __cplusplus
}
#endif

#endif /* FP8Z1_H */
