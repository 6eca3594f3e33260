/*
 * dspark_ctx_kv.h -- C ABI of the DSpark draft-model context-KV write on one
 * GB300 GPU (sm_103a).
 *
 * The write (sglang PR #31986 summary page, "write_target_hidden_kv" snippet;
 * sglang PR #31847 summary page, "fused_kv_norm_rope_write" snippet):
 *
 *   for every draft layer l, token t, kv head h, d in [0, D):
 *     yK = ctx_hidden[t] . W_qkv,l[q_size + h*D + d]        (+ bias)
 *     yV = ctx_hidden[t] . W_qkv,l[q_size + KV + h*D + d]   (+ bias)
 *     n  = yK / sqrt(mean_d(yK^2) + eps) * k_norm_l[d]        (fp32 weights)
 *     K  = neox rotation of n by the cos/sin row positions[t] of the table
 *     if cache_loc[t] >= 0 (and, in window mode, t's column < commit_lens[row]):
 *       K_pool_l[cache_loc[t]][h][:] = K,  V_pool_l[cache_loc[t]][h][:] = yV
 *
 * computed as ONE dense product of ctx_hidden with the row-stacked K|V slices
 * of every layer (the inputs are shared, so stacking is exact: PR #31986 page,
 * "Motivation") followed by a fused norm / rotation / scatter epilogue.
 *
 * Conventions
 *  - Pointers are DEVICE pointers unless marked (host).  Element strides are
 *    counted in elements, not bytes.
 *  - Every call returns a dspark_status (0 = success).  Argument errors are
 *    detected on the host before any GPU work is enqueued; nothing is
 *    allocated or written when a call is refused.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  Writes
 *    are asynchronous and stream-ordered; caller-owned buffers must stay
 *    alive until the stream work completes.
 *  - The library has no CPU fallback: without a usable sm_103 GPU the GPU
 *    calls return DSPARK_E_CUDA / DSPARK_E_DEVICE.
 */
#ifndef DSPARK_CTX_KV_H
#define DSPARK_CTX_KV_H

#include <stdint.h>

#if defined(__GNUC__)
#define DSPARK_API __attribute__((visibility("default")))
#else
#define DSPARK_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* element types */
#define DSPARK_DTYPE_BF16 1
#define DSPARK_DTYPE_FP16 2
#define DSPARK_DTYPE_FP32 3   /* accepted for k_norm weights only */
/* Any other weight_dtype code (e.g. a quantized format) marks the layer's
 * qkv weight as non-sliceable and the pack is refused. */

typedef enum dspark_status {
  DSPARK_OK = 0,
  DSPARK_E_INVALID_ARG = 1,       /* NULL pointer, negative size, ... */
  DSPARK_E_NO_LAYERS = 2,         /* num_layers == 0 */
  DSPARK_E_NOT_SLICEABLE = 3,     /* a qkv weight is not plain bf16/fp16 (quantized) */
  DSPARK_E_EPS_MISMATCH = 4,      /* layers disagree on the k_norm epsilon */
  DSPARK_E_DTYPE_MISMATCH = 5,    /* layers / activations / pools of different dtype */
  DSPARK_E_SHAPE_MISMATCH = 6,    /* layers disagree on q_size, num_kv_heads or head_dim,
                                     or a weight has fewer rows than q_size + 2*kv_size */
  DSPARK_E_HEAD_DIM = 7,          /* head_dim not 64 or 128 */
  DSPARK_E_BIAS_MISMATCH = 8,     /* bias on some layers only */
  DSPARK_E_COMMIT_ARGS = 9,       /* commit_lens and loc_row_width not given together */
  DSPARK_E_NUMEL = 10,            /* num_windows * loc_row_width != num_tokens */
  DSPARK_E_ALIGNMENT = 11,        /* a buffer or stride breaks the 16-byte rules below */
  DSPARK_E_POOL_LAYOUT = 12,      /* pool row stride < num_kv_heads * head_dim */
  DSPARK_E_TOO_MANY_LAYERS = 13,  /* num_layers > DSPARK_MAX_LAYERS */
  DSPARK_E_DEVICE = 14,           /* no sm_103 device, or not the bundle's device */
  DSPARK_E_CUDA = 15,             /* a CUDA runtime call failed */
  DSPARK_E_DEVICE_FAULT = 16,     /* a device-side check fired (see status flags) */
  DSPARK_E_SCRATCH_LIMIT = 17     /* dspark_write_ctx_kv_noalloc: the launch would need more
                                     scratch than the library's static array holds */
} dspark_status;

#define DSPARK_MAX_LAYERS 32

/* Bits of the device status word (dspark_get_device_status).  The write skips
 * the offending token and sets the bit; other tokens are still written. */
#define DSPARK_FLAG_POS_RANGE 0x1u   /* positions[t] < 0 or >= max_pos */
#define DSPARK_FLAG_LOC_RANGE 0x2u   /* cache_loc[t] >= pool_slots */
#define DSPARK_FLAG_TIMEOUT   0x4u   /* an in-kernel wait exceeded its bound; output incomplete */

/* One draft layer's attention parameters, as the model holds them
 * (PR #31986 page, _stacked_ctx_kv_params; PR #31847 page,
 * _build_fused_kv_write_bundle).  (host) struct, device buffers. */
typedef struct dspark_layer_desc {
  const void* qkv_weight;     /* [qkv_rows, hidden] row-major, out-by-in (F.linear);
                                 rows [q_size, q_size+kv_size) are K, the next kv_size are V */
  int64_t qkv_rows;           /* rows in qkv_weight, >= q_size + 2*kv_size */
  int64_t qkv_row_stride;     /* elements between rows, >= hidden */
  const void* qkv_bias;       /* NULL or [qkv_rows] in weight_dtype */
  const void* k_norm_weight;  /* [head_dim] in k_norm_dtype; converted to fp32 */
  int32_t weight_dtype;       /* DSPARK_DTYPE_BF16 | DSPARK_DTYPE_FP16, else non-sliceable */
  int32_t k_norm_dtype;       /* BF16 | FP16 | FP32 */
  int32_t q_size;             /* Q rows that precede the K rows */
  int32_t num_kv_heads;       /* NH; kv_size = NH * head_dim */
  int32_t head_dim;           /* D: 64 or 128 */
  float eps;                  /* k_norm variance epsilon */
} dspark_layer_desc;

typedef struct dspark_bundle* dspark_bundle_t;

/* Read-only view of a packed bundle. (host) */
typedef struct dspark_bundle_info {
  int32_t num_layers, hidden, num_kv_heads, head_dim, dtype, has_bias, device;
  float eps;
  int64_t stacked_rows;       /* N = num_layers * 2 * num_kv_heads * head_dim */
} dspark_bundle_info;

/*
 * dspark_check_ctx_kv_layers -- host-only eligibility check of a set of layers.
 * Touches no GPU and reads no device memory.  Returns DSPARK_OK or the first
 * refusal, in this order: E_INVALID_ARG, E_NO_LAYERS, E_TOO_MANY_LAYERS, then
 * per layer E_NOT_SLICEABLE, E_EPS_MISMATCH, E_DTYPE_MISMATCH,
 * E_SHAPE_MISMATCH, E_HEAD_DIM, and finally E_BIAS_MISMATCH.  The refusals
 * follow PR #31986's _stacked_ctx_kv_params (quantized weight, eps mismatch,
 * partial bias -> no stacked bundle) and PR #31847's bundle builder (same
 * head_dim and kv_size on every layer).
 */
DSPARK_API int dspark_check_ctx_kv_layers(const dspark_layer_desc* layers /* (host) [num_layers] */,
                               int32_t num_layers, int32_t hidden);

/*
 * dspark_pack_ctx_kv -- build the immutable stacked bundle.
 * Copies rows [q_size, q_size + 2*kv_size) of every layer's qkv weight into one
 * bundle-owned [N, hidden] matrix (rows l0:K, l0:V, l1:K, ...), the matching
 * bias rows (when every layer has a bias), and the k_norm weights as fp32
 * [L, head_dim]; records eps.  Runs the check above first and allocates
 * nothing on refusal.  The bundle is owned by the library: free it with
 * dspark_free_bundle.  It is bound to the device current at the call.  The
 * copies run on `stream` and the call synchronises that stream before it
 * returns, so the bundle is ready for use on any stream (writes with one
 * bundle must still be ordered: see dspark_write_ctx_kv).  The bundle keeps a
 * snapshot: if the model's weights change, pack again (PR #31986 page, Risks:
 * the cached stack assumes frozen weights).
 */
DSPARK_API int dspark_pack_ctx_kv(const dspark_layer_desc* layers /* (host) [num_layers] */,
                       int32_t num_layers, int32_t hidden, void* stream,
                       dspark_bundle_t* out /* (host) */);

/*
 * dspark_write_ctx_kv -- project, normalise, rotate and scatter K/V of
 * num_tokens tokens into every layer's pool (PR #31847 page,
 * fused_kv_norm_rope_write: loc < 0 is skipped; with commit_lens the locs are
 * a flattened [num_windows, loc_row_width] verify window and only the first
 * commit_lens[b] columns of row b are written).
 *
 *  ctx_hidden      [num_tokens, hidden] in the bundle dtype, row stride
 *                  hidden_row_stride (>= hidden); base and row pitch 16-byte aligned
 *  positions       [num_tokens] int64, each in [0, max_pos)
 *  cos_sin         [max_pos, head_dim] fp32, row p = [cos(p*f_0..f_{D/2-1}) | sin(...)],
 *                  16-byte aligned.  Neox pairing, full rotary dimension.
 *  cache_loc       [num_tokens] int64 pool slots; < 0 = skip
 *  commit_lens     NULL, or [num_windows] int32 (<= 0 writes nothing, > width acts as width)
 *  loc_row_width   0 when commit_lens is NULL, else the window width W > 0
 *  num_windows     0 when commit_lens is NULL, else bs with bs * W == num_tokens
 *  k_pools/v_pools (host) arrays of num_layers device pointers, each pool
 *                  [pool_slots, num_kv_heads, head_dim] with row stride
 *                  k_row_strides[l] / v_row_strides[l] (host arrays, elements,
 *                  >= num_kv_heads*head_dim, multiple of 8) and head/dim
 *                  strides head_dim / 1; 16-byte aligned bases
 *  pool_dtype      must equal the bundle dtype
 * Written non-negative locs must be distinct.  A position outside the table or
 * a loc >= pool_slots is a caller error: that token is skipped and a device
 * status flag is set.  num_tokens == 0 returns DSPARK_OK at once.
 * Enqueues one kernel on `stream`; no host synchronisation and no device
 * allocation (the bundle's scratch is allocated by dspark_pack_ctx_kv), so the
 * call can be captured in a CUDA graph and replayed; a replay reads the
 * buffers' current contents.
 *
 * Concurrency.  Every write with a bundle uses that bundle's scratch: the
 * partial tiles of the work split, their arrival counters and the status
 * word.  Writes with the same bundle must therefore be ordered on the GPU
 * (one stream, or streams ordered by events); two that overlap race on the
 * scratch and write wrong values.  Writes with different bundles may overlap.
 * The grid is sized to what the device can hold resident at once (one CTA, or
 * CTA pair, per SM or SM pair), and a CTA may wait, bounded, for parts that
 * other CTAs of the same launch publish.  If other work holds SMs while the
 * write runs (a concurrent kernel, an MPS thread limit, a green context) those
 * waits can run out: the write then stops, sets DSPARK_FLAG_TIMEOUT and leaves
 * some rows unwritten rather than hanging; dspark_clear_device_status makes the
 * bundle usable again.
 */
DSPARK_API int dspark_write_ctx_kv(dspark_bundle_t bundle,
                        const void* ctx_hidden, int64_t num_tokens,
                        int64_t hidden_row_stride, int32_t hidden_dtype,
                        const int64_t* positions,
                        const float* cos_sin, int64_t max_pos,
                        const int64_t* cache_loc,
                        const int32_t* commit_lens, int64_t loc_row_width,
                        int64_t num_windows,
                        void* const* k_pools, void* const* v_pools,
                        const int64_t* k_row_strides, const int64_t* v_row_strides,
                        int32_t pool_dtype, int64_t pool_slots,
                        void* stream);

/*
 * dspark_write_ctx_kv_noalloc -- the same write for callers that must not
 * allocate device memory.  (The pages have no counterpart: their write always
 * runs inside a serving framework that allocates freely.)
 *
 * Some callers cannot call cudaMalloc: frameworks whose own pool allocator
 * owns all device memory (an allocation behind its back escapes its accounting
 * and can fragment or exhaust the pool), and latency-critical loops that
 * cannot afford cudaMalloc's implicit device-wide synchronisation.  They cannot
 * use dspark_pack_ctx_kv either, since the bundle is allocated.  This entry
 * point allocates nothing: the caller passes the stacked parameters the pack
 * would build, every input and every output, and the kernel's scratch (the
 * partial-tile workspace of the split schedule and its arrival counters) lives
 * in a file-scope device array of 16 MiB + 4 KiB that the library reserves on
 * every GPU it is loaded on, until the process exits.
 *
 *  stacked_weight    [N, hidden], N = num_layers*2*num_kv_heads*head_dim, rows
 *                    l0:K, l0:V, l1:K, ... (the pack's layout), row stride
 *                    weight_row_stride elements (16-byte pitch), 16-byte aligned
 *  stacked_bias      NULL or [N] in dtype
 *  k_norm_weight     [num_layers, head_dim] fp32, 16-byte aligned
 *  dtype             DSPARK_DTYPE_BF16 or DSPARK_DTYPE_FP16 (weights, hidden, pools)
 *  status_flags      a device uint32 the kernel ORs DSPARK_FLAG_* bits into, or NULL:
 *                    then the flags (out-of-range positions or slots, a wait that ran
 *                    out) go to a word inside the library's array that no call reads
 *                    back, so those errors are discarded
 *  other arguments   as for dspark_write_ctx_kv
 * The sizes of the caller's buffers are not known to this call (there is no
 * bundle to check them against): they must match the arguments.
 *
 * A call runs on at most 64 SMs, the CTAs whose partial tiles fit in the
 * array.  The scratch a launch uses depends on its CTA count only, not on the
 * token count or the model's sizes, so every problem fits;
 * DSPARK_E_SCRATCH_LIMIT is a guard that valid arguments never reach.  All
 * calls share the one array and it keeps the
 * previous call's contents: each call clears the arrival counters (a
 * stream-ordered memset) before its kernel, and two calls whose kernels
 * overlap on the GPU race and give wrong results, so keep the calls on a
 * device ordered.  The first call on each device looks up the array's address
 * and sets the kernel's shared-memory limit; make that first call before any
 * stream capture begins.
 */
DSPARK_API int dspark_write_ctx_kv_noalloc(
    const void* stacked_weight, int64_t weight_row_stride, const void* stacked_bias,
    const float* k_norm_weight, float eps, int32_t num_layers, int32_t hidden,
    int32_t num_kv_heads, int32_t head_dim, int32_t dtype,
    const void* ctx_hidden, int64_t num_tokens, int64_t hidden_row_stride,
    const int64_t* positions, const float* cos_sin, int64_t max_pos,
    const int64_t* cache_loc, const int32_t* commit_lens, int64_t loc_row_width,
    int64_t num_windows, void* const* k_pools, void* const* v_pools,
    const int64_t* k_row_strides, const int64_t* v_row_strides, int64_t pool_slots,
    uint32_t* status_flags, void* stream);

/* Copy the bundle's device status word (DSPARK_FLAG_* bits, OR-ed over all
 * writes since the last clear) to *flags, ordered after prior work on
 * `stream`; synchronises `stream`. */
DSPARK_API int dspark_get_device_status(dspark_bundle_t bundle, void* stream, uint32_t* flags /* (host) */);

/* As dspark_get_device_status, without waiting: enqueue on `stream` the copy
 * of the status word to *flags and return.  *flags must stay valid until the
 * copy has run, and is meaningful only after `stream` (or an event recorded
 * on it after this call) has been synchronised; for the copy to be truly
 * asynchronous *flags should be page-locked host memory.  This lets a
 * pipelined caller read every write's status without a synchronisation per
 * write.  Returns DSPARK_E_INVALID_ARG for a NULL bundle or flags, else
 * DSPARK_OK or DSPARK_E_CUDA (enqueueing failed). */
DSPARK_API int dspark_read_device_status_async(dspark_bundle_t bundle, void* stream, uint32_t* flags /* (host) */);

/* Reset the device status word to 0 and the split-tile arrival counters
 * (stream-ordered, asynchronous).  Call it after a write that reported
 * DSPARK_FLAG_TIMEOUT: such a write may leave counters set. */
DSPARK_API int dspark_clear_device_status(dspark_bundle_t bundle, void* stream);

/* Kernel variant used by later writes with this bundle.
 *  PAIR:   256-token x 256-column tiles computed by two CTAs of a cluster with
 *          tcgen05.mma.cta_group::2 (each CTA stages half of the weight tile).
 *  SINGLE: 128 x 256 tiles, one CTA each.
 *  STREAM: for num_tokens <= 256 (and num_kv_heads*head_dim a multiple of 128):
 *          128 weight rows x all tokens per tile, weights streamed by every SM;
 *          a write that does not meet those limits returns DSPARK_E_INVALID_ARG.
 *  AUTO (the default): STREAM when it applies and num_tokens <= 64, or
 *        num_tokens <= 128 and the CTA pairs would get fewer tiles than half
 *        their number (every tile cut); else PAIR.
 * Results agree within rounding; the choice only changes speed.  Returns
 * DSPARK_E_INVALID_ARG for other values. */
#define DSPARK_VARIANT_AUTO 0
#define DSPARK_VARIANT_SINGLE 1
#define DSPARK_VARIANT_PAIR 2
#define DSPARK_VARIANT_STREAM 3
DSPARK_API int dspark_set_kernel_variant(dspark_bundle_t bundle, int32_t variant);

/* Diagnostics: make later writes with this bundle record a per-CTA timeline
 * into `buf` (device, uint64 [SMs x 64]: globaltimer ns at CTA start and end,
 * the number of work items, then per work item its tile, its k-block range and
 * kind, and the times its accumulator became ready and was released; the last
 * word: when the CTA finished its rows of the leftover split tiles).  `words`
 * is the buffer length; NULL turns tracing off (the default).  Tracing adds a
 * few global stores per work item and does not change results. */
DSPARK_API int dspark_set_trace_buffer(dspark_bundle_t bundle, uint64_t* buf, int64_t words);

/* Diagnostics for tests of the timeout path: later writes with this bundle
 * wait for `missing_arrivals` more published parts of every tile that is cut
 * between CTAs than there are contributors (a count that no CTA will reach),
 * and give up on each such wait after `limit_ns` nanoseconds (1 .. 2e9)
 * instead of the normal 2 s.  Those waits then run out: the write stops,
 * sets DSPARK_FLAG_TIMEOUT and returns with the rows of those tiles (and
 * possibly others) unwritten.  Every other wait keeps its normal bound, and
 * each CTA still waits for its own copies and tensor-core work before it
 * exits, so the GPU stays usable.  A write without cut tiles is unaffected.
 * missing_arrivals = 0 restores normal writes.  Returns DSPARK_E_INVALID_ARG
 * for a negative count, more than 1024, or a limit outside 1 .. 2e9 ns. */
DSPARK_API int dspark_set_split_wait_test(dspark_bundle_t bundle, int32_t missing_arrivals, uint64_t limit_ns);

DSPARK_API int dspark_bundle_get_info(dspark_bundle_t bundle, dspark_bundle_info* info /* (host) */);

/* Work split of the tiled kernels (host only; needs no GPU). (host) */
typedef struct dspark_schedule_info {
  int32_t workers;        /* workers launched (CTAs, or CTA pairs) */
  int32_t whole_tiles;    /* tiles 0 .. whole_tiles-1 are computed whole, tile w, w+workers, ... by worker w */
  int64_t split_units;    /* k-blocks of the remaining tiles, cut into contiguous ranges */
  int32_t split_workers;  /* workers 0 .. split_workers-1 take one range each (equal shares) */
  int32_t split_first;    /* 1: ranges before whole tiles, every contributor finishes rows of its
                             cut tiles; 0: whole tiles first, a cut tile finished by the owner of
                             its last k-block */
} dspark_schedule_info;

/*
 * dspark_describe_schedule -- the work split a write (or the combine product)
 * uses for a problem of `tiles` output tiles with `num_kb` 64-deep k-blocks
 * each on up to `workers` workers (SMs for single-CTA tiles, SM pairs for CTA
 * pairs).  `split_first_allowed` is 1 for the tiled kernels and 0 for the
 * weight-streaming kernel.  Diagnostics: the kernels compute the same split
 * themselves.  With `split_first_allowed` the split is the tiled write's,
 * which gives every tile whole to one worker (and leaves the others idle)
 * when there are fewer tiles than workers but at least half as many; the
 * combine product and the allocation-free write cut those tiles instead.
 * One refinement is not shown: in the split-first order with
 * one whole tile per worker, the write hands the leftover only to the
 * workers whose whole tile holds V heads (when each then takes 2 to 8
 * k-blocks), reordering the whole tiles so that those workers come first.
 * Returns DSPARK_E_INVALID_ARG for non-positive sizes or a NULL `out`.
 */
DSPARK_API int dspark_describe_schedule(int64_t tiles, int32_t num_kb, int32_t workers,
                                        int32_t split_first_allowed, dspark_schedule_info* out /* (host) */);

/* Release the bundle's device memory (synchronises the device first). NULL is a no-op. */
DSPARK_API void dspark_free_bundle(dspark_bundle_t bundle);

/* Static English text for a status code. */
DSPARK_API const char* dspark_status_string(int code);

#ifdef __cplusplus
}
#endif
#endif /* DSPARK_CTX_KV_H */
