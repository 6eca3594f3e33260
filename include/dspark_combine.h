/*
 * dspark_combine.h -- C ABI of the draft model's combine_hidden_states on one
 * GB300 GPU (sm_103a): the context hidden state that dspark_write_ctx_kv
 * consumes.
 *
 * The operation (vLLM PR #46995 summary page, "Key source snippets": the
 * DSpark draft model's __init__ and combine_hidden_states):
 *
 *   y          = aux . W^T        aux [T, aux_dim]: the target model's auxiliary
 *                                 hidden states of its chosen layers, concatenated;
 *                                 W [hidden, aux_dim]: main_proj (no bias)
 *   ctx_hidden = y / sqrt(mean(y^2) + eps) * w      main_norm over hidden
 *
 * y is rounded to the model dtype (the linear layer's output) before the
 * norm; ctx_hidden is stored in the model dtype.  The product runs on the same
 * tcgen05 kernel as the KV write, in a plain mode whose epilogue stores y and
 * its per-row sums of squares per 256-column tile; a second, elementwise
 * kernel applies the norm in place.
 *
 * Conventions as in dspark_ctx_kv.h (device pointers unless marked (host),
 * strides in elements, dspark_status codes, host-side argument checks,
 * asynchronous and stream-ordered, no CPU fallback).
 */
#ifndef DSPARK_COMBINE_H
#define DSPARK_COMBINE_H

#include "dspark_ctx_kv.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct dspark_combine* dspark_combine_t;

/*
 * dspark_pack_combine -- prepare main_proj / main_norm for later calls.
 *
 *  main_proj_weight  [hidden, aux_dim] row-major (rows weight_row_stride
 *                    elements apart), `dtype` BF16 or FP16.  NOT copied: it
 *                    must stay alive and unchanged while the handle is used.
 *  main_norm_weight  [hidden] in norm_dtype (BF16 | FP16 | FP32), copied as fp32.
 *  hidden            a multiple of 32; aux_dim a multiple of 8; base 16-byte
 *                    aligned, weight_row_stride a multiple of 8, >= aux_dim.
 *  stream            used for the copies; synchronised before returning.
 *
 * Allocates the handle's device memory (fp32 norm weight, the split
 * schedule's workspace and counters, a status word).  Returns
 * DSPARK_E_INVALID_ARG, DSPARK_E_DTYPE_MISMATCH, DSPARK_E_SHAPE_MISMATCH,
 * DSPARK_E_ALIGNMENT, DSPARK_E_DEVICE or DSPARK_E_CUDA.
 */
DSPARK_API int dspark_pack_combine(const void* main_proj_weight, int64_t hidden, int64_t aux_dim,
                                   int64_t weight_row_stride, int32_t dtype, const void* main_norm_weight,
                                   int32_t norm_dtype, float eps, void* stream, dspark_combine_t* out /*host*/);

/*
 * dspark_combine_hidden_states -- ctx_hidden = main_norm(main_proj(aux)).
 *
 *  aux         [num_tokens, aux_dim] in the handle's dtype, rows aux_row_stride
 *              elements apart (a multiple of 8), 16-byte aligned.
 *  ctx_hidden  [num_tokens, hidden] out, rows out_row_stride apart (a multiple
 *              of 8, >= hidden), 16-byte aligned.
 *
 * The first call with more tokens than any earlier one grows the handle's
 * per-row scratch (cudaMalloc).  Enqueues two kernels on `stream`.  Returns
 * DSPARK_E_INVALID_ARG, DSPARK_E_ALIGNMENT, DSPARK_E_DEVICE or DSPARK_E_CUDA;
 * num_tokens == 0 is a successful no-op.
 */
DSPARK_API int dspark_combine_hidden_states(dspark_combine_t c, const void* aux, int64_t num_tokens,
                                            int64_t aux_row_stride, void* ctx_hidden, int64_t out_row_stride,
                                            void* stream);

/* The handle's device status word (DSPARK_FLAG_TIMEOUT if an in-kernel wait
 * ran out); synchronises `stream`. */
DSPARK_API int dspark_combine_get_status(dspark_combine_t c, void* stream, uint32_t* flags /*host*/);

/* Free the handle (synchronises its device).  NULL is a no-op. */
DSPARK_API void dspark_free_combine(dspark_combine_t c);

/*
 * combine_hidden_states fused into the context-KV write: one launch per step
 * from the target's auxiliary hidden states to the written pools, ctx_hidden
 * never formed.
 *
 * With y = aux . W^T rounded to the model dtype, s_t = 1/sqrt(mean(y_t^2) + eps)
 * and w main_norm's weight, ctx_hidden = y * s_t * w and the write's
 * projection ctx_hidden . W_kv^T equals s_t * (y . (W_kv diag(w))^T).  The
 * pack scales the stacked K|V weights by w once (rounded to the model dtype);
 * each write runs main_proj on the tensor cores (y and its per-row sums of
 * squares into the handle's scratch, which stays in L2 for decode-sized
 * batches) and then, after every CTA is done with it, the write over y with
 * each token row scaled by s_t before the bias, the K norm and the rotation.
 * The result equals dspark_combine_hidden_states followed by
 * dspark_write_ctx_kv up to rounding: ctx_hidden is not rounded to the model
 * dtype here, the scaled weights are.
 */
typedef struct dspark_fused* dspark_fused_t;

/*
 * dspark_pack_fused_ctx_kv -- main_proj_weight [hidden, aux_dim] (rows
 * weight_row_stride elements apart, the layers' dtype; NOT copied: it must stay
 * alive and unchanged while the handle is used), main_norm_weight [hidden] in
 * norm_dtype (BF16 | FP16 | FP32), norm_eps, and the draft layers as for
 * dspark_pack_ctx_kv (checked the same way, same refusal codes).  hidden a
 * multiple of 32, aux_dim a multiple of 8, weight base 16-byte aligned and
 * weight_row_stride a multiple of 8.  Allocates the handle's device memory;
 * the copies run on `stream`, which is synchronised before returning.
 */
DSPARK_API int dspark_pack_fused_ctx_kv(const void* main_proj_weight, int64_t aux_dim, int64_t weight_row_stride,
                                        const void* main_norm_weight, int32_t norm_dtype, float norm_eps,
                                        const dspark_layer_desc* layers /* (host) */, int32_t num_layers,
                                        int32_t hidden, void* stream, dspark_fused_t* out /* (host) */);

/*
 * dspark_combine_write_ctx_kv -- the write of dspark_write_ctx_kv with
 * ctx_hidden = main_norm(main_proj(aux)): aux [num_tokens, aux_dim] in the
 * handle's dtype, rows aux_row_stride elements apart (a multiple of 8),
 * 16-byte aligned; every other argument as for dspark_write_ctx_kv.  One
 * kernel launch (CTA pairs).  The first call with more tokens than any earlier
 * one grows the handle's scratch (cudaMalloc, after a device synchronise).
 * Writes with one handle must be ordered on the GPU (they share its scratch);
 * the grid-wide step between the two products assumes every CTA resident (as
 * the write's split tiles do) and ends on its 2 s bound, with
 * DSPARK_FLAG_TIMEOUT, if it is not.
 */
DSPARK_API int dspark_combine_write_ctx_kv(dspark_fused_t f, const void* aux, int64_t num_tokens,
                                           int64_t aux_row_stride, const int64_t* positions, const float* cos_sin,
                                           int64_t max_pos, const int64_t* cache_loc, const int32_t* commit_lens,
                                           int64_t loc_row_width, int64_t num_windows, void* const* k_pools,
                                           void* const* v_pools, const int64_t* k_row_strides,
                                           const int64_t* v_row_strides, int32_t pool_dtype, int64_t pool_slots,
                                           void* stream);

/* Status word of the handle's writes (DSPARK_FLAG_* bits), synchronising
 * `stream`; and its reset (also of the handle's counters: call it after a
 * write that reported DSPARK_FLAG_TIMEOUT). */
DSPARK_API int dspark_fused_get_status(dspark_fused_t f, void* stream, uint32_t* flags /* (host) */);
DSPARK_API int dspark_fused_clear_status(dspark_fused_t f, void* stream);

/* Free the handle (synchronises its device).  NULL is a no-op. */
DSPARK_API void dspark_free_fused(dspark_fused_t f);

#ifdef __cplusplus
}
#endif

#endif /* DSPARK_COMBINE_H */
