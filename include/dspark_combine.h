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

#ifdef __cplusplus
}
#endif

#endif /* DSPARK_COMBINE_H */
