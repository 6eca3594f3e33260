/*
 * dspark_qk_norm_rope.h -- C ABI of the in-place QK RMSNorm + table neox RoPE
 * that a DSpark (or DFlash) draft layer applies to its own fused QKV tensor,
 * on one GB300 GPU (sm_103a).
 *
 * The operation (sglang PR #31847 summary page, "Key source snippets",
 * dflash_utils.py: `_table_qk_norm_rope_kernel` and `table_qk_norm_rope_`):
 *
 *   for every token t and every head h of the first num_q_heads + num_k_heads
 *   heads of row t (Q heads first, then K heads; the V heads that follow are
 *   not touched), with x the head's head_dim values and w the Q norm weight
 *   for Q heads, the K norm weight for K heads:
 *     inv = 1 / sqrt(mean(x^2) + eps)                     (fp32)
 *     x1  = round(x[:D/2] * inv * w[:D/2]),  x2 = round(x[D/2:] * inv * w[D/2:])
 *     c = cos_sin[positions[t]][:D/2],  s = cos_sin[positions[t]][D/2:]
 *     head[:D/2] = x1 * c - x2 * s,  head[D/2:] = x2 * c + x1 * s     (stored)
 *   round(): the intermediate rounding to the model dtype that the page keeps
 *   so that the fused kernel matches the eager path.
 *
 * Conventions as in dspark_ctx_kv.h: device pointers unless marked (host),
 * strides in elements, dspark_status return codes, argument errors detected
 * on the host before any GPU work, asynchronous and stream-ordered, no CPU
 * fallback.
 */
#ifndef DSPARK_QK_NORM_ROPE_H
#define DSPARK_QK_NORM_ROPE_H

#include "dspark_ctx_kv.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * dspark_qk_norm_rope -- normalise and rotate the Q and K heads of a fused
 * QKV tensor in place.
 *
 *  qkv            [num_tokens, row_stride] elements of `dtype` (BF16 | FP16),
 *                 read and written in place; each row holds num_q_heads Q
 *                 heads then num_k_heads K heads of head_dim elements from
 *                 column 0 (the page's q_size = num_q_heads * head_dim);
 *                 columns from (num_q_heads + num_k_heads) * head_dim on are
 *                 left untouched.  Base 16-byte aligned, row_stride a multiple
 *                 of 8 and >= (num_q_heads + num_k_heads) * head_dim.
 *  positions      int64 [num_tokens], each in [0, max_pos).
 *  q_weight, k_weight  [head_dim] each, in `dtype`, 16-byte aligned.
 *  cos_sin        fp32 [max_pos, head_dim], row = [cos(0..D/2-1) | sin(0..D/2-1)],
 *                 16-byte aligned.
 *  head_dim       64 or 128; num_q_heads >= 0, num_k_heads >= 0.
 *  status_flags   NULL, or a device word to which DSPARK_FLAG_POS_RANGE is
 *                 OR-ed when a token's position is outside the table; that
 *                 token's row is left untouched and the others are processed.
 *  stream         cudaStream_t.
 *
 * num_tokens == 0 (or no heads) is a successful no-op.  Returns
 * DSPARK_E_INVALID_ARG (NULL pointer, negative size), DSPARK_E_HEAD_DIM,
 * DSPARK_E_DTYPE_MISMATCH (dtype not BF16 / FP16), DSPARK_E_POOL_LAYOUT
 * (row_stride shorter than the Q and K heads), DSPARK_E_ALIGNMENT,
 * DSPARK_E_DEVICE (no sm_103 device current) or DSPARK_E_CUDA (launch).
 */
DSPARK_API int dspark_qk_norm_rope(void* qkv, int64_t num_tokens, int64_t row_stride, int32_t dtype,
                                   const int64_t* positions, const void* q_weight, const void* k_weight,
                                   const float* cos_sin, int64_t max_pos, int32_t num_q_heads,
                                   int32_t num_k_heads, int32_t head_dim, float eps,
                                   uint32_t* status_flags, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DSPARK_QK_NORM_ROPE_H */
