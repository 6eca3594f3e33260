/*
 * dspark_attention.h -- C ABI of the draft model's attention over the written
 * KV pool, on one GB300 GPU (sm_103a).
 *
 * The operation (sglang PR #35499 summary page, K3 DSpark draft attention:
 * "Implementation breakdown" items 2-3 and the verify_mla.py snippets of the
 * shared-KV split-KV kernels): qwen3-style GQA, bidirectional.  For request
 * b, query row i of its draft block (block rows), query head h, with
 * g = h / (num_q_heads / num_kv_heads):
 *
 *   keys   = k_pool[kv_indices[kv_start[b] .. kv_start[b+1]-1]][g]  then  k_ext[b*block .. b*block+block-1][g]
 *   values = the same rows of v_pool / v_ext
 *   out[b*block + i][h] = softmax(sm_scale * keys . q[b*block + i][h]) . values
 *
 * Every query sees every key (no causal mask).  The context part is split
 * into chunks processed in parallel and merged with the usual log-sum-exp
 * rescaling, through a caller-provided workspace.  The per-split products
 * run on the tcgen05 tensor cores with the accumulators in tensor memory.
 *
 * Conventions as in dspark_ctx_kv.h (device pointers unless marked (host),
 * strides in elements, dspark_status codes, host-side argument checks,
 * asynchronous and stream-ordered, no CPU fallback).
 */
#ifndef DSPARK_ATTENTION_H
#define DSPARK_ATTENTION_H

#include "dspark_ctx_kv.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Status bit (OR-ed into status_flags): a request's context is longer than
 * max_context (its tail is not attended). */
#define DSPARK_FLAG_CONTEXT_RANGE 0x8u

/*
 * dspark_draft_attention_workspace_bytes -- bytes of workspace that
 * dspark_draft_attention needs for these sizes (0 on invalid sizes).
 * Host-only; needs no GPU.
 */
DSPARK_API int64_t dspark_draft_attention_workspace_bytes(int64_t batch, int32_t block, int32_t num_q_heads,
                                                          int32_t num_kv_heads, int32_t head_dim,
                                                          int64_t max_context);

/*
 * dspark_draft_attention -- the attention above for every request.
 *
 *  q              [batch*block, num_q_heads, head_dim] contiguous, `dtype`.
 *  k_ext, v_ext   [batch*block, num_kv_heads, head_dim] contiguous: the block's
 *                 own keys and values.
 *  k_pool, v_pool [pool_slots, num_kv_heads, head_dim] with row stride
 *                 pool_row_stride (>= num_kv_heads*head_dim, a multiple of 8):
 *                 the layer's pools as dspark_write_ctx_kv fills them.
 *  kv_indices     int64 pool slots of every request's context, request after
 *                 request; kv_start int64 [batch + 1], non-decreasing, request
 *                 b's context is kv_indices[kv_start[b] .. kv_start[b+1]-1].
 *  max_context    (host) upper bound on any request's context length; it
 *                 sizes the split of the context and the workspace.
 *  out            [batch*block, num_q_heads, head_dim] contiguous, `dtype`.
 *  workspace      device buffer of at least
 *                 dspark_draft_attention_workspace_bytes(...) bytes, 16-byte
 *                 aligned; its contents on entry do not matter.
 *  status_flags   NULL or a device word: DSPARK_FLAG_LOC_RANGE is OR-ed when a
 *                 kv index is outside [0, pool_slots) (that key is skipped),
 *                 DSPARK_FLAG_CONTEXT_RANGE when a context exceeds max_context.
 *
 * Supported shapes: head_dim 64 or 128; num_q_heads a multiple of
 * num_kv_heads; rows per KV head (block * num_q_heads / num_kv_heads) 16 or
 * 32 (they are the N side of the tensor-core products; the keys, 128 per
 * step, are the M side); block <= 128; batch <= 65535; dtype BF16 or FP16.
 * batch == 0 is a successful no-op.  Returns DSPARK_E_INVALID_ARG
 * (NULL pointer, sizes), DSPARK_E_HEAD_DIM, DSPARK_E_SHAPE_MISMATCH (an
 * unsupported head / block combination), DSPARK_E_DTYPE_MISMATCH,
 * DSPARK_E_POOL_LAYOUT, DSPARK_E_ALIGNMENT, DSPARK_E_SCRATCH_LIMIT
 * (workspace too small), DSPARK_E_DEVICE or DSPARK_E_CUDA.
 *
 * Enqueues two kernels on `stream`: the split kernel, then the merge as a
 * programmatic dependent launch (its blocks may be scheduled while the split
 * kernel's last blocks run, and read the workspace only once that kernel has
 * completed).  No host synchronisation and no allocation: the call can be
 * captured in a CUDA graph and replayed.  Calls that share a workspace must be
 * ordered on the GPU.
 */
DSPARK_API int dspark_draft_attention(const void* q, const void* k_ext, const void* v_ext, const void* k_pool,
                                      const void* v_pool, int64_t pool_row_stride, int64_t pool_slots,
                                      const int64_t* kv_indices, const int64_t* kv_start, int64_t batch,
                                      int32_t block, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                      int32_t dtype, float sm_scale, int64_t max_context, void* out,
                                      void* workspace, int64_t workspace_bytes, uint32_t* status_flags,
                                      void* stream);

/*
 * dspark_draft_attention_set_wait_test -- diagnostics: with limit_ns > 0,
 * every later dspark_draft_attention call in this process makes its split
 * kernel's MMA issuer wait (bounded by limit_ns) on a barrier that nothing
 * arrives on, so that every role of the kernel takes its timeout path: the
 * call returns, DSPARK_FLAG_TIMEOUT is OR-ed into status_flags and the output
 * is incomplete.  0 switches it off (the default).  Not for production use;
 * process-wide, not synchronised with calls in flight on other threads.
 * Returns DSPARK_OK.
 */
DSPARK_API int dspark_draft_attention_set_wait_test(uint64_t limit_ns);

#ifdef __cplusplus
}
#endif

#endif /* DSPARK_ATTENTION_H */
