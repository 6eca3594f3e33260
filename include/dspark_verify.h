/*
 * dspark_verify.h -- C ABI of the speculative verify step's accepted-draft
 * count and bonus token, on one GB300 GPU (sm_103a).
 *
 * The sglang PR #31847 summary page ("Implementation breakdown", item 2,
 * dflash_utils.py: compute_dflash_correct_drafts_and_bonus and its single-
 * launch kernel) describes the step as finding, per request, the first
 * position where draft and target disagree.  The page prints neither the
 * kernel nor the tensors; this library takes the plainest reading:
 *
 *   candidates[b][0] is request b's last verified token, candidates[b][1..B-1]
 *   its draft tokens; target[b][i] is the target model's greedy token at
 *   position i (its prediction for position i + 1).
 *   correct[b] = number of leading i in [0, B-1) with
 *                candidates[b][i+1] == target[b][i]
 *   bonus[b]   = target[b][correct[b]]
 *
 * Conventions as in dspark_ctx_kv.h (device pointers, element strides,
 * dspark_status codes, host-side argument checks, stream-ordered).
 */
#ifndef DSPARK_VERIFY_H
#define DSPARK_VERIFY_H

#include "dspark_ctx_kv.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * dspark_correct_drafts_and_bonus -- per request, the accepted-draft count
 * and the bonus token.
 *
 *  candidates     int64 [batch, block] rows `candidates_stride` elements apart.
 *  target         int64 [batch, block] rows `target_stride` elements apart.
 *  block          B >= 1 tokens per request (1: no drafts, bonus = target[b][0]).
 *  correct        int32 [batch] out; bonus int64 [batch] out.
 *  stream         cudaStream_t.
 *
 * batch == 0 is a successful no-op.  Returns DSPARK_E_INVALID_ARG (NULL
 * pointer, batch < 0, block < 1, a stride < block), DSPARK_E_DEVICE (no
 * sm_103 device current) or DSPARK_E_CUDA (launch).
 */
DSPARK_API int dspark_correct_drafts_and_bonus(const int64_t* candidates, int64_t candidates_stride,
                                               const int64_t* target, int64_t target_stride, int64_t batch,
                                               int32_t block, int32_t* correct, int64_t* bonus, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DSPARK_VERIFY_H */
