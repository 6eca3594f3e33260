"""Oracle for the speculative verify step's accepted-draft count and bonus token.

TEST INFRASTRUCTURE ONLY (see the package docstring).

The sglang PR #31847 summary page ("Implementation breakdown", item 2,
dflash_utils.py) describes compute_dflash_correct_drafts_and_bonus: on CUDA a
single kernel finds, per request, the first position where the draft and the
target disagree (a minimum over positions of "position, or BLOCK where they
agree"); the CPU branch keeps a cumulative product of the matches.  The page
prints neither the kernel nor the tensors, so this oracle takes the plainest
reading, which is also what the design notes record:

  candidates [bs, B]: column 0 is the request's last verified token, columns
                      1..B-1 its draft tokens;
  target     [bs, B]: the target model's greedy token at each of the B
                      positions (the prediction for the following position);
  correct[b] = number of leading i in [0, B-1) with candidates[b, i+1] ==
               target[b, i]    (the cumulative-product form, written as a loop)
  bonus[b]   = target[b, correct[b]]   (the target's token after the accepted
               drafts: the correction at the first mismatch, or the token
               after the last draft when every draft is accepted)
"""
from __future__ import annotations

import numpy as np


def correct_drafts_and_bonus(candidates: np.ndarray, target: np.ndarray):
    """(correct int32 [bs], bonus int64 [bs]) for int64 [bs, B] inputs, B >= 1."""
    candidates = np.asarray(candidates)
    target = np.asarray(target)
    if candidates.shape != target.shape or candidates.ndim != 2 or candidates.shape[1] < 1:
        raise ValueError("candidates and target must both be [bs, B] with B >= 1")
    bs, B = candidates.shape
    correct = np.zeros(bs, dtype=np.int32)
    bonus = np.zeros(bs, dtype=np.int64)
    for b in range(bs):
        still = 1
        n = 0
        for i in range(B - 1):
            still *= int(candidates[b, i + 1] == target[b, i])
            n += still
        correct[b] = n
        bonus[b] = target[b, n]
    return correct, bonus
