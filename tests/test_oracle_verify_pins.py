"""Pins for the verify-step oracle (oracle/verify.py).

Hand-worked cases (tests/golden/verify_accept.json), and invariants that any
correct implementation of "count the leading accepted drafts, then take the
target's token there" satisfies: tokens after the first mismatch do not
matter, the bonus is the target token at the count, and a block whose drafts
are the target's own tokens is accepted whole.
"""
import json
import os

import numpy as np

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))


def test_golden_cases():
    cases = json.load(open(os.path.join(HERE, "golden", "verify_accept.json")))["cases"]
    for c in cases:
        cand = np.array([c["candidates"]], dtype=np.int64)
        tgt = np.array([c["target"]], dtype=np.int64)
        correct, bonus = oracle.correct_drafts_and_bonus(cand, tgt)
        assert (int(correct[0]), int(bonus[0])) == (c["correct"], c["bonus"]), c["why"]


def test_invariants_on_random_blocks():
    rng = np.random.default_rng(0)
    bs, B = 200, 16
    tgt = rng.integers(0, 50, size=(bs, B))
    cand = np.concatenate([rng.integers(0, 50, size=(bs, 1)), tgt[:, :-1]], axis=1)
    # drafts equal to the target's own tokens: everything accepted
    correct, bonus = oracle.correct_drafts_and_bonus(cand, tgt)
    assert np.all(correct == B - 1) and np.all(bonus == tgt[:, -1])
    # break each row at a random position k: exactly k accepted
    k = rng.integers(0, B - 1, size=bs)
    bad = cand.copy()
    bad[np.arange(bs), k + 1] = tgt[np.arange(bs), k] + 1000
    correct, bonus = oracle.correct_drafts_and_bonus(bad, tgt)
    np.testing.assert_array_equal(correct, k)
    np.testing.assert_array_equal(bonus, tgt[np.arange(bs), k])
    # anything after the first mismatch is irrelevant
    scrambled = bad.copy()
    for b in range(bs):
        scrambled[b, k[b] + 2:] = rng.integers(0, 50, size=B - k[b] - 2)
    c2, b2 = oracle.correct_drafts_and_bonus(scrambled, tgt)
    np.testing.assert_array_equal(c2, correct)
    np.testing.assert_array_equal(b2, bonus)
