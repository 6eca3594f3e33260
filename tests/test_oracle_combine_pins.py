"""Pins for the combine_hidden_states oracle (oracle/combine.py).

Closed forms and invariants: an identity block in the weight selects one
auxiliary state (constant rows then give sign(c) * w exactly, which catches
a transposed weight or the wrong block), one-hot auxiliary rows select weight
columns, scaling the inputs leaves the output unchanged (eps 0), the mean
square of out / w is ms / (ms + eps), and y is rounded to the model dtype
before the norm (a constant row whose product is not representable).
"""
import numpy as np
import pytest

import oracle
from synthetic import f32_to_bf16_bits

H, NAUX = 64, 3


def bits(x):
    return f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


def test_identity_block_selects_one_auxiliary_state():
    """W = [0 | I | 0] picks the second auxiliary state: rows that are
    constant there give sign(c) * w with eps 0."""
    W = np.zeros((H, NAUX * H))
    W[:, H:2 * H] = np.eye(H)
    rng = np.random.default_rng(0)
    aux = rng.standard_normal((5, NAUX * H))
    c = np.array([1.5, -2.0, 0.25, 4.0, -0.125])
    aux[:, H:2 * H] = c[:, None]
    w = 1 + 0.1 * rng.standard_normal(H)
    out = oracle.combine_hidden_states(bits(aux), bits(W), bits(w), 0.0, "bf16")
    np.testing.assert_array_equal(out, np.sign(c)[:, None] * oracle.widen(bits(w), "bf16")[None, :])


def test_one_hot_rows_select_weight_columns():
    rng = np.random.default_rng(1)
    W = rng.standard_normal((H, NAUX * H)) * 0.1
    Wb = bits(W)
    aux = np.zeros((3, NAUX * H))
    cols = [0, 70, 191]
    for r, c in enumerate(cols):
        aux[r, c] = 1.0
    one = bits(np.ones(H))
    out = oracle.combine_hidden_states(bits(aux), Wb, one, 0.0, "bf16")
    for r, c in enumerate(cols):
        y = oracle.widen(Wb, "bf16")[:, c]
        np.testing.assert_allclose(out[r], y / np.sqrt(np.mean(y * y)), rtol=1e-12)


def test_scale_invariance_and_mean_square():
    rng = np.random.default_rng(2)
    W = bits(rng.standard_normal((H, NAUX * H)) * 0.1)
    aux = rng.standard_normal((8, NAUX * H))
    one = bits(np.ones(H))
    a = oracle.combine_hidden_states(bits(aux), W, one, 0.0, "bf16")
    b = oracle.combine_hidden_states(bits(aux * 4.0), W, one, 0.0, "bf16")   # powers of two: exact
    np.testing.assert_allclose(a, b, rtol=1e-12)
    eps = 0.05
    o = oracle.combine_hidden_states(bits(aux), W, one, eps, "bf16")
    y = oracle.round_to(oracle.widen(bits(aux), "bf16") @ oracle.widen(W, "bf16").T, "bf16")
    ms = np.mean(y * y, axis=1)
    np.testing.assert_allclose(np.mean(o * o, axis=1), ms / (ms + eps), rtol=1e-12)


def test_linear_output_is_rounded_before_the_norm():
    """aux row of 1.0 against a weight row summing to 1 + 2**-9 (not a bf16
    value): y rounds to 1.0, so a head of equal rows normalises to exactly
    1.0 * w; without the rounding the row would not be constant."""
    W = np.zeros((H, NAUX * H))
    W[:, 0] = 1.0
    W[:, 1] = 2.0 ** -9
    W[0, 1] = 0.0                       # row 0 sums to 1, the others to 1 + 2**-9 -> 1.0 after rounding
    aux = np.zeros((1, NAUX * H))
    aux[0, :2] = 1.0
    one = bits(np.ones(H))
    out = oracle.combine_hidden_states(bits(aux), bits(W), one, 0.0, "bf16")
    np.testing.assert_array_equal(out, np.ones((1, H)))
