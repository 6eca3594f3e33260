"""Pins for the draft-attention oracle (oracle/draft_attention.py).

Closed forms and invariants of softmax attention that catch the plausible
mistakes: a wrong query-head -> KV-head mapping (per-KV-head constant values),
a missing or doubled scale (two-key weight ratio), a causal mask over the
block (a later extend key must be visible to query 0), dropping either key
source (single-key and equal-key cases), and order dependence (permuting the
context's slots).
"""
import numpy as np
import pytest

import oracle
from synthetic import f32_to_bf16_bits

D = 64


def bits(x):
    return f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


def val(b):
    return oracle.widen(b, "bf16")


def build(bs, E, nq, nk, ctx, slots, rng, scale=0.5):
    q = bits(rng.standard_normal((bs * E, nq, D)) * scale)
    ke = bits(rng.standard_normal((bs * E, nk, D)) * scale)
    ve = bits(rng.standard_normal((bs * E, nk, D)))
    kp = bits(rng.standard_normal((slots, nk, D)) * scale)
    vp = bits(rng.standard_normal((slots, nk, D)))
    idx = rng.permutation(slots)[:sum(ctx)].astype(np.int64)
    start = np.concatenate([[0], np.cumsum(ctx)]).astype(np.int64)
    return q, ke, ve, kp, vp, idx, start


def test_single_key_returns_its_value():
    """Empty context and a block of one: the only key gets weight 1."""
    rng = np.random.default_rng(0)
    q, ke, ve, kp, vp, idx, start = build(3, 1, 4, 2, [0, 0, 0], 16, rng)
    out = oracle.draft_attention(q, ke, ve, kp, vp, idx, start, "bf16", 4, 2, D, 0.125)
    for h in range(4):
        np.testing.assert_allclose(out[:, h], val(ve)[:, h // 2], rtol=0, atol=1e-12)


def test_equal_keys_average_the_values():
    """Every key equal (context and block): uniform weights, the mean of the
    values of the request's keys."""
    rng = np.random.default_rng(1)
    bs, E, nq, nk = 2, 4, 4, 2
    q, ke, ve, kp, vp, idx, start = build(bs, E, nq, nk, [5, 3], 32, rng)
    ke[:] = bits(np.ones((bs * E, nk, D)) * 0.25)
    kp[:] = bits(np.ones((32, nk, D)) * 0.25)
    out = oracle.draft_attention(q, ke, ve, kp, vp, idx, start, "bf16", nq, nk, D, 0.125)
    for b in range(bs):
        rows = np.concatenate([val(vp)[idx[start[b]:start[b + 1]]], val(ve)[b * E:(b + 1) * E]])
        for h in range(nq):
            np.testing.assert_allclose(out[b * E:(b + 1) * E, h], np.broadcast_to(rows[:, h // 2].mean(0), (E, D)),
                                       rtol=0, atol=1e-12)


def test_gqa_head_mapping():
    """Values constant per KV head g (value g + 1 everywhere): any weights give
    g + 1, so query head h must return h // (nq / nk) + 1."""
    rng = np.random.default_rng(2)
    bs, E, nq, nk = 2, 8, 8, 2
    q, ke, ve, kp, vp, idx, start = build(bs, E, nq, nk, [20, 7], 64, rng)
    for g in range(nk):
        ve[:, g] = bits(np.full((bs * E, D), g + 1.0))
        vp[:, g] = bits(np.full((64, D), g + 1.0))
    out = oracle.draft_attention(q, ke, ve, kp, vp, idx, start, "bf16", nq, nk, D, 0.1)
    for h in range(nq):
        np.testing.assert_allclose(out[:, h], h // (nq // nk) + 1.0, rtol=0, atol=1e-12)


def test_two_key_weight_ratio_is_exp_scale_times_score_gap():
    """One context key and one block key; values e_0 and e_1: the output's
    first two components are the weights, whose ratio is exp(sm_scale * (s0 - s1))."""
    qv = np.zeros((1, 1, D)); qv[0, 0, :4] = 1.0
    k0 = np.zeros((1, 1, D)); k0[0, 0, :4] = 2.0        # score 8
    k1 = np.zeros((1, 1, D)); k1[0, 0, :4] = 0.5        # score 2
    v0 = np.zeros((1, 1, D)); v0[0, 0, 0] = 1.0
    v1 = np.zeros((1, 1, D)); v1[0, 0, 1] = 1.0
    for scale in (0.125, 0.3, 1.0):
        out = oracle.draft_attention(bits(qv), bits(k1), bits(v1), bits(k0), bits(v0), np.array([0]),
                                     np.array([0, 1]), "bf16", 1, 1, D, scale)
        w0, w1 = out[0, 0, 0], out[0, 0, 1]
        assert w0 + w1 == pytest.approx(1.0, abs=1e-12)
        assert w0 / w1 == pytest.approx(np.exp(scale * 6.0), rel=1e-12)


def test_block_is_not_causal():
    """Query 0 of a block sees the block's last key: make that key dominant for
    it and the output is (nearly) that key's value."""
    E = 8
    q = np.zeros((E, 1, D)); q[0, 0, 0] = 4.0
    ke = np.zeros((E, 1, D)); ke[E - 1, 0, 0] = 4.0
    ve = np.zeros((E, 1, D)); ve[E - 1, 0, 5] = 1.0
    out = oracle.draft_attention(bits(q), bits(ke), bits(ve), bits(np.zeros((4, 1, D))), bits(np.zeros((4, 1, D))),
                                 np.array([0, 1, 2]), np.array([0, 3]), "bf16", 1, 1, D, 1.0)
    # weights: exp(16) for the last key, exp(0) for the other 7 + 3 keys
    w = np.exp(16.0) / (np.exp(16.0) + 10)
    assert out[0, 0, 5] == pytest.approx(w, rel=1e-12)


def test_context_order_does_not_matter():
    rng = np.random.default_rng(3)
    q, ke, ve, kp, vp, idx, start = build(2, 4, 4, 2, [30, 17], 128, rng)
    a = oracle.draft_attention(q, ke, ve, kp, vp, idx, start, "bf16", 4, 2, D, 0.125)
    idx2 = idx.copy()
    idx2[:30] = idx2[:30][::-1]
    idx2[30:] = rng.permutation(idx2[30:])
    b = oracle.draft_attention(q, ke, ve, kp, vp, idx2, start, "bf16", 4, 2, D, 0.125)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)
    with pytest.raises(ValueError):
        oracle.draft_attention(q, ke, ve, kp, vp, idx + 1000, start, "bf16", 4, 2, D, 0.125)
