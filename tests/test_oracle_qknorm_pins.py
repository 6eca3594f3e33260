"""Pins for the QK RMSNorm + table neox RoPE oracle (oracle/qk_norm_rope.py).

The pages print no worked example for this kernel, so each pin is a closed
form, an exhaustive check or an invariant, chosen so that a plausible mistake
fails one of them: Q and K weights swapped or Q/K heads offset (distinct
weights), a dropped intermediate rounding (identity-row outputs must be
representable), GPT-J pairing or a sign flip (quarter-turn row), eps outside
the square root or a D-1 divisor (eps closed form), and a wrong rotation
(pair norm, multiplication by exp(i*theta)).
"""
import numpy as np
import pytest

import oracle
from synthetic import f32_to_bf16_bits, f32_to_fp16_bits

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def bf16_value(bits):
    return (np.asarray(bits, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)


def test_round_to_bf16_exhaustive():
    """Every bf16 value is a fixed point; every midpoint between neighbours
    goes to the neighbour with an even last bit; just off the midpoint goes to
    the nearer one."""
    bits = np.arange(0x0001, 0x7F80, dtype=np.uint32)          # positive finite
    v = bf16_value(bits)
    np.testing.assert_array_equal(oracle.round_to(v, "bf16"), v)
    np.testing.assert_array_equal(oracle.round_to(-v, "bf16"), -v)
    lo, hi = v[:-1], v[1:]
    mid = (lo + hi) / 2                                        # exact in float64
    even = np.where(bits[:-1] % 2 == 0, lo, hi)
    np.testing.assert_array_equal(oracle.round_to(mid, "bf16"), even)
    gap = hi - lo
    np.testing.assert_array_equal(oracle.round_to(mid - gap / 64, "bf16"), lo)
    np.testing.assert_array_equal(oracle.round_to(mid + gap / 64, "bf16"), hi)


def test_round_to_fp16_matches_numpy_conversion():
    """numpy converts float64 to float16 with round to nearest even, subnormals
    included; compare on every fp16 value, every midpoint and random values."""
    h = np.arange(0x0000, 0x7C00, dtype=np.uint16).view(np.float16).astype(np.float64)
    mids = (h[:-1] + h[1:]) / 2
    rng = np.random.default_rng(0)
    x = np.concatenate([h, mids, rng.standard_normal(100000) * 100, rng.standard_normal(10000) * 1e-6])
    x = np.concatenate([x, -x])
    np.testing.assert_array_equal(oracle.round_to(x, "fp16"), x.astype(np.float16).astype(np.float64))


def identity_and_quarter_table(D):
    """Row 0: cos 1, sin 0 (identity).  Row 1: cos 0, sin 1 (quarter turn)."""
    t = np.zeros((2, D), dtype=np.float32)
    t[0, :D // 2] = 1.0
    t[1, D // 2:] = 1.0
    return t


def const_heads(T, nq, nk, nv, D, values, dtype):
    """qkv bits whose every head is a constant (values[t, h]); V heads 7."""
    x = np.repeat(np.asarray(values, dtype=np.float32)[:, :, None], D, axis=2).reshape(T, (nq + nk) * D)
    x = np.concatenate([x, np.full((T, nv * D), 7.0, dtype=np.float32)], axis=1)
    return f32_to_bf16_bits(x) if dtype == "bf16" else f32_to_fp16_bits(x)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("D", [64, 128])
def test_identity_row_constant_heads_give_sign_times_weight(dtype, D):
    """Constant head c, eps 0, identity row: x * inv = sign(c) exactly, so the
    output is sign(c) * w, with the Q weight on Q heads and the K weight on K
    heads (2 and 0.5 here, so a swap or a head offset shows)."""
    nq, nk, T = 4, 2, 3
    vals = np.array([[1.5, -3.0, 0.25, -1.0, 2.0, -0.5],
                     [-2.0, 4.0, -8.0, 16.0, -0.125, 1.0],
                     [3.0, 3.0, -3.0, -3.0, 5.0, -5.0]])
    qkv = const_heads(T, nq, nk, 2, D, vals, dtype)
    to_bits = f32_to_bf16_bits if dtype == "bf16" else f32_to_fp16_bits
    wq = to_bits(np.full(D, 2.0, np.float32))
    wk = to_bits(np.full(D, 0.5, np.float32))
    out = oracle.table_qk_norm_rope(qkv, dtype, np.zeros(T, np.int64), wq, wk,
                                    identity_and_quarter_table(D), nq, nk, D, 0.0)
    expect = np.sign(vals)[:, :, None] * np.array([2.0] * nq + [0.5] * nk)[None, :, None]
    np.testing.assert_array_equal(out, np.broadcast_to(expect, out.shape))


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_identity_row_outputs_are_representable(dtype):
    """At the identity row the output is the intermediate value itself, which
    the page rounds to the model dtype: every element must be representable
    (random inputs almost never give representable x * inv * w)."""
    rng = np.random.default_rng(1)
    T, nq, nk, D = 16, 4, 2, 128
    to_bits = f32_to_bf16_bits if dtype == "bf16" else f32_to_fp16_bits
    qkv = to_bits(rng.standard_normal((T, (nq + 2 * nk) * D), dtype=np.float32))
    wq = to_bits(1 + 0.1 * rng.standard_normal(D, dtype=np.float32))
    wk = to_bits(1 + 0.1 * rng.standard_normal(D, dtype=np.float32))
    out = oracle.table_qk_norm_rope(qkv, dtype, np.zeros(T, np.int64), wq, wk,
                                    identity_and_quarter_table(D), nq, nk, D, 1e-6)
    if dtype == "bf16":
        rt = bf16_value(f32_to_bf16_bits(out.astype(np.float32)))
    else:
        rt = out.astype(np.float16).astype(np.float64)
    np.testing.assert_array_equal(rt, out)
    assert np.all(out != 0)


def test_quarter_turn_is_neox_rotate_half():
    """Quarter-turn row (cos 0, sin 1): out = (-x2, x1) where x1 / x2 are the
    first / second half.  Halves of +1 and +2 (eps 0, w 1) give first half
    -2/r and second half +1/r with r = sqrt(2.5); adjacent-pair pairing or a
    sign flip gives something else."""
    D, nq, nk = 128, 1, 1
    x = np.concatenate([np.ones(D // 2), 2 * np.ones(D // 2)]).astype(np.float32)
    qkv = f32_to_bf16_bits(np.tile(x, (1, nq + nk + 1)))
    one = f32_to_bf16_bits(np.ones(D, np.float32))
    out = oracle.table_qk_norm_rope(qkv, "bf16", np.array([1]), one, one,
                                    identity_and_quarter_table(D), nq, nk, D, 0.0)
    r = np.sqrt(2.5)
    x1 = oracle.round_to(np.array([1 / r]), "bf16")[0]
    x2 = oracle.round_to(np.array([2 / r]), "bf16")[0]
    expect = np.concatenate([-x2 * np.ones(D // 2), x1 * np.ones(D // 2)])
    for h in range(nq + nk):
        np.testing.assert_array_equal(out[0, h], expect)


def test_eps_inside_the_square_root_and_mean_over_head_dim():
    """Constant head 1 with eps 3: mean(x^2) + eps = 4, inv = 1/2, output 0.5
    exactly.  eps outside the root gives 1/(1+3)... = 4 or 0.25-type values and
    a D-1 divisor gives a value that is not 0.5."""
    D = 64
    qkv = const_heads(1, 1, 1, 1, D, np.array([[1.0, -1.0]]), "bf16")
    one = f32_to_bf16_bits(np.ones(D, np.float32))
    out = oracle.table_qk_norm_rope(qkv, "bf16", np.array([0]), one, one,
                                    identity_and_quarter_table(D), 1, 1, D, 3.0)
    np.testing.assert_array_equal(out[0, 0], 0.5 * np.ones(D))
    np.testing.assert_array_equal(out[0, 1], -0.5 * np.ones(D))


def test_rotation_preserves_pair_norm_and_is_exp_i_theta():
    """Against the identity-row output r (the rounded, normalised heads), the
    output at position p is (r1 + i r2) * (c + i s) with c, s the table row:
    each pair's norm is kept up to the table's rounding, and the complex
    product computed in complex128 agrees to float64 rounding."""
    rng = np.random.default_rng(2)
    T, nq, nk, D = 12, 3, 2, 128
    qkv = f32_to_bf16_bits(rng.standard_normal((T, (nq + 2 * nk) * D), dtype=np.float32))
    wq = f32_to_bf16_bits(1 + 0.1 * rng.standard_normal(D, dtype=np.float32))
    wk = f32_to_bf16_bits(1 + 0.1 * rng.standard_normal(D, dtype=np.float32))
    max_pos = 5000
    ang = np.arange(max_pos)[:, None] * (1e6 ** (-np.arange(D // 2) * 2.0 / D))[None, :]
    table = np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32)
    table[0, :D // 2], table[0, D // 2:] = 1.0, 0.0
    pos = rng.integers(1, max_pos, size=T)
    r = oracle.table_qk_norm_rope(qkv, "bf16", np.zeros(T, np.int64), wq, wk, table, nq, nk, D, 1e-6)
    o = oracle.table_qk_norm_rope(qkv, "bf16", pos, wq, wk, table, nq, nk, D, 1e-6)
    h = D // 2
    rz = r[..., :h] + 1j * r[..., h:]
    cs = table[pos].astype(np.float64)
    rot = (cs[:, None, :h] + 1j * cs[:, None, h:])
    oz = o[..., :h] + 1j * o[..., h:]
    np.testing.assert_allclose(oz, rz * rot, rtol=0, atol=1e-12)
    norm_err = np.abs(np.abs(rot) - 1).max()
    np.testing.assert_allclose(np.abs(oz), np.abs(rz), rtol=2 * norm_err + 1e-12, atol=1e-12)


def test_v_heads_and_tail_are_not_inputs():
    """Only the Q and K heads enter: changing V columns leaves the output
    unchanged; a short row or a position off the table is refused."""
    rng = np.random.default_rng(3)
    T, nq, nk, D = 4, 2, 1, 64
    qkv = f32_to_bf16_bits(rng.standard_normal((T, (nq + 2 * nk) * D), dtype=np.float32))
    w = f32_to_bf16_bits(np.ones(D, np.float32))
    tab = identity_and_quarter_table(D)
    a = oracle.table_qk_norm_rope(qkv, "bf16", np.zeros(T, np.int64), w, w, tab, nq, nk, D, 1e-6)
    qkv2 = qkv.copy()
    qkv2[:, (nq + nk) * D:] ^= 0x1234
    b = oracle.table_qk_norm_rope(qkv2, "bf16", np.zeros(T, np.int64), w, w, tab, nq, nk, D, 1e-6)
    np.testing.assert_array_equal(a, b)
    with pytest.raises(ValueError):
        oracle.table_qk_norm_rope(qkv[:, :D], "bf16", np.zeros(T, np.int64), w, w, tab, nq, nk, D, 1e-6)
    with pytest.raises(ValueError):
        oracle.table_qk_norm_rope(qkv, "bf16", np.full(T, 2), w, w, tab, nq, nk, D, 1e-6)
