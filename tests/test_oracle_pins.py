"""Pins of the oracle to facts that do not come from the oracle itself.

Each test names the fact it uses: brute force on exact small-integer inputs,
closed forms of special cases, invariants (RMS of a normalised vector, norm of
a rotated pair), an independent library routine (complex multiplication), and
hand-worked examples stored under tests/golden/.  Together they are chosen so
that a dropped term, a wrong sign or index, a transposed operand, a K/V swap,
a layer mix-up or an off-by-one in the window rule fails at least one of them.
"""
import functools
import json
import math
import os

import numpy as np
import pytest

import oracle
import synthetic
from oracle import LayerDesc
from synthetic import f32_to_bf16_bits, f32_to_fp16_bits

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def bf(x):
    return f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


def make_layer(wk, wv, knw, eps=1e-6, q_rows=3, bias=None, dtype="bf16", fill_q=np.nan):
    """A layer whose qkv weight holds q_rows Q rows (filled with fill_q), then wk, then wv."""
    wk = np.asarray(wk, dtype=np.float32)
    wv = np.asarray(wv, dtype=np.float32)
    H = wk.shape[1]
    q = np.full((q_rows, H), fill_q, dtype=np.float32)
    enc = bf if dtype == "bf16" else (lambda a: f32_to_fp16_bits(np.asarray(a, np.float32)))
    w = np.concatenate([enc(q), enc(wk), enc(wv)], axis=0)
    b = None
    if bias is not None:
        b = np.concatenate([enc(np.full(q_rows, np.nan)), enc(bias)])
    D = len(knw)
    return LayerDesc(qkv_weight=w, qkv_bias=b, k_norm_weight=enc(knw), eps=eps,
                     weight_dtype=dtype, q_size=q_rows, num_kv_heads=wk.shape[0] // D,
                     head_dim=D)


def identity_table(max_pos, D):
    t = np.zeros((max_pos, D), dtype=np.float32)
    t[:, :D // 2] = 1.0
    return t


# ---------------------------------------------------------------------------
# projection and stacking
# ---------------------------------------------------------------------------

def test_projection_matches_brute_force_triple_loop_exactly():
    """Brute force: small-integer inputs make every dot product exact in fp64,
    so the oracle's projection must equal a pure-Python triple loop bit for bit."""
    rng = np.random.default_rng(11)
    T, H, NH, D = 3, 5, 1, 4
    x = rng.integers(-3, 4, size=(T, H)).astype(np.float32)
    wk = rng.integers(-3, 4, size=(NH * D, H))
    wv = rng.integers(-3, 4, size=(NH * D, H))
    lay = make_layer(wk, wv, np.ones(D), q_rows=2)
    k, v = oracle.kv_proj_only(oracle.widen(bf(x), "bf16"), oracle.widen(lay.qkv_weight, "bf16"),
                               None, lay.q_size, NH * D)
    for t in range(T):
        for r in range(NH * D):
            sk = sum(float(x[t, j]) * float(wk[r, j]) for j in range(H))
            sv = sum(float(x[t, j]) * float(wv[r, j]) for j in range(H))
            assert k[t, r] == sk and v[t, r] == sv


def test_stacked_equals_per_layer_bit_exact_on_integer_inputs():
    """The stacking identity (shared input => concatenated rows give the same
    columns) holds exactly when all products are exact.  Layers get distinct
    weights, norm weights and a fixed per-layer offset so order mix-ups show."""
    rng = np.random.default_rng(5)
    T, H, NH, D, L = 4, 8, 2, 64, 3
    layers = []
    for l in range(L):
        wk = rng.integers(-2, 3, size=(NH * D, H)) + (l + 1)
        wv = rng.integers(-2, 3, size=(NH * D, H)) - (l + 1)
        layers.append(make_layer(wk, wv, 1.0 + 0.25 * rng.integers(0, 4, size=D), q_rows=5))
    x = bf(rng.integers(-2, 3, size=(T, H)))
    tab = synthetic.rope_cos_sin_table(64, D, 1e6)
    pos = rng.integers(0, 64, size=T)
    st, why = oracle.stacked_ctx_kv_params(layers)
    assert why == "ok" and st.weight.shape == (L * 2 * NH * D, H)
    ks, vs = oracle.per_layer_reference(x, layers, pos, tab)
    ks2, vs2 = oracle.project_stacked(x, st, pos, tab)
    for l in range(L):
        np.testing.assert_array_equal(ks[l], ks2[l])
        np.testing.assert_array_equal(vs[l], vs2[l])
    # layers really differ (the order check above is not vacuous)
    assert not np.array_equal(vs[0], vs[1])


def test_value_identity_weight_gives_hidden_columns():
    """Closed form: with W_v = c_l * [I | 0] the stored V of layer l is exactly
    c_l * ctx_hidden[:, :kv_size]; Q rows are NaN and K rows random, so
    reading the wrong slice, swapping K and V or mixing layers fails."""
    rng = np.random.default_rng(3)
    T, H, NH, D = 6, 200, 1, 128
    x = bf(rng.standard_normal((T, H)))
    layers = []
    for l in range(3):
        wv = np.zeros((NH * D, H))
        wv[:, :NH * D] = np.eye(NH * D) * (l + 1)
        layers.append(make_layer(rng.standard_normal((NH * D, H)), wv, np.ones(D), q_rows=7))
    tab = synthetic.rope_cos_sin_table(16, D, 1e6)
    ks, vs = oracle.per_layer_reference(x, layers, rng.integers(0, 16, size=T), tab)
    xv = oracle.widen(x, "bf16")
    for l in range(3):
        np.testing.assert_array_equal(vs[l].reshape(T, -1), (l + 1) * xv[:, :NH * D])
        assert np.isfinite(ks[l]).all()


def test_one_hot_hidden_selects_weight_column():
    """Closed form: a one-hot hidden row e_j projects to column j of W_v
    (catches a transposed weight: W_v is not square here)."""
    rng = np.random.default_rng(4)
    H, D = 96, 64
    wv = rng.standard_normal((D, H)).astype(np.float32)
    lay = make_layer(rng.standard_normal((D, H)), wv, np.ones(D), q_rows=1)
    for j in (0, 17, 95):
        x = np.zeros((1, H), np.float32)
        x[0, j] = 1.0
        _, vs = oracle.per_layer_reference(bf(x), [lay], np.zeros(1, np.int64),
                                           identity_table(1, D))
        np.testing.assert_array_equal(vs[0].reshape(-1), oracle.widen(bf(wv[:, j]), "bf16"))


# ---------------------------------------------------------------------------
# RMSNorm
# ---------------------------------------------------------------------------

def test_rmsnorm_of_constant_head_is_sign_times_weight():
    """Closed form: a head whose values are all c has mean square c^2, so with
    eps = 0 the normalised head is sign(c) * w exactly (up to rounding).  Two
    heads with different constants catch a norm taken over the whole KV row;
    per-layer weights catch a wrong k_norm index."""
    D, NH = 64, 2
    rng = np.random.default_rng(8)
    w_layers = [1.0 + 0.1 * rng.standard_normal(D) for _ in range(2)]
    for consts in ((3.0, -0.25), (-7.0, 0.5)):
        y = np.concatenate([np.full(D, consts[0]), np.full(D, consts[1])])[None, :]
        for wl in w_layers:
            w32 = wl.astype(np.float32).astype(np.float64)
            n = oracle.apply_k_norm(y, w32, 0.0, NH, D)
            expect = np.concatenate([np.sign(consts[0]) * w32, np.sign(consts[1]) * w32])
            np.testing.assert_allclose(n[0], expect, rtol=1e-14, atol=0)


def test_rmsnorm_mean_square_invariant_with_eps():
    """Invariant: with unit weights the normalised head has mean square
    ms / (ms + eps), where ms is the input's mean square (from numpy's norm)."""
    rng = np.random.default_rng(9)
    D, NH = 128, 4
    y = rng.standard_normal((5, NH * D)) * 0.01
    for eps in (0.0, 1e-6, 1e-4):
        n = oracle.apply_k_norm(y, np.ones(D), eps, NH, D).reshape(5, NH, D)
        ms = np.linalg.norm(y.reshape(5, NH, D), axis=-1) ** 2 / D
        np.testing.assert_allclose((n ** 2).mean(axis=-1), ms / (ms + eps), rtol=1e-12)


def test_rmsnorm_scale_invariant_without_eps():
    rng = np.random.default_rng(10)
    D = 64
    y = rng.standard_normal((3, 2 * D))
    w = rng.standard_normal(D)
    a = oracle.apply_k_norm(y, w, 0.0, 2, D)
    b = oracle.apply_k_norm(12.5 * y, w, 0.0, 2, D)
    np.testing.assert_allclose(a, b, rtol=1e-13)


# ---------------------------------------------------------------------------
# table RoPE
# ---------------------------------------------------------------------------

def test_rope_position_zero_is_identity():
    """Row 0 of any angle table is [1..1 | 0..0] exactly, so position 0 leaves
    the head unchanged."""
    rng = np.random.default_rng(12)
    D = 128
    tab = synthetic.rope_cos_sin_table(8, D, 1e6)
    assert (tab[0, :D // 2] == 1).all() and (tab[0, D // 2:] == 0).all()
    k = rng.standard_normal((4, 3 * D))
    out = oracle.apply_k_rope(np.zeros(4, np.int64), k, tab, 3, D)
    np.testing.assert_array_equal(out, k)


def test_rope_equals_complex_rotation_and_keeps_pair_norms():
    """Independent routine: pairing element i with i + D/2 as the complex
    number n_i + 1j * n_(i+D/2) and multiplying by exp(1j * theta_i(p)) with
    theta formed in fp64 must give the same pair (to the table's fp32 rounding);
    |pair| is preserved (invariant)."""
    rng = np.random.default_rng(13)
    D, NH, base = 64, 3, 1e6
    tab = synthetic.rope_cos_sin_table(5000, D, base)
    pos = rng.integers(0, 5000, size=7)
    n = rng.standard_normal((7, NH * D))
    out = oracle.apply_k_rope(pos, n, tab, NH, D).reshape(7, NH, D)
    nn = n.reshape(7, NH, D)
    i = np.arange(D // 2)
    theta = pos[:, None].astype(np.float64) * base ** (-2.0 * i / D)[None, :]
    z = (nn[..., :D // 2] + 1j * nn[..., D // 2:]) * np.exp(1j * theta)[:, None, :]
    np.testing.assert_allclose(out[..., :D // 2], z.real, atol=2e-6 * np.abs(nn).max())
    np.testing.assert_allclose(out[..., D // 2:], z.imag, atol=2e-6 * np.abs(nn).max())
    pair_in = nn[..., :D // 2] ** 2 + nn[..., D // 2:] ** 2
    pair_out = out[..., :D // 2] ** 2 + out[..., D // 2:] ** 2
    np.testing.assert_allclose(pair_out, pair_in, rtol=1e-6)


def test_rope_quarter_turn_moves_second_half_to_first_with_sign():
    """cos = 0, sin = 1: neox rotate-half sends (x1, x2) to (-x2, x1); an
    interleaved (GPT-J) pairing or a flipped sign would not."""
    D = 64
    tab = np.zeros((2, D), np.float32)
    tab[1, D // 2:] = 1.0
    x = np.arange(D, dtype=np.float64)[None, :] + 1
    out = oracle.apply_k_rope(np.array([1]), x, tab, 1, D)
    np.testing.assert_array_equal(out[0, :D // 2], -x[0, D // 2:])
    np.testing.assert_array_equal(out[0, D // 2:], x[0, :D // 2])


def _eval(expr):
    return float(eval(expr, {"__builtins__": {}}, {"sqrt": math.sqrt}))


def test_k_path_hand_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "k_path_worked.json")))
    lay = make_layer(g["w_k"], g["w_v"], g["k_norm_weight"], eps=g["eps"], q_rows=g["q_rows"])
    tab = np.asarray(g["table"], np.float32)
    ks, vs = oracle.per_layer_reference(bf([g["hidden"]]), [lay], np.array([g["position"]]), tab)
    np.testing.assert_allclose(ks[0].reshape(-1), [_eval(e) for e in g["expected_k"]],
                               atol=g["tolerance"], rtol=0)
    np.testing.assert_allclose(vs[0].reshape(-1), [_eval(e) for e in g["expected_v"]],
                               atol=0, rtol=0)


# ---------------------------------------------------------------------------
# bias
# ---------------------------------------------------------------------------

def test_bias_enters_k_before_norm_and_v_as_is():
    """Closed form: zero weights and a per-head constant bias b give
    V = bias exactly and, at position 0 with eps = 0, K = sign(b) * w."""
    D, NH, H = 64, 2, 32
    consts = [0.75, -2.0]
    bk = np.concatenate([np.full(D, c) for c in consts])
    bv = np.linspace(-1, 1, NH * D).astype(np.float32)
    w = (1.0 + 0.125 * np.arange(D) / D).astype(np.float32)
    lay = make_layer(np.zeros((NH * D, H)), np.zeros((NH * D, H)), w, eps=0.0, q_rows=4,
                     bias=np.concatenate([bk, bv]))
    x = bf(np.random.default_rng(1).standard_normal((3, H)))
    ks, vs = oracle.per_layer_reference(x, [lay], np.zeros(3, np.int64), identity_table(1, D))
    np.testing.assert_array_equal(vs[0].reshape(3, -1), np.tile(oracle.widen(bf(bv), "bf16"), (3, 1)))
    wb = oracle.widen(bf(w), "bf16")
    expect = np.concatenate([np.sign(c) * wb for c in consts])
    np.testing.assert_allclose(ks[0].reshape(3, -1), np.tile(expect, (3, 1)), rtol=1e-14)


# ---------------------------------------------------------------------------
# scatter rule
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("case", json.load(open(os.path.join(GOLDEN, "window_scatter.json")))["cases"],
                         ids=lambda c: c["name"])
def test_window_scatter_golden(case):
    loc = np.asarray(case["cache_loc"], np.int64)
    cl = None if case["commit_lens"] is None else np.asarray(case["commit_lens"], np.int32)
    toks = oracle.written_tokens(loc, cl, case["loc_row_width"], pool_slots=64)
    assert toks.tolist() == case["tokens"]
    assert loc[toks].tolist() == case["slots"]


def test_write_places_rows_only_in_written_slots():
    """Every written row carries the value of its own token; a token that is
    skipped contributes nothing (checked against an independent per-token call)."""
    w = synthetic.make_workload("tiny")
    loc = w.cache_loc.copy()
    loc[[3, 9, 10]] = -1
    descs = oracle.layer_descs(w)
    res = oracle.write_target_hidden_kv(w.ctx_hidden, descs, w.positions, w.cos_sin, loc,
                                        w.pool_slots)
    assert set(res.tokens.tolist()) == set(range(w.T)) - {3, 9, 10}
    for j, t in enumerate(res.tokens[:5]):
        ks, vs = oracle.per_layer_reference(w.ctx_hidden[t:t + 1], descs,
                                            w.positions[t:t + 1], w.cos_sin)
        for l in range(w.L):
            np.testing.assert_array_equal(res.k[l, j], ks[l][0])
            np.testing.assert_array_equal(res.v[l, j], vs[l][0])


def test_write_argument_errors():
    loc = np.arange(6, dtype=np.int64)
    with pytest.raises(oracle.WriteArgError):
        oracle.written_tokens(loc, np.array([1, 2], np.int32), None)
    with pytest.raises(oracle.WriteArgError):
        oracle.written_tokens(np.array([1, 1], np.int64))          # duplicate written slot
    with pytest.raises(oracle.WriteArgError):
        oracle.written_tokens(np.array([1, 70], np.int64), pool_slots=64)
    # a duplicate that is masked out is fine
    assert oracle.written_tokens(np.array([1, 1], np.int64), np.array([1], np.int32), 2).tolist() == [0]


def test_position_outside_table_is_an_error():
    w = synthetic.make_workload("tiny")
    pos = w.positions.copy()
    pos[4] = w.max_pos
    with pytest.raises(oracle.WriteArgError):
        oracle.write_target_hidden_kv(w.ctx_hidden, oracle.layer_descs(w), pos, w.cos_sin,
                                      w.cache_loc, w.pool_slots)


# ---------------------------------------------------------------------------
# refusals (PR #31986 test: quantized, eps mismatch, bias mismatch -> None)
# ---------------------------------------------------------------------------

def _tiny_layers(n=3, **kw):
    rng = np.random.default_rng(21)
    return [make_layer(rng.standard_normal((128, 16)), rng.standard_normal((128, 16)),
                       np.ones(64), **kw) for _ in range(n)]


def test_refusals():
    ok, why = oracle.stacked_ctx_kv_params(_tiny_layers())
    assert why == "ok" and ok is not None
    assert oracle.stacked_ctx_kv_params([]) == (None, "no_layers")
    lay = _tiny_layers()
    lay[1].weight_dtype = "fp8_e4m3"
    assert oracle.stacked_ctx_kv_params(lay) == (None, "not_sliceable")
    lay = _tiny_layers()
    lay[2].eps = 1e-5
    assert oracle.stacked_ctx_kv_params(lay) == (None, "eps_mismatch")
    lay = _tiny_layers()
    lay[1].qkv_bias = np.zeros(lay[1].qkv_weight.shape[0], np.uint16)
    assert oracle.stacked_ctx_kv_params(lay) == (None, "bias_mismatch")
    lay = _tiny_layers() + _tiny_layers(1, dtype="fp16")
    assert oracle.stacked_ctx_kv_params(lay) == (None, "dtype_mismatch")
    lay = _tiny_layers()
    lay[1].head_dim = 128
    lay[1].num_kv_heads = 1
    assert oracle.stacked_ctx_kv_params(lay) == (None, "shape_mismatch")
    rng = np.random.default_rng(2)
    odd = [make_layer(rng.standard_normal((32, 16)), rng.standard_normal((32, 16)), np.ones(32))]
    assert oracle.stacked_ctx_kv_params(odd) == (None, "head_dim")
    # all layers biased is accepted, and the bias is stacked K then V per layer
    lay = _tiny_layers()
    for l in lay:
        l.qkv_bias = np.arange(l.qkv_weight.shape[0], dtype=np.uint16)
    st, why = oracle.stacked_ctx_kv_params(lay)
    assert why == "ok" and st.bias.shape == (3 * 256,)
    assert st.k_norm_weight.shape == (3, 64)


# ---------------------------------------------------------------------------
# tolerance is meaningful: fp32 arithmetic sits far inside it
# ---------------------------------------------------------------------------

def test_fp32_oracle_within_small_fraction_of_tolerance():
    w = synthetic.make_workload("tiny")
    r64 = oracle.run_workload(w)
    r32 = oracle.run_workload(w, acc=np.float32)
    err = np.abs(r64.k - r32.k.astype(np.float64)).max()
    err_v = np.abs(r64.v - r32.v.astype(np.float64)).max()
    assert err < 2e-2 / 100 and err_v < 2e-2 / 100


# ---------------------------------------------------------------------------
# the eager-rounding reading (diagnostic mode of the oracle)
# ---------------------------------------------------------------------------

def test_eager_rounding_rounds_the_projection_and_the_normed_k():
    """Closed forms for where the eager reading rounds.  V: hidden [1, 1] and
    a V row [1, 2**-10] give 1 + 2**-10, which bf16 (8 significant bits)
    rounds to 1.0 -- the pure reading keeps 1 + 2**-10.  K: a constant head of
    3 with eps 0 normalises to w exactly (no rounding to see), while a head
    [3, 4, 0, ...] normalises to (3, 4) / rms and the eager reading rounds those
    values to bf16 before the (identity) rotation."""
    D, H = 64, 2
    wv = np.zeros((D, H), np.float32)
    wv[0] = [1.0, 2.0 ** -10]
    wk = np.zeros((D, H), np.float32)
    wk[:, 0] = 3.0
    lay = make_layer(wk, wv, np.ones(D), eps=0.0, q_rows=2)
    x = bf(np.array([[1.0, 1.0]], np.float32))
    pos = np.zeros(1, np.int64)
    tab = identity_table(1, D)
    ks, vs = oracle.per_layer_reference(x, [lay], pos, tab)
    ke, ve = oracle.per_layer_reference(x, [lay], pos, tab, eager=True)
    assert vs[0][0, 0, 0] == 1.0 + 2.0 ** -10 and ve[0][0, 0, 0] == 1.0
    np.testing.assert_array_equal(ks[0], ke[0])           # 3 / 3 * 1: representable
    wk2 = np.zeros((D, H), np.float32)
    wk2[0, 0], wk2[1, 0] = 3.0, 4.0
    lay2 = make_layer(wk2, wv, np.ones(D), eps=0.0, q_rows=2)
    ks2, _ = oracle.per_layer_reference(x, [lay2], pos, tab)
    ke2, _ = oracle.per_layer_reference(x, [lay2], pos, tab, eager=True)
    r = math.sqrt(25.0 / D)
    np.testing.assert_allclose(ks2[0][0, 0, :2], [3 / r, 4 / r], rtol=1e-15)
    np.testing.assert_array_equal(ke2[0][0, 0, :2], oracle.round_to(np.array([3 / r, 4 / r]), "bf16"))


@functools.lru_cache(maxsize=1)
def _decode_shapes_8():
    return synthetic.make_workload("decode512", tokens=8)


def test_eager_and_pure_readings_agree_within_the_tolerance():
    """The two readings of the unshown fused kernel's rounding differ by far
    less than the parity tolerance, so either is a valid reference."""
    w = _decode_shapes_8()
    a = oracle.run_workload(w)
    b = oracle.run_workload(w, eager=True)
    for x, y in ((a.k, b.k), (a.v, b.v)):
        assert np.all(np.abs(x - y) <= 2e-2 + 2e-2 * np.abs(x))
    assert not np.array_equal(a.k, b.k)
