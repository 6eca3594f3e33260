"""GPU parity: the CUDA path (through the C ABI) against the oracle.

Placement is checked bit-exactly: the set of pool slots whose bits changed
must equal the set the oracle writes, every other slot keeps the sentinel.
Values are checked element by element within rtol = atol = 2e-2 (bf16) or
5e-3 (fp16), the tolerances of the stacked-vs-per-layer parity test on the
sglang PR #31986 summary page.  Small cases compare every written row; the
full-size workloads compare a sample of tokens (tile edges plus random ones)
that the oracle computes one by one, and the complete placement.
"""
import functools

import numpy as np
import pytest

import oracle
import synthetic
from synthetic.device import make_pools, sentinel_int16, stage

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from draft_model_kv_gb300 import build
    build.build()


@functools.lru_cache(maxsize=4)
def workload(name, **kw):
    return synthetic.make_workload(name, **dict(kw))


def tol(w):
    return (2e-2, 2e-2) if w.dtype == "bf16" else (5e-3, 5e-3)


def run_gpu(w, row_pad=0, hidden_pad=0, st=None, variant="auto"):
    import draft_model_kv_gb300 as dk
    st = st or stage(w, row_pad=row_pad)
    x = st["ctx_hidden"]
    if hidden_pad:
        wide = torch.zeros((w.T, w.H + hidden_pad), dtype=x.dtype, device=x.device)
        wide[:, :w.H] = x
        x = wide[:, :w.H]
    b = dk.dspark_pack_ctx_kv(st["layers"], w.H)
    dk.dspark_set_kernel_variant(b, variant)
    dk.dspark_clear_device_status(b)
    dk.dspark_write_ctx_kv(b, x, st["positions"], st["cos_sin"], st["cache_loc"], st["k_pools"],
                           st["v_pools"], commit_lens=st["commit_lens"],
                           loc_row_width=st["loc_row_width"])
    torch.cuda.synchronize()
    flags = dk.dspark_get_device_status(b)
    return st, b, flags


def touched_slots(pool):
    bits = pool.view(torch.int16).reshape(pool.shape[0], -1)
    return torch.nonzero((bits != sentinel_int16()).any(dim=1)).flatten().cpu().numpy()


def check_placement(w, st):
    toks = oracle.written_tokens(w.cache_loc, w.commit_lens,
                                 w.loc_row_width if w.commit_lens is not None else None,
                                 w.pool_slots)
    expect = np.sort(w.cache_loc[toks])
    for pool in list(st["k_pools"]) + list(st["v_pools"]):
        np.testing.assert_array_equal(touched_slots(pool), expect)
    return toks


def check_values(w, st, sample=None):
    res = oracle.run_workload(w, sample=sample)
    rtol, atol = tol(w)
    slots = torch.from_numpy(res.slots).to("cuda")
    assert res.slots.size > 0
    for l in range(w.L):
        gk = st["k_pools"][l][slots].double().cpu().numpy()
        gv = st["v_pools"][l][slots].double().cpu().numpy()
        np.testing.assert_allclose(gk, res.k[l], rtol=rtol, atol=atol, err_msg=f"K layer {l}")
        np.testing.assert_allclose(gv, res.v[l], rtol=rtol, atol=atol, err_msg=f"V layer {l}")
    return res


def edge_sample(T, n_random=192, seed=0):
    edges = [0, 1, 126, 127, 128, 129, 255, 256, T // 2, T - 129, T - 128, T - 2, T - 1]
    rng = np.random.default_rng(seed)
    s = np.concatenate([[e for e in edges if 0 <= e < T], rng.integers(0, T, size=n_random)])
    return np.unique(s)


# ------------------------------------------------------------------ small cases, all rows

VARIANTS = ["single", "pair", "stream"]


def skip_if_unsupported(variant, T):
    if variant == "stream" and T > 256:
        pytest.skip("the weight-streaming kernel takes at most 256 tokens")


@pytest.mark.parametrize("variant", VARIANTS)
def test_tiny_full(variant):
    w = workload("tiny")
    st, _, flags = run_gpu(w, variant=variant)
    assert flags == 0
    check_placement(w, st)
    check_values(w, st)


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("T", [1, 7, 127, 128, 129, 255, 256, 257, 300])
def test_tiny_ragged_token_counts(T, variant):
    skip_if_unsupported(variant, T)
    w = workload("tiny", tokens=T)
    st, _, flags = run_gpu(w, variant=variant)
    assert flags == 0
    check_placement(w, st)
    check_values(w, st)


@pytest.mark.parametrize("variant", VARIANTS)
def test_decode_shapes_ragged_window_all_rows(variant):
    """Qwen3-8B-shaped decode (H=4096, 5 layers, 8x128) with 37 windows of 8:
    token tiles with a ragged tail, 40 column tiles, commit_lens truncation."""
    skip_if_unsupported(variant, 296)
    w = workload("decode512", tokens=296)
    st, _, flags = run_gpu(w, variant=variant)
    assert flags == 0
    check_placement(w, st)
    check_values(w, st)


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("T", [16, 64])
def test_decode_shapes_small_token_counts(T, variant):
    """Small T: every column tile is split across several CTAs (up to ~4
    contributors per tile), so the partial-tile fixup carries the result."""
    w = workload("decode512", tokens=T)
    st, _, flags = run_gpu(w, variant=variant)
    assert flags == 0
    check_placement(w, st)
    check_values(w, st)


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("T", [64, 256, 512])
def test_many_contributors_per_split_tile(T, variant):
    skip_if_unsupported(variant, T)
    """Few column tiles (N=512) over a long K (H=4096): every tile is cut
    across about 8 CTAs, too many parts for the finisher's staging area, so
    it reads them from the workspace directly (the staged path, up to 3-5
    other parts, is taken by the decode-shape small-T cases)."""
    w = workload("tiny", tokens=T, H=4096, pool_slots=512)
    st, _, flags = run_gpu(w, variant=variant)
    assert flags == 0
    check_placement(w, st)
    check_values(w, st)


@pytest.mark.parametrize("name,T", [("k3gqa", 64), ("fp16bias", 48), ("decode512", 200),
                                    ("decode512", 256)])
def test_small_token_counts_other_shapes(name, T):
    """The weight-streaming kernel (chosen automatically at T <= 64) on head
    dim 64, fp16 with bias, and token counts that are not a multiple of 32."""
    w = workload(name, tokens=T)
    st, _, flags = run_gpu(w, variant="stream")
    assert flags == 0
    check_placement(w, st)
    check_values(w, st)


def test_decode512_full():
    w = workload("decode512")
    st, _, flags = run_gpu(w)
    assert flags == 0
    check_placement(w, st)
    check_values(w, st)


def test_strided_hidden_and_padded_pool_rows():
    w = workload("tiny", tokens=200)
    st, _, flags = run_gpu(w, row_pad=64, hidden_pad=24)
    assert flags == 0
    check_placement(w, st)
    check_values(w, st)


# ------------------------------------------------------------------ full-size, sampled rows

def test_prefill32k_sampled():
    w = workload("prefill32k")
    st, _, flags = run_gpu(w)
    assert flags == 0
    check_placement(w, st)
    check_values(w, st, sample=edge_sample(w.T))


def test_fp16bias_sampled():
    w = workload("fp16bias")
    st, _, flags = run_gpu(w)
    assert flags == 0
    check_placement(w, st)
    check_values(w, st, sample=edge_sample(w.T))


def test_k3gqa_sampled():
    w = workload("k3gqa")
    st, _, flags = run_gpu(w)
    assert flags == 0
    check_placement(w, st)
    check_values(w, st, sample=edge_sample(w.T))


# ------------------------------------------------------------------ one-wave problems

@pytest.mark.parametrize("variant", ["single", "pair"])
@pytest.mark.parametrize("name,kw", [("decode512", ()), ("fp16bias", (("tokens", 304),)),
                                     ("k3gqa", (("tokens", 1000),)), ("tiny", (("tokens", 12000),)),
                                     ("tiny", (("tokens", 12000), ("H", 64)))])
def test_one_wave_problems(name, kw, variant):
    """Between one and two waves of tiles: the leftover tiles' k-blocks are
    spread over every worker and each contributor finishes a share of their
    rows (bias, head_dim 64, a ragged last token block, and with H = 64 a
    single k-block per tile, where no tile is cut at all)."""
    w = workload(name, **dict(kw))
    st, _, flags = run_gpu(w, variant=variant)
    assert flags == 0
    check_placement(w, st)
    check_values(w, st)


@pytest.mark.parametrize("variant", ["single", "pair"])
def test_one_wave_repeat_is_bitwise_deterministic(variant):
    w = workload("k3gqa", tokens=1000)
    st1, _, _ = run_gpu(w, variant=variant)
    st2, _, _ = run_gpu(w, variant=variant)
    for a, b in zip(st1["k_pools"] + st1["v_pools"], st2["k_pools"] + st2["v_pools"]):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


# ------------------------------------------------------------------ edge cases and errors

def test_zero_tokens_is_a_noop():
    import draft_model_kv_gb300 as dk
    w = workload("tiny")
    st = stage(w)
    b = dk.dspark_pack_ctx_kv(st["layers"], w.H)
    empty = st["ctx_hidden"][:0]
    dk.dspark_write_ctx_kv(b, empty, st["positions"][:0], st["cos_sin"], st["cache_loc"][:0],
                           st["k_pools"], st["v_pools"])
    torch.cuda.synchronize()
    for p in st["k_pools"] + st["v_pools"]:
        assert touched_slots(p).size == 0


def test_all_tokens_masked_writes_nothing():
    import draft_model_kv_gb300 as dk
    w = workload("decode512", tokens=64)
    st = stage(w)
    b = dk.dspark_pack_ctx_kv(st["layers"], w.H)
    zero = torch.zeros_like(st["commit_lens"])
    dk.dspark_write_ctx_kv(b, st["ctx_hidden"], st["positions"], st["cos_sin"], st["cache_loc"],
                           st["k_pools"], st["v_pools"], commit_lens=zero, loc_row_width=8)
    st["cache_loc"].fill_(-1)
    dk.dspark_write_ctx_kv(b, st["ctx_hidden"], st["positions"], st["cos_sin"], st["cache_loc"],
                           st["k_pools"], st["v_pools"])
    torch.cuda.synchronize()
    for p in st["k_pools"] + st["v_pools"]:
        assert touched_slots(p).size == 0


def test_out_of_range_position_and_loc_are_flagged_and_skipped():
    import draft_model_kv_gb300 as dk
    w = workload("tiny")
    st = stage(w)
    st["positions"][3] = w.max_pos          # outside the table
    st["positions"][5] = -2
    st["cache_loc"][7] = w.pool_slots + 10  # outside the pool
    b = dk.dspark_pack_ctx_kv(st["layers"], w.H)
    dk.dspark_clear_device_status(b)
    dk.dspark_write_ctx_kv(b, st["ctx_hidden"], st["positions"], st["cos_sin"], st["cache_loc"],
                           st["k_pools"], st["v_pools"])
    # the asynchronous read (pinned host word, no synchronisation of its own)
    # and the synchronous one agree
    word = torch.full((1,), -1, dtype=torch.int32).pin_memory()
    dk.dspark_read_device_status_async(b, word)
    torch.cuda.synchronize()
    assert int(word[0]) == (dk.FLAG_POS_RANGE | dk.FLAG_LOC_RANGE)
    flags = dk.dspark_get_device_status(b)
    assert flags == (dk.FLAG_POS_RANGE | dk.FLAG_LOC_RANGE)
    expect = np.sort(np.delete(w.cache_loc, [3, 5, 7]))
    for p in st["k_pools"] + st["v_pools"]:
        np.testing.assert_array_equal(touched_slots(p), expect)
    dk.dspark_clear_device_status(b)
    assert dk.dspark_get_device_status(b) == 0


@pytest.mark.parametrize("variant", VARIANTS)
def test_repeat_is_bitwise_deterministic(variant):
    w = workload("decode512", tokens=128)
    st1, _, _ = run_gpu(w, variant=variant)
    st2, _, _ = run_gpu(w, variant=variant)
    for a, b in zip(st1["k_pools"] + st1["v_pools"], st2["k_pools"] + st2["v_pools"]):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_argument_refusals():
    import draft_model_kv_gb300 as dk
    w = workload("decode512", tokens=64)
    st = stage(w)
    b = dk.dspark_pack_ctx_kv(st["layers"], w.H)
    args = (b, st["ctx_hidden"], st["positions"], st["cos_sin"], st["cache_loc"], st["k_pools"],
            st["v_pools"])
    with pytest.raises(dk.DSparkError) as e:
        dk.dspark_write_ctx_kv(*args, commit_lens=st["commit_lens"], loc_row_width=None)
    assert e.value.name == "E_COMMIT_ARGS"
    with pytest.raises(dk.DSparkError) as e:
        dk.dspark_write_ctx_kv(*args, commit_lens=None, loc_row_width=8)
    assert e.value.name == "E_COMMIT_ARGS"
    with pytest.raises(dk.DSparkError) as e:
        dk.dspark_write_ctx_kv(*args, commit_lens=st["commit_lens"][:-1], loc_row_width=8)
    assert e.value.name == "E_NUMEL"
    with pytest.raises(dk.DSparkError) as e:
        dk.dspark_write_ctx_kv(b, st["ctx_hidden"].half(), *args[2:])
    assert e.value.name == "E_DTYPE_MISMATCH"
    mis = torch.empty(w.T * w.H + 1, dtype=torch.bfloat16, device="cuda")[1:].view(w.T, w.H)
    with pytest.raises(dk.DSparkError) as e:
        dk.dspark_write_ctx_kv(b, mis, *args[2:])
    assert e.value.name == "E_ALIGNMENT"
    bad_layers = [l for l in st["layers"]]
    bad_layers[2].eps = 1e-3
    with pytest.raises(dk.DSparkError) as e:
        dk.dspark_pack_ctx_kv(bad_layers, w.H)
    assert e.value.name == "E_EPS_MISMATCH"
    torch.cuda.synchronize()
    for p in st["k_pools"] + st["v_pools"]:
        assert touched_slots(p).size == 0


def test_bundle_info_and_q_rows_never_read():
    """The synthetic Q rows are NaN: finite outputs everywhere show that the
    pack slices exactly rows [q_size, q_size + 2*kv_size)."""
    w = workload("tiny")
    st, b, _ = run_gpu(w)
    assert (b.num_layers, b.hidden, b.num_kv_heads, b.head_dim) == (w.L, w.H, w.NH, w.D)
    assert b.stacked_rows == w.N and not b.has_bias
    slots = torch.from_numpy(w.cache_loc).cuda()
    for p in st["k_pools"] + st["v_pools"]:
        assert torch.isfinite(p[slots].float()).all()


def test_bound_pools_write_the_same_bits():
    """A PoolSet (pools checked and marshalled once) writes exactly what the
    per-call pool lists write."""
    import draft_model_kv_gb300 as dk
    w = workload("decode512", tokens=296)
    st, b, flags = run_gpu(w)
    assert flags == 0
    pools = make_pools(w, "cuda")
    kp, vp = pools[0::2], pools[1::2]
    ps = dk.dspark_bind_pools(b, kp, vp)
    dk.dspark_write_ctx_kv(b, st["ctx_hidden"], st["positions"], st["cos_sin"], st["cache_loc"], ps,
                           commit_lens=st["commit_lens"], loc_row_width=st["loc_row_width"])
    torch.cuda.synchronize()
    assert dk.dspark_get_device_status(b) == 0
    for got, ref in zip(kp + vp, list(st["k_pools"]) + list(st["v_pools"])):
        assert torch.equal(got.view(torch.int16), ref.view(torch.int16))
    with pytest.raises(ValueError):
        dk.dspark_write_ctx_kv(b, st["ctx_hidden"], st["positions"], st["cos_sin"], st["cache_loc"], ps,
                               st["v_pools"], commit_lens=st["commit_lens"],
                               loc_row_width=st["loc_row_width"])
