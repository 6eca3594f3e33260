"""Parity of combine_hidden_states (main_proj on the tcgen05 kernel in plain
mode, then the in-place norm) with its oracle, within the model dtype's
tolerance (bf16 2e-2, fp16 5e-3, rtol = atol; the outputs are normalised to
unit mean square), on the context-KV workloads' shapes."""
import numpy as np
import pytest

import oracle
import synthetic
from synthetic.device import bits_to_tensor

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from draft_model_kv_gb300 import build
    build.build()


def run(cw, pad=0):
    import draft_model_kv_gb300 as dk
    dt = torch.bfloat16 if cw.dtype == "bf16" else torch.float16
    W = bits_to_tensor(cw.weight, dt, "cuda")
    c = dk.dspark_pack_combine(W, bits_to_tensor(cw.norm_weight, dt, "cuda"), cw.eps)
    aux = bits_to_tensor(cw.aux, dt, "cuda")
    out = torch.full((cw.T, cw.hidden + pad), 7.0, dtype=dt, device="cuda")
    dk.dspark_combine_hidden_states(c, aux, out=out[:, :cw.hidden])
    torch.cuda.synchronize()
    assert dk.dspark_combine_get_status(c) == 0
    c.free()
    return out


def check(cw, out, rows=None):
    rows = np.arange(cw.T) if rows is None else np.asarray(rows)
    ref = oracle.combine_hidden_states(cw.aux[rows], cw.weight, cw.norm_weight, cw.eps, cw.dtype)
    got = out[torch.from_numpy(rows).cuda(), :cw.hidden].double().cpu().numpy()
    tol = 2e-2 if cw.dtype == "bf16" else 5e-3
    np.testing.assert_allclose(got, ref, rtol=tol, atol=tol)


@pytest.mark.parametrize("T", [1, 7, 130, 300])
def test_small_hidden_ragged_tokens(T):
    cw = synthetic.make_combine_workload("tiny", tokens=T, hidden=512)
    out = run(cw, pad=8)
    check(cw, out)
    np.testing.assert_array_equal(out[:, cw.hidden:].float().cpu().numpy(), 7.0)   # padding untouched


def test_decode512_shapes_sampled():
    cw = synthetic.make_combine_workload("decode512")
    out = run(cw)
    rows = np.sort(np.random.default_rng(4).choice(cw.T, size=48, replace=False))
    check(cw, out, rows=np.concatenate([[0], rows, [cw.T - 1]]))


def test_4096_tokens_sampled():
    # the bench's second configuration: 16 x 16 pair tiles (three waves and a
    # leftover, whole tiles first); rows of the first, middle and last blocks
    cw = synthetic.make_combine_workload("prefill32k", tokens=4096)
    out = run(cw)
    rows = np.sort(np.random.default_rng(5).choice(cw.T, size=40, replace=False))
    check(cw, out, rows=np.concatenate([[0, 255, 256, 2047], rows, [cw.T - 1]]))


@pytest.mark.parametrize("name,T", [("fp16bias", 64), ("k3gqa", 40)])
def test_other_shapes(name, T):
    cw = synthetic.make_combine_workload(name, tokens=T)
    out = run(cw)
    check(cw, out)


def test_one_wave_of_tiles():
    # 94 tiles of 256 x 256 on 76 CTA pairs: the leftover tiles are split over
    # every pair and each contributor stores its share of their rows
    cw = synthetic.make_combine_workload("tiny", tokens=12000, hidden=512)
    out = run(cw)
    check(cw, out)
    again = run(cw)
    assert torch.equal(out.view(torch.int16), again.view(torch.int16))


def test_deterministic():
    cw = synthetic.make_combine_workload("tiny", tokens=200, hidden=1024)
    a = run(cw)
    b = run(cw)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_combine_then_write_matches_the_oracle_pipeline():
    """The draft step's front half: combine_hidden_states produces ctx_hidden
    on the device and the context-KV write consumes it.  The oracle side runs
    the same two steps from the same inputs (its ctx_hidden rounded to the
    model dtype by the oracle's own rounding), never from device values."""
    import dataclasses
    import draft_model_kv_gb300 as dk
    from synthetic.device import stage
    w = synthetic.make_workload("decode512", tokens=64)
    cw = synthetic.make_combine_workload("decode512", tokens=64)
    # the write's input is the oracle's combine output, in the model dtype
    ref_hidden = oracle.round_to(oracle.combine_hidden_states(cw.aux, cw.weight, cw.norm_weight, cw.eps,
                                                              cw.dtype), cw.dtype)
    w_ref = dataclasses.replace(w, ctx_hidden=synthetic.f32_to_bf16_bits(ref_hidden.astype(np.float32)))
    ref = oracle.run_workload(w_ref)
    st = stage(w)
    dt = torch.bfloat16
    c = dk.dspark_pack_combine(bits_to_tensor(cw.weight, dt, "cuda"), bits_to_tensor(cw.norm_weight, dt, "cuda"),
                               cw.eps)
    hidden = dk.dspark_combine_hidden_states(c, bits_to_tensor(cw.aux, dt, "cuda"))
    b = dk.dspark_pack_ctx_kv(st["layers"], w.H)
    dk.dspark_write_ctx_kv(b, hidden, st["positions"], st["cos_sin"], st["cache_loc"], st["k_pools"],
                           st["v_pools"], commit_lens=st["commit_lens"], loc_row_width=st["loc_row_width"])
    torch.cuda.synchronize()
    assert dk.dspark_get_device_status(b) == 0 and dk.dspark_combine_get_status(c) == 0
    slots = torch.from_numpy(ref.slots).cuda()
    for l in range(w.L):
        np.testing.assert_allclose(st["k_pools"][l][slots].double().cpu().numpy(), ref.k[l], rtol=2e-2, atol=2e-2)
        np.testing.assert_allclose(st["v_pools"][l][slots].double().cpu().numpy(), ref.v[l], rtol=2e-2, atol=2e-2)
    b.free()
    c.free()
