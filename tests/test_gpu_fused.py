"""combine_hidden_states fused into the context-KV write (one launch) against
the oracle pipeline.

The oracle side runs the two steps the pages describe, from the same host
inputs: oracle.combine_hidden_states (main_proj, y rounded to the model dtype,
main_norm), ctx_hidden rounded to the model dtype, then the per-layer write
(oracle.run_workload).  The fused path computes the same quantity with
main_norm's weight folded into the stacked K|V weights and each token row
scaled by 1/rms(y); its rounding points differ (ctx_hidden is not rounded, the
scaled weights are), by a few units of the model dtype's last place, well
inside the write's tolerance.  Placement is compared bit-exactly, values
element by element at rtol = atol = 2e-2 (bf16) or 5e-3 (fp16).
"""
import dataclasses

import numpy as np
import pytest

import oracle
import synthetic
from synthetic.device import bits_to_tensor, sentinel_int16, stage

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from draft_model_kv_gb300 import build
    build.build()


def touched(pool):
    bits = pool.view(torch.int16).reshape(pool.shape[0], -1)
    return torch.nonzero((bits != sentinel_int16()).any(dim=1)).flatten().cpu().numpy()


def run_fused(w, cw):
    import draft_model_kv_gb300 as dk
    st = stage(w)
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float16
    f = dk.dspark_pack_fused_ctx_kv(bits_to_tensor(cw.weight, dt, "cuda"), bits_to_tensor(cw.norm_weight, dt, "cuda"),
                                    cw.eps, st["layers"])
    dk.dspark_fused_clear_status(f)
    dk.dspark_combine_write_ctx_kv(f, bits_to_tensor(cw.aux, dt, "cuda"), st["positions"], st["cos_sin"],
                                   st["cache_loc"], st["k_pools"], st["v_pools"], commit_lens=st["commit_lens"],
                                   loc_row_width=st["loc_row_width"])
    torch.cuda.synchronize()
    flags = dk.dspark_fused_get_status(f)
    return st, f, flags


def oracle_pipeline(w, cw, sample=None):
    hidden = oracle.round_to(oracle.combine_hidden_states(cw.aux, cw.weight, cw.norm_weight, cw.eps, cw.dtype),
                             cw.dtype)
    w_ref = dataclasses.replace(w, ctx_hidden=synthetic.to_bits(hidden.astype(np.float32), w.dtype))
    return oracle.run_workload(w_ref, sample=sample)


def check(w, st, ref):
    toks = oracle.written_tokens(w.cache_loc, w.commit_lens,
                                 w.loc_row_width if w.commit_lens is not None else None, w.pool_slots)
    expect = np.sort(w.cache_loc[toks])
    for pool in list(st["k_pools"]) + list(st["v_pools"]):
        np.testing.assert_array_equal(touched(pool), expect)
    tol = 2e-2 if w.dtype == "bf16" else 5e-3
    slots = torch.from_numpy(ref.slots).cuda()
    for l in range(w.L):
        np.testing.assert_allclose(st["k_pools"][l][slots].double().cpu().numpy(), ref.k[l], rtol=tol, atol=tol,
                                   err_msg=f"K layer {l}")
        np.testing.assert_allclose(st["v_pools"][l][slots].double().cpu().numpy(), ref.v[l], rtol=tol, atol=tol,
                                   err_msg=f"V layer {l}")


# decode shapes at 64 and 296 tokens (both products cut over the CTA pairs),
# decode512 in full (split-first write), head_dim 64 (k3gqa) and fp16 with
# bias (fp16bias); tiny: hidden 256, one column tile of main_proj.
CASES = [("decode512", 64), ("decode512", 296), ("decode512", None), ("k3gqa", 40), ("fp16bias", 48),
         ("tiny", None)]


@pytest.mark.parametrize("name,tokens", CASES, ids=[f"{n}-{t}" for n, t in CASES])
def test_fused_matches_the_oracle_pipeline(name, tokens):
    w = synthetic.make_workload(name, **({} if tokens is None else {"tokens": tokens}))
    cw = synthetic.make_combine_workload(name, tokens=w.T)
    st, f, flags = run_fused(w, cw)
    assert flags == 0
    sample = None if w.T <= 300 else np.unique(np.concatenate([[0, 255, 256, w.T - 1],
                                                               np.random.default_rng(3).integers(0, w.T, 96)]))
    check(w, st, oracle_pipeline(w, cw, sample))
    f.free()


def test_fused_is_deterministic_and_reusable():
    """Two writes with one handle (its scratch and counters reused) store the
    same bits."""
    import draft_model_kv_gb300 as dk
    from synthetic.device import make_pools
    w = synthetic.make_workload("decode512", tokens=296)
    cw = synthetic.make_combine_workload("decode512", tokens=w.T)
    st, f, flags = run_fused(w, cw)
    assert flags == 0
    pools = make_pools(w, "cuda")
    kp, vp = pools[0::2], pools[1::2]
    dt = torch.bfloat16
    dk.dspark_combine_write_ctx_kv(f, bits_to_tensor(cw.aux, dt, "cuda"), st["positions"], st["cos_sin"],
                                   st["cache_loc"], kp, vp, commit_lens=st["commit_lens"],
                                   loc_row_width=st["loc_row_width"])
    torch.cuda.synchronize()
    assert dk.dspark_fused_get_status(f) == 0
    for a, b in zip(kp + vp, list(st["k_pools"]) + list(st["v_pools"])):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    f.free()
