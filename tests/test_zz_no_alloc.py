"""The allocation-free entry point against the regular one.

dspark_write_ctx_kv_noalloc serves callers that cannot allocate device memory
(their own pool allocator owns it all, or they cannot afford cudaMalloc's
device-wide synchronisation).  It takes the stacked parameters from the caller
and keeps the kernel's scratch in a static device array.  Two calls in a row
must each reproduce what dspark_write_ctx_kv (bundle-owned scratch) writes:
the same pool slots, values within the parity tolerance.  The first workload
splits tiles between CTAs, so the static scratch is really used, and the
second call starts from the first call's leftovers in it.

This file is collected last on purpose: if it fails, every other GPU test has
already run.
"""
import numpy as np
import pytest

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


def touched(pool):
    bits = pool.view(torch.int16).reshape(pool.shape[0], -1)
    return torch.nonzero((bits != sentinel_int16()).any(dim=1)).flatten().cpu().numpy()


def write_with_bundle(w, st):
    import draft_model_kv_gb300 as dk
    b = dk.dspark_pack_ctx_kv(st["layers"], w.H)
    dk.dspark_write_ctx_kv(b, st["ctx_hidden"], st["positions"], st["cos_sin"], st["cache_loc"],
                           st["k_pools"], st["v_pools"], commit_lens=st["commit_lens"],
                           loc_row_width=st["loc_row_width"])
    torch.cuda.synchronize()
    assert dk.dspark_get_device_status(b) == 0
    b.free()


def stacked_params(w, st):
    kv = w.NH * w.D
    rows = slice(w.q_size, w.q_size + 2 * kv)
    weight = torch.cat([l.qkv_weight[rows] for l in st["layers"]], dim=0).contiguous()
    bias = None
    if st["layers"][0].qkv_bias is not None:
        bias = torch.cat([l.qkv_bias[rows] for l in st["layers"]], dim=0).contiguous()
    knorm = torch.stack([l.k_norm_weight.float() for l in st["layers"]], dim=0).contiguous()
    return weight, bias, knorm


# decode-split: 296 tokens, 120 tiles of 128 x 256 on at most 64 CTAs, the
# tail cut between CTAs (whole tiles first).  split-first: 200 tokens, 80
# tiles, one wave of 64 whole tiles and 16 leftover tiles cut over all 64 CTAs
# (every contributor finishes rows of the leftover).  fp16-bias: 48 tokens,
# every tile cut.  tiny: fewer tiles than CTAs.
@pytest.mark.parametrize("name,kw", [("decode512", {"tokens": 296}), ("decode512", {"tokens": 200}),
                                     ("fp16bias", {"tokens": 48}), ("tiny", {})],
                         ids=["decode-split", "split-first", "fp16-bias", "tiny"])
def test_noalloc_matches_regular_write_on_two_calls(name, kw):
    import draft_model_kv_gb300 as dk
    import oracle
    w = synthetic.make_workload(name, **kw)
    st = stage(w)
    write_with_bundle(w, st)
    ref_k, ref_v = st["k_pools"], st["v_pools"]
    weight, bias, knorm = stacked_params(w, st)
    rtol, atol = (2e-2, 2e-2) if w.dtype == "bf16" else (5e-3, 5e-3)
    expect = oracle.run_workload(w)
    for call in range(2):
        pools = make_pools(w, "cuda")
        kp, vp = pools[0::2], pools[1::2]
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        dk.dspark_write_ctx_kv_noalloc(weight, knorm, w.eps, w.L, w.NH, w.D, st["ctx_hidden"],
                                       st["positions"], st["cos_sin"], st["cache_loc"], kp, vp,
                                       stacked_bias=bias, commit_lens=st["commit_lens"],
                                       loc_row_width=st["loc_row_width"], status_flags=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0, f"call {call}: device status {int(status.item()):#x}"
        # against the oracle directly as well: the written slots and values
        idx = torch.from_numpy(expect.slots).cuda()
        for l in range(w.L):
            np.testing.assert_array_equal(touched(kp[l]), np.sort(expect.slots))
            np.testing.assert_allclose(kp[l][idx].double().cpu().numpy(), expect.k[l], rtol=rtol, atol=atol,
                                       err_msg=f"call {call} layer {l} K vs oracle")
            np.testing.assert_allclose(vp[l][idx].double().cpu().numpy(), expect.v[l], rtol=rtol, atol=atol,
                                       err_msg=f"call {call} layer {l} V vs oracle")
        for l in range(w.L):
            for got, ref in ((kp[l], ref_k[l]), (vp[l], ref_v[l])):
                slots = touched(ref)
                assert slots.size > 0
                np.testing.assert_array_equal(touched(got), slots, err_msg=f"call {call} layer {l}")
                idx = torch.from_numpy(slots).cuda()
                np.testing.assert_allclose(got[idx].double().cpu().numpy(),
                                           ref[idx].double().cpu().numpy(), rtol=rtol, atol=atol,
                                           err_msg=f"call {call} layer {l}")


def test_noalloc_refuses_bad_arguments_without_running():
    import draft_model_kv_gb300 as dk
    w = synthetic.make_workload("tiny")
    st = stage(w)
    weight, bias, knorm = stacked_params(w, st)
    with pytest.raises(dk.DSparkError) as e:
        dk.dspark_write_ctx_kv_noalloc(weight, knorm, w.eps, w.L, w.NH, w.D, st["ctx_hidden"],
                                       st["positions"], st["cos_sin"], st["cache_loc"],
                                       st["k_pools"], st["v_pools"], loc_row_width=8)
    assert e.value.name == "E_COMMIT_ARGS"
    torch.cuda.synchronize()
    for p in st["k_pools"] + st["v_pools"]:
        assert touched(p).size == 0


def test_noalloc_without_status_word_writes_the_same():
    """status_flags=None: the device flags go to the library's own word (and
    are discarded); the write itself is unchanged."""
    import draft_model_kv_gb300 as dk
    w = synthetic.make_workload("decode512", tokens=296)
    st = stage(w)
    weight, bias, knorm = stacked_params(w, st)
    outs = []
    for status in (torch.zeros(1, dtype=torch.int32, device="cuda"), None):
        pools = make_pools(w, "cuda")
        kp, vp = pools[0::2], pools[1::2]
        dk.dspark_write_ctx_kv_noalloc(weight, knorm, w.eps, w.L, w.NH, w.D, st["ctx_hidden"],
                                       st["positions"], st["cos_sin"], st["cache_loc"], kp, vp,
                                       commit_lens=st["commit_lens"], loc_row_width=st["loc_row_width"],
                                       status_flags=status)
        torch.cuda.synchronize()
        if status is not None:
            assert int(status.item()) == 0
        outs.append(kp + vp)
    for a, b in zip(*outs):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
