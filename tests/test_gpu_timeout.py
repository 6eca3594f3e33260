"""The timeout branch of the write, reached on purpose (through the C ABI).

Every in-kernel wait is bounded: a wait that runs out sets DSPARK_FLAG_TIMEOUT
in the bundle's status word, the CTA stops its work, waits for its own copies
and tensor-core work, frees its tensor memory and returns.  Here the waits for
the parts other CTAs publish of a cut tile are made to run out: the
diagnostics entry point dspark_set_split_wait_test makes them wait for one
arrival more than there are contributors (a count no CTA reaches), bounded by
20 microseconds.  No fault, trap or endless wait is involved.

Each case checks that the call returns, that the write reports the timeout,
and that the bundle is usable afterwards: after dspark_clear_device_status and
back in normal mode, a write into fresh pools matches the oracle (placement
bit-exact, values within the bf16 tolerance).  The cases cover each kernel and
each finishing order: the weight-streaming kernel (every tile cut, the owner of
a tile's last k-block finishes it), single CTAs with cut tiles only, CTA pairs
in the split-first order (contributors finish rows of the leftover tiles while
their whole tile is still on the tensor cores) and CTA pairs with whole tiles
first.
"""
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


def touched(pool):
    bits = pool.view(torch.int16).reshape(pool.shape[0], -1)
    return torch.nonzero((bits != sentinel_int16()).any(dim=1)).flatten().cpu().numpy()


def write(dk, b, w, st, kp, vp):
    dk.dspark_write_ctx_kv(b, st["ctx_hidden"], st["positions"], st["cos_sin"], st["cache_loc"], kp, vp,
                           commit_lens=st["commit_lens"], loc_row_width=st["loc_row_width"])


def check_against_oracle(w, kp, vp, sample=None):
    toks = oracle.written_tokens(w.cache_loc, w.commit_lens,
                                 w.loc_row_width if w.commit_lens is not None else None, w.pool_slots)
    expect = np.sort(w.cache_loc[toks])
    for pool in list(kp) + list(vp):
        np.testing.assert_array_equal(touched(pool), expect)
    res = oracle.run_workload(w, sample=sample)
    idx = torch.from_numpy(res.slots).cuda()
    for l in range(w.L):
        np.testing.assert_allclose(kp[l][idx].double().cpu().numpy(), res.k[l], rtol=2e-2, atol=2e-2)
        np.testing.assert_allclose(vp[l][idx].double().cpu().numpy(), res.v[l], rtol=2e-2, atol=2e-2)


CASES = [
    ("stream", 16), ("stream", 64),   # weight streaming: every weight tile cut between ~2 SMs
    ("single", 120),                  # 40 tiles on 152 SMs: all cut, finished by their last owner
    ("pair", 512),                    # 80 tiles on 76 pairs: split-first, leftover on the V-tile pairs
    ("pair", 1024),                   # 160 tiles: one wave of whole tiles, then 84 cut tiles
]


@pytest.mark.parametrize("variant,tokens", CASES, ids=[f"{v}-{t}" for v, t in CASES])
def test_split_wait_runs_out_and_bundle_recovers(variant, tokens):
    import draft_model_kv_gb300 as dk
    w = synthetic.make_workload("decode512", tokens=tokens)
    st = stage(w)
    b = dk.dspark_pack_ctx_kv(st["layers"], w.H)
    dk.dspark_set_kernel_variant(b, variant)
    dk.dspark_clear_device_status(b)

    dk.dspark_set_split_wait_test(b, 1, 20_000)
    write(dk, b, w, st, st["k_pools"], st["v_pools"])      # returns: the launch itself succeeds
    torch.cuda.synchronize()
    flags = dk.dspark_get_device_status(b)
    assert flags & dk.FLAG_TIMEOUT, f"expected the timeout flag, got {flags:#x}"
    assert not flags & (dk.FLAG_POS_RANGE | dk.FLAG_LOC_RANGE)

    # back to normal: the same bundle writes correct pools again
    dk.dspark_set_split_wait_test(b, 0)
    dk.dspark_clear_device_status(b)
    pools = make_pools(w, "cuda")
    kp, vp = pools[0::2], pools[1::2]
    write(dk, b, w, st, kp, vp)
    torch.cuda.synchronize()
    assert dk.dspark_get_device_status(b) == 0
    sample = None if w.T <= 512 else np.unique(np.linspace(0, w.T - 1, 160).astype(np.int64))
    check_against_oracle(w, kp, vp, sample)
    b.free()


@pytest.mark.parametrize("name,tokens", [("tiny", None), ("decode512", 296)], ids=["tiny", "single-296"])
def test_split_wait_test_leaves_uncut_writes_alone(name, tokens):
    """tiny: 2 tiles of 4 k-blocks go to one CTA whole; 296 tokens on single
    CTAs: 120 tiles for 152 SMs, at least half as many tiles as workers, so
    each goes whole to one CTA.  No wait for other CTAs exists and the
    diagnostic mode changes nothing."""
    import draft_model_kv_gb300 as dk
    w = synthetic.make_workload(name, **({} if tokens is None else {"tokens": tokens}))
    st = stage(w)
    b = dk.dspark_pack_ctx_kv(st["layers"], w.H)
    dk.dspark_set_kernel_variant(b, "single")
    dk.dspark_clear_device_status(b)
    dk.dspark_set_split_wait_test(b, 1, 20_000)
    write(dk, b, w, st, st["k_pools"], st["v_pools"])
    torch.cuda.synchronize()
    assert dk.dspark_get_device_status(b) == 0
    check_against_oracle(w, st["k_pools"], st["v_pools"])
    b.free()


def test_split_wait_test_refuses_bad_limits():
    import draft_model_kv_gb300 as dk
    w = synthetic.make_workload("tiny")
    st = stage(w)
    b = dk.dspark_pack_ctx_kv(st["layers"], w.H)
    for missing, limit in ((1, 0), (1, 3_000_000_000), (-1, 1000), (2000, 1000)):
        with pytest.raises(dk.DSparkError) as e:
            dk.dspark_set_split_wait_test(b, missing, limit)
        assert e.value.name == "E_INVALID_ARG"
    b.free()
