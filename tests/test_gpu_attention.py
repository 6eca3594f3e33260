"""Parity of the draft attention over the pool with its oracle.

dspark_draft_attention (through the C ABI) against oracle.draft_attention on
seeded synthetic pools and blocks, element by element.  Tolerance from the
arithmetic: scores and sums in fp32, the softmax weights rounded to the model
dtype before the P.V product (relative 2**-9 for bf16, 2**-12 for fp16) and
the output rounded once: rtol 2e-2 / atol 2e-3 for bf16, 5e-3 / 5e-4 for
fp16 (outputs are weighted means of N(0,1) values, mostly well below 1).
"""
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


def run(a, max_context=None, kv_indices=None):
    import draft_model_kv_gb300 as dk
    dt = torch.bfloat16 if a.dtype == "bf16" else torch.float16
    dev = "cuda"
    t = lambda x: bits_to_tensor(x, dt, dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    idx = a.kv_indices if kv_indices is None else kv_indices
    out = dk.dspark_draft_attention(t(a.q), t(a.k_ext), t(a.v_ext), t(a.k_pool), t(a.v_pool),
                                    torch.from_numpy(idx).to(dev), torch.from_numpy(a.kv_start).to(dev),
                                    a.sm_scale, a.max_context if max_context is None else max_context,
                                    status_flags=status)
    torch.cuda.synchronize()
    return out, int(status.item())


def check(a, out, requests=None, kv_start=None, kv_indices=None):
    ref = oracle.draft_attention(a.q, a.k_ext, a.v_ext, a.k_pool, a.v_pool,
                                 a.kv_indices if kv_indices is None else kv_indices,
                                 a.kv_start if kv_start is None else kv_start, a.dtype, a.num_q_heads,
                                 a.num_kv_heads, a.D, a.sm_scale, requests=requests)
    got = out.double().cpu().numpy()
    if requests is not None:
        got = np.concatenate([got[b * a.block:(b + 1) * a.block] for b in requests])
    rtol, atol = (2e-2, 2e-3) if a.dtype == "bf16" else (5e-3, 5e-4)
    np.testing.assert_allclose(got, ref, rtol=rtol, atol=atol)


@pytest.mark.parametrize("batch,block,nq,nkv,D,lo,hi,dtype", [
    (4, 8, 32, 8, 128, 10, 300, "bf16"),      # decode shapes, ragged chunks
    (3, 8, 32, 8, 64, 1, 200, "bf16"),        # head_dim 64
    (2, 8, 32, 8, 128, 3000, 5000, "bf16"),   # many context splits to merge
    (5, 16, 16, 8, 128, 0, 40, "bf16"),       # block 16, group 2, empty contexts
    (6, 4, 16, 4, 128, 17, 90, "bf16"),       # 16 rows per KV head (8 warps)
    (3, 8, 32, 8, 128, 50, 400, "fp16"),
    (1, 8, 32, 8, 128, 29000, 30000, "bf16"),  # one request: more than 32 splits to merge
], ids=["decode", "d64", "long", "block16", "rows16", "fp16", "splits34"])
def test_matches_oracle(batch, block, nq, nkv, D, lo, hi, dtype):
    a = synthetic.make_attention_workload(batch, block, nq, nkv, D, lo, hi, dtype=dtype)
    out, status = run(a)
    assert status == 0
    check(a, out)


def _widen_bf16(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32)


@pytest.mark.parametrize("lo,hi", [(600, 900), (2500, 3000)], ids=["one-split", "splits"])
def test_growing_scores_force_rescales(lo, hi):
    """Keys whose magnitude grows from chunk to chunk (x(1 + 4c) for the keys
    of the c-th 128-key chunk of every context, x40 for the block's own keys):
    every 32-key group's running maximum then grows by more than 2^8 in most
    chunks, so the lazy rescale of O^T (by all warps of a warpgroup, for the
    groups whose maximum grew) runs in every chunk, within a split, across
    context splits and in the chunk of the block's own keys."""
    import dataclasses
    a = synthetic.make_attention_workload(3 if hi < 2048 else 2, 8, 32, 8, 128, lo, hi)
    kp = _widen_bf16(a.k_pool)
    for b in range(a.batch):
        s0, s1 = int(a.kv_start[b]), int(a.kv_start[b + 1])
        grow = 1.0 + 4.0 * (np.arange(s1 - s0) // 128)
        kp[a.kv_indices[s0:s1]] *= grow[:, None, None].astype(np.float32)
    a = dataclasses.replace(a, k_pool=synthetic.to_bits(kp, "bf16"),
                            k_ext=synthetic.to_bits(_widen_bf16(a.k_ext) * np.float32(40.0), "bf16"))
    out, status = run(a)
    assert status == 0
    check(a, out)


def test_timeout_branch_returns_flags_and_leaves_the_context_usable():
    """A split-kernel wait that nothing completes (diagnostics switch, 20 us
    bound): the call returns with DSPARK_FLAG_TIMEOUT (0x4) in the status word;
    afterwards, switched off, the same inputs give the oracle's output."""
    import draft_model_kv_gb300 as dk
    a = synthetic.make_attention_workload(3, 8, 32, 8, 128, 300, 700)
    dk.dspark_draft_attention_set_wait_test(20_000)
    try:
        _, status = run(a)
    finally:
        dk.dspark_draft_attention_set_wait_test(0)
    assert status & 0x4
    out, status = run(a)
    assert status == 0
    check(a, out)


def test_bench_launch_configuration_sampled():
    """The bench's launch configuration (64 requests of 8 x 32 heads over 8 KV
    heads of 128, bf16, contexts up to 32768: the same context split and
    waves) with one 32768-token context and 63 short ones; the long request
    and two short ones are checked against the oracle."""
    ctx = [32768] + [int(c) for c in np.random.default_rng(11).integers(1, 200, size=63)]
    a = synthetic.make_attention_workload(64, 8, 32, 8, 128, 0, 0, contexts=ctx)
    out, flags = run(a, max_context=32768)
    assert flags == 0
    check(a, out, requests=[0, 1, 63])


@pytest.mark.parametrize("D,dtype", [(128, "fp16"), (64, "bf16")], ids=["fp16", "d64"])
def test_full_size_launch_other_dtype_and_head_dim_sampled(D, dtype):
    """The bench's launch shape (64 requests, 32 query / 8 KV heads, contexts
    up to 32768: sixteen context splits) in fp16 and with head_dim 64: one
    32768-token context, one of 20000 (a ragged last split) and 62 short ones;
    those two and a short one are checked against the oracle."""
    ctx = [32768, 20000] + [int(c) for c in np.random.default_rng(12).integers(1, 300, size=62)]
    a = synthetic.make_attention_workload(64, 8, 32, 8, D, 0, 0, contexts=ctx, dtype=dtype)
    out, flags = run(a, max_context=32768)
    assert flags == 0
    check(a, out, requests=[0, 1, 40])


def test_bad_index_is_flagged_and_skipped():
    a = synthetic.make_attention_workload(3, 8, 32, 8, 128, 20, 60)
    idx = a.kv_indices.copy()
    b0, b1 = a.kv_start[1], a.kv_start[2]
    idx[b0 + 3] = a.k_pool.shape[0] + 5          # request 1, key 3: outside the pool
    out, status = run(a, kv_indices=idx)
    assert status == 0x2                          # DSPARK_FLAG_LOC_RANGE
    # request 1 equals attention without that key; the others are untouched by it
    keep = np.concatenate([idx[:b0 + 3], idx[b0 + 4:]])
    start = a.kv_start.copy()
    start[2:] -= 1
    check(a, out, requests=[0, 1, 2], kv_start=start, kv_indices=keep)


def test_context_beyond_max_context_is_flagged():
    a = synthetic.make_attention_workload(2, 8, 32, 8, 128, 100, 120)
    out, status = run(a, max_context=64)
    assert status & 0x8                           # DSPARK_FLAG_CONTEXT_RANGE


def test_workspace_size_and_refusals():
    import draft_model_kv_gb300 as dk
    assert dk.dspark_draft_attention_workspace_bytes(64, 8, 32, 8, 128, 32768) > 0
    assert dk.dspark_draft_attention_workspace_bytes(64, 8, 32, 8, 96, 1000) == 0     # head_dim
    assert dk.dspark_draft_attention_workspace_bytes(64, 3, 32, 8, 128, 1000) == 0    # 12 rows per head
    a = synthetic.make_attention_workload(2, 8, 32, 8, 128, 10, 20)
    dt = torch.bfloat16
    t = lambda x: bits_to_tensor(x, dt, "cuda")
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(dk.DSparkError) as e:
        dk.dspark_draft_attention(t(a.q), t(a.k_ext), t(a.v_ext), t(a.k_pool), t(a.v_pool),
                                  torch.from_numpy(a.kv_indices).cuda(), torch.from_numpy(a.kv_start).cuda(),
                                  a.sm_scale, a.max_context, workspace=small)
    assert e.value.name == "E_SCRATCH_LIMIT"
