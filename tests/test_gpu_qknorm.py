"""Parity of the in-place QK RMSNorm + table RoPE kernel with its oracle.

The CUDA path (dspark_qk_norm_rope through the C ABI) runs on the seeded
synthetic QKV rows of each workload's shapes; the Q and K heads are compared
with oracle.table_qk_norm_rope element by element within the model dtype's
tolerance (bf16 2e-2, fp16 5e-3, rtol = atol), every V column and any row
padding must keep its bits, and an out-of-table position leaves its row
untouched and sets the status flag.
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


def tdtype(q):
    return torch.bfloat16 if q.dtype == "bf16" else torch.float16


def run(q, pad=0, positions=None):
    """Apply the kernel to q's rows (row stride row + pad); returns the
    device tensor [T, row + pad] and the status word."""
    import draft_model_kv_gb300 as dk
    dt = tdtype(q)
    full = np.zeros((q.T, q.row + pad), dtype=np.uint16)
    full[:, :q.row] = q.qkv
    if pad:
        full[:, q.row:] = 0x3F80                  # padding columns: a recognisable pattern
    x = bits_to_tensor(full, dt, "cuda")
    pos = torch.from_numpy(q.positions if positions is None else positions).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    dk.dspark_qk_norm_rope(x, pos, bits_to_tensor(q.q_weight, dt, "cuda"), bits_to_tensor(q.k_weight, dt, "cuda"),
                           torch.from_numpy(q.cos_sin).cuda(), q.num_q_heads, q.num_k_heads, q.D, q.eps,
                           status_flags=status)
    torch.cuda.synchronize()
    return x, int(status.item()), full


def check(q, x, full, tokens=None):
    nqk = (q.num_q_heads + q.num_k_heads) * q.D
    got_bits = x.view(torch.int16).cpu().numpy().view(np.uint16)
    # V heads and padding keep their bits
    np.testing.assert_array_equal(got_bits[:, nqk:], full[:, nqk:])
    t_idx = np.arange(q.T) if tokens is None else np.asarray(tokens)
    ref = oracle.table_qk_norm_rope(q.qkv, q.dtype, q.positions, q.q_weight, q.k_weight, q.cos_sin,
                                    q.num_q_heads, q.num_k_heads, q.D, q.eps, tokens=t_idx)
    got = oracle.widen(got_bits[t_idx, :nqk], q.dtype).reshape(ref.shape)
    tol = 2e-2 if q.dtype == "bf16" else 5e-3
    np.testing.assert_allclose(got, ref, rtol=tol, atol=tol)


@pytest.mark.parametrize("name,kw", [("tiny", {}), ("decode512", {}), ("k3gqa", {"tokens": 256}),
                                     ("fp16bias", {"tokens": 512}), ("decode512", {"tokens": 8})],
                         ids=["tiny", "decode512", "k3gqa-256", "fp16bias-512", "decode-8"])
def test_matches_oracle(name, kw):
    q = synthetic.make_qknorm_workload(name, **kw)
    x, status, full = run(q)
    assert status == 0
    check(q, x, full)


@pytest.mark.parametrize("T", [1, 3, 33])
def test_ragged_token_counts_and_padded_rows(T):
    """Token counts that leave a partial last block, and rows with 8 extra
    columns after the V heads."""
    q = synthetic.make_qknorm_workload("tiny", tokens=T)
    x, status, full = run(q, pad=8)
    assert status == 0
    check(q, x, full)


def test_prefill32k_sampled():
    """The 32768-token shape in one launch (grid-stride over 1.3 M heads);
    compared on a seeded sample of tokens, every V column everywhere."""
    q = synthetic.make_qknorm_workload("prefill32k")
    x, status, full = run(q)
    assert status == 0
    sample = np.sort(np.random.default_rng(7).choice(q.T, size=256, replace=False))
    check(q, x, full, tokens=np.concatenate([[0], sample, [q.T - 1]]))


def test_out_of_table_position_is_flagged_and_skipped():
    q = synthetic.make_qknorm_workload("tiny", tokens=16)
    pos = q.positions.copy()
    bad = [2, 9]
    pos[2] = q.cos_sin.shape[0]
    pos[9] = -1
    x, status, full = run(q, positions=pos)
    assert status == 0x1                          # DSPARK_FLAG_POS_RANGE
    got = x.view(torch.int16).cpu().numpy().view(np.uint16)
    np.testing.assert_array_equal(got[bad], full[bad])
    good = np.array([t for t in range(q.T) if t not in bad])
    check(q, x, full, tokens=good)


def test_deterministic_and_zero_tokens():
    import draft_model_kv_gb300 as dk
    q = synthetic.make_qknorm_workload("decode512", tokens=64)
    a, _, _ = run(q)
    b, _, _ = run(q)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    empty = torch.empty((0, q.row), dtype=tdtype(q), device="cuda")
    w = torch.ones(q.D, dtype=tdtype(q), device="cuda")
    dk.dspark_qk_norm_rope(empty, torch.empty(0, dtype=torch.int64, device="cuda"), w, w,
                           torch.from_numpy(q.cos_sin).cuda(), q.num_q_heads, q.num_k_heads, q.D, q.eps)
