"""Size checks of the Python binding that run before the library is called.

The C entry points take buffer sizes on trust (a pointer carries none), so a
tensor that is too short for the arguments would make a kernel read past it.
The binding compares every size it can against the arguments and raises
ValueError before anything is launched.  These checks need no GPU: CPU
tensors stand in, and no call reaches the library.
"""
import pytest

torch = pytest.importorskip("torch")

import draft_model_kv_gb300 as dk  # noqa: E402

L, NH, D, H, T, SLOTS = 2, 2, 64, 256, 8, 32
N = L * 2 * NH * D


def noalloc_args(**over):
    a = dict(
        stacked_weight=torch.zeros((N, H), dtype=torch.bfloat16),
        k_norm_weight=torch.ones((L, D), dtype=torch.float32),
        eps=1e-6, num_layers=L, num_kv_heads=NH, head_dim=D,
        ctx_hidden=torch.zeros((T, H), dtype=torch.bfloat16),
        positions=torch.zeros(T, dtype=torch.int64),
        cos_sin=torch.zeros((64, D), dtype=torch.float32),
        cache_loc=torch.arange(T, dtype=torch.int64),
        k_pools=[torch.zeros((SLOTS, NH, D), dtype=torch.bfloat16) for _ in range(L)],
        v_pools=[torch.zeros((SLOTS, NH, D), dtype=torch.bfloat16) for _ in range(L)],
    )
    a.update(over)
    return a


@pytest.mark.parametrize("over,msg", [
    (dict(stacked_weight=torch.zeros((N - 128, H), dtype=torch.bfloat16)), "rows"),
    (dict(k_norm_weight=torch.ones((L, D // 2), dtype=torch.float32)), "k_norm_weight"),
    (dict(stacked_bias=torch.zeros(N - 1, dtype=torch.bfloat16)), "stacked_bias"),
    (dict(cos_sin=torch.zeros((64, D // 2), dtype=torch.float32)), "cos_sin"),
    (dict(positions=torch.zeros(T - 1, dtype=torch.int64)), "one entry per token"),
    (dict(cache_loc=torch.zeros(T + 1, dtype=torch.int64)), "one entry per token"),
    (dict(ctx_hidden=torch.zeros((T, H - 64), dtype=torch.bfloat16)), "columns"),
    (dict(k_pools=[torch.zeros((SLOTS, NH, D // 2), dtype=torch.bfloat16) for _ in range(L)]), "pools"),
    (dict(v_pools=[torch.zeros((SLOTS, NH - 1, D), dtype=torch.bfloat16) for _ in range(L)]), "pools"),
], ids=["short-weight", "k-norm", "bias", "cos-sin", "positions", "cache-loc", "hidden", "k-pool", "v-pool"])
def test_noalloc_wrapper_refuses_mismatched_sizes(over, msg, monkeypatch):
    def no_library():
        raise AssertionError("the library was called before the size check")
    monkeypatch.setattr(dk, "load", no_library)
    with pytest.raises(ValueError, match=msg):
        dk.dspark_write_ctx_kv_noalloc(**noalloc_args(**over))


def test_write_wrapper_refuses_mismatched_token_sizes(monkeypatch):
    def no_library():
        raise AssertionError("the library was called before the size check")
    monkeypatch.setattr(dk, "load", no_library)

    class FakeBundle:
        hidden, head_dim, num_layers, num_kv_heads = H, D, L, NH
    a = noalloc_args()
    for over, msg in ((dict(positions=torch.zeros(T + 3, dtype=torch.int64)), "one entry per token"),
                      (dict(cos_sin=torch.zeros((64, 2 * D), dtype=torch.float32)), "cos_sin"),
                      (dict(ctx_hidden=torch.zeros((T, H + 8), dtype=torch.bfloat16)), "columns")):
        b = dict(a, **over)
        with pytest.raises(ValueError, match=msg):
            dk.dspark_write_ctx_kv(FakeBundle(), b["ctx_hidden"], b["positions"], b["cos_sin"], b["cache_loc"],
                                   b["k_pools"], b["v_pools"])
