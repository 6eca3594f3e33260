"""Host-side checks of the C ABI library (no GPU needed).

The library must load, export every entry point that include/*.h declares,
and refuse ineligible layer sets with the same verdicts as the oracle's
bundle rules, without touching a GPU.
"""
import ctypes
import glob
import os
import re

import numpy as np
import pytest

import oracle
from draft_model_kv_gb300 import _abi, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _abi.load()


def declared_symbols():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        names += re.findall(r"DSPARK_API\s+[\w\s\*]+?\b(dspark_\w+)\s*\(", text)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(lib):
    names = declared_symbols()
    assert len(names) >= 8
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) >= set(_abi.EXPORTS)


def test_status_strings(lib):
    for code in _abi.STATUS:
        s = lib.dspark_status_string(code).decode()
        assert s and s != "unknown status"
    assert lib.dspark_status_string(999).decode() == "unknown status"


FAKE = 0x10000  # never dereferenced: the check reads host fields only


def desc(dtype=_abi.DTYPE_BF16, eps=1e-6, bias=False, q=256, nh=2, d=64, rows=None, hidden=64,
         kn_dtype=None):
    return _abi.LayerDesc(qkv_weight=FAKE, qkv_rows=rows if rows is not None else q + 4 * nh * d // 2 * 2,
                          qkv_row_stride=hidden, qkv_bias=FAKE if bias else None,
                          k_norm_weight=FAKE, weight_dtype=dtype,
                          k_norm_dtype=kn_dtype if kn_dtype is not None else dtype,
                          q_size=q, num_kv_heads=nh, head_dim=d, eps=eps)


def check(lib, descs, hidden=64):
    arr = (_abi.LayerDesc * max(1, len(descs)))(*descs)
    return _abi.STATUS[lib.dspark_check_ctx_kv_layers(arr, len(descs), hidden)]


def test_layer_check_refusals(lib):
    assert check(lib, [desc(), desc(), desc()]) == "OK"
    assert check(lib, []) == "E_NO_LAYERS"
    assert check(lib, [desc(), desc(dtype=_abi.DTYPE_OTHER)]) == "E_NOT_SLICEABLE"
    assert check(lib, [desc(), desc(dtype=_abi.DTYPE_FP32)]) == "E_NOT_SLICEABLE"
    assert check(lib, [desc(), desc(eps=1e-5)]) == "E_EPS_MISMATCH"
    assert check(lib, [desc(), desc(dtype=_abi.DTYPE_FP16)]) == "E_DTYPE_MISMATCH"
    assert check(lib, [desc(), desc(nh=1, d=128)]) == "E_SHAPE_MISMATCH"
    assert check(lib, [desc(d=32, nh=4)]) == "E_HEAD_DIM"
    assert check(lib, [desc(bias=True), desc()]) == "E_BIAS_MISMATCH"
    assert check(lib, [desc(bias=True), desc(bias=True)]) == "OK"
    assert check(lib, [desc(rows=256 + 255)]) == "E_SHAPE_MISMATCH"
    assert check(lib, [desc()] * 33) == "E_TOO_MANY_LAYERS"
    assert check(lib, [desc(kn_dtype=_abi.DTYPE_FP32)]) == "OK"
    assert check(lib, [desc(kn_dtype=7)]) == "E_INVALID_ARG"
    assert check(lib, [desc()], hidden=0) == "E_INVALID_ARG"
    d = desc()
    d.qkv_row_stride = 32
    assert check(lib, [d]) == "E_INVALID_ARG"


def test_layer_check_agrees_with_oracle_rules(lib):
    """The same ineligible sets are refused by the library and by the oracle's
    bundle rules (the page-1 test's three cases plus dtype / shape / head_dim)."""
    rng = np.random.default_rng(0)
    H, NH, D, q = 16, 2, 64, 8

    def olayer(**kw):
        w = rng.integers(0, 2 ** 14, size=(q + 2 * NH * D, H)).astype(np.uint16)
        base = dict(qkv_weight=w, qkv_bias=None, k_norm_weight=np.zeros(D, np.uint16), eps=1e-6,
                    weight_dtype="bf16", q_size=q, num_kv_heads=NH, head_dim=D)
        base.update(kw)
        return oracle.LayerDesc(**base)

    to_code = {"bf16": _abi.DTYPE_BF16, "fp16": _abi.DTYPE_FP16}
    cases = [
        [olayer(), olayer()],
        [olayer(), olayer(weight_dtype="int8")],
        [olayer(), olayer(eps=1e-5)],
        [olayer(qkv_bias=np.zeros(q + 2 * NH * D, np.uint16)), olayer()],
        [olayer(), olayer(weight_dtype="fp16")],
        [olayer(), olayer(num_kv_heads=1, head_dim=128)],
        [olayer(num_kv_heads=4, head_dim=32)],
        [],
    ]
    names = {"ok": "OK", "no_layers": "E_NO_LAYERS", "not_sliceable": "E_NOT_SLICEABLE",
             "eps_mismatch": "E_EPS_MISMATCH", "bias_mismatch": "E_BIAS_MISMATCH",
             "dtype_mismatch": "E_DTYPE_MISMATCH", "shape_mismatch": "E_SHAPE_MISMATCH",
             "head_dim": "E_HEAD_DIM"}
    for layers in cases:
        _, why = oracle.stacked_ctx_kv_params(layers)
        descs = [_abi.LayerDesc(qkv_weight=FAKE, qkv_rows=l.qkv_weight.shape[0], qkv_row_stride=H,
                                qkv_bias=FAKE if l.qkv_bias is not None else None,
                                k_norm_weight=FAKE, weight_dtype=to_code.get(l.weight_dtype, 100),
                                k_norm_dtype=_abi.DTYPE_BF16, q_size=l.q_size,
                                num_kv_heads=l.num_kv_heads, head_dim=l.head_dim, eps=l.eps)
                 for l in layers]
        assert check(lib, descs, hidden=H) == names[why], (why, layers and layers[-1].weight_dtype)


def test_write_refuses_null_bundle_without_gpu(lib):
    null = ctypes.c_void_p(0)
    L = 1
    arr = (ctypes.c_void_p * L)()
    strides = (ctypes.c_int64 * L)()
    code = lib.dspark_write_ctx_kv(null, None, 4, 64, 1, None, None, 1, None, None, 0, 0, arr, arr,
                                   strides, strides, 1, 16, None)
    assert _abi.STATUS[code] == "E_INVALID_ARG"
    lib.dspark_free_bundle(null)  # NULL is a no-op
    flags = ctypes.c_uint32(7)
    assert _abi.STATUS[lib.dspark_get_device_status(null, None, ctypes.byref(flags))] == "E_INVALID_ARG"


def test_pack_refusal_needs_no_gpu(lib):
    """Refusals are decided before any CUDA call, so they work on a GPU-less host."""
    out = ctypes.c_void_p(123)
    arr = (_abi.LayerDesc * 2)(desc(), desc(eps=1e-3))
    assert _abi.STATUS[lib.dspark_pack_ctx_kv(arr, 2, 64, None, ctypes.byref(out))] == "E_EPS_MISMATCH"
    assert out.value is None


def test_bind_pools_checks_shapes_once():
    """dspark_bind_pools (host only) refuses pools that do not match the
    bundle's layers, heads and head_dim, and records pointers and strides."""
    import types
    import torch
    import draft_model_kv_gb300 as dk
    b = types.SimpleNamespace(handle=None, num_layers=2, num_kv_heads=2, head_dim=64)
    kp = [torch.zeros(8, 2, 64, dtype=torch.bfloat16) for _ in range(2)]
    vp = [torch.zeros(8, 2, 64, dtype=torch.bfloat16) for _ in range(2)]
    ps = dk.dspark_bind_pools(b, kp, vp)
    assert ps.slots == 8 and ps.num_layers == 2 and list(ps.k_strides) == [128, 128]
    assert ps.k_ptrs[1] == kp[1].data_ptr()
    with pytest.raises(ValueError):
        dk.dspark_bind_pools(b, kp[:1], vp)
    with pytest.raises(ValueError):
        dk.dspark_bind_pools(b, kp, [torch.zeros(8, 2, 32, dtype=torch.bfloat16)] * 2)
    with pytest.raises(TypeError):
        dk.dspark_bind_pools(b, kp, [torch.zeros(8, 2, 64, dtype=torch.float16)] * 2)


def test_qk_norm_rope_refuses_bad_arguments_before_any_gpu_work(lib):
    """dspark_qk_norm_rope checks its arguments on the host, before it looks
    for a device: these refusals need no GPU."""
    assert "dspark_qk_norm_rope" in declared_symbols()
    buf = ctypes.create_string_buffer(4096 + 16)
    base = (ctypes.addressof(buf) + 15) // 16 * 16
    f = lib.dspark_qk_norm_rope

    def call(qkv=base, T=4, stride=1024, dtype=1, pos=base, qw=base, kw=base, cs=base, max_pos=8,
             nq=4, nk=2, D=128, eps=1e-6):
        return _abi.STATUS[f(qkv, T, stride, dtype, pos, qw, kw, cs, max_pos, nq, nk, D, eps, None, None)]

    assert call(T=0, qkv=None) == "OK"                       # nothing to do
    assert call(nq=0, nk=0) == "OK"
    assert call(D=96) == "E_HEAD_DIM"
    assert call(dtype=3) == "E_DTYPE_MISMATCH"
    assert call(T=-1) == "E_INVALID_ARG"
    assert call(pos=None) == "E_INVALID_ARG"
    assert call(stride=6 * 128 - 8) == "E_POOL_LAYOUT"       # shorter than the Q and K heads
    assert call(qkv=base + 2) == "E_ALIGNMENT"
    assert call(stride=6 * 128 + 4) == "E_ALIGNMENT"


def test_correct_drafts_refuses_bad_arguments_before_any_gpu_work(lib):
    buf = ctypes.create_string_buffer(1024)
    p = ctypes.addressof(buf)
    f = lib.dspark_correct_drafts_and_bonus

    def call(c=p, cs=8, t=p, ts=8, batch=4, block=8, out_c=p, out_b=p):
        return _abi.STATUS[f(c, cs, t, ts, batch, block, out_c, out_b, None)]

    assert call(batch=0, c=None) == "OK"
    assert call(block=0) == "E_INVALID_ARG"
    assert call(batch=-1) == "E_INVALID_ARG"
    assert call(cs=7) == "E_INVALID_ARG"
    assert call(t=None) == "E_INVALID_ARG"
    assert call(out_b=None) == "E_INVALID_ARG"


def test_draft_attention_sizes_and_refusals_need_no_gpu(lib):
    """The workspace size query and the shape refusals run on the host."""
    ws = lib.dspark_draft_attention_workspace_bytes
    assert ws(64, 8, 32, 8, 128, 32768) > 0
    assert ws(64, 8, 32, 8, 96, 1000) == 0          # head_dim
    assert ws(64, 8, 30, 8, 128, 1000) == 0         # heads not grouped
    assert ws(64, 3, 32, 8, 128, 1000) == 0         # 12 rows per KV head
    assert ws(64, 16, 32, 8, 128, 1000) == 0        # 64 rows per KV head x 8 heads: 32 warps
    f = lib.dspark_draft_attention
    buf = ctypes.create_string_buffer(64)
    p = (ctypes.addressof(buf) + 15) // 16 * 16

    def call(D=128, dtype=1, block=8, nq=32, nkv=8, stride=1024, wsb=1 << 30, q=p):
        return _abi.STATUS[f(q, p, p, p, p, stride, 100, p, p, 4, block, nq, nkv, D, dtype, 0.1, 64, p, p, wsb,
                             None, None)]

    assert call(D=96) == "E_HEAD_DIM"
    assert call(dtype=3) == "E_DTYPE_MISMATCH"
    assert call(block=3) == "E_SHAPE_MISMATCH"
    assert call(stride=1000) == "E_POOL_LAYOUT"
    assert call(stride=1028) == "E_ALIGNMENT"
    assert call(q=p + 4) == "E_ALIGNMENT"
    assert call(wsb=16) == "E_SCRATCH_LIMIT"


def test_combine_refuses_bad_arguments_before_any_gpu_work(lib):
    buf = ctypes.create_string_buffer(64)
    p = (ctypes.addressof(buf) + 15) // 16 * 16
    out = ctypes.c_void_p()
    f = lib.dspark_pack_combine

    def pack(w=p, H=4096, K=12288, stride=12288, dtype=1, nw=p, ndt=3, eps=1e-6):
        return _abi.STATUS[f(w, H, K, stride, dtype, nw, ndt, eps, None, ctypes.byref(out))]

    assert pack(w=None) == "E_INVALID_ARG"
    assert pack(dtype=3) == "E_DTYPE_MISMATCH"
    assert pack(ndt=9) == "E_DTYPE_MISMATCH"
    assert pack(H=4016) == "E_SHAPE_MISMATCH"       # not a multiple of 32
    assert pack(stride=100) == "E_SHAPE_MISMATCH"
    assert pack(w=p + 2) == "E_ALIGNMENT"
    assert pack(eps=-1.0) == "E_INVALID_ARG"
    assert _abi.STATUS[lib.dspark_combine_hidden_states(None, p, 4, 8, p, 8, None)] == "E_INVALID_ARG"
    lib.dspark_free_combine(None)
