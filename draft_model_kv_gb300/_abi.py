"""ctypes declarations of the C ABI in include/dspark_ctx_kv.h.

Loading fails loudly when the shared library has not been built: there is no
CPU fallback for any entry point.
"""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libdspark_ctx_kv.so")

DTYPE_BF16 = 1
DTYPE_FP16 = 2
DTYPE_FP32 = 3
DTYPE_OTHER = 100
VARIANT_AUTO, VARIANT_SINGLE, VARIANT_PAIR, VARIANT_STREAM = 0, 1, 2, 3          # any non-bf16/fp16 weight: the pack refuses it as non-sliceable
MAX_LAYERS = 32

FLAG_POS_RANGE = 0x1
FLAG_LOC_RANGE = 0x2
FLAG_TIMEOUT = 0x4

STATUS = {
    0: "OK", 1: "E_INVALID_ARG", 2: "E_NO_LAYERS", 3: "E_NOT_SLICEABLE", 4: "E_EPS_MISMATCH",
    5: "E_DTYPE_MISMATCH", 6: "E_SHAPE_MISMATCH", 7: "E_HEAD_DIM", 8: "E_BIAS_MISMATCH",
    9: "E_COMMIT_ARGS", 10: "E_NUMEL", 11: "E_ALIGNMENT", 12: "E_POOL_LAYOUT",
    13: "E_TOO_MANY_LAYERS", 14: "E_DEVICE", 15: "E_CUDA", 16: "E_DEVICE_FAULT",
    17: "E_SCRATCH_LIMIT",
}
CODE = {v: k for k, v in STATUS.items()}

EXPORTS = (
    "dspark_check_ctx_kv_layers", "dspark_pack_ctx_kv", "dspark_write_ctx_kv",
    "dspark_get_device_status", "dspark_read_device_status_async", "dspark_clear_device_status",
    "dspark_bundle_get_info",
    "dspark_free_bundle", "dspark_status_string", "dspark_set_trace_buffer",
    "dspark_write_ctx_kv_noalloc", "dspark_set_kernel_variant", "dspark_describe_schedule",
    "dspark_set_split_wait_test",
)


class LayerDesc(ctypes.Structure):
    _fields_ = [
        ("qkv_weight", ctypes.c_void_p),
        ("qkv_rows", ctypes.c_int64),
        ("qkv_row_stride", ctypes.c_int64),
        ("qkv_bias", ctypes.c_void_p),
        ("k_norm_weight", ctypes.c_void_p),
        ("weight_dtype", ctypes.c_int32),
        ("k_norm_dtype", ctypes.c_int32),
        ("q_size", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("eps", ctypes.c_float),
    ]


class ScheduleInfo(ctypes.Structure):
    _fields_ = [
        ("workers", ctypes.c_int32), ("whole_tiles", ctypes.c_int32), ("split_units", ctypes.c_int64),
        ("split_workers", ctypes.c_int32), ("split_first", ctypes.c_int32),
    ]


class BundleInfo(ctypes.Structure):
    _fields_ = [
        ("num_layers", ctypes.c_int32), ("hidden", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
        ("dtype", ctypes.c_int32), ("has_bias", ctypes.c_int32), ("device", ctypes.c_int32),
        ("eps", ctypes.c_float), ("stacked_rows", ctypes.c_int64),
    ]


_lib = None


def load() -> ctypes.CDLL:
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it with `python -m draft_model_kv_gb300.build` "
            "(the context-KV write has no CPU fallback)")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    lib.dspark_check_ctx_kv_layers.argtypes = [ctypes.POINTER(LayerDesc), i32, i32]
    lib.dspark_check_ctx_kv_layers.restype = ctypes.c_int
    lib.dspark_pack_ctx_kv.argtypes = [ctypes.POINTER(LayerDesc), i32, i32, vp, ctypes.POINTER(vp)]
    lib.dspark_pack_ctx_kv.restype = ctypes.c_int
    lib.dspark_write_ctx_kv.argtypes = [
        vp, vp, i64, i64, i32, vp, vp, i64, vp, vp, i64, i64,
        ctypes.POINTER(vp), ctypes.POINTER(vp), ctypes.POINTER(i64), ctypes.POINTER(i64),
        i32, i64, vp]
    lib.dspark_write_ctx_kv.restype = ctypes.c_int
    lib.dspark_get_device_status.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_uint32)]
    lib.dspark_get_device_status.restype = ctypes.c_int
    lib.dspark_read_device_status_async.argtypes = [vp, vp, vp]
    lib.dspark_read_device_status_async.restype = ctypes.c_int
    lib.dspark_clear_device_status.argtypes = [vp, vp]
    lib.dspark_clear_device_status.restype = ctypes.c_int
    lib.dspark_bundle_get_info.argtypes = [vp, ctypes.POINTER(BundleInfo)]
    lib.dspark_bundle_get_info.restype = ctypes.c_int
    lib.dspark_free_bundle.argtypes = [vp]
    lib.dspark_free_bundle.restype = None
    lib.dspark_write_ctx_kv_noalloc.argtypes = [
        vp, i64, vp, vp, ctypes.c_float, i32, i32, i32, i32, i32,
        vp, i64, i64, vp, vp, i64, vp, vp, i64, i64,
        ctypes.POINTER(vp), ctypes.POINTER(vp), ctypes.POINTER(i64), ctypes.POINTER(i64), i64,
        vp, vp]
    lib.dspark_write_ctx_kv_noalloc.restype = ctypes.c_int
    lib.dspark_set_kernel_variant.argtypes = [vp, i32]
    lib.dspark_set_kernel_variant.restype = ctypes.c_int
    lib.dspark_describe_schedule.argtypes = [i64, i32, i32, i32, ctypes.POINTER(ScheduleInfo)]
    lib.dspark_describe_schedule.restype = ctypes.c_int
    lib.dspark_set_trace_buffer.argtypes = [vp, vp, i64]
    lib.dspark_set_trace_buffer.restype = ctypes.c_int
    lib.dspark_set_split_wait_test.argtypes = [vp, i32, ctypes.c_uint64]
    lib.dspark_set_split_wait_test.restype = ctypes.c_int
    lib.dspark_qk_norm_rope.argtypes = [vp, i64, i64, i32, vp, vp, vp, vp, i64, i32, i32, i32,
                                        ctypes.c_float, vp, vp]
    lib.dspark_qk_norm_rope.restype = ctypes.c_int
    lib.dspark_correct_drafts_and_bonus.argtypes = [vp, i64, vp, i64, i64, i32, vp, vp, vp]
    lib.dspark_correct_drafts_and_bonus.restype = ctypes.c_int
    lib.dspark_draft_attention_workspace_bytes.argtypes = [i64, i32, i32, i32, i32, i64]
    lib.dspark_draft_attention_workspace_bytes.restype = i64
    lib.dspark_draft_attention.argtypes = [vp, vp, vp, vp, vp, i64, i64, vp, vp, i64, i32, i32, i32, i32, i32,
                                           ctypes.c_float, i64, vp, vp, i64, vp, vp]
    lib.dspark_draft_attention.restype = ctypes.c_int
    lib.dspark_draft_attention_set_wait_test.argtypes = [ctypes.c_uint64]
    lib.dspark_draft_attention_set_wait_test.restype = ctypes.c_int
    lib.dspark_pack_combine.argtypes = [vp, i64, i64, i64, i32, vp, i32, ctypes.c_float, vp, ctypes.POINTER(vp)]
    lib.dspark_pack_combine.restype = ctypes.c_int
    lib.dspark_combine_hidden_states.argtypes = [vp, vp, i64, i64, vp, i64, vp]
    lib.dspark_combine_hidden_states.restype = ctypes.c_int
    lib.dspark_combine_get_status.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_uint32)]
    lib.dspark_combine_get_status.restype = ctypes.c_int
    lib.dspark_free_combine.argtypes = [vp]
    lib.dspark_free_combine.restype = None
    lib.dspark_pack_fused_ctx_kv.argtypes = [vp, i64, i64, vp, i32, ctypes.c_float, ctypes.POINTER(LayerDesc), i32,
                                             i32, vp, ctypes.POINTER(vp)]
    lib.dspark_pack_fused_ctx_kv.restype = ctypes.c_int
    lib.dspark_combine_write_ctx_kv.argtypes = [
        vp, vp, i64, i64, vp, vp, i64, vp, vp, i64, i64,
        ctypes.POINTER(vp), ctypes.POINTER(vp), ctypes.POINTER(i64), ctypes.POINTER(i64), i32, i64, vp]
    lib.dspark_combine_write_ctx_kv.restype = ctypes.c_int
    lib.dspark_fused_get_status.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_uint32)]
    lib.dspark_fused_get_status.restype = ctypes.c_int
    lib.dspark_fused_clear_status.argtypes = [vp, vp]
    lib.dspark_fused_clear_status.restype = ctypes.c_int
    lib.dspark_free_fused.argtypes = [vp]
    lib.dspark_free_fused.restype = None
    lib.dspark_status_string.argtypes = [ctypes.c_int]
    lib.dspark_status_string.restype = ctypes.c_char_p
    _lib = lib
    return lib


class DSparkError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        self.name = STATUS.get(code, str(code))
        text = load().dspark_status_string(code).decode()
        super().__init__(f"{where}: DSPARK_{self.name} ({text})")


def check(code: int, where: str) -> None:
    if code != 0:
        raise DSparkError(code, where)
