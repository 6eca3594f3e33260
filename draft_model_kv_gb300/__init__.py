"""DSpark draft-model context-KV write on one GB300 (sm_103a).

Python binding of the C ABI declared in include/dspark_ctx_kv.h, with the
same entry-point names.  It only marshals arguments: torch tensors supply
device pointers, strides and the current CUDA stream; every step of the write
runs in the library's CUDA kernels.  Importing works without a GPU (the
host-only eligibility check can run); GPU calls raise when the library is not
built or no sm_103 device is present.  There is no CPU fallback.
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass
from typing import Optional, Sequence

from . import _abi
from ._abi import (DSparkError, FLAG_LOC_RANGE, FLAG_POS_RANGE, FLAG_TIMEOUT,  # noqa: F401
                   LayerDesc, load)

__all__ = [
    "DSparkError", "Layer", "Bundle", "dspark_check_ctx_kv_layers", "dspark_pack_ctx_kv",
    "dspark_write_ctx_kv", "dspark_get_device_status", "dspark_read_device_status_async",
    "dspark_clear_device_status",
    "dspark_status_string", "dspark_set_trace_buffer", "dspark_write_ctx_kv_noalloc", "dspark_set_split_wait_test",
    "dspark_set_kernel_variant", "dspark_describe_schedule", "dspark_bind_pools", "PoolSet", "dspark_qk_norm_rope",
    "dspark_correct_drafts_and_bonus", "dspark_draft_attention", "dspark_draft_attention_workspace_bytes",
    "dspark_draft_attention_set_wait_test",
    "Combine", "dspark_pack_combine", "dspark_combine_hidden_states", "dspark_combine_get_status",
    "Fused", "dspark_pack_fused_ctx_kv", "dspark_combine_write_ctx_kv", "dspark_fused_get_status",
    "dspark_fused_clear_status",
    "FLAG_POS_RANGE", "FLAG_LOC_RANGE", "FLAG_TIMEOUT",
]


def _dtype_code(t) -> int:
    import torch
    return {torch.bfloat16: _abi.DTYPE_BF16, torch.float16: _abi.DTYPE_FP16,
            torch.float32: _abi.DTYPE_FP32}.get(t, _abi.DTYPE_OTHER)


def _stream_handle(stream) -> Optional[int]:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


@dataclass
class Layer:
    """One draft layer's attention parameters (device tensors)."""
    qkv_weight: object                 # [q_size + 2*kv_size (or more), hidden]
    k_norm_weight: object              # [head_dim]
    eps: float
    q_size: int
    num_kv_heads: int
    head_dim: int
    qkv_bias: object = None            # [rows] or None

    def desc(self) -> LayerDesc:
        w = self.qkv_weight
        if w.dim() != 2 or w.stride(1) != 1:
            raise ValueError("qkv_weight must be a 2-D tensor with unit column stride")
        return LayerDesc(
            qkv_weight=w.data_ptr(), qkv_rows=w.shape[0], qkv_row_stride=w.stride(0),
            qkv_bias=None if self.qkv_bias is None else self.qkv_bias.data_ptr(),
            k_norm_weight=self.k_norm_weight.data_ptr(), weight_dtype=_dtype_code(w.dtype),
            k_norm_dtype=_dtype_code(self.k_norm_weight.dtype), q_size=self.q_size,
            num_kv_heads=self.num_kv_heads, head_dim=self.head_dim, eps=self.eps)


def _desc_array(layers: Sequence) -> ctypes.Array:
    descs = [l if isinstance(l, LayerDesc) else l.desc() for l in layers]
    arr = (LayerDesc * max(1, len(descs)))()
    for i, d in enumerate(descs):
        arr[i] = d
    return arr


def dspark_check_ctx_kv_layers(layers: Sequence, hidden: int) -> int:
    """Host-only eligibility check; returns the status code (0 = stackable)."""
    arr = _desc_array(layers)
    return load().dspark_check_ctx_kv_layers(arr, len(layers), hidden)


def dspark_status_string(code: int) -> str:
    return load().dspark_status_string(code).decode()


class Bundle:
    """Owner of a packed dspark_bundle_t (freed on garbage collection)."""

    def __init__(self, handle: int):
        self.handle = ctypes.c_void_p(handle)
        info = _abi.BundleInfo()
        _abi.check(load().dspark_bundle_get_info(self.handle, ctypes.byref(info)),
                   "dspark_bundle_get_info")
        self.num_layers = info.num_layers
        self.hidden = info.hidden
        self.num_kv_heads = info.num_kv_heads
        self.head_dim = info.head_dim
        self.dtype_code = info.dtype
        self.has_bias = bool(info.has_bias)
        self.device = info.device
        self.eps = info.eps
        self.stacked_rows = info.stacked_rows

    def free(self) -> None:
        if self.handle is not None and self.handle.value:
            load().dspark_free_bundle(self.handle)
        self.handle = None

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass


def dspark_pack_ctx_kv(layers: Sequence, hidden: int, stream=None) -> Bundle:
    """Stack every layer's K|V projection slice into a library-owned bundle."""
    arr = _desc_array(layers)
    out = ctypes.c_void_p()
    _abi.check(load().dspark_pack_ctx_kv(arr, len(layers), hidden, _stream_handle(stream),
                                         ctypes.byref(out)), "dspark_pack_ctx_kv")
    return Bundle(out.value)


def _ptr_array(tensors):
    arr = (ctypes.c_void_p * len(tensors))()
    for i, t in enumerate(tensors):
        arr[i] = t.data_ptr()
    return arr


class PoolSet:
    """Every layer's K and V pool, checked once against a bundle.

    Built by dspark_bind_pools; pass it as `k_pools` (with `v_pools` None) to
    dspark_write_ctx_kv to skip the per-call checks and pointer marshalling of
    the pools.  It keeps references to the pool tensors, whose device pointers
    and row strides it records.
    """
    __slots__ = ("k_pools", "v_pools", "k_ptrs", "v_ptrs", "k_strides", "v_strides", "slots",
                 "dtype_code", "num_layers")


def dspark_bind_pools(bundle: Bundle, k_pools, v_pools) -> PoolSet:
    """Check one [slots, num_kv_heads, head_dim] pool per layer for K and V
    (head/dim strides (head_dim, 1), one dtype, one slot count) and record
    their pointers and row strides."""
    if len(k_pools) != bundle.num_layers or len(v_pools) != bundle.num_layers:
        raise ValueError("one K and one V pool per layer")
    slots = k_pools[0].shape[0]
    for p in list(k_pools) + list(v_pools):
        if p.dtype != k_pools[0].dtype:
            raise TypeError("all pools must share one dtype")
        if (p.dim() != 3 or p.shape[0] != slots or p.shape[1] != bundle.num_kv_heads
                or p.shape[2] != bundle.head_dim or p.stride(1) != bundle.head_dim or p.stride(2) != 1):
            raise ValueError("pools must be [slots, num_kv_heads, head_dim] with strides (*, head_dim, 1)")
    ps = PoolSet()
    L = bundle.num_layers
    ps.k_pools, ps.v_pools = tuple(k_pools), tuple(v_pools)
    ps.k_ptrs, ps.v_ptrs = _ptr_array(k_pools), _ptr_array(v_pools)
    ps.k_strides = (ctypes.c_int64 * L)(*[p.stride(0) for p in k_pools])
    ps.v_strides = (ctypes.c_int64 * L)(*[p.stride(0) for p in v_pools])
    ps.slots, ps.dtype_code, ps.num_layers = slots, _dtype_code(k_pools[0].dtype), L
    return ps


def _check_token_shapes(ctx_hidden, positions, cache_loc, cos_sin, hidden: int, head_dim: int) -> None:
    """The sizes the C ABI takes on trust: one position and one loc per token,
    hidden columns, and cos/sin rows of head_dim values."""
    T = ctx_hidden.shape[0]
    if ctx_hidden.shape[1] != hidden:
        raise ValueError(f"ctx_hidden has {ctx_hidden.shape[1]} columns, the layers take {hidden}")
    if positions.numel() != T or cache_loc.numel() != T:
        raise ValueError("positions and cache_loc must hold one entry per token")
    if cos_sin.dim() != 2 or cos_sin.shape[1] != head_dim or cos_sin.shape[0] < 1:
        raise ValueError(f"cos_sin must be [max_pos, head_dim={head_dim}]")


def dspark_write_ctx_kv(bundle: Bundle, ctx_hidden, positions, cos_sin, cache_loc, k_pools,
                        v_pools=None, commit_lens=None, loc_row_width: Optional[int] = None,
                        stream=None) -> None:
    """Write K (normed, roped) and V of every token into every layer's pool.

    ctx_hidden [T, hidden] (bundle dtype, unit column stride); positions and
    cache_loc int64 [T]; cos_sin fp32 [max_pos, head_dim]; commit_lens int32
    [bs] with loc_row_width W (bs * W == T) or neither; k_pools / v_pools: one
    [slots, num_kv_heads, head_dim] tensor per layer with head/dim strides
    (head_dim, 1), or k_pools a PoolSet from dspark_bind_pools and v_pools
    None.  Asynchronous on `stream` (default: torch's current stream).
    """
    import torch
    T = ctx_hidden.shape[0]
    if ctx_hidden.dim() != 2 or (T > 0 and ctx_hidden.stride(1) != 1):
        raise ValueError("ctx_hidden must be [T, hidden] with unit column stride")
    for name, t, dt in (("positions", positions, torch.int64), ("cache_loc", cache_loc, torch.int64),
                        ("cos_sin", cos_sin, torch.float32)):
        if t.dtype != dt or not t.is_contiguous():
            raise TypeError(f"{name} must be a contiguous {dt} tensor")
    if commit_lens is not None and (commit_lens.dtype != torch.int32 or not commit_lens.is_contiguous()):
        raise TypeError("commit_lens must be a contiguous int32 tensor")
    _check_token_shapes(ctx_hidden, positions, cache_loc, cos_sin, bundle.hidden, bundle.head_dim)
    if isinstance(k_pools, PoolSet):
        if v_pools is not None or k_pools.num_layers != bundle.num_layers:
            raise ValueError("a PoolSet of this bundle's layer count goes alone in k_pools")
        ps = k_pools
    else:
        ps = dspark_bind_pools(bundle, k_pools, v_pools)
    width = 0 if loc_row_width is None else int(loc_row_width)
    nwin = 0 if commit_lens is None else commit_lens.numel()
    code = load().dspark_write_ctx_kv(
        bundle.handle, ctx_hidden.data_ptr(), T, ctx_hidden.stride(0) if T > 0 else ctx_hidden.shape[1],
        _dtype_code(ctx_hidden.dtype), positions.data_ptr(), cos_sin.data_ptr(), cos_sin.shape[0],
        cache_loc.data_ptr(), None if commit_lens is None else commit_lens.data_ptr(), width, nwin,
        ps.k_ptrs, ps.v_ptrs, ps.k_strides, ps.v_strides, ps.dtype_code, ps.slots,
        _stream_handle(stream))
    _abi.check(code, "dspark_write_ctx_kv")


def dspark_get_device_status(bundle: Bundle, stream=None) -> int:
    flags = ctypes.c_uint32(0)
    _abi.check(load().dspark_get_device_status(bundle.handle, _stream_handle(stream),
                                               ctypes.byref(flags)), "dspark_get_device_status")
    return flags.value


def dspark_read_device_status_async(bundle: Bundle, out, stream=None) -> None:
    """Enqueue on `stream` the copy of the bundle's status word into `out`, a
    one-element int32/uint32 CPU tensor (pinned for a truly asynchronous
    copy); read `out` only after synchronising the stream."""
    import torch
    if out.device.type != "cpu" or out.numel() < 1 or out.element_size() != 4 or not out.is_contiguous():
        raise ValueError("out must be a contiguous CPU tensor of 4-byte elements")
    _abi.check(load().dspark_read_device_status_async(bundle.handle, _stream_handle(stream), out.data_ptr()),
               "dspark_read_device_status_async")


def dspark_clear_device_status(bundle: Bundle, stream=None) -> None:
    _abi.check(load().dspark_clear_device_status(bundle.handle, _stream_handle(stream)),
               "dspark_clear_device_status")


def dspark_set_trace_buffer(bundle: Bundle, buf) -> None:
    """Record per-CTA timelines of later writes into `buf` (a uint64-sized
    CUDA tensor of at least SMs x 64 words), or stop recording (None)."""
    if buf is None:
        code = load().dspark_set_trace_buffer(bundle.handle, None, 0)
    else:
        code = load().dspark_set_trace_buffer(bundle.handle, buf.data_ptr(), buf.numel())
    _abi.check(code, "dspark_set_trace_buffer")


def dspark_set_split_wait_test(bundle: Bundle, missing_arrivals: int, limit_ns: int = 0) -> None:
    """Diagnostics for tests of the timeout path: later writes with `bundle`
    wait for `missing_arrivals` more published parts of every cut tile than
    exist, each such wait bounded by `limit_ns`, so those waits run out and the
    write reports DSPARK_FLAG_TIMEOUT.  0 restores normal writes."""
    _abi.check(load().dspark_set_split_wait_test(bundle.handle, int(missing_arrivals), int(limit_ns)),
               "dspark_set_split_wait_test")


def dspark_write_ctx_kv_noalloc(stacked_weight, k_norm_weight, eps: float, num_layers: int,
                                num_kv_heads: int, head_dim: int, ctx_hidden, positions, cos_sin,
                                cache_loc, k_pools, v_pools, stacked_bias=None, commit_lens=None,
                                loc_row_width: Optional[int] = None, status_flags=None,
                                stream=None) -> None:
    """The write for callers that must not allocate device memory.

    For frameworks whose own allocator owns all device memory, or loops that
    cannot afford cudaMalloc's device-wide synchronisation.  The caller passes
    the stacked weight [N, hidden] (rows l0:K, l0:V, l1:K, ...), the fp32
    k_norm weights [num_layers, head_dim], optional stacked bias [N], every
    input and the pools; the kernel's scratch lives in a fixed 16 MiB + 4 KiB
    device array inside the library (at most 64 SMs per call).  Calls share
    that array, so calls whose kernels overlap on the GPU race: keep them
    ordered.  Make the first call on a device before any stream capture.
    status_flags: a one-element int32 CUDA tensor that receives the device
    flags (out-of-range position or slot, a wait that ran out); with None
    those flags are discarded and cannot be read back.  Sizes are checked
    here, before the library is called, since the C entry point has no
    bundle to check them against.
    """
    import torch
    T = ctx_hidden.shape[0]
    if stacked_weight.dim() != 2 or stacked_weight.stride(1) != 1:
        raise ValueError("stacked_weight must be [N, hidden] with unit column stride")
    if k_norm_weight.dtype != torch.float32 or not k_norm_weight.is_contiguous():
        raise TypeError("k_norm_weight must be a contiguous float32 [num_layers, head_dim] tensor")
    if ctx_hidden.dim() != 2 or (T > 0 and ctx_hidden.stride(1) != 1):
        raise ValueError("ctx_hidden must be [T, hidden] with unit column stride")
    for name, t, dt in (("positions", positions, torch.int64), ("cache_loc", cache_loc, torch.int64),
                        ("cos_sin", cos_sin, torch.float32)):
        if t.dtype != dt or not t.is_contiguous():
            raise TypeError(f"{name} must be a contiguous {dt} tensor")
    if commit_lens is not None and (commit_lens.dtype != torch.int32 or not commit_lens.is_contiguous()):
        raise TypeError("commit_lens must be a contiguous int32 tensor")
    if len(k_pools) != num_layers or len(v_pools) != num_layers:
        raise ValueError("one K and one V pool per layer")
    # the C ABI takes these sizes on trust (there is no bundle to check them
    # against): a mismatch would make the kernel read past a tensor
    n_rows = num_layers * 2 * num_kv_heads * head_dim
    hidden = stacked_weight.shape[1]
    if stacked_weight.shape[0] != n_rows:
        raise ValueError(f"stacked_weight must have num_layers*2*num_kv_heads*head_dim = {n_rows} rows, "
                         f"got {stacked_weight.shape[0]}")
    if tuple(k_norm_weight.shape) != (num_layers, head_dim):
        raise ValueError(f"k_norm_weight must be [num_layers, head_dim] = [{num_layers}, {head_dim}]")
    if stacked_bias is not None and (stacked_bias.numel() != n_rows or not stacked_bias.is_contiguous()):
        raise ValueError(f"stacked_bias must be a contiguous [{n_rows}] tensor")
    _check_token_shapes(ctx_hidden, positions, cache_loc, cos_sin, hidden, head_dim)
    slots = k_pools[0].shape[0]
    for p in list(k_pools) + list(v_pools):
        if (p.dim() != 3 or p.shape[0] != slots or p.shape[1] != num_kv_heads or p.shape[2] != head_dim
                or p.stride(1) != head_dim or p.stride(2) != 1):
            raise ValueError("pools must be [slots, num_kv_heads, head_dim] with strides (*, head_dim, 1) "
                             "and one slot count")
    if status_flags is not None and (status_flags.numel() < 1 or status_flags.element_size() != 4):
        raise TypeError("status_flags must be a 4-byte integer CUDA tensor")
    dt = stacked_weight.dtype
    for t in [ctx_hidden] + list(k_pools) + list(v_pools) + ([] if stacked_bias is None else [stacked_bias]):
        if t.dtype != dt:
            raise TypeError("weights, hidden, bias and pools must share one dtype")
    width = 0 if loc_row_width is None else int(loc_row_width)
    nwin = 0 if commit_lens is None else commit_lens.numel()
    kstr = (ctypes.c_int64 * num_layers)(*[p.stride(0) for p in k_pools])
    vstr = (ctypes.c_int64 * num_layers)(*[p.stride(0) for p in v_pools])
    code = load().dspark_write_ctx_kv_noalloc(
        stacked_weight.data_ptr(), stacked_weight.stride(0),
        None if stacked_bias is None else stacked_bias.data_ptr(), k_norm_weight.data_ptr(),
        eps, num_layers, stacked_weight.shape[1], num_kv_heads, head_dim, _dtype_code(dt),
        ctx_hidden.data_ptr(), T, ctx_hidden.stride(0) if T > 0 else ctx_hidden.shape[1],
        positions.data_ptr(), cos_sin.data_ptr(), cos_sin.shape[0], cache_loc.data_ptr(),
        None if commit_lens is None else commit_lens.data_ptr(), width, nwin,
        _ptr_array(k_pools), _ptr_array(v_pools), kstr, vstr, slots,
        None if status_flags is None else status_flags.data_ptr(), _stream_handle(stream))
    _abi.check(code, "dspark_write_ctx_kv_noalloc")


def dspark_qk_norm_rope(qkv, positions, q_weight, k_weight, cos_sin, num_q_heads: int,
                        num_k_heads: int, head_dim: int, eps: float, status_flags=None,
                        stream=None) -> None:
    """In place: RMSNorm (Q or K weight) then table neox RoPE on the first
    num_q_heads + num_k_heads heads of every row of a fused QKV tensor; the V
    heads after them are untouched.

    qkv [T, row] bf16 or fp16 (unit column stride, row stride a multiple of 8);
    positions int64 [T]; q_weight / k_weight [head_dim] in qkv's dtype; cos_sin
    fp32 [max_pos, head_dim]; status_flags: optional int32 CUDA tensor of one
    element to which an out-of-table position is reported (that token is left
    untouched).  Asynchronous on `stream` (default: torch's current stream).
    """
    import torch
    if qkv.dim() != 2 or (qkv.shape[0] > 0 and qkv.stride(1) != 1):
        raise ValueError("qkv must be [T, row] with unit column stride")
    if positions.dtype != torch.int64 or not positions.is_contiguous():
        raise TypeError("positions must be a contiguous int64 tensor")
    if cos_sin.dtype != torch.float32 or not cos_sin.is_contiguous():
        raise TypeError("cos_sin must be a contiguous float32 tensor")
    for name, w in (("q_weight", q_weight), ("k_weight", k_weight)):
        if w.dtype != qkv.dtype or not w.is_contiguous() or w.numel() != head_dim:
            raise TypeError(f"{name} must be a contiguous [head_dim] tensor in qkv's dtype")
    code = load().dspark_qk_norm_rope(
        qkv.data_ptr(), qkv.shape[0], qkv.stride(0) if qkv.shape[0] > 0 else qkv.shape[1],
        _dtype_code(qkv.dtype), positions.data_ptr(), q_weight.data_ptr(), k_weight.data_ptr(),
        cos_sin.data_ptr(), cos_sin.shape[0], num_q_heads, num_k_heads, head_dim, eps,
        None if status_flags is None else status_flags.data_ptr(), _stream_handle(stream))
    _abi.check(code, "dspark_qk_norm_rope")


def dspark_correct_drafts_and_bonus(candidates, target, stream=None):
    """Per request: how many leading drafts the target accepts, and the
    target's token after them.  candidates / target: int64 [batch, block] CUDA
    tensors (unit column stride); candidates[:, 0] is the last verified token.
    Returns (correct int32 [batch], bonus int64 [batch]) on the same device."""
    import torch
    for name, t in (("candidates", candidates), ("target", target)):
        if t.dtype != torch.int64 or t.dim() != 2 or (t.numel() and t.stride(1) != 1):
            raise TypeError(f"{name} must be an int64 [batch, block] tensor with unit column stride")
    if candidates.shape != target.shape:
        raise ValueError("candidates and target must have the same shape")
    batch, block = candidates.shape
    correct = torch.empty(batch, dtype=torch.int32, device=candidates.device)
    bonus = torch.empty(batch, dtype=torch.int64, device=candidates.device)
    code = load().dspark_correct_drafts_and_bonus(
        candidates.data_ptr(), candidates.stride(0) if batch else block, target.data_ptr(),
        target.stride(0) if batch else block, batch, block, correct.data_ptr(), bonus.data_ptr(),
        _stream_handle(stream))
    _abi.check(code, "dspark_correct_drafts_and_bonus")
    return correct, bonus


def dspark_draft_attention_workspace_bytes(batch: int, block: int, num_q_heads: int, num_kv_heads: int,
                                           head_dim: int, max_context: int) -> int:
    """Workspace bytes dspark_draft_attention needs (0: unsupported sizes)."""
    return int(load().dspark_draft_attention_workspace_bytes(batch, block, num_q_heads, num_kv_heads, head_dim,
                                                             max_context))


def dspark_draft_attention(q, k_ext, v_ext, k_pool, v_pool, kv_indices, kv_start, sm_scale: float,
                           max_context: int, out=None, workspace=None, status_flags=None, stream=None):
    """Non-causal GQA attention of each request's draft block over its
    context in the pool (kv_indices[kv_start[b]:kv_start[b+1]]) and the block's
    own keys.  q [batch*block, Hq, D]; k_ext / v_ext [batch*block, Hkv, D];
    k_pool / v_pool [slots, Hkv, D] (row stride a multiple of 8); kv_indices /
    kv_start int64 CUDA tensors; max_context bounds every context length.
    Returns out [batch*block, Hq, D] (allocated when not given); the workspace
    is allocated when not given (dspark_draft_attention_workspace_bytes)."""
    import torch
    nq, D = q.shape[1], q.shape[2]
    nkv = k_ext.shape[1]
    batch = kv_start.numel() - 1
    block = q.shape[0] // batch if batch > 0 else 1
    for name, t in (("q", q), ("k_ext", k_ext), ("v_ext", v_ext), ("out", out)):
        if t is not None and not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    for name, t in (("k_pool", k_pool), ("v_pool", v_pool)):
        if t.dim() != 3 or t.shape[1] != nkv or t.shape[2] != D or t.stride(1) != D or t.stride(2) != 1:
            raise ValueError(f"{name} must be [slots, num_kv_heads, head_dim] with strides (*, head_dim, 1)")
    if k_pool.stride(0) != v_pool.stride(0) or k_pool.shape[0] != v_pool.shape[0]:
        raise ValueError("k_pool and v_pool must share slots and row stride")
    for name, t in (("kv_indices", kv_indices), ("kv_start", kv_start)):
        if t.dtype != torch.int64 or not t.is_contiguous():
            raise TypeError(f"{name} must be a contiguous int64 tensor")
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        nbytes = dspark_draft_attention_workspace_bytes(max(batch, 1), block, nq, nkv, D, max_context)
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=q.device)
    code = load().dspark_draft_attention(
        q.data_ptr(), k_ext.data_ptr(), v_ext.data_ptr(), k_pool.data_ptr(), v_pool.data_ptr(), k_pool.stride(0),
        k_pool.shape[0], kv_indices.data_ptr(), kv_start.data_ptr(), batch, block, nq, nkv, D,
        _dtype_code(q.dtype), sm_scale, max_context, out.data_ptr(), workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), None if status_flags is None else status_flags.data_ptr(),
        _stream_handle(stream))
    _abi.check(code, "dspark_draft_attention")
    return out


def dspark_draft_attention_set_wait_test(limit_ns: int) -> None:
    """Diagnostics: with limit_ns > 0, later dspark_draft_attention calls take
    their timeout path after a wait of limit_ns (DSPARK_FLAG_TIMEOUT in the
    status word, output incomplete); 0 switches it off."""
    _abi.check(load().dspark_draft_attention_set_wait_test(int(limit_ns)), "dspark_draft_attention_set_wait_test")


class Combine:
    """Handle of dspark_pack_combine (main_proj / main_norm of the draft
    model); keeps the main_proj weight tensor alive, as the library does not
    copy it."""

    def __init__(self, handle, weight, hidden: int, aux_dim: int, dtype):
        self.handle = handle
        self.weight = weight
        self.hidden = hidden
        self.aux_dim = aux_dim
        self.dtype = dtype

    def free(self) -> None:
        if self.handle:
            load().dspark_free_combine(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass


def dspark_pack_combine(main_proj_weight, main_norm_weight, eps: float, stream=None) -> Combine:
    """main_proj_weight [hidden, aux_dim] (bf16 / fp16, unit column stride),
    main_norm_weight [hidden] (bf16 / fp16 / fp32)."""
    w = main_proj_weight
    if w.dim() != 2 or w.stride(1) != 1:
        raise ValueError("main_proj_weight must be [hidden, aux_dim] with unit column stride")
    if main_norm_weight.numel() != w.shape[0] or not main_norm_weight.is_contiguous():
        raise ValueError("main_norm_weight must be a contiguous [hidden] tensor")
    out = ctypes.c_void_p()
    code = load().dspark_pack_combine(w.data_ptr(), w.shape[0], w.shape[1], w.stride(0), _dtype_code(w.dtype),
                                      main_norm_weight.data_ptr(), _dtype_code(main_norm_weight.dtype), eps,
                                      _stream_handle(stream), ctypes.byref(out))
    _abi.check(code, "dspark_pack_combine")
    return Combine(out.value, w, w.shape[0], w.shape[1], w.dtype)


def dspark_combine_hidden_states(c: Combine, aux, out=None, stream=None):
    """ctx_hidden = main_norm(main_proj(aux)); aux [T, aux_dim] in the handle's
    dtype.  Returns out [T, hidden] (allocated when not given)."""
    import torch
    if aux.dim() != 2 or aux.shape[1] != c.aux_dim or (aux.shape[0] and aux.stride(1) != 1):
        raise ValueError("aux must be [T, aux_dim] with unit column stride")
    if aux.dtype != c.dtype:
        raise TypeError("aux must be in the handle's dtype")
    if out is None:
        out = torch.empty((aux.shape[0], c.hidden), dtype=aux.dtype, device=aux.device)
    code = load().dspark_combine_hidden_states(c.handle, aux.data_ptr(), aux.shape[0],
                                               aux.stride(0) if aux.shape[0] else c.aux_dim, out.data_ptr(),
                                               out.stride(0) if out.shape[0] else c.hidden,
                                               _stream_handle(stream))
    _abi.check(code, "dspark_combine_hidden_states")
    return out


def dspark_combine_get_status(c: Combine, stream=None) -> int:
    flags = ctypes.c_uint32(0)
    _abi.check(load().dspark_combine_get_status(c.handle, _stream_handle(stream), ctypes.byref(flags)),
               "dspark_combine_get_status")
    return flags.value


class Fused:
    """Handle of dspark_pack_fused_ctx_kv (combine_hidden_states fused into the
    write); keeps the main_proj weight tensor alive, as the library does not
    copy it."""

    def __init__(self, handle, weight, hidden: int, aux_dim: int, dtype, num_layers: int, num_kv_heads: int,
                 head_dim: int):
        self.handle = handle
        self.weight = weight
        self.hidden = hidden
        self.aux_dim = aux_dim
        self.dtype = dtype
        self.num_layers = num_layers
        self.num_kv_heads = num_kv_heads
        self.head_dim = head_dim

    def free(self) -> None:
        if self.handle:
            load().dspark_free_fused(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass


def dspark_pack_fused_ctx_kv(main_proj_weight, main_norm_weight, norm_eps: float, layers: Sequence, stream=None) -> Fused:
    """main_proj_weight [hidden, aux_dim] (the layers' dtype, unit column
    stride), main_norm_weight [hidden]; layers as for dspark_pack_ctx_kv."""
    w = main_proj_weight
    if w.dim() != 2 or w.stride(1) != 1:
        raise ValueError("main_proj_weight must be [hidden, aux_dim] with unit column stride")
    if main_norm_weight.numel() != w.shape[0] or not main_norm_weight.is_contiguous():
        raise ValueError("main_norm_weight must be a contiguous [hidden] tensor")
    arr = _desc_array(layers)
    out = ctypes.c_void_p()
    code = load().dspark_pack_fused_ctx_kv(w.data_ptr(), w.shape[1], w.stride(0), main_norm_weight.data_ptr(),
                                           _dtype_code(main_norm_weight.dtype), norm_eps, arr, len(layers),
                                           w.shape[0], _stream_handle(stream), ctypes.byref(out))
    _abi.check(code, "dspark_pack_fused_ctx_kv")
    l0 = layers[0]
    return Fused(out.value, w, w.shape[0], w.shape[1], w.dtype, len(layers), l0.num_kv_heads, l0.head_dim)


def dspark_combine_write_ctx_kv(f: Fused, aux, positions, cos_sin, cache_loc, k_pools, v_pools,
                                commit_lens=None, loc_row_width: Optional[int] = None, stream=None) -> None:
    """The write with ctx_hidden = main_norm(main_proj(aux)) in one launch:
    aux [T, aux_dim] in the handle's dtype (unit column stride); the other
    arguments as for dspark_write_ctx_kv (pools as lists)."""
    import torch
    T = aux.shape[0]
    if aux.dim() != 2 or aux.shape[1] != f.aux_dim or (T > 0 and aux.stride(1) != 1):
        raise ValueError("aux must be [T, aux_dim] with unit column stride")
    if aux.dtype != f.dtype:
        raise TypeError("aux must be in the handle's dtype")
    for name, t, dt in (("positions", positions, torch.int64), ("cache_loc", cache_loc, torch.int64),
                        ("cos_sin", cos_sin, torch.float32)):
        if t.dtype != dt or not t.is_contiguous():
            raise TypeError(f"{name} must be a contiguous {dt} tensor")
    if commit_lens is not None and (commit_lens.dtype != torch.int32 or not commit_lens.is_contiguous()):
        raise TypeError("commit_lens must be a contiguous int32 tensor")
    if positions.numel() != T or cache_loc.numel() != T:
        raise ValueError("positions and cache_loc must hold one entry per token")
    if cos_sin.dim() != 2 or cos_sin.shape[1] != f.head_dim:
        raise ValueError(f"cos_sin must be [max_pos, head_dim={f.head_dim}]")
    if len(k_pools) != f.num_layers or len(v_pools) != f.num_layers:
        raise ValueError("one K and one V pool per layer")
    slots = k_pools[0].shape[0]
    for p in list(k_pools) + list(v_pools):
        if (p.dim() != 3 or p.shape[0] != slots or p.shape[1] != f.num_kv_heads or p.shape[2] != f.head_dim
                or p.stride(1) != f.head_dim or p.stride(2) != 1 or p.dtype != f.dtype):
            raise ValueError("pools must be [slots, num_kv_heads, head_dim] in the handle's dtype with strides "
                             "(*, head_dim, 1)")
    L = f.num_layers
    kstr = (ctypes.c_int64 * L)(*[p.stride(0) for p in k_pools])
    vstr = (ctypes.c_int64 * L)(*[p.stride(0) for p in v_pools])
    width = 0 if loc_row_width is None else int(loc_row_width)
    nwin = 0 if commit_lens is None else commit_lens.numel()
    code = load().dspark_combine_write_ctx_kv(
        f.handle, aux.data_ptr(), T, aux.stride(0) if T > 0 else f.aux_dim, positions.data_ptr(),
        cos_sin.data_ptr(), cos_sin.shape[0], cache_loc.data_ptr(),
        None if commit_lens is None else commit_lens.data_ptr(), width, nwin, _ptr_array(k_pools),
        _ptr_array(v_pools), kstr, vstr, _dtype_code(f.dtype), slots, _stream_handle(stream))
    _abi.check(code, "dspark_combine_write_ctx_kv")


def dspark_fused_get_status(f: Fused, stream=None) -> int:
    flags = ctypes.c_uint32(0)
    _abi.check(load().dspark_fused_get_status(f.handle, _stream_handle(stream), ctypes.byref(flags)),
               "dspark_fused_get_status")
    return flags.value


def dspark_fused_clear_status(f: Fused, stream=None) -> None:
    _abi.check(load().dspark_fused_clear_status(f.handle, _stream_handle(stream)), "dspark_fused_clear_status")


def dspark_describe_schedule(tiles: int, num_kb: int, workers: int, split_first_allowed: bool = True) -> dict:
    """The work split of the tiled kernels for `tiles` output tiles of
    `num_kb` k-blocks on up to `workers` workers (host only): workers,
    whole_tiles, split_units, split_workers, split_first."""
    import ctypes
    info = _abi.ScheduleInfo()
    _abi.check(load().dspark_describe_schedule(int(tiles), int(num_kb), int(workers), int(bool(split_first_allowed)),
                                               ctypes.byref(info)), "dspark_describe_schedule")
    return {name: getattr(info, name) for name, _ in info._fields_}


def dspark_set_kernel_variant(bundle: Bundle, variant: str) -> None:
    """Select the kernel of later writes: "auto" (default), "single" (one CTA
    per 128 x 256 tile), "pair" (CTA pairs per 256 x 256 tile) or "stream"
    (weight streaming, at most 256 tokens)."""
    code = {"auto": _abi.VARIANT_AUTO, "single": _abi.VARIANT_SINGLE, "pair": _abi.VARIANT_PAIR,
            "stream": _abi.VARIANT_STREAM}[variant]
    _abi.check(load().dspark_set_kernel_variant(bundle.handle, code), "dspark_set_kernel_variant")
