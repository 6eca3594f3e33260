"""Stage a synthetic workload's host buffers on a CUDA device (torch tensors).

Pure data movement: bit patterns are copied as they are; pools are filled
with the sentinel bit pattern so that untouched slots can be recognised.
"""
from __future__ import annotations

from typing import Dict, List

import numpy as np

from . import POOL_SENTINEL, Workload


def torch_dtype(w: Workload):
    import torch
    return torch.bfloat16 if w.dtype == "bf16" else torch.float16


def bits_to_tensor(bits: np.ndarray, dtype, device):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.to(device).view(dtype)


def sentinel_int16() -> int:
    return POOL_SENTINEL - 0x10000 if POOL_SENTINEL >= 0x8000 else POOL_SENTINEL


def make_pools(w: Workload, device, row_pad: int = 0) -> List:
    """2*L pools [slots, NH, D] filled with the sentinel; row_pad extra
    elements per slot give a row stride larger than NH*D."""
    import torch
    pools = []
    for _ in range(2 * w.L):
        buf = torch.full((w.pool_slots, w.NH * w.D + row_pad), sentinel_int16(), dtype=torch.int16,
                         device=device)
        pools.append(buf[:, :w.NH * w.D].view(torch_dtype(w)).view(w.pool_slots, w.NH, w.D)
                     if row_pad == 0 else
                     buf.view(torch_dtype(w))[:, :w.NH * w.D].unflatten(1, (w.NH, w.D)))
    return pools


def stage(w: Workload, device="cuda", row_pad: int = 0) -> Dict[str, object]:
    """Device copies of every input of the write, plus fresh sentinel pools."""
    import torch
    from draft_model_kv_gb300 import Layer
    dt = torch_dtype(w)
    layers = []
    for lay in w.layers:
        layers.append(Layer(
            qkv_weight=bits_to_tensor(lay.qkv_weight, dt, device),
            qkv_bias=None if lay.qkv_bias is None else bits_to_tensor(lay.qkv_bias, dt, device),
            k_norm_weight=bits_to_tensor(lay.k_norm_weight, dt, device),
            eps=lay.eps, q_size=w.q_size, num_kv_heads=w.NH, head_dim=w.D))
    pools = make_pools(w, device, row_pad)
    return {
        "layers": layers,
        "ctx_hidden": bits_to_tensor(w.ctx_hidden, dt, device),
        "positions": torch.from_numpy(w.positions).to(device),
        "cos_sin": torch.from_numpy(w.cos_sin).to(device),
        "cache_loc": torch.from_numpy(w.cache_loc).to(device),
        "commit_lens": None if w.commit_lens is None else torch.from_numpy(w.commit_lens).to(device),
        "loc_row_width": w.loc_row_width if w.commit_lens is not None else None,
        "k_pools": pools[0::2],
        "v_pools": pools[1::2],
    }
