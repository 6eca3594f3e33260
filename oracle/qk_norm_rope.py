"""Oracle for the in-place QK RMSNorm + table neox RoPE of the draft layers.

TEST INFRASTRUCTURE ONLY.  A plain, slow CPU restatement used to check the
CUDA path; only the tests, the smoke check and the benchmark's CPU-baseline
leg may import it.  It shares no code with the library.

What it computes follows the ``_table_qk_norm_rope_kernel`` /
``table_qk_norm_rope_`` snippet on the sglang PR #31847 summary page ("Key
source snippets", dflash_utils.py), which the DFlash and DSpark draft models
share.  The fused QKV row of token t holds num_q_heads Q heads, then
num_k_heads K heads, then the V heads; V is left alone.  For every Q or K head
of every token, with x the head's head_dim values:

  inv = 1 / sqrt(mean(x^2) + eps)
  x1  = round(x[:D/2] * inv * w[:D/2]),  x2 = round(x[D/2:] * inv * w[D/2:])
  c, s = table[pos][:D/2], table[pos][D/2:]
  out[:D/2] = x1 * c - x2 * s,  out[D/2:] = x2 * c + x1 * s

w is the Q norm weight for Q heads and the K norm weight for K heads.
``round`` is the page's intermediate rounding to the model dtype ("round back
to bf16 first, to match the eager path"); the outputs are then stored in the
model dtype.

Readings where the page is silent or narrower (also listed in the design
notes):
  * The page's kernel is bf16 only.  For an fp16 model the intermediate
    rounding goes to fp16, and the weights are in the model dtype.
  * Arithmetic here is float64 apart from that rounding, which is a correctly
    rounded (round to nearest, ties to even) conversion of the float64 value.
  * A position outside [0, max_pos) is a caller error: the oracle raises.

Pins (tests/test_oracle_qknorm_pins.py): identity table row gives exactly
representable outputs and the closed form sign(c) * w on constant heads with
distinct Q and K weights; the quarter-turn row gives (-x2, x1); eps placement
closed form; rotation preserves each pair's norm and equals multiplication by
exp(i*theta) of the identity-row output.
"""
from __future__ import annotations

from typing import Optional

import numpy as np

from .ctx_kv import widen

# significand bits (including the implicit one) and smallest normal exponent
# (x = m * 2**e with 0.5 <= |m| < 1) of the 16-bit formats
_FORMATS = {"bf16": (8, -125), "fp16": (11, -13)}
_MAX = {"bf16": float(np.finfo(np.float32).max), "fp16": 65504.0}


def round_to(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round float64 values to the nearest bf16 / fp16 value (ties to even),
    returned as float64.  Finite inputs; fp16 overflow saturates to inf."""
    bits, emin = _FORMATS[dtype]
    x = np.asarray(x, dtype=np.float64)
    _, e = np.frexp(x)
    e = np.maximum(e, emin)                      # below the normal range: fixed quantum
    quantum = np.ldexp(1.0, e - bits)
    r = np.rint(x / quantum) * quantum           # np.rint rounds half to even
    if dtype == "fp16":
        r = np.where(np.abs(r) > _MAX[dtype], np.sign(r) * np.inf, r)
    return r


def table_qk_norm_rope(qkv: np.ndarray, dtype: str, positions: np.ndarray, q_weight: np.ndarray,
                       k_weight: np.ndarray, cos_sin: np.ndarray, num_q_heads: int,
                       num_k_heads: int, head_dim: int, eps: float,
                       tokens: Optional[np.ndarray] = None) -> np.ndarray:
    """Rotated, normalised Q and K heads before the store rounding.

    qkv: bits [T, row] (row >= (num_q_heads + num_k_heads) * head_dim); q_weight
    and k_weight: bits [head_dim] in ``dtype``; cos_sin: fp32 [max_pos, head_dim];
    tokens: optional subset of token indices.  Returns float64
    [len(tokens), num_q_heads + num_k_heads, head_dim].
    """
    D = head_dim
    half = D // 2
    nh = num_q_heads + num_k_heads
    if D % 2 or qkv.shape[1] < nh * D:
        raise ValueError("row too short for the Q and K heads")
    t_idx = np.arange(qkv.shape[0]) if tokens is None else np.asarray(tokens)
    pos = np.asarray(positions)[t_idx]
    if np.any(pos < 0) or np.any(pos >= cos_sin.shape[0]):
        raise ValueError("position outside the cos/sin table")
    x = widen(qkv[t_idx, :nh * D], dtype).reshape(len(t_idx), nh, D)
    w = np.stack([widen(q_weight, dtype)] * num_q_heads + [widen(k_weight, dtype)] * num_k_heads)
    inv = 1.0 / np.sqrt(np.mean(x * x, axis=2, keepdims=True) + eps)
    x1 = round_to(x[:, :, :half] * inv * w[None, :, :half], dtype)
    x2 = round_to(x[:, :, half:] * inv * w[None, :, half:], dtype)
    table = np.asarray(cos_sin, dtype=np.float32).astype(np.float64)[pos]
    c = table[:, None, :half]
    s = table[:, None, half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=2)
