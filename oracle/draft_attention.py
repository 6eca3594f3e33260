"""Oracle for the draft model's attention over the written KV pool.

TEST INFRASTRUCTURE ONLY (see the package docstring).

The sglang PR #35499 summary page (K3 DSpark draft attention on ROCm) routes
the draft layers' attention to the shared-KV split-KV kernels: the draft
attention is qwen3-style GQA, bidirectional (non-causal), every query of a
request's draft block attends to the request's context KV, gathered from the
pool through a kv_indices table, and to the block's own keys ("Implementation
breakdown" items 2-3 and the verify_mla.py snippets: the KV head of a query
head is head // KV_GROUP_NUM; IS_CAUSAL = 0 removes the causal mask so every
token sees the whole KV sequence).  The kernels' softmax body is not printed;
this oracle writes out plain scaled-dot-product attention:

  for request b, query row i of its block (E rows), query head h, with
  g = h // (num_q_heads / num_kv_heads):
    keys   = K_pool[kv_indices[kv_start[b] : kv_start[b+1]], g]  then  K_ext[b*E : b*E+E, g]
    values = the same rows of V_pool / V_ext
    s = sm_scale * keys . q[b*E + i, h];  p = softmax(s);  out[b*E + i, h] = p . values

in float64 from the exact widened inputs (the output before its rounding to
the model dtype).
"""
from __future__ import annotations

from typing import Optional, Sequence

import numpy as np

from .ctx_kv import widen


def draft_attention(q: np.ndarray, k_ext: np.ndarray, v_ext: np.ndarray, k_pool: np.ndarray,
                    v_pool: np.ndarray, kv_indices: np.ndarray, kv_start: np.ndarray, dtype: str,
                    num_q_heads: int, num_kv_heads: int, head_dim: int, sm_scale: float,
                    requests: Optional[Sequence[int]] = None) -> np.ndarray:
    """Attention output (float64) of the requested requests' query rows.

    q: bits [bs*E, num_q_heads, D]; k_ext / v_ext: bits [bs*E, num_kv_heads, D];
    k_pool / v_pool: bits [slots, num_kv_heads, D]; kv_indices int64; kv_start
    int64 [bs + 1] (request b's context is kv_indices[kv_start[b]:kv_start[b+1]]).
    Returns [len(requests) * E, num_q_heads, D] in request order.
    """
    if num_q_heads % num_kv_heads:
        raise ValueError("num_q_heads must be a multiple of num_kv_heads")
    group = num_q_heads // num_kv_heads
    bs = len(kv_start) - 1
    E = q.shape[0] // bs
    reqs = range(bs) if requests is None else requests
    out = []
    for b in reqs:
        slots = np.asarray(kv_indices[kv_start[b]:kv_start[b + 1]])
        if np.any(slots < 0) or np.any(slots >= k_pool.shape[0]):
            raise ValueError("kv index outside the pool")
        kb = np.concatenate([widen(k_pool[slots], dtype), widen(k_ext[b * E:(b + 1) * E], dtype)], axis=0)
        vb = np.concatenate([widen(v_pool[slots], dtype), widen(v_ext[b * E:(b + 1) * E], dtype)], axis=0)
        qb = widen(q[b * E:(b + 1) * E], dtype)                 # [E, NHQ, D]
        ob = np.empty((E, num_q_heads, head_dim))
        for h in range(num_q_heads):
            g = h // group
            s = sm_scale * (qb[:, h, :] @ kb[:, g, :].T)        # [E, keys]
            s = s - s.max(axis=1, keepdims=True)
            p = np.exp(s)
            p /= p.sum(axis=1, keepdims=True)
            ob[:, h, :] = p @ vb[:, g, :]
        out.append(ob)
    return np.concatenate(out, axis=0)
