"""Oracle for the draft model's combine_hidden_states (main_proj + main_norm).

TEST INFRASTRUCTURE ONLY (see the package docstring).

The vLLM PR #46995 page (DSpark in vLLM, "Key source snippets": the draft
model's __init__ and combine_hidden_states) defines the context hidden state
the KV write consumes: the target model's auxiliary hidden states of its
len(target_layer_ids) layers, concatenated, go through main_proj (a linear
layer from hidden * len(target_layer_ids) to hidden, no bias) and then
main_norm (an RMSNorm over hidden with the model's rms_norm_eps):

  y   = aux . W^T                      W: [hidden, aux_dim] (out by in)
  out = y / sqrt(mean(y^2) + eps) * w  per token, over the hidden dimension

Readings (also in the design notes): the linear layer's output is in the
model dtype, so y is rounded to it before the norm (a plain F.linear); the
norm computes in float from those values and its output is stored in the
model dtype (returned here before that rounding); w multiplies as given.
The snippet's trailing ``[0]`` after main_proj is read as taking the layer's
output (the layer is built with return_bias=False).  Float64 apart from the
rounding of y, which is a correctly rounded conversion (oracle.round_to).
"""
from __future__ import annotations

import numpy as np

from .ctx_kv import widen
from .qk_norm_rope import round_to


def combine_hidden_states(aux: np.ndarray, weight: np.ndarray, norm_weight: np.ndarray, eps: float,
                          dtype: str) -> np.ndarray:
    """aux bits [T, aux_dim]; weight bits [hidden, aux_dim]; norm_weight bits
    [hidden] (model dtype).  Returns float64 [T, hidden]."""
    y = round_to(widen(aux, dtype) @ widen(weight, dtype).T, dtype)
    inv = 1.0 / np.sqrt(np.mean(y * y, axis=1, keepdims=True) + eps)
    return y * inv * widen(norm_weight, dtype)[None, :]
