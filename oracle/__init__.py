"""Oracle package: a plain fp64 CPU restatement of the DSpark context-KV write.

TEST INFRASTRUCTURE ONLY.  Imported by ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py``; never by the library, which has no
CPU fallback.  It shares no code with the CUDA path.

Parity status of each function (what pins it, in ``tests/test_oracle_pins.py``):
  stacked_ctx_kv_params  refusal cases + stacked == per-layer (exact, brute force)
  kv_proj_only           brute-force triple loop (exact), identity / one-hot closed forms
  apply_k_norm           constant-vector closed form, mean-square and scale invariants
  apply_k_rope           position-0 identity, pair-norm, complex-rotation equality,
                         quarter-turn table, hand-worked golden example
  written_tokens         hand-worked window golden example, -1 / commit edge cases
  write_target_hidden_kv composition of the above + bias closed form
  eager=True (diagnostic) closed forms for both rounding points (projection,
                         normed K); agrees with the pure reading within the
                         parity tolerance

and of the in-place QK RMSNorm + table RoPE (``qk_norm_rope.py``, pinned in
``tests/test_oracle_qknorm_pins.py``):
  round_to               exhaustive agreement with numpy's float16 conversion
                         and with bf16 bit truncation plus ties on all patterns
  table_qk_norm_rope     identity-row closed forms with distinct Q/K weights,
                         representable identity-row outputs, quarter-turn row,
                         eps placement, pair norm, exp(i*theta) rotation

and of the verify step's accepted-draft count (``verify.py``, pinned in
``tests/test_oracle_verify_pins.py``):
  correct_drafts_and_bonus  hand-worked golden cases, suffix independence,
                            bonus-at-count and all-accepted invariants

and of the draft attention over the pool (``draft_attention.py``, pinned in
``tests/test_oracle_attention_pins.py``):
  draft_attention        single key, equal keys (mean of values), per-KV-head
                         constant values (GQA head mapping), two-key weight
                         ratio exp(sm_scale * diff), non-causal extend keys,
                         key permutation invariance, dominant key

and of the draft model's combine_hidden_states (``combine.py``, pinned in
``tests/test_oracle_combine_pins.py``):
  combine_hidden_states  identity-block weight closed form (sign(c) * w on
                         constant rows), one-hot columns, scale invariance,
                         mean-square invariant, representable rounding of y
"""
from .ctx_kv import (  # noqa: F401
    LayerDesc, Stacked, WriteArgError, WriteResult, apply_k_norm, apply_k_rope,
    kv_proj_only, layer_descs, per_layer_reference, project_stacked, run_workload,
    stacked_ctx_kv_params, widen, write_target_hidden_kv, written_tokens,
)
from .qk_norm_rope import round_to, table_qk_norm_rope  # noqa: F401,E402
from .verify import correct_drafts_and_bonus  # noqa: F401,E402
from .draft_attention import draft_attention  # noqa: F401,E402
from .combine import combine_hidden_states  # noqa: F401,E402
