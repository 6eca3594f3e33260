"""Oracle for the DSpark draft-model context-KV write.

TEST INFRASTRUCTURE ONLY.  This is a plain, slow CPU restatement of what the
write computes, used to check the CUDA path.  Only the tests, the smoke check
and the benchmark's CPU-baseline leg may import it; the library never does.

Arithmetic is numpy float64 (``acc=np.float32`` gives a single-precision
variant used to show that the tolerances are meaningful).  Inputs arrive as
the raw bf16/fp16 bit patterns that the model would hold; they are widened
exactly before any arithmetic.  The only library primitive used as a step is
the matrix product of the projection.

The steps follow the per-layer reference path that the sglang PR #31986
summary page uses as ground truth ("Key source snippets",
``write_target_hidden_kv`` fallback branch and the test's
``_per_layer_reference``): ``kv_proj_only`` -> ``apply_k_norm`` ->
``apply_k_rope`` -> view as [T, num_kv_heads, head_dim], followed by the pool
write that the sglang PR #31847 page describes for
``fused_kv_norm_rope_write`` (docstring: skip ``loc < 0``; with
``commit_lens`` the locs are a flattened [bs, W] window and only the first
``commit_lens[b]`` columns of row b are written).

Readings taken where the pages are silent (each also listed in the design
notes):
  * RMSNorm is ``y * (1/sqrt(mean(y^2) + eps)) * w`` per head over head_dim,
    w multiplied as given (not 1+w), matching the ``_table_qk_norm_rope_kernel``
    arithmetic on the PR #31847 page.
  * The bias, when present, is part of the linear: added to K and V before the
    norm (PR #31986 page, ``_stacked_ctx_kv_params`` stacks it with the weight).
  * k_norm weights are converted to fp32 (PR #31986 page: stacked ``.float()``).
  * No intermediate rounding: values stay in the accumulation precision until
    the store (the fused kernel's body is not shown on the PR #31847 page).
    ``eager=True`` is the other reading, kept as a diagnostic: the eager path
    rounds the projection (the linear layer's output) and the normalised K
    (the PR #31847 QK kernel rounds before the rotation "to match eager") to
    the model dtype.
  * In window mode a token is also skipped when its loc is -1; commit_lens[b]
    above W acts as W, and 0 writes nothing.
  * pos outside [0, max_pos), loc >= pool_slots and duplicate written locs are
    caller errors: the oracle raises.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional, Sequence, Tuple

import numpy as np

# ---------------------------------------------------------------------------
# storage formats
# ---------------------------------------------------------------------------


def widen(bits: np.ndarray, dtype: str, acc=np.float64) -> np.ndarray:
    """Exact value of bf16 / fp16 bit patterns (or pass fp32 through) in ``acc``."""
    if dtype == "bf16":
        return (np.asarray(bits).astype(np.uint32) << 16).view(np.float32).astype(acc)
    if dtype == "fp16":
        return np.asarray(bits).astype(np.uint16).view(np.float16).astype(acc)
    if dtype == "fp32":
        return np.asarray(bits, dtype=np.float32).astype(acc)
    raise ValueError(f"unknown dtype {dtype!r}")


# ---------------------------------------------------------------------------
# bundle: which layers may be stacked (PR #31986 page, _stacked_ctx_kv_params;
# PR #31847 page, _build_fused_kv_write_bundle)
# ---------------------------------------------------------------------------

SLICEABLE = ("bf16", "fp16")


@dataclasses.dataclass
class LayerDesc:
    """A draft layer's attention parameters as the bundle builder sees them."""
    qkv_weight: np.ndarray          # bits [q_size + 2*kv_size, H]
    qkv_bias: Optional[np.ndarray]  # bits [q_size + 2*kv_size] or None
    k_norm_weight: np.ndarray       # bits [head_dim] in k_norm_dtype
    eps: float
    weight_dtype: str               # "bf16" | "fp16" | anything else = quantized
    q_size: int
    num_kv_heads: int
    head_dim: int
    k_norm_dtype: str = ""          # defaults to weight_dtype


@dataclasses.dataclass
class Stacked:
    weight: np.ndarray              # [L*2*KV, H], rows l0:K, l0:V, l1:K, ...
    bias: Optional[np.ndarray]      # [L*2*KV] or None
    k_norm_weight: np.ndarray       # [L, head_dim], values of the fp32 conversion
    eps: float
    dtype: str
    num_layers: int
    num_kv_heads: int
    head_dim: int


def stacked_ctx_kv_params(layers: Sequence[LayerDesc], acc=np.float64
                          ) -> Tuple[Optional[Stacked], str]:
    """Stack every layer's K|V slice, or say why the layers cannot be stacked.

    Returns ``(stacked, "ok")`` or ``(None, reason)``.  Reasons, in the order
    the checks run: ``no_layers`` (empty model, PR #31847 bundle builder),
    ``not_sliceable`` (quantized qkv_proj, both pages), ``eps_mismatch``
    (layers disagree on k_norm epsilon, both pages), ``dtype_mismatch``,
    ``shape_mismatch`` (head_dim / kv_size differ, PR #31847 page),
    ``head_dim`` (not 64 or 128: the sizes the CUDA path instantiates),
    ``bias_mismatch`` (bias on some layers only, PR #31986 page).
    """
    if len(layers) == 0:
        return None, "no_layers"
    eps = None
    first = layers[0]
    weights, biases, knws = [], [], []
    for lay in layers:
        if lay.weight_dtype not in SLICEABLE:
            return None, "not_sliceable"
        if eps is not None and lay.eps != eps:
            return None, "eps_mismatch"
        eps = lay.eps
        if lay.weight_dtype != first.weight_dtype:
            return None, "dtype_mismatch"
        if (lay.head_dim != first.head_dim or lay.num_kv_heads != first.num_kv_heads
                or lay.q_size != first.q_size):
            return None, "shape_mismatch"
        if lay.head_dim not in (64, 128):
            return None, "head_dim"
        kv_size = lay.num_kv_heads * lay.head_dim
        kv_slice = slice(lay.q_size, lay.q_size + 2 * kv_size)
        weights.append(widen(lay.qkv_weight[kv_slice], lay.weight_dtype, acc))
        biases.append(None if lay.qkv_bias is None
                      else widen(lay.qkv_bias[kv_slice], lay.weight_dtype, acc))
        kn_dtype = lay.k_norm_dtype or lay.weight_dtype
        # k_norm weights are stacked and converted to fp32
        knws.append(widen(lay.k_norm_weight, kn_dtype, np.float32).astype(acc))
    has_bias = [b is not None for b in biases]
    if any(has_bias) and not all(has_bias):
        return None, "bias_mismatch"
    return Stacked(weight=np.concatenate(weights, axis=0),
                   bias=np.concatenate(biases, axis=0) if all(has_bias) else None,
                   k_norm_weight=np.stack(knws, axis=0), eps=float(eps),
                   dtype=first.weight_dtype, num_layers=len(layers),
                   num_kv_heads=first.num_kv_heads, head_dim=first.head_dim), "ok"


# ---------------------------------------------------------------------------
# per-layer reference path (PR #31986 page, _per_layer_reference)
# ---------------------------------------------------------------------------


def kv_proj_only(ctx_hidden: np.ndarray, qkv_weight: np.ndarray,
                 qkv_bias: Optional[np.ndarray], q_size: int, kv_size: int
                 ) -> Tuple[np.ndarray, np.ndarray]:
    """K and V columns of the qkv projection: rows [q_size, q_size + 2*kv_size)
    of the out-by-in weight, K first, then V (F.linear convention)."""
    w_k = qkv_weight[q_size:q_size + kv_size]
    w_v = qkv_weight[q_size + kv_size:q_size + 2 * kv_size]
    k = ctx_hidden @ w_k.T
    v = ctx_hidden @ w_v.T
    if qkv_bias is not None:
        k = k + qkv_bias[q_size:q_size + kv_size]
        v = v + qkv_bias[q_size + kv_size:q_size + 2 * kv_size]
    return k, v


def apply_k_norm(k: np.ndarray, k_norm_weight: np.ndarray, eps: float,
                 num_kv_heads: int, head_dim: int) -> np.ndarray:
    """Per-head RMSNorm over head_dim: y / sqrt(mean(y^2) + eps) * w."""
    acc = k.dtype.type
    y = k.reshape(k.shape[0], num_kv_heads, head_dim)
    ms = (y * y).sum(axis=-1, keepdims=True) / acc(head_dim)
    inv = acc(1.0) / np.sqrt(ms + acc(eps))
    return (y * inv * k_norm_weight.astype(k.dtype)).reshape(k.shape)


def apply_k_rope(positions: np.ndarray, k: np.ndarray, cos_sin: np.ndarray,
                 num_kv_heads: int, head_dim: int) -> np.ndarray:
    """Neox (rotate-half) RoPE with cos/sin looked up in the precomputed table.

    Element i of each head pairs with element i + D/2 and turns through the
    angle whose cosine is ``table[pos][i]`` and sine ``table[pos][D/2 + i]``.
    """
    acc = k.dtype.type
    half = head_dim // 2
    rows = cos_sin[positions].astype(acc)            # [T, D]
    cos = rows[:, None, :half]
    sin = rows[:, None, half:]
    y = k.reshape(k.shape[0], num_kv_heads, head_dim)
    x1, x2 = y[..., :half], y[..., half:]
    o1 = x1 * cos - x2 * sin
    o2 = x2 * cos + x1 * sin
    return np.concatenate([o1, o2], axis=-1).reshape(k.shape)


def _round(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round to the nearest value of the model dtype (ties to even), in the
    accumulation precision."""
    from .qk_norm_rope import round_to
    return round_to(x, dtype).astype(x.dtype)


def per_layer_reference(ctx_hidden: np.ndarray, layers: Sequence[LayerDesc],
                        positions: np.ndarray, cos_sin: np.ndarray, acc=np.float64,
                        eager: bool = False) -> Tuple[List[np.ndarray], List[np.ndarray]]:
    """K (normed, roped) and V of every layer as [T, num_kv_heads, head_dim].
    With ``eager`` the projection and the normalised K are rounded to the
    model dtype (the eager path's intermediate roundings)."""
    ks, vs = [], []
    for lay in layers:
        dt = lay.weight_dtype
        x = widen(ctx_hidden, dt, acc)
        kv_size = lay.num_kv_heads * lay.head_dim
        # only the K|V rows are ever read: widen those (Q rows stay untouched)
        rows = slice(lay.q_size, lay.q_size + 2 * kv_size)
        w = widen(lay.qkv_weight[rows], dt, acc)
        b = None if lay.qkv_bias is None else widen(lay.qkv_bias[rows], dt, acc)
        k, v = kv_proj_only(x, w, b, 0, kv_size)
        if eager:
            k, v = _round(k, dt), _round(v, dt)
        kn = widen(lay.k_norm_weight, lay.k_norm_dtype or dt, np.float32).astype(acc)
        k = apply_k_norm(k, kn, lay.eps, lay.num_kv_heads, lay.head_dim)
        if eager:
            k = _round(k, dt)
        k = apply_k_rope(positions, k, cos_sin, lay.num_kv_heads, lay.head_dim)
        ks.append(k.reshape(-1, lay.num_kv_heads, lay.head_dim))
        vs.append(v.reshape(-1, lay.num_kv_heads, lay.head_dim))
    return ks, vs


def project_stacked(ctx_hidden: np.ndarray, st: Stacked, positions: np.ndarray,
                    cos_sin: np.ndarray, acc=np.float64
                    ) -> Tuple[List[np.ndarray], List[np.ndarray]]:
    """The stacked form: one product with the row-stacked weight, split per
    layer, then the same norm and rotation (PR #31986 page, implementation
    item 2).  Used to pin that stacking changes nothing."""
    x = widen(ctx_hidden, st.dtype, acc)
    y = x @ st.weight.astype(acc).T
    if st.bias is not None:
        y = y + st.bias.astype(acc)
    kv = st.num_kv_heads * st.head_dim
    ks, vs = [], []
    for l in range(st.num_layers):
        k = y[:, l * 2 * kv:l * 2 * kv + kv]
        v = y[:, l * 2 * kv + kv:(l + 1) * 2 * kv]
        k = apply_k_norm(k, st.k_norm_weight[l].astype(acc), st.eps, st.num_kv_heads,
                         st.head_dim)
        k = apply_k_rope(positions, k, cos_sin, st.num_kv_heads, st.head_dim)
        ks.append(k.reshape(-1, st.num_kv_heads, st.head_dim))
        vs.append(v.reshape(-1, st.num_kv_heads, st.head_dim))
    return ks, vs


# ---------------------------------------------------------------------------
# pool write (PR #31847 page, fused_kv_norm_rope_write docstring and checks)
# ---------------------------------------------------------------------------


class WriteArgError(ValueError):
    pass


def written_tokens(cache_loc: np.ndarray, commit_lens: Optional[np.ndarray] = None,
                   loc_row_width: Optional[int] = None,
                   pool_slots: Optional[int] = None) -> np.ndarray:
    """Indices t of the tokens whose K/V rows land in the pool, ascending.

    A token is written when ``cache_loc[t] >= 0`` and, in window mode, when its
    column ``t mod W`` is below ``commit_lens[t div W]``.
    """
    cache_loc = np.asarray(cache_loc, dtype=np.int64)
    if (commit_lens is None) != (loc_row_width is None):
        raise WriteArgError("commit_lens and loc_row_width must be passed together")
    keep = []
    for t in range(cache_loc.shape[0]):
        if cache_loc[t] < 0:
            continue
        if commit_lens is not None:
            b, col = divmod(t, loc_row_width)
            if col >= int(commit_lens[b]):
                continue
        keep.append(t)
    keep = np.asarray(keep, dtype=np.int64)
    locs = cache_loc[keep]
    if pool_slots is not None and locs.size and locs.max() >= pool_slots:
        raise WriteArgError("cache_loc beyond the pool")
    if np.unique(locs).size != locs.size:
        raise WriteArgError("two written tokens share a pool slot")
    return keep


@dataclasses.dataclass
class WriteResult:
    tokens: np.ndarray        # [n] token index of each written row
    slots: np.ndarray         # [n] pool slot of each written row
    k: np.ndarray             # [L, n, NH, D] value stored in each K pool row
    v: np.ndarray             # [L, n, NH, D] value stored in each V pool row


def write_target_hidden_kv(ctx_hidden: np.ndarray, layers: Sequence[LayerDesc],
                           positions: np.ndarray, cos_sin: np.ndarray,
                           cache_loc: np.ndarray, pool_slots: int,
                           commit_lens: Optional[np.ndarray] = None,
                           loc_row_width: Optional[int] = None,
                           sample: Optional[np.ndarray] = None,
                           acc=np.float64, eager: bool = False) -> WriteResult:
    """The whole write: what every pool row holds afterwards.

    The pool slot set is decided from cache_loc / commit_lens over all tokens;
    ``sample`` restricts the (expensive) values to a subset of the written
    tokens (each token's rows depend on its own hidden row alone).
    """
    T = ctx_hidden.shape[0]
    if cache_loc.shape[0] != T or positions.shape[0] != T:
        raise WriteArgError("positions / cache_loc must have one entry per token")
    if commit_lens is not None and loc_row_width is not None:
        if commit_lens.shape[0] * loc_row_width != T:
            raise WriteArgError("locs must be a flattened [bs, W] window")
    toks = written_tokens(cache_loc, commit_lens, loc_row_width, pool_slots)
    if sample is not None:
        toks = np.intersect1d(toks, np.asarray(sample, dtype=np.int64))
    pos = positions[toks]
    if pos.size and (pos.min() < 0 or pos.max() >= cos_sin.shape[0]):
        raise WriteArgError("position outside the cos/sin table")
    ks, vs = per_layer_reference(ctx_hidden[toks], layers, pos, cos_sin, acc, eager)
    return WriteResult(tokens=toks, slots=cache_loc[toks], k=np.stack(ks), v=np.stack(vs))


def layer_descs(workload) -> List[LayerDesc]:
    """LayerDesc view of a synthetic workload's layers."""
    return [LayerDesc(qkv_weight=l.qkv_weight, qkv_bias=l.qkv_bias,
                      k_norm_weight=l.k_norm_weight, eps=l.eps,
                      weight_dtype=workload.dtype, q_size=workload.q_size,
                      num_kv_heads=workload.NH, head_dim=workload.D)
            for l in workload.layers]


def run_workload(workload, sample=None, acc=np.float64, eager: bool = False) -> WriteResult:
    w = workload
    return write_target_hidden_kv(
        w.ctx_hidden, layer_descs(w), w.positions, w.cos_sin, w.cache_loc, w.pool_slots,
        w.commit_lens, w.loc_row_width if w.commit_lens is not None else None,
        sample=sample, acc=acc, eager=eager)
