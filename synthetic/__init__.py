"""Seeded synthetic inputs for the DSpark context-KV write.

This module only draws random numbers and lays them out in the storage formats
that both sides consume (raw bf16/fp16 bit patterns, int64 indices, an fp32
cos/sin table).  It holds none of the write's arithmetic: no projection, no
norm, no rotation, no scatter rule.  The oracle and the CUDA path each read the
same host buffers produced here.

Shapes follow the draft-model context-KV write described on the sglang PR
#31986 summary page ("write_target_hidden_kv" snippet: ctx_hidden [T, H],
per-layer qkv_proj.weight [q_size + 2*kv_size, H], k_norm weight [head_dim])
and the sglang PR #31847 summary page ("_build_fused_kv_write_bundle" and
"fused_kv_norm_rope_write" snippets: pools [slots, num_kv_heads, head_dim],
cos/sin cache rows [cos | sin] of width head_dim, flattened [bs, W] verify
windows with commit_lens).

Five named workloads:

* ``tiny``       T=32,    H=256,  L=2, NH=2, D=64,  bf16, no bias, 1-D locs
* ``decode512``  T=512,   H=4096, L=5, NH=8, D=128, bf16, 64 requests x 8 window
* ``prefill32k`` T=32768, H=4096, L=5, NH=8, D=128, bf16, 8 requests x 4096, 1% -1
* ``fp16bias``   T=4096,  H=5120, L=8, NH=8, D=128, fp16 + bias, 256 x 16 window
* ``k3gqa``      T=2048,  H=7168, L=5, NH=8, D=64,  bf16, 256 x 8 window

``make_workload(name, seed=None, **overrides)`` builds one; overrides change
T-independent sizes for sweeps (``tokens`` keeps the decode shapes but changes
the request count).
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional, Sequence

import numpy as np

BF16 = "bf16"
FP16 = "fp16"

# Bit pattern written into every pool slot before a write; any slot that the
# write must not touch keeps it.  0xDEAD is a finite bf16 / a finite fp16.
POOL_SENTINEL = 0xDEAD
# Quiet-NaN bit pattern for the Q rows of the synthetic qkv weights, so that a
# path which reads outside the KV slice produces NaN outputs.
QNAN_BITS = {BF16: 0x7FC1, FP16: 0x7E01}


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (round to nearest, ties to even); finite inputs."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return (u >> 16).astype(np.uint16)


def f32_to_fp16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to IEEE fp16 (numpy's conversion rounds to nearest even)."""
    return np.ascontiguousarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)


def to_bits(x: np.ndarray, dtype: str) -> np.ndarray:
    return f32_to_bf16_bits(x) if dtype == BF16 else f32_to_fp16_bits(x)


@dataclasses.dataclass
class Layer:
    """One draft layer's attention parameters as a model would hold them."""
    qkv_weight: np.ndarray            # uint16 bits [q_size + 2*kv_size, H]
    qkv_bias: Optional[np.ndarray]    # uint16 bits [q_size + 2*kv_size] or None
    k_norm_weight: np.ndarray         # uint16 bits [head_dim] (model dtype)
    eps: float


@dataclasses.dataclass
class Workload:
    name: str
    seed: int
    dtype: str                        # "bf16" | "fp16"
    T: int
    H: int
    L: int
    NH: int
    D: int
    q_size: int
    layers: List[Layer]
    ctx_hidden: np.ndarray            # uint16 bits [T, H]
    positions: np.ndarray             # int64 [T]
    cos_sin: np.ndarray               # float32 [max_pos, D], row = [cos | sin]
    cache_loc: np.ndarray             # int64 [T] (flattened [bs, W] in window mode)
    commit_lens: Optional[np.ndarray]  # int32 [bs] or None
    loc_row_width: int                # W in window mode, 0 otherwise
    pool_slots: int
    rope_base: float

    @property
    def KV(self) -> int:
        return self.NH * self.D

    @property
    def N(self) -> int:
        return self.L * 2 * self.KV

    @property
    def max_pos(self) -> int:
        return int(self.cos_sin.shape[0])

    @property
    def eps(self) -> float:
        return self.layers[0].eps

    @property
    def has_bias(self) -> bool:
        return self.layers[0].qkv_bias is not None


def rope_cos_sin_table(max_pos: int, head_dim: int, base: float) -> np.ndarray:
    """Precomputed neox cos/sin cache, fp32, one row per position.

    Row p holds cos(p * base**(-2i/D)) for i < D/2, then the matching sines
    (the layout the table-lookup kernels on the sglang PR #31847 page index as
    ``pos * D + i`` and ``pos * D + D/2 + i``).  Angles are formed in fp64 and
    the cos/sin values rounded once to fp32.  The table is an input of the
    write: it is built here, outside both implementations.
    """
    half = head_dim // 2
    inv_freq = base ** (-np.arange(half, dtype=np.float64) * 2.0 / head_dim)
    ang = np.arange(max_pos, dtype=np.float64)[:, None] * inv_freq[None, :]
    return np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32)


def _layers(rng, dtype, L, H, q_size, KV, D, eps, bias_std):
    layers = []
    rows = q_size + 2 * KV
    for _ in range(L):
        w = np.empty((rows, H), dtype=np.uint16)
        w[:q_size] = QNAN_BITS[dtype]
        w[q_size:] = to_bits(rng.standard_normal((2 * KV, H), dtype=np.float32)
                             * np.float32(H ** -0.5), dtype)
        b = None
        if bias_std is not None:
            b = np.empty((rows,), dtype=np.uint16)
            b[:q_size] = QNAN_BITS[dtype]
            b[q_size:] = to_bits(rng.standard_normal(2 * KV, dtype=np.float32)
                                 * np.float32(bias_std), dtype)
        knw = to_bits(1.0 + 0.1 * rng.standard_normal(D, dtype=np.float32), dtype)
        layers.append(Layer(qkv_weight=w, qkv_bias=b, k_norm_weight=knw, eps=eps))
    return layers


def _hidden(rng, T, H, dtype):
    return to_bits(rng.standard_normal((T, H), dtype=np.float32), dtype)


def _distinct_slots(rng, n, slots):
    return rng.permutation(slots)[:n].astype(np.int64)


def _window_commit(rng, bs, lo, hi):
    return rng.integers(lo, hi + 1, size=bs).astype(np.int32)


def make_workload(name: str, seed: Optional[int] = None, **kw) -> Workload:
    """Build one named synthetic workload (bit-identical for a given seed)."""
    seeds = {"tiny": 0, "decode512": 1, "prefill32k": 2, "fp16bias": 3, "k3gqa": 4}
    if name not in seeds:
        raise KeyError(f"unknown workload {name!r}; have {sorted(seeds)}")
    seed = seeds[name] if seed is None else seed
    rng = np.random.default_rng(seed)

    if name == "tiny":
        dtype, H, L, NH, D = BF16, kw.get("H", 256), kw.get("L", 2), 2, 64
        T = kw.get("tokens", 32)
        KV, q_size, eps, base, max_pos = NH * D, 2 * NH * D, 1e-6, 1e6, 4096
        slots = kw.get("pool_slots", max(256, T))
        layers = _layers(rng, dtype, L, H, q_size, KV, D, eps, None)
        x = _hidden(rng, T, H, dtype)
        pos = rng.integers(0, 4000, size=T).astype(np.int64)
        loc = _distinct_slots(rng, T, slots)
        commit, width = None, 0

    elif name in ("decode512", "k3gqa"):
        if name == "decode512":
            dtype, H, L, NH, D = BF16, 4096, 5, 8, 128
            q_size, slots, max_pos = 4 * NH * D, 65536, 65536
        else:
            dtype, H, L, NH, D = BF16, 7168, 5, 8, 64
            q_size, slots, max_pos = 4 * NH * D, 262144, 131072
        width = 8
        T = kw.get("tokens", 512 if name == "decode512" else 2048)
        if T % width:
            raise ValueError("window-mode token count must be a multiple of 8")
        bs = T // width
        KV, eps, base = NH * D, 1e-6, 1e6
        slots = kw.get("pool_slots", slots)
        layers = _layers(rng, dtype, L, H, q_size, KV, D, eps, None)
        x = _hidden(rng, T, H, dtype)
        if name == "decode512":
            ctx = rng.integers(1024, 32768 + 1, size=bs).astype(np.int64)
            pos = (ctx[:, None] + np.arange(width, dtype=np.int64)[None, :]).reshape(-1)
        else:
            pos = rng.integers(0, 131071, size=T).astype(np.int64)
        loc = _distinct_slots(rng, T, slots)
        commit = _window_commit(rng, bs, 1, width)

    elif name == "prefill32k":
        dtype, H, L, NH, D = BF16, 4096, 5, 8, 128
        req_len = kw.get("req_len", 4096)
        nreq = kw.get("requests", kw["tokens"] // req_len if "tokens" in kw else 8)
        T = nreq * req_len
        KV, q_size, eps, base, max_pos = NH * D, 4 * NH * D, 1e-6, 1e6, 4096
        slots = kw.get("pool_slots", 40000 if T <= 40000 else T + T // 5)
        layers = _layers(rng, dtype, L, H, q_size, KV, D, eps, None)
        x = _hidden(rng, T, H, dtype)
        pos = np.tile(np.arange(req_len, dtype=np.int64), nreq)
        # non-overlapping contiguous slot ranges, random order, random gaps
        spare = slots - T
        cuts = np.sort(rng.integers(0, spare + 1, size=nreq))
        order = rng.permutation(nreq)
        bases = np.empty(nreq, dtype=np.int64)
        for k, r in enumerate(order):
            bases[r] = cuts[k] + k * req_len
        loc = (bases[:, None] + np.arange(req_len, dtype=np.int64)[None, :]).reshape(-1)
        loc[rng.random(T) < 0.01] = -1
        commit, width = None, 0

    else:  # fp16bias
        dtype, H, L, NH, D = FP16, 5120, 8, 8, 128
        width = 16
        T = kw.get("tokens", 4096)
        bs = T // width
        KV, q_size, eps, base, max_pos = NH * D, 4 * NH * D, 1e-5, 1e6, 131072
        slots = kw.get("pool_slots", 65536)
        layers = _layers(rng, dtype, L, H, q_size, KV, D, eps, 0.02)
        x = _hidden(rng, T, H, dtype)
        start = rng.integers(0, 131056, size=bs).astype(np.int64)
        pos = (start[:, None] + np.arange(width, dtype=np.int64)[None, :]).reshape(-1)
        loc = _distinct_slots(rng, T, slots)
        commit = _window_commit(rng, bs, 0, width)

    return Workload(
        name=name, seed=seed, dtype=dtype, T=T, H=H, L=L, NH=NH, D=D, q_size=q_size,
        layers=layers, ctx_hidden=x, positions=pos.astype(np.int64),
        cos_sin=rope_cos_sin_table(max_pos, D, base), cache_loc=loc.astype(np.int64),
        commit_lens=commit, loc_row_width=width, pool_slots=slots, rope_base=base)


WORKLOADS = ("tiny", "decode512", "prefill32k", "fp16bias", "k3gqa")


@dataclasses.dataclass
class QkWorkload:
    """Inputs of the in-place QK RMSNorm + table RoPE of one draft layer."""
    name: str
    seed: int
    dtype: str
    T: int
    num_q_heads: int
    num_k_heads: int
    D: int
    qkv: np.ndarray          # bits [T, (num_q_heads + 2*num_k_heads) * D]: Q, K, V heads
    positions: np.ndarray    # int64 [T]
    cos_sin: np.ndarray      # float32 [max_pos, D]
    q_weight: np.ndarray     # bits [D]
    k_weight: np.ndarray     # bits [D]
    eps: float

    @property
    def row(self) -> int:
        return (self.num_q_heads + 2 * self.num_k_heads) * self.D


def make_qknorm_workload(name: str, seed: Optional[int] = None, **kw) -> QkWorkload:
    """The draft layer's fused QKV rows for the shapes of a named context-KV
    workload: its tokens, positions, cos/sin table, dtype and eps, with
    q_size / head_dim Q heads and num_kv_heads K and V heads.  QKV values are
    N(0,1); the Q and K norm weights 1 + 0.1 N(0,1), in the model dtype."""
    w = make_workload(name, seed, **kw)
    rng = np.random.default_rng(w.seed + 1000)
    nq, nk, D = w.q_size // w.D, w.NH, w.D
    qkv = to_bits(rng.standard_normal((w.T, (nq + 2 * nk) * D), dtype=np.float32), w.dtype)
    qw = to_bits(1.0 + 0.1 * rng.standard_normal(D, dtype=np.float32), w.dtype)
    kwt = to_bits(1.0 + 0.1 * rng.standard_normal(D, dtype=np.float32), w.dtype)
    return QkWorkload(name=name, seed=w.seed, dtype=w.dtype, T=w.T, num_q_heads=nq, num_k_heads=nk, D=D,
                      qkv=qkv, positions=w.positions, cos_sin=w.cos_sin, q_weight=qw, k_weight=kwt,
                      eps=w.eps)


def describe(w: Workload) -> Dict[str, object]:
    return {"workload": w.name, "tokens": w.T, "hidden": w.H, "layers": w.L,
            "kv_heads": w.NH, "head_dim": w.D, "dtype": w.dtype, "bias": w.has_bias,
            "window": w.loc_row_width, "pool_slots": w.pool_slots, "max_pos": w.max_pos,
            "seed": w.seed}


def make_verify_workload(batch: int, block: int, seed: int = 5, vocab: int = 151936):
    """Verify-step inputs: int64 target [batch, block] uniform over the vocab;
    candidates [batch, block] whose column 0 is random and whose drafts copy
    the target's previous-position token up to a first disagreement at a
    uniform position in [0, block-1] (block-1: every draft agrees); the
    tokens after it are random."""
    rng = np.random.default_rng(seed)
    target = rng.integers(0, vocab, size=(batch, block), dtype=np.int64)
    cand = rng.integers(0, vocab, size=(batch, block), dtype=np.int64)
    k = rng.integers(0, block, size=batch)
    for b in range(batch):
        cand[b, 1:k[b] + 1] = target[b, :k[b]]
        if k[b] < block - 1:
            cand[b, k[b] + 1] = (target[b, k[b]] + 1 + rng.integers(0, vocab - 1)) % vocab
    return cand, target


@dataclasses.dataclass
class AttnWorkload:
    """Inputs of the draft attention over a pool (bit patterns in ``dtype``)."""
    dtype: str
    batch: int
    block: int
    num_q_heads: int
    num_kv_heads: int
    D: int
    q: np.ndarray            # [batch*block, Hq, D]
    k_ext: np.ndarray        # [batch*block, Hkv, D]
    v_ext: np.ndarray
    k_pool: np.ndarray       # [slots, Hkv, D]
    v_pool: np.ndarray
    kv_indices: np.ndarray   # int64 [sum of context lengths]
    kv_start: np.ndarray     # int64 [batch + 1]
    sm_scale: float

    @property
    def max_context(self) -> int:
        return int(np.diff(self.kv_start).max()) if self.batch else 0


def make_attention_workload(batch: int, block: int, num_q_heads: int, num_kv_heads: int, D: int,
                            ctx_lo: int, ctx_hi: int, slack: int = 64, dtype: str = BF16,
                            seed: int = 6, contexts: Optional[Sequence[int]] = None) -> AttnWorkload:
    """Per request a context length U[ctx_lo, ctx_hi] (or the given
    `contexts`) of distinct random pool slots (pool = total context + slack
    slots); q, keys and values N(0,1) in the model dtype; sm_scale = D**-0.5."""
    rng = np.random.default_rng(seed)
    ctx = rng.integers(ctx_lo, ctx_hi + 1, size=batch)
    if contexts is not None:
        ctx = np.asarray(contexts, dtype=np.int64)
        assert ctx.shape == (batch,)
    slots = int(ctx.sum()) + slack
    idx = rng.permutation(slots)[:int(ctx.sum())].astype(np.int64)
    start = np.concatenate([[0], np.cumsum(ctx)]).astype(np.int64)
    rows = batch * block

    def draw(*shape):
        return to_bits(rng.standard_normal(shape, dtype=np.float32), dtype)

    return AttnWorkload(dtype=dtype, batch=batch, block=block, num_q_heads=num_q_heads,
                        num_kv_heads=num_kv_heads, D=D, q=draw(rows, num_q_heads, D),
                        k_ext=draw(rows, num_kv_heads, D), v_ext=draw(rows, num_kv_heads, D),
                        k_pool=draw(slots, num_kv_heads, D), v_pool=draw(slots, num_kv_heads, D),
                        kv_indices=idx, kv_start=start, sm_scale=float(D) ** -0.5)


@dataclasses.dataclass
class CombineWorkload:
    """Inputs of combine_hidden_states (bit patterns in ``dtype``)."""
    dtype: str
    T: int
    hidden: int
    n_aux: int
    aux: np.ndarray          # [T, n_aux * hidden]
    weight: np.ndarray       # [hidden, n_aux * hidden]
    norm_weight: np.ndarray  # [hidden]
    eps: float


def make_combine_workload(name: str = "decode512", tokens: Optional[int] = None, n_aux: int = 3,
                          hidden: Optional[int] = None, seed: Optional[int] = None) -> CombineWorkload:
    """The draft model's main_proj / main_norm inputs for a workload's shapes:
    n_aux auxiliary hidden states of the target, each N(0,1); main_proj
    weight std (n_aux * hidden)**-0.5; norm weight 1 + 0.1 N(0,1)."""
    w = make_workload(name, seed, **({} if tokens is None else {"tokens": tokens}))
    H = w.H if hidden is None else hidden
    rng = np.random.default_rng(w.seed + 2000)
    K = n_aux * H
    return CombineWorkload(dtype=w.dtype, T=w.T, hidden=H, n_aux=n_aux,
                           aux=to_bits(rng.standard_normal((w.T, K), dtype=np.float32), w.dtype),
                           weight=to_bits(rng.standard_normal((H, K), dtype=np.float32) * np.float32(K ** -0.5),
                                          w.dtype),
                           norm_weight=to_bits(1.0 + 0.1 * rng.standard_normal(H, dtype=np.float32), w.dtype),
                           eps=w.eps)
