"""Planted mistakes in the oracle must fail its pins.

The oracle is only trusted because its pins (tests/test_oracle_*pins.py) tie
it to facts from outside it.  This module checks that the pins are strong
enough: each case below rewrites one line of an oracle source file into a
plausible mistake (a dropped term, a wrong sign, index or operand, a K/V swap,
a layer mix-up, an off-by-one in the window rule, a misplaced eps), loads the
rewritten module in place of the real one (CPU only: nothing here touches the
CUDA path) and runs that file's pins; at least one pin must fail.  A case whose
line no longer appears in the oracle fails too, so the list follows the oracle.
"""
import importlib
import inspect
import itertools
import os
import sys
import types

import pytest

import oracle

ORACLE_DIR = os.path.dirname(oracle.__file__)
pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")

# oracle source file -> (pin module, [(case, exact original text, mistake)])
CASES = {
    "ctx_kv.py": ("test_oracle_pins", [
        ("K rows taken from the V slice",
         "w_k = qkv_weight[q_size:q_size + kv_size]",
         "w_k = qkv_weight[q_size + kv_size:q_size + 2 * kv_size]"),
        ("K rows taken from the Q slice",
         "w_k = qkv_weight[q_size:q_size + kv_size]",
         "w_k = qkv_weight[0:kv_size]"),
        ("K bias dropped",
         "k = k + qkv_bias[q_size:q_size + kv_size]",
         "k = k + 0 * qkv_bias[q_size:q_size + kv_size]"),
        ("V bias from the K slice",
         "v = v + qkv_bias[q_size + kv_size:q_size + 2 * kv_size]",
         "v = v + qkv_bias[q_size:q_size + kv_size]"),
        ("mean over D - 1",
         "ms = (y * y).sum(axis=-1, keepdims=True) / acc(head_dim)",
         "ms = (y * y).sum(axis=-1, keepdims=True) / acc(head_dim - 1)"),
        ("eps outside the square root",
         "inv = acc(1.0) / np.sqrt(ms + acc(eps))",
         "inv = acc(1.0) / (np.sqrt(ms) + acc(eps))"),
        ("norm weight dropped",
         "return (y * inv * k_norm_weight.astype(k.dtype)).reshape(k.shape)",
         "return (y * inv).reshape(k.shape)"),
        ("norm weight read as 1 + w",
         "return (y * inv * k_norm_weight.astype(k.dtype)).reshape(k.shape)",
         "return (y * inv * (1 + k_norm_weight.astype(k.dtype))).reshape(k.shape)"),
        ("first rotation sign",
         "o1 = x1 * cos - x2 * sin",
         "o1 = x1 * cos + x2 * sin"),
        ("second rotation sign",
         "o2 = x2 * cos + x1 * sin",
         "o2 = x2 * cos - x1 * sin"),
        ("cos and sin halves swapped",
         "cos = rows[:, None, :half]\n    sin = rows[:, None, half:]",
         "sin = rows[:, None, :half]\n    cos = rows[:, None, half:]"),
        ("interleaved (GPT-J) pairing",
         "x1, x2 = y[..., :half], y[..., half:]",
         "x1, x2 = y[..., 0::2], y[..., 1::2]"),
        ("table row of the next position",
         "rows = cos_sin[positions].astype(acc)",
         "rows = cos_sin[positions + 1].astype(acc)"),
        ("window rule off by one",
         "if col >= int(commit_lens[b]):",
         "if col > int(commit_lens[b]):"),
        ("window row and column swapped",
         "b, col = divmod(t, loc_row_width)",
         "col, b = divmod(t, loc_row_width)"),
        ("loc -1 not skipped",
         "if cache_loc[t] < 0:",
         "if cache_loc[t] < -1:"),
        ("stacked layers read at the wrong stride",
         "k = y[:, l * 2 * kv:l * 2 * kv + kv]",
         "k = y[:, l * kv:l * kv + kv]"),
        ("first layer's k_norm for every layer",
         "k = apply_k_norm(k, st.k_norm_weight[l].astype(acc)",
         "k = apply_k_norm(k, st.k_norm_weight[0].astype(acc)"),
        ("bf16 widened with a wrong shift",
         "(np.asarray(bits).astype(np.uint32) << 16)",
         "(np.asarray(bits).astype(np.uint32) << 15)"),
        ("mixed eps accepted",
         "if eps is not None and lay.eps != eps:",
         "if False:"),
    ]),
    "qk_norm_rope.py": ("test_oracle_qknorm_pins", [
        ("Q and K weights swapped",
         "[widen(q_weight, dtype)] * num_q_heads + [widen(k_weight, dtype)] * num_k_heads",
         "[widen(k_weight, dtype)] * num_q_heads + [widen(q_weight, dtype)] * num_k_heads"),
        ("no rounding of the normalised first half",
         "x1 = round_to(x[:, :, :half] * inv * w[None, :, :half], dtype)",
         "x1 = x[:, :, :half] * inv * w[None, :, :half]"),
        ("eps outside the square root",
         "inv = 1.0 / np.sqrt(np.mean(x * x, axis=2, keepdims=True) + eps)",
         "inv = 1.0 / (np.sqrt(np.mean(x * x, axis=2, keepdims=True)) + eps)"),
        ("mean over D - 1",
         "np.mean(x * x, axis=2, keepdims=True)",
         "(np.sum(x * x, axis=2, keepdims=True) / (D - 1))"),
        ("first rotation sign",
         "[x1 * c - x2 * s, x2 * c + x1 * s]",
         "[x1 * c + x2 * s, x2 * c + x1 * s]"),
        ("second rotation sign",
         "[x1 * c - x2 * s, x2 * c + x1 * s]",
         "[x1 * c - x2 * s, x2 * c - x1 * s]"),
        ("cos and sin halves swapped",
         "c = table[:, None, :half]\n    s = table[:, None, half:]",
         "s = table[:, None, :half]\n    c = table[:, None, half:]"),
        ("heads read one head late",
         "x = widen(qkv[t_idx, :nh * D], dtype)",
         "x = widen(qkv[t_idx, D:(nh + 1) * D], dtype)"),
        ("rounding half away from zero",
         "r = np.rint(x / quantum) * quantum",
         "r = np.trunc(x / quantum + np.sign(x) * 0.5) * quantum"),
    ]),
    "verify.py": ("test_oracle_verify_pins", [
        ("draft compared with the target at its own index",
         "still *= int(candidates[b, i + 1] == target[b, i])",
         "still *= int(candidates[b, i] == target[b, i])"),
        ("matches not cumulative",
         "still *= int(candidates[b, i + 1] == target[b, i])",
         "still = int(candidates[b, i + 1] == target[b, i])"),
        ("bonus one position early",
         "bonus[b] = target[b, n]",
         "bonus[b] = target[b, n - 1]"),
        ("every draft counted",
         "n += still",
         "n += 1"),
    ]),
    "draft_attention.py": ("test_oracle_attention_pins", [
        ("KV head of a query head taken modulo",
         "g = h // group",
         "g = h % num_kv_heads"),
        ("scale dropped",
         "s = sm_scale * (qb[:, h, :] @ kb[:, g, :].T)",
         "s = (qb[:, h, :] @ kb[:, g, :].T)"),
        ("block's own keys dropped",
         "widen(k_ext[b * E:(b + 1) * E], dtype)], axis=0)",
         "widen(k_ext[b * E:(b + 1) * E], dtype)[:0]], axis=0)"),
        ("causal mask inside the block",
         "p = np.exp(s)",
         "p = np.exp(s); p[:, s.shape[1] - E:] *= np.tril(np.ones((E, E)))"),
        ("softmax normalised over the queries",
         "p /= p.sum(axis=1, keepdims=True)",
         "p /= p.sum(axis=0, keepdims=True)"),
        ("keys used as values",
         "ob[:, h, :] = p @ vb[:, g, :]",
         "ob[:, h, :] = p @ kb[:, g, :]"),
    ]),
    "combine.py": ("test_oracle_combine_pins", [
        ("projection not rounded to the model dtype",
         "y = round_to(widen(aux, dtype) @ widen(weight, dtype).T, dtype)",
         "y = widen(aux, dtype) @ widen(weight, dtype).T"),
        ("eps outside the square root",
         "inv = 1.0 / np.sqrt(np.mean(y * y, axis=1, keepdims=True) + eps)",
         "inv = 1.0 / (np.sqrt(np.mean(y * y, axis=1, keepdims=True)) + eps)"),
        ("mean over the tokens",
         "np.mean(y * y, axis=1, keepdims=True)",
         "np.mean(y * y, axis=0, keepdims=True)"),
        ("norm weight dropped",
         "return y * inv * widen(norm_weight, dtype)[None, :]",
         "return y * inv"),
    ]),
}


def _calls(fn):
    """Every argument combination of a pin (its parametrize marks expanded)."""
    marks = [m for m in getattr(fn, "pytestmark", []) if m.name == "parametrize"]
    axes = []
    for m in marks:
        names, values = m.args[0], m.args[1]
        names = [n.strip() for n in names.split(",")] if isinstance(names, str) else list(names)
        rows = []
        for v in values:
            v = v.values if hasattr(v, "values") and not isinstance(v, dict) else v
            v = v if len(names) > 1 else (v,)
            rows.append(dict(zip(names, v)))
        axes.append(rows)
    for combo in itertools.product(*axes):
        kw = {}
        for part in combo:
            kw.update(part)
        yield kw


def _pins_fail(pin_module):
    """True if at least one pin of the module fails (raises) under the
    current oracle."""
    mod = importlib.import_module(pin_module)
    for name, fn in sorted(vars(mod).items()):
        if not name.startswith("test_") or not callable(fn):
            continue
        assert not set(inspect.signature(fn).parameters) - {
            n for kw in _calls(fn) for n in kw}, f"{name} needs a fixture"
        for kw in _calls(fn):
            try:
                fn(**kw)
            except Exception:   # a pin failed (assertion or an error the mistake caused)
                return True
    return False


def _load_mutated(fname, old, new, monkeypatch):
    path = os.path.join(ORACLE_DIR, fname)
    src = open(path).read()
    assert src.count(old) == 1, f"{fname}: the text to rewrite must appear once: {old!r}"
    mod = types.ModuleType(f"oracle._mutated_{fname[:-3]}")
    mod.__package__ = "oracle"
    mod.__file__ = path
    monkeypatch.setitem(sys.modules, mod.__name__, mod)   # dataclasses look their module up
    exec(compile(src.replace(old, new, 1), path + " (mutated)", "exec"), mod.__dict__)
    return mod


def _exported(fname):
    real = importlib.import_module("oracle." + fname[:-3])
    return [n for n in dir(oracle) if not n.startswith("_") and getattr(real, n, None) is getattr(oracle, n)]


@pytest.mark.parametrize("fname,case,old,new",
                         [(f, c, o, n) for f, (_, cases) in CASES.items() for c, o, n in cases],
                         ids=[f"{f[:-3]}: {c}" for f, (_, cases) in CASES.items() for c, _, _ in cases])
def test_planted_mistake_fails_a_pin(fname, case, old, new, monkeypatch):
    pins, _ = CASES[fname]
    assert not _pins_fail(pins), "the pins must pass on the oracle as it is"
    mutated = _load_mutated(fname, old, new, monkeypatch)
    for name in _exported(fname):
        monkeypatch.setattr(oracle, name, getattr(mutated, name))
    # functions of other oracle files that call into this one see the
    # rewritten module through the package attributes patched above
    assert _pins_fail(pins), f"no pin caught: {case}"
