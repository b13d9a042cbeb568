"""Plant plausible mistakes in copies of the oracle and check the pins catch each.

Every mutant is the oracle's source with one edit (a dropped term, a wrong sign
or index, a transposed reduction, a reversed tie rule ...), loaded as a separate
module on the CPU. The real oracle is untouched. A mutant survives only if
every pin in test_oracle_pins passes on it, which fails this test.
"""
import inspect
import os
import sys
import types

import pytest

import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle",
                   "h2o_oracle.py")

MUTANTS = {
    "new token left out of attention": ("    s = c.scale * (K @ q)\n",
                                        "    s = c.scale * (K @ q)\n    s[-1] = -np.inf\n"),
    "candidate mask off by one": ("pos <= t - c.r", "pos < t - c.r"),
    "row sums instead of column sums": ("colsum[:i1] += P.sum(axis=0)",
                                        "colsum[i0:i1] += P.sum(axis=1)"),
    "decode logits unscaled": ("    s = c.scale * (K @ q)\n", "    s = (K @ q)\n"),
    "decode tie rule reversed": ("np.lexsort((pos[cand], score[cand]))",
                                 "np.lexsort((-pos[cand], score[cand]))"),
    "scores not accumulated": ("score = np.append(c.score + p[:-1], p[-1])",
                               "score = np.append(c.score, p[-1])"),
    "new token starts at score zero": ("score = np.append(c.score + p[:-1], p[-1])",
                                       "score = np.append(c.score + p[:-1], 0.0)"),
    "recent window shifted": ("np.arange(n_cand, T)])", "np.arange(n_cand - 1, T - 1)])"),
    "prefill keeps the lowest scores": ("heavy = order[n_drop:]", "heavy = order[:h]"),
    "causal mask leaks one future key": ("cols <= rows", "cols <= rows + 1"),
    "decode evicts the maximum": ("e_idx = order[0]", "e_idx = order[-1]"),
    "softmax not normalised": ("p = e / e.sum()", "p = e / (e.sum() + 1e-3)"),
    "prefill tie rule reversed": ("np.lexsort((cand, colsum[:n_cand]))",
                                  "np.lexsort((-cand, colsum[:n_cand]))"),
    "prefill scale ignored": ("S = scale * (Q[i0:i1] @ K[:i1].T)", "S = (Q[i0:i1] @ K[:i1].T)"),
    "prefill values from keys": ("O[i0:i1] = P @ V[:i1]", "O[i0:i1] = P @ K[:i1, :V.shape[1]]"),
    # the near-tie margin (steps below the threshold are excused from exact comparison)
    "decode margin forced to zero": ("margin = (s2 - s1) / s2 if s2 > 0 else 0.0", "margin = 0.0"),
    "prefill margin forced to zero": ("margin = (s_keep - s_drop) / s_keep if s_keep > 0 else 0.0",
                                      "margin = 0.0"),
    "decode margin over every attended token": ("s1, s2 = score[order[0]], score[order[1]]",
                                                "s1, s2 = np.sort(score)[:2]"),
    "decode margin not relative": ("margin = (s2 - s1) / s2 if s2 > 0 else 0.0",
                                   "margin = (s2 - s1) if s2 > 0 else 0.0"),
    "prefill margin against the wrong dropped key": ("s_drop = colsum[order[n_drop - 1]]",
                                                     "s_drop = colsum[order[max(n_drop - 2, 0)]]"),
    "prefill margin relative to the dropped key": (
        "margin = (s_keep - s_drop) / s_keep if s_keep > 0 else 0.0",
        "margin = (s_keep - s_drop) / s_drop if s_drop > 0 else 0.0"),
}


def _load_mutant(name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name!r} not unique"
    src = src.replace(old, new)
    modname = "oracle_mutant_" + "".join(ch if ch.isalnum() else "_" for ch in name)
    mod = types.ModuleType(modname)
    mod.__file__ = SRC
    mod.__package__ = "oracle"  # the oracle's relative imports resolve in its package
    sys.modules[modname] = mod
    try:
        exec(compile(src, SRC, "exec"), mod.__dict__)
    except Exception:
        del sys.modules[modname]
        raise
    return mod


def _pin_calls():
    """(check function, args) for every pin and each of its parametrize cases."""
    calls = []
    for name, fn in inspect.getmembers(pins, inspect.isfunction):
        if not name.startswith("check_"):
            continue
        test = getattr(pins, "test_" + name[len("check_"):])
        marks = getattr(test, "pytestmark", [])
        cases = [()]
        for m in marks:
            if m.name == "parametrize":
                argvals = m.args[1]
                cases = [tuple(v) if isinstance(v, (tuple, list)) else (v,) for v in argvals]
        for c in cases:
            calls.append((fn, c))
    return calls


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name):
    old, new = MUTANTS[name]
    mod = _load_mutant(name, old, new)
    try:
        caught = []
        for fn, args in _pin_calls():
            try:
                fn(mod, *args)
            except Exception as e:  # an assertion or a crash both count as caught
                caught.append((fn.__name__, type(e).__name__))
                break
        assert caught, f"mutant {name!r} passes every pin"
    finally:
        sys.modules.pop(mod.__name__, None)
