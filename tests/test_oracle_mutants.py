"""Planted mistakes in the oracle must be caught by its pins.

Each case edits one line of the oracle's source (a dropped term, a flipped
sign, a wrong index, a wrong normaliser), loads the edited copy as a separate
module on the CPU, and checks that at least one pin fails on it.  This shows
that the pins constrain every formula the oracle implements.
"""
import importlib.util
import os
import types

import pytest

from tests import oracle_pins as P

pytest.importorskip("mpmath")

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "vloss_oracle.py")

MUTANTS = {
    "ce loss sign": ("loss[t] = lse[t] - s[int(labels[t])]", "loss[t] = s[int(labels[t])] - lse[t]"),
    "lse without log": ("return float(m + np.log(S))", "return float(m + S)"),
    "lse without max": ("return float(m + np.log(S))", "return float(np.log(S))"),
    "ce grad drops onehot": ("        g[t] = scale * (p - oh)", "        g[t] = scale * p"),
    "ce grad drops scale": ("        g[t] = scale * (p - oh)", "        g[t] = (p - oh)"),
    "ce label off by one": ("j = int(labels[t]) - col0", "j = int(labels[t]) - col0 + 1"),
    "ce mean over all rows": ("    n = loss_end - loss_start\n", "    n = loss_end\n"),
    "kl loss drops lse": ("loss[t] += pt * (np.log(pt) - (s_full[j] - l))", "loss[t] += pt * (np.log(pt) - s_full[j])"),
    "kl loss flips ln p": ("loss[t] += pt * (np.log(pt) - (s_full[j] - l))", "loss[t] += pt * (-np.log(pt) - (s_full[j] - l))"),
    "kl scatter sign": ("row[j - col0] -= coef * pt", "row[j - col0] += coef * pt"),
    "kl student term drops coef": ("row = coef * p_s", "row = p_s.copy()"),
    "kl ignores window": ("        if not win[t]:\n            continue\n        s_full", "        s_full"),
    "kl fold drops onehot": ("row += ce_coef * (p_s - oh)", "row += ce_coef * p_s"),
    "topk ties to higher id": ("order = np.argsort(-s, kind=\"stable\")[:k]",
                               "order = (len(s) - 1 - np.argsort(-s[::-1], kind=\"stable\"))[:k]"),
    "topk probs over the row": ("probs[t] = e / e.sum()", "probs[t] = e / np.exp(s - v[0]).sum()"),
    "topk ascending": ("order = np.argsort(-s, kind=\"stable\")[:k]", "order = np.argsort(s, kind=\"stable\")[:k]"),
    "ce forward ignores window": ("        if win[t]:\n            loss[t] = lse[t]", "        if True:\n            loss[t] = lse[t]"),
    "ce backward ignores window": ("        if not win[t]:\n            continue\n        s = logits[t, col0",
                                   "        s = logits[t, col0"),
    "ce mean of empty window": ("    if n <= 0:\n        return 0.0\n", ""),
    "ce slice part drops lse": ("part[t] = float(lse[t]) - s[j]", "part[t] = -s[j]"),
    "topk ignores window": ("        if not win[t]:\n            continue\n        s = logits[t].astype(np.float64)\n        order",
                            "        s = logits[t].astype(np.float64)\n        order"),
    "kl keeps zero probabilities": ("            if pt > 0.0:\n                loss[t] +=", "            if True:\n                loss[t] +="),
    "kl slice start excluded": ("if not (col0 <= j < col0 + ncols):", "if not (col0 < j < col0 + ncols):"),
    "lse sum drops the max term": ("S = np.exp(s - m).sum()", "S = np.exp(s - m).sum() - 1.0"),
    "acc_add subtracts": ("return (a.astype(np.float64) + b.astype(np.float64)).astype(np.float32)",
                          "return (a.astype(np.float64) - b.astype(np.float64)).astype(np.float32)"),
    "acc_add truncates": ("return (a.astype(np.float64) + b.astype(np.float64)).astype(np.float32)",
                          "return np.trunc((a.astype(np.float64) + b.astype(np.float64))).astype(np.float32)"),
}


def _load_mutant(old, new):
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation site not found: {old!r}"
    src = src.replace(old, new)
    mod = types.ModuleType("vloss_oracle_mutant")
    exec(compile(src, "vloss_oracle_mutant.py", "exec"), mod.__dict__)
    return mod


@pytest.mark.filterwarnings("ignore::RuntimeWarning")      # a broken formula may take the log of 0
@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name):
    mod = _load_mutant(*MUTANTS[name])
    failed = []
    for pin in P.ALL_PINS:
        try:
            pin(mod)
        except (AssertionError, ValueError, IndexError, FloatingPointError) as e:
            failed.append(pin.__name__)
    assert failed, f"no pin catches the planted mistake '{name}'"
