"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Each ``pin_*`` function takes an oracle module (the real one, or a copy with a
planted mistake) and raises AssertionError when the oracle disagrees with:

* the hand-derived closed forms in tests/golden/closed_forms.json,
* brute force at 50 significant digits (mpmath) written from the plain
  definitions (-ln softmax, sum p ln(p/q)), not from the max-shifted form,
* central finite differences of the oracle's own loss (which pins the
  gradient formula to the loss formula),
* invariants: gradient rows sum to zero, KL >= 0, KL = 0 at a match,
  top-k equal to a pure-Python sort, sliced = unsliced,
* exact rational arithmetic (acc_add).
"""
from __future__ import annotations

import json
import math
import os
from fractions import Fraction

import numpy as np

from top_kl_distill_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "closed_forms.json")


def golden():
    with open(GOLDEN) as f:
        return json.load(f)


def _close(a, b, tol, what):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, f"{what}: shape {a.shape} vs {b.shape}"
    err = np.max(np.abs(a - b)) if a.size else 0.0
    assert err <= tol, f"{what}: max abs error {err:.3e} > {tol:.1e}"


# ----------------------------------------------------------------- golden


def pin_golden_ce(O):
    for c in golden()["ce"]:
        if "logits_const" in c:
            s = np.full((1, c["V"]), c["logits_const"], dtype=np.float64)
        else:
            s = np.array([c["logits"]], dtype=np.float64)
        lab = np.array([c["label"]])
        loss, lse, g, mean = O.ce_fused(s, lab, 0, 1, c["scale"])
        _close(loss, [c["loss"]], 1e-12, c["case"] + " loss")
        _close(lse, [c["lse"]], 1e-12, c["case"] + " lse")
        _close(mean, c["loss"], 1e-12, c["case"] + " mean")
        if "grad" in c:
            _close(g[0], c["grad"], 1e-12, c["case"] + " grad")
        else:
            want = np.full(c["V"], c["grad_other"])
            want[c["label"]] = c["grad_label"]
            _close(g[0], want, 1e-12, c["case"] + " grad")


def pin_golden_kl(O):
    for c in golden()["kl"]:
        s = np.array([c["logits"]], dtype=np.float64)
        tid = np.array([c["tid"]])
        tp = np.array([c["tp"]], dtype=np.float64)
        loss, g = O.kl_topk(s, tid, tp, c["coef"])
        _close(loss, [c["loss"]], 1e-12, c["case"] + " loss")
        _close(g[0], c["grad"], 1e-12, c["case"] + " grad")


def pin_golden_topk(O):
    for c in golden()["topk"]:
        s = np.array([c["logits"]], dtype=np.float32)
        ids, probs, valid = O.topk_rows(s, c["k"])
        assert valid.all()
        assert ids[0].tolist() == c["ids"], f"{c['case']}: ids {ids[0].tolist()} vs {c['ids']}"
        u = np.array(c["probs_unnormalised"])
        _close(probs[0], u / u.sum(), 1e-15, c["case"] + " probs")


# ----------------------------------------------------------------- brute force (mpmath)


def _mp():
    import mpmath
    mpmath.mp.dps = 50
    return mpmath


def pin_ce_brute_force(O):
    mp = _mp()
    for V in (1, 2, 7, 33, 200):
        s = W.random_logits(4, V, seed=100 + V, sigma=3.0)
        lab = W.random_labels(4, V, seed=200 + V)
        loss, lse = O.ce_forward(s, lab, 0, 4)
        for t in range(4):
            ex = [mp.e ** mp.mpf(float(x)) for x in s[t]]
            Z = mp.fsum(ex)
            want_loss = -mp.log(ex[int(lab[t])] / Z)
            want_lse = mp.log(Z)
            assert abs(float(want_loss) - loss[t]) <= 1e-12 * max(1.0, abs(float(want_loss))), "CE loss vs -ln softmax"
            assert abs(float(want_lse) - lse[t]) <= 1e-12 * max(1.0, abs(float(want_lse))), "lse vs ln sum exp"


def pin_ce_mean_page_case(O):
    """The page's tiny parity case: seq 4, vocab 8, logits sin(0.3 i), labels [2, 5, 1, 7]."""
    mp = _mp()
    s = np.array([math.sin(0.3 * i) for i in range(32)], dtype=np.float32).reshape(4, 8)
    lab = np.array([2, 5, 1, 7])
    loss, lse, g, mean = O.ce_fused(s, lab, 0, 4, 0.25)
    tot = mp.mpf(0)
    for t in range(4):
        ex = [mp.e ** mp.mpf(float(x)) for x in s[t]]
        tot += -mp.log(ex[int(lab[t])] / mp.fsum(ex))
    assert abs(float(tot / 4) - mean) < 1e-13, "mean CE of the page's case"
    # empty window: mean 0, loss 0, gradient 0
    loss, lse, g, mean = O.ce_fused(s, lab, 2, 2, 1.0)
    assert mean == 0.0 and not loss.any() and not g.any(), "empty window"


def pin_kl_brute_force(O):
    mp = _mp()
    for V, k in ((5, 3), (40, 7), (300, 16)):
        s = W.random_logits(3, V, seed=300 + V, sigma=2.0)
        tid, tp = W.random_teacher(3, V, k, seed=400 + V)
        loss, g = O.kl_topk(s, tid, tp, 1.0)
        for t in range(3):
            ex = [mp.e ** mp.mpf(float(x)) for x in s[t]]
            Z = mp.fsum(ex)
            want = mp.fsum(mp.mpf(float(p)) * mp.log(mp.mpf(float(p)) / (ex[int(j)] / Z))
                           for j, p in zip(tid[t], tp[t]) if p > 0)
            assert abs(float(want) - loss[t]) <= 1e-12 * max(1.0, abs(float(want))), "KL vs sum p ln(p/q)"


def pin_topk_probs_full_softmax(O):
    mp = _mp()
    s = W.random_logits(2, 12, seed=7, sigma=2.0)
    ids, probs, _ = O.topk_rows(s, 12)
    for t in range(2):
        ex = [mp.e ** mp.mpf(float(x)) for x in s[t]]
        Z = mp.fsum(ex)
        want = [float(ex[int(j)] / Z) for j in ids[t]]
        _close(probs[t], want, 1e-15, "k = V probabilities are the softmax")


# ----------------------------------------------------------------- finite differences


def _fd(f, x, h=1e-6):
    g = np.zeros_like(x)
    for idx in np.ndindex(x.shape):
        xp = x.copy(); xp[idx] += h
        xm = x.copy(); xm[idx] -= h
        g[idx] = (f(xp) - f(xm)) / (2 * h)
    return g


def pin_ce_grad_fd(O):
    ntok, V, ls, le, scale = 5, 9, 1, 4, 0.37
    s = W.random_logits(ntok, V, seed=11).astype(np.float64)
    lab = W.random_labels(ntok, V, seed=12)

    def total(x):
        loss, _ = O.ce_forward(x, lab, ls, le)
        return scale * loss.sum()

    _, lse = O.ce_forward(s, lab, ls, le)
    g, _ = O.ce_backward(s, lab, lse, ls, le, scale)
    _close(g, _fd(total, s), 2e-8, "CE gradient vs finite differences")
    _, _, gf, _ = O.ce_fused(s, lab, ls, le, scale)
    _close(gf, _fd(total, s), 2e-8, "fused CE gradient vs finite differences")


def pin_kl_grad_fd(O):
    ntok, V, coef = 4, 11, 0.61
    s = W.random_logits(ntok, V, seed=13).astype(np.float64)
    # dyadic teacher probabilities: they sum to exactly 1 in binary
    tp = np.array([[0.5, 0.25, 0.125, 0.125]] * ntok)
    tid = np.array([[3, 0, 7, 10], [1, 2, 3, 4], [10, 9, 8, 0], [5, 6, 2, 1]])

    def total(x):
        loss, _ = O.kl_topk(x, tid, tp, coef)
        return coef * loss.sum()

    _, g = O.kl_topk(s, tid, tp, coef)
    _close(g, _fd(total, s), 2e-8, "KL gradient vs finite differences")
    # a window: rows outside contribute nothing, their gradient is 0
    def total_w(x):
        loss, _ = O.kl_topk(x, tid, tp, coef, 1, 3)
        return coef * loss.sum()

    _, gw = O.kl_topk(s, tid, tp, coef, 1, 3)
    _close(gw, _fd(total_w, s), 2e-8, "windowed KL gradient vs finite differences")


def pin_combined_grad_fd(O):
    """CE folded into the KL pass: gradient of ce_coef*CE + coef*KL."""
    ntok, V, coef, ce_coef = 3, 8, 0.3, 0.7
    s = W.random_logits(ntok, V, seed=14).astype(np.float64)
    lab = W.random_labels(ntok, V, seed=15)
    tp = np.array([[0.75, 0.25]] * ntok)
    tid = np.array([[1, 6], [0, 3], [7, 2]])

    def total(x):
        kl, _ = O.kl_topk(x, tid, tp, coef)
        ce, _ = O.ce_forward(x, lab, 0, ntok)
        return coef * kl.sum() + ce_coef * ce.sum()

    _, g = O.kl_topk(s, tid, tp, coef, labels=lab, ce_coef=ce_coef)
    _close(g, _fd(total, s), 2e-8, "combined CE + KL gradient vs finite differences")


# ----------------------------------------------------------------- invariants


def pin_ce_invariants(O):
    ntok, V, ls, le, scale = 16, 300, 3, 13, 0.125
    s = W.random_logits(ntok, V, seed=21, sigma=3.0)
    lab = W.random_labels(ntok, V, seed=22)
    loss, lse, g, mean = O.ce_fused(s, lab, ls, le, scale)
    rs = g.sum(axis=1)
    assert np.all(np.abs(rs) < 1e-15), "CE gradient rows sum to 0"
    assert np.all(g[:ls] == 0) and np.all(g[le:] == 0), "rows outside the window are 0"
    assert np.all(loss[:ls] == 0) and np.all(loss[le:] == 0), "loss outside the window is 0"
    assert np.all(loss[ls:le] > 0), "CE > 0 for V > 1"
    assert np.all(lse >= s.max(axis=1)), "lse >= max"
    assert np.all(lse <= s.max(axis=1) + math.log(V) + 1e-12), "lse <= max + ln V"
    assert abs(mean - loss.sum() / (le - ls)) < 1e-12
    # uniform logits: loss = ln V on every in-window row
    u = np.full((4, 64), -1.5, dtype=np.float32)
    loss, lse, g, _ = O.ce_fused(u, np.array([0, 5, 63, 17]), 0, 4, 1.0)
    _close(loss, [math.log(64)] * 4, 1e-13, "uniform logits give ln V")
    # slices of the backward concatenate to the full gradient, loss parts add up
    _, lse = O.ce_forward(s, lab, ls, le)
    full, part = O.ce_backward(s, lab, lse, ls, le, scale)
    cuts = [(0, 100), (100, 128), (228, 72)]
    pieces, parts = [], np.zeros(ntok)
    for c0, w in cuts:
        gp, pp = O.ce_backward(s, lab, lse, ls, le, scale, c0, w)
        pieces.append(gp)
        parts += pp
    _close(np.concatenate(pieces, axis=1), full, 0.0, "sliced CE gradient = full")
    loss2, _ = O.ce_forward(s, lab, ls, le)
    _close(parts, loss2, 1e-12, "slice loss parts add up to the loss")


def pin_kl_invariants(O):
    ntok, V, k, coef = 12, 500, 24, 0.5
    s = W.random_logits(ntok, V, seed=31, sigma=2.0)
    tid, tp = W.random_teacher(ntok, V, k, seed=32)
    loss, g = O.kl_topk(s, tid, tp, coef)
    assert np.all(loss >= 0), "KL >= 0"
    sum_tp = tp.astype(np.float64).sum(axis=1)
    _close(g.sum(axis=1), coef * (1.0 - sum_tp), 1e-15, "KL gradient rows sum to coef (1 - sum p_T)")
    # k = V, p_T = softmax(s): KL = 0 and gradient 0
    s2 = W.random_logits(2, 30, seed=33).astype(np.float64)
    e = np.exp(s2 - s2.max(axis=1, keepdims=True))
    p = e / e.sum(axis=1, keepdims=True)
    ids = np.tile(np.arange(30), (2, 1))
    l2, g2 = O.kl_topk(s2, ids, p, 1.0)
    _close(l2, [0, 0], 1e-14, "KL at p_T = p_S over the whole vocabulary")
    _close(g2, np.zeros_like(g2), 1e-15, "gradient at p_T = p_S")
    # repeated teacher ids add up: gradient equals that of the merged support
    tid_d = np.array([[4, 9, 4, 2]])
    tp_d = np.array([[0.25, 0.25, 0.25, 0.25]])
    tid_m = np.array([[4, 9, 2]])
    tp_m = np.array([[0.5, 0.25, 0.25]])
    sd = W.random_logits(1, 12, seed=34)
    _, gd = O.kl_topk(sd, tid_d, tp_d, 1.0)
    lm, gm = O.kl_topk(sd, tid_m, tp_m, 1.0)
    _close(gd, gm, 1e-16, "repeated ids add their contributions")
    # zero teacher probability: no loss term (0 ln 0 = 0, the guard of kl_rows), no
    # gradient change
    lz, gz = O.kl_topk(sd, np.array([[4, 9, 2, 7]]), np.array([[0.5, 0.25, 0.25, 0.0]]), 1.0)
    _close(gz, gm, 1e-16, "p_T = 0 entries change the gradient by nothing")
    _close(lz, lm, 1e-16, "p_T = 0 entries add no loss term")
    # window: rows outside [loss_start, loss_end) have loss 0 and a zero gradient,
    # rows inside equal the unwindowed result
    lw, gw = O.kl_topk(s, tid, tp, coef, 2, 9)
    assert not lw[:2].any() and not lw[9:].any(), "KL loss outside the window is 0"
    assert not gw[:2].any() and not gw[9:].any(), "KL gradient outside the window is 0"
    _close(lw[2:9], loss[2:9], 0.0, "in-window KL rows are unchanged")
    _close(gw[2:9], g[2:9], 0.0, "in-window KL gradient rows are unchanged")


def pin_kl_sliced(O):
    """The page's host-reference shape: v = 1024, 45 tokens, k = 16, three slices (384, 384, 256),
    teacher ids (37 t + 61 q) mod v."""
    from top_kl_distill_gb300.slicing import vocab_cuts
    v, ntok, k = 1024, 45, 16
    s = W.random_logits(ntok, v, seed=41, sigma=2.0)
    tid = np.array([[(t * 37 + q * 61) % v for q in range(k)] for t in range(ntok)])
    _, tp = W.random_teacher(ntok, v, k, seed=42)
    lab = W.random_labels(ntok, v, seed=43)
    coef, ce_coef = 1.0 / ntok, 0.25
    full_loss, full_g = O.kl_topk(s, tid, tp, coef, labels=lab, ce_coef=ce_coef)
    _, lse = O.ce_forward(s, lab, 0, ntok)
    cuts = vocab_cuts(v, max_rows=384)
    assert [w for _, w in cuts] == [384, 384, 256]
    acc = np.zeros(ntok, dtype=np.float64)
    pieces = []
    for c0, w in cuts:
        l, g = O.kl_topk(s, tid, tp, coef, lse=lse, col0=c0, ncols=w, labels=lab, ce_coef=ce_coef)
        pieces.append(g)
        acc += l
    _close(np.concatenate(pieces, axis=1), full_g, 1e-15, "sliced KL + CE gradient = unsliced")
    _close(acc, full_loss, 1e-12, "slice KL losses add up to the unsliced KL")
    # the CE fold is exactly ce_coef / scale times the CE gradient
    kl_only_loss, kl_only = O.kl_topk(s, tid, tp, coef)
    ce_g, _ = O.ce_backward(s, lab, lse, 0, ntok, 1.0)
    _close(full_g, kl_only + ce_coef * ce_g, 1e-15, "CE fold = KL gradient + ce_coef * CE gradient")
    _close(full_loss, kl_only_loss, 0.0, "the CE fold leaves the KL loss unchanged")


def _brute_topk(row, k):
    return sorted(range(len(row)), key=lambda j: (-float(row[j]), j))[:k]


def pin_topk_sort(O):
    cases = [W.random_logits(3, 257, seed=51), W.tie_heavy_logits(3, 300, seed=52),
             W.tie_heavy_logits(2, 64, seed=53, step=1.0)]
    for s in cases:
        for k in (1, 5, 64, s.shape[1]):
            ids, probs, _ = O.topk_rows(s, k)
            for t in range(s.shape[0]):
                assert ids[t].tolist() == _brute_topk(s[t], k), "top-k vs a pure-Python sort"
                assert abs(probs[t].sum() - 1.0) < 1e-14, "probabilities sum to 1"
                assert np.all(np.diff(probs[t]) <= 0), "probabilities descend"
            if k == 1:
                assert ids[:, 0].tolist() == np.argmax(s.astype(np.float64), axis=1).tolist(), "k = 1 is argmax"
                assert np.all(probs == 1.0)
    # window: rows outside are not produced
    ids, probs, valid = O.topk_rows(cases[0], 3, 1, 2)
    assert valid.tolist() == [False, True, False] and np.all(ids[0] == -1)


def pin_acc_add(O):
    g = np.random.default_rng(5)
    a = (g.standard_normal(4000) * 10.0 ** g.integers(-6, 6, 4000)).astype(np.float32)
    b = (g.standard_normal(4000) * 10.0 ** g.integers(-6, 6, 4000)).astype(np.float32)
    out = O.acc_add(a, b)
    assert out.dtype == np.float32
    for x, y, z in zip(a, b, out):
        exact = Fraction(float(x)) + Fraction(float(y))
        # z must be the fp32 value nearest to the exact sum (ties to even)
        lo = np.nextafter(z, np.float32(-np.inf))
        hi = np.nextafter(z, np.float32(np.inf))
        dz = abs(Fraction(float(z)) - exact)
        assert dz <= abs(Fraction(float(lo)) - exact) and dz <= abs(Fraction(float(hi)) - exact), \
            "acc_add is the correctly rounded fp32 sum"


def pin_memory_figure(O=None):
    m = golden()["memory_figure"]
    b = m["seq"] * m["vocab"] * 4
    assert b == m["bytes"] and b / 2 ** 20 == m["mib"]


ALL_PINS = [
    pin_golden_ce, pin_golden_kl, pin_golden_topk,
    pin_ce_brute_force, pin_ce_mean_page_case, pin_kl_brute_force, pin_topk_probs_full_softmax,
    pin_ce_grad_fd, pin_kl_grad_fd, pin_combined_grad_fd,
    pin_ce_invariants, pin_kl_invariants, pin_kl_sliced, pin_topk_sort, pin_acc_add,
]
