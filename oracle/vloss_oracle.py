"""CPU oracle for the fused vocabulary-row losses.  TEST INFRASTRUCTURE ONLY.

This module is the slow, plain definition that the CUDA path is checked
against.  Only the tests, the smoke check and the benchmark's CPU-baseline leg
may import it; the library never does, and it shares no code with the library.

Everything is float64 numpy, one row at a time, in the order the pages state
the steps.  Inputs are the fp32 (or uint32) arrays the library receives; the
oracle widens them to float64 once and never rounds in between.  Results are
float64 (ids are int64) so that a test can measure the fp32 error of the CUDA
path against them.

Sources (page, item):

* [TH]  cortiq-engine 0.8.21, ``src/gpu_wgpu/train_head.rs``: the module
        doc (loss and gradient of the top-k distillation KL), the ``kl_rows``
        shader (max, sum of exponentials, log-sum-exp, loss over the teacher
        support, gradient write then scatter), the ``acc_add`` shader, the
        ``topk_rows`` shader (top-k and probabilities renormalised over the
        k) and the float64 host reference of ``head_kl_matches_host``.
* [CE]  aprender-train 0.36.0, ``entrenar/autograd/wgpu_cross_entropy.rs``:
        the module doc (loss = logsumexp - logit[label]; gradient
        softmax - onehot written in place), ``CEForwardParams`` /
        ``CEBackwardParams`` (loss window), ``read_loss`` (mean over the
        window) and ``backward`` (scale = 1 / max(1, window)).

Readings where the pages are silent (each one is listed in the design notes):

* Rows outside the window [loss_start, loss_end) have loss 0 and a gradient
  of exactly 0; their log-sum-exp is still produced by the CE forward.
  Top-k leaves such rows unwritten (here: marked invalid).
* The CE gradient scale and the KL coefficient are explicit arguments.
* Teacher ids that repeat within a row add their contributions.
* Top-k ties go to the lower column; -0.0 and +0.0 are equal.
* A vocabulary slice [col0, col0 + ncols) of a row uses the full-row
  log-sum-exp; the KL loss of a slice sums only the support ids inside it.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "row_lse", "ce_forward", "ce_backward", "ce_fused", "ce_mean",
    "kl_topk", "topk_rows", "acc_add",
]


def _window(ntok: int, loss_start: int, loss_end: int) -> np.ndarray:
    if not (0 <= loss_start <= loss_end <= ntok):
        raise ValueError("window must satisfy 0 <= loss_start <= loss_end <= ntok")
    w = np.zeros(ntok, dtype=bool)
    w[loss_start:loss_end] = True
    return w


def row_lse(s: np.ndarray) -> float:
    """log-sum-exp of one row: m = max s, S = sum exp(s - m), lse = m + ln S  [TH kl_rows]."""
    s = np.asarray(s, dtype=np.float64)
    m = s.max()
    S = np.exp(s - m).sum()
    return float(m + np.log(S))


# --------------------------------------------------------------------- CE


def ce_forward(logits: np.ndarray, labels: np.ndarray, loss_start: int, loss_end: int):
    """Per-token CE loss and log-sum-exp  [CE module doc, forward_async].

    loss_t = lse_t - s_t[label_t] for t in the window, 0 elsewhere; lse_t for
    every row.  Returns (loss[ntok], lse[ntok]) as float64.
    """
    ntok = logits.shape[0]
    win = _window(ntok, loss_start, loss_end)
    loss = np.zeros(ntok)
    lse = np.zeros(ntok)
    for t in range(ntok):
        s = logits[t].astype(np.float64)
        lse[t] = row_lse(s)
        if win[t]:
            loss[t] = lse[t] - s[int(labels[t])]
    return loss, lse


def ce_mean(loss: np.ndarray, loss_start: int, loss_end: int) -> float:
    """Mean loss over the window, 0 for an empty window  [CE read_loss]."""
    n = loss_end - loss_start
    if n <= 0:
        return 0.0
    return float(np.sum(np.asarray(loss, dtype=np.float64)) / n)


def ce_backward(logits: np.ndarray, labels: np.ndarray, lse: np.ndarray, loss_start: int,
                loss_end: int, scale: float, col0: int = 0, ncols: int | None = None):
    """CE gradient over columns [col0, col0+ncols)  [CE backward].

    g_t,j = scale * (exp(s_t,j - lse_t) - [j == label_t]) in the window, 0
    elsewhere.  Also returns the slice's share of the loss: lse_t - s_t[label]
    when the label falls inside the slice (and t is in the window), else 0.
    Returns (grad[ntok][ncols], loss_part[ntok]) as float64.
    """
    ntok, V = logits.shape
    ncols = V - col0 if ncols is None else ncols
    win = _window(ntok, loss_start, loss_end)
    g = np.zeros((ntok, ncols))
    part = np.zeros(ntok)
    for t in range(ntok):
        if not win[t]:
            continue
        s = logits[t, col0:col0 + ncols].astype(np.float64)
        p = np.exp(s - float(lse[t]))
        j = int(labels[t]) - col0
        oh = np.zeros(ncols)
        if 0 <= j < ncols:
            oh[j] = 1.0
            part[t] = float(lse[t]) - s[j]
        g[t] = scale * (p - oh)
    return g, part


def ce_fused(logits: np.ndarray, labels: np.ndarray, loss_start: int, loss_end: int, scale: float):
    """Forward and in-place backward in one call.  Returns (loss, lse, grad, mean)."""
    loss, lse = ce_forward(logits, labels, loss_start, loss_end)
    g, _ = ce_backward(logits, labels, lse, loss_start, loss_end, scale)
    return loss, lse, g, ce_mean(loss, loss_start, loss_end)


# --------------------------------------------------------------------- KL


def kl_topk(logits: np.ndarray, tid: np.ndarray, tp: np.ndarray, coef: float,
            loss_start: int = 0, loss_end: int | None = None, lse: np.ndarray | None = None,
            col0: int = 0, ncols: int | None = None, labels: np.ndarray | None = None,
            ce_coef: float = 0.0):
    """Top-k distillation KL and its gradient  [TH module doc, kl_rows, head_kl_matches_host].

    Per row t (in the window) with lse over the FULL row:

      loss_t = sum_q [p_q > 0] p_q (ln p_q - (s[id_q] - lse))
               (only q with id_q inside the slice when sliced)
      g_j    = coef * exp(s_j - lse)                     for j in the slice,
      g[id_q] -= coef * p_q                              for each q, in q order.

    With ``labels`` the CE gradient ce_coef * (exp(s_j - lse) - [j == label])
    is added to g (the loss stays the KL alone).  Rows outside the window:
    loss 0, g = 0.  Returns (loss[ntok], grad[ntok][ncols]) as float64.
    """
    ntok, V = logits.shape
    loss_end = ntok if loss_end is None else loss_end
    ncols = V - col0 if ncols is None else ncols
    win = _window(ntok, loss_start, loss_end)
    k = tid.shape[1]
    loss = np.zeros(ntok)
    g = np.zeros((ntok, ncols))
    for t in range(ntok):
        if not win[t]:
            continue
        s_full = logits[t].astype(np.float64)
        l = row_lse(s_full) if lse is None else float(lse[t])
        s = s_full[col0:col0 + ncols]
        p_s = np.exp(s - l)
        row = coef * p_s
        for q in range(k):
            j = int(tid[t, q])
            pt = float(tp[t, q])
            if not (col0 <= j < col0 + ncols):
                continue
            if pt > 0.0:
                loss[t] += pt * (np.log(pt) - (s_full[j] - l))
            row[j - col0] -= coef * pt
        if labels is not None and ce_coef != 0.0:
            oh = np.zeros(ncols)
            jl = int(labels[t]) - col0
            if 0 <= jl < ncols:
                oh[jl] = 1.0
            row += ce_coef * (p_s - oh)
        g[t] = row
    return loss, g


# --------------------------------------------------------------------- top-k


def topk_rows(logits: np.ndarray, k: int, loss_start: int = 0, loss_end: int | None = None):
    """Teacher top-k: ids of the k largest values, descending, ties to the lower id,
    and probabilities renormalised over the k  [TH topk_rows].

    The order is a full stable sort of the row by value, descending (numpy's
    stable argsort of -s; -0.0 and +0.0 compare equal).  prob_q =
    exp(v_q - v_0) / sum_r exp(v_r - v_0).  Rows outside the window are not
    produced: returns (ids[ntok][k] int64, probs[ntok][k] float64, valid[ntok]).
    """
    ntok, V = logits.shape
    loss_end = ntok if loss_end is None else loss_end
    if not (1 <= k <= V):
        raise ValueError("need 1 <= k <= V")
    win = _window(ntok, loss_start, loss_end)
    ids = np.full((ntok, k), -1, dtype=np.int64)
    probs = np.full((ntok, k), np.nan)
    for t in range(ntok):
        if not win[t]:
            continue
        s = logits[t].astype(np.float64)
        order = np.argsort(-s, kind="stable")[:k]
        v = s[order]
        e = np.exp(v - v[0])
        ids[t] = order
        probs[t] = e / e.sum()
    return ids, probs, win


# --------------------------------------------------------------------- acc_add


def acc_add(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """a + b rounded to fp32: the elementwise partial-sum add  [TH acc_add]."""
    a = np.asarray(a, dtype=np.float32)
    b = np.asarray(b, dtype=np.float32)
    return (a.astype(np.float64) + b.astype(np.float64)).astype(np.float32)
