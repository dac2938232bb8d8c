"""Seeded synthetic inputs shaped like the workloads of the fused vocabulary-row losses.

This module only draws random numbers.  It holds none of the loss arithmetic:
both the CUDA path and the CPU oracle are fed from here, and nothing here
depends on either of them.

Every tensor is generated in blocks of ``BLOCK_ROWS`` rows.  Block ``b`` of a
tensor is drawn from its own generator, seeded by ``(seed, tensor tag, b)``,
so any row range can be regenerated on its own (the full-size parity tests
use this to give the oracle only the rows they sample) and blocks can be
drawn on several host threads with the same result.

Workloads (one entry of ``WORKLOADS`` each):

* ``ce_tiny``   fused CE, 64 x 1024, logits N(0, 2^2), window [8, 64), scale 1/56.
* ``ce_lm``     fused CE, 512 x 32000, logits N(0, 3^2) plus 8 at the row's
                label with probability 0.3, window [128, 512), scale 1/384.
* ``kl``        top-k KL, 2048 x 32000, k = 64, student N(0, 2^2), teacher ids
                k distinct uniform ids, teacher probs the normalised exponentials
                of N(0, 1.5^2) draws over the k, coef 1/2048.
* ``topk``      teacher top-k, 4096 x 128256, k = 256 (2048 in the sweep),
                logits 4 z + 1e-3 pi(j) with pi a seeded permutation of the
                columns, then nudged upward until every row holds distinct
                fp32 values.
* ``large_v``   CE + top-k KL over 8192 x 128256, logits 2 t_4 (Student t,
                4 degrees of freedom), labels uniform, teacher as ``kl`` with
                k = 128, two vocabulary slices of 64128 columns.
"""
from __future__ import annotations

import concurrent.futures as _cf
import os
from dataclasses import dataclass, field

import numpy as np

BLOCK_ROWS = 64

# tensor tags: one independent stream per tensor of a workload
_T_LOGITS, _T_LABELS, _T_PEAK, _T_TID, _T_TPRAW, _T_PERM = 1, 2, 3, 4, 5, 6


@dataclass(frozen=True)
class Workload:
    name: str
    kind: str                 # "ce", "kl", "topk", "ce_kl_sliced"
    ntok: int
    V: int
    seed: int
    window: tuple = (0, None)  # (loss_start, loss_end); None = ntok
    scale: float = 0.0        # CE gradient scale
    k: int = 0
    coef: float = 0.0         # KL gradient coefficient
    ce_coef: float = 0.0      # CE gradient coefficient folded into the KL pass
    slices: int = 1           # vocabulary slices of the large-vocabulary step
    extra: dict = field(default_factory=dict)

    @property
    def loss_start(self) -> int:
        return int(self.window[0])

    @property
    def loss_end(self) -> int:
        return int(self.ntok if self.window[1] is None else self.window[1])

    def scaled(self, ntok: int) -> "Workload":
        """Same recipe and seed with ``ntok`` rows; the window is clipped to it."""
        ls = min(self.loss_start, ntok)
        le = min(self.loss_end, ntok)
        d = dict(self.__dict__)
        d.update(ntok=ntok, window=(ls, le))
        return Workload(**d)


WORKLOADS = {
    "ce_tiny": Workload("ce_tiny", "ce", 64, 1024, seed=0x7C0DE001, window=(8, 64),
                        scale=1.0 / 56, extra=dict(sigma=2.0)),
    "ce_lm": Workload("ce_lm", "ce", 512, 32000, seed=0x7C0DE002, window=(128, 512),
                      scale=1.0 / 384, extra=dict(sigma=3.0, peak=8.0, peak_prob=0.3)),
    "kl": Workload("kl", "kl", 2048, 32000, seed=0x7C0DE003, k=64, coef=1.0 / 2048,
                   extra=dict(sigma=2.0, teacher_sigma=1.5)),
    "topk": Workload("topk", "topk", 4096, 128256, seed=0x7C0DE004, k=256,
                     extra=dict(sigma=4.0, jitter=1e-3, k_sweep=2048)),
    "large_v": Workload("large_v", "ce_kl_sliced", 8192, 128256, seed=0x7C0DE005, k=128,
                        coef=1.0 / 8192, ce_coef=1.0 / 8192, slices=2,
                        extra=dict(t_scale=2.0, t_dof=4.0, teacher_sigma=1.5)),
}


def _gen(seed: int, tag: int, block: int) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence([seed & 0xFFFFFFFF, tag, block]))


def _blocks(r0: int, r1: int):
    b0, b1 = r0 // BLOCK_ROWS, (r1 + BLOCK_ROWS - 1) // BLOCK_ROWS
    for b in range(b0, b1):
        lo, hi = b * BLOCK_ROWS, (b + 1) * BLOCK_ROWS
        yield b, lo, hi, max(lo, r0), min(hi, r1)


def _threads() -> int:
    return max(1, min(16, os.cpu_count() or 1))


def _fill_rows(out: np.ndarray, r0: int, r1: int, ntok: int, block_fn, threads: int | None = None):
    """Fill ``out[0:r1-r0]`` with rows r0..r1 by drawing whole blocks."""
    jobs = []
    for b, lo, hi, a, z in _blocks(r0, r1):
        hi = min(hi, ntok)
        jobs.append((b, lo, hi, a, z))

    def one(job):
        b, lo, hi, a, z = job
        blk = block_fn(b, hi - lo)
        out[a - r0:z - r0] = blk[a - lo:z - lo]

    nthr = threads if threads is not None else _threads()
    if nthr <= 1 or len(jobs) <= 1:
        for j in jobs:
            one(j)
    else:
        with _cf.ThreadPoolExecutor(nthr) as ex:
            list(ex.map(one, jobs))
    return out


# ---------------------------------------------------------------- labels


def labels(w: Workload, r0: int = 0, r1: int | None = None) -> np.ndarray:
    """Row labels, uniform in [0, V), uint32."""
    r1 = w.ntok if r1 is None else r1
    out = np.empty(r1 - r0, dtype=np.uint32)

    def blk(b, n):
        return _gen(w.seed, _T_LABELS, b).integers(0, w.V, size=n, dtype=np.uint32)

    return _fill_rows(out, r0, r1, w.ntok, blk, threads=1)


# ---------------------------------------------------------------- logits


def logits(w: Workload, r0: int = 0, r1: int | None = None, out: np.ndarray | None = None,
           threads: int | None = None) -> np.ndarray:
    """fp32 logits rows [r0, r1) of workload ``w``, shape [r1-r0][V]."""
    r1 = w.ntok if r1 is None else r1
    if out is None:
        out = np.empty((r1 - r0, w.V), dtype=np.float32)
    V = w.V
    ex = w.extra

    if "peak" in ex:
        lab_all = labels(w, 0, w.ntok)

        def blk(b, n):
            g = _gen(w.seed, _T_LOGITS, b)
            x = g.standard_normal((n, V), dtype=np.float32)
            x *= np.float32(ex["sigma"])
            hit = _gen(w.seed, _T_PEAK, b).random(n) < ex["peak_prob"]
            rows = np.nonzero(hit)[0]
            lab = lab_all[b * BLOCK_ROWS + rows]
            x[rows, lab] += np.float32(ex["peak"])
            return x
    elif w.kind == "topk":
        def blk(b, n):
            g = _gen(w.seed, _T_LOGITS, b)
            gp = _gen(w.seed, _T_PERM, b)
            x = g.standard_normal((n, V), dtype=np.float32)
            x *= np.float32(ex["sigma"])
            perm = gp.permuted(np.broadcast_to(np.arange(V, dtype=np.int32), (n, V)), axis=1)
            x += perm.astype(np.float32) * np.float32(ex["jitter"])
            return make_distinct_rows(x)
    elif "t_dof" in ex:
        def blk(b, n):
            g = _gen(w.seed, _T_LOGITS, b)
            x = g.standard_t(ex["t_dof"], size=(n, V)).astype(np.float32)
            x *= np.float32(ex["t_scale"])
            return x
    else:
        def blk(b, n):
            g = _gen(w.seed, _T_LOGITS, b)
            x = g.standard_normal((n, V), dtype=np.float32)
            x *= np.float32(ex["sigma"])
            return x

    return _fill_rows(out, r0, r1, w.ntok, blk, threads)


def make_distinct_rows(x: np.ndarray) -> np.ndarray:
    """Nudge equal fp32 values within each row of ``x`` upward (nextafter) until all differ.

    In place.  Among equal values the one at the lowest column keeps its value;
    each later duplicate moves up by one ulp and the check repeats.
    """
    assert x.dtype == np.float32 and x.ndim == 2
    while True:
        order = np.argsort(x, axis=1, kind="stable")
        srt = np.take_along_axis(x, order, axis=1)
        r, c = np.nonzero(srt[:, 1:] == srt[:, :-1])
        if r.size == 0:
            return x
        cols = order[r, c + 1]
        x[r, cols] = np.nextafter(x[r, cols], np.float32(np.inf))


def make_distinct(row: np.ndarray) -> np.ndarray:
    """make_distinct_rows for one row."""
    make_distinct_rows(row.reshape(1, -1))
    return row


# ---------------------------------------------------------------- teacher


def teacher(w: Workload, r0: int = 0, r1: int | None = None):
    """Teacher top-k support: ids [n][k] uint32 (k distinct per row) and probs [n][k] fp32.

    The probabilities are exp(u_q - max u) / sum over the k, u ~ N(0, sigma^2),
    computed in float64 and rounded to fp32.
    """
    r1 = w.ntok if r1 is None else r1
    k, V = w.k, w.V
    ids = np.empty((r1 - r0, k), dtype=np.uint32)
    tp = np.empty((r1 - r0, k), dtype=np.float32)
    sig = w.extra.get("teacher_sigma", 1.5)

    def blk_ids(b, n):
        g = _gen(w.seed, _T_TID, b)
        return np.stack([g.choice(V, size=k, replace=False) for _ in range(n)]).astype(np.uint32)

    def blk_tp(b, n):
        g = _gen(w.seed, _T_TPRAW, b)
        u = g.standard_normal((n, k)) * sig
        e = np.exp(u - u.max(axis=1, keepdims=True))
        return (e / e.sum(axis=1, keepdims=True)).astype(np.float32)

    _fill_rows(ids, r0, r1, w.ntok, blk_ids, threads=1)
    _fill_rows(tp, r0, r1, w.ntok, blk_tp, threads=1)
    return ids, tp


# ---------------------------------------------------------------- test-only shapes


def tie_heavy_logits(n: int, V: int, seed: int, step: float = 0.125, sigma: float = 2.0) -> np.ndarray:
    """Logits quantised to multiples of ``step`` (many exact ties), with signed zeros mixed in."""
    g = _gen(seed, 77, 0)
    x = (np.round(g.standard_normal((n, V)) * sigma / step) * step).astype(np.float32)
    z = g.random((n, V)) < 0.5
    x[(x == 0) & z] = np.float32(-0.0)
    return x


def random_logits(n: int, V: int, seed: int, sigma: float = 2.0) -> np.ndarray:
    """Plain N(0, sigma^2) fp32 logits for ad-hoc test shapes."""
    return (_gen(seed, 78, 0).standard_normal((n, V)) * sigma).astype(np.float32)


def random_labels(n: int, V: int, seed: int) -> np.ndarray:
    return _gen(seed, 79, 0).integers(0, V, size=n, dtype=np.uint32)


def random_teacher(n: int, V: int, k: int, seed: int, sigma: float = 1.5, distinct: bool = True):
    g = _gen(seed, 80, 0)
    if distinct:
        ids = np.stack([g.choice(V, size=k, replace=False) for _ in range(n)]).astype(np.uint32)
    else:
        ids = g.integers(0, V, size=(n, k), dtype=np.uint32)
    u = g.standard_normal((n, k)) * sigma
    e = np.exp(u - u.max(axis=1, keepdims=True))
    return ids, (e / e.sum(axis=1, keepdims=True)).astype(np.float32)
