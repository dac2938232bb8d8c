"""Benchmark of the fused vocabulary-row losses on GB300 (one JSON line on stdout).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--no-sweep]
    python bench.py --impl reference ...      # the CPU oracle arm

Headline workload: fused cross-entropy over 512 token rows x 32000 vocabulary
fp32 logits, window [128, 512), scale 1/384 -- one step is one vl_ce_fused call
(loss, lse, in-place gradient, windowed mean) over the whole batch.  `value` is
token-rows per second over all ranks; each rank runs its own copy of the batch
(rows are independent, so ranks share no data and scaling is weak).

Timing: every timed step reads a freshly restored copy of the pristine inputs
(the kernels overwrite the logits with the gradient).  Restores happen outside
the events, followed by a write of a buffer larger than L2, so every step
starts with a cold L2.  CUDA events on the launching stream bracket each step;
the dominant kernel is also timed alone, launch by launch, for the roofline.

The sweep (on by default) measures the other workloads the same way and
reports them under "sweep": top-k KL 2048 x 32000 (k 64), teacher top-k
4096 x 128256 (k 256 and 2048), and the large-vocabulary step 8192 x 128256
(CE forward, two vocabulary slices of KL + CE gradient, acc_add).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from top_kl_distill_gb300 import workloads as W  # noqa: E402
from top_kl_distill_gb300.slicing import cuts_for_slices  # noqa: E402
from top_kl_distill_gb300.dist import max_over_ranks, world  # noqa: E402

METRIC = "token-rows/sec and achieved HBM GB/s (% of GB300 peak) at 32000/128256 vocab"
UNIT = "token-rows/s"
L2_FLUSH_BYTES = 512 << 20


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def bf16_peak():
    """Dense bf16 TFLOP/s of a kernel timed alone (the burst figure), measured or fallback."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        if "bf16_tflops" in d:
            return float(d["bf16_tflops"]), "measured"
    return 1900.0, "fallback"


def head_gemm_line(torch, flush, M=2048, N=128256, K=4096, reps=10):
    """The vocabulary head's logits GEMM (a chunk of 2048 hidden rows of 4096 against a
    128256 x 4096 weight plane, bf16 in, fp32 out) on the tensor-core kernel, timed alone
    with CUDA events after an L2 flush; cuBLAS (torch.matmul, bf16 out) on the same shape
    as context."""
    from top_kl_distill_gb300 import vloss as vl
    g = torch.Generator(device="cuda").manual_seed(20260)
    A = torch.randn(M, K, device="cuda", generator=g).to(torch.bfloat16)
    B = torch.randn(N, K, device="cuda", generator=g).to(torch.bfloat16)
    D = torch.empty(M, N, device="cuda")
    Dr = torch.empty(M, N, device="cuda", dtype=torch.bfloat16)

    def timed(fn):
        for _ in range(2):
            fn()
        ms = []
        for _ in range(reps):
            flush()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            ms.append(e0.elapsed_time(e1))
        return sorted(ms)[len(ms) // 2]

    ms = timed(lambda: vl.vl_gemm_bf16_tn(A, B, D, M, N, K, N, 1.0))
    ms_ref = timed(lambda: torch.matmul(A, B.t(), out=Dr))
    peak, kind = bf16_peak()
    tf = 2.0 * M * N * K / (ms * 1e-3) / 1e12
    out = {"shape": f"M {M} x N {N} x K {K}, bf16 in, fp32 out", "ms": round(ms, 4),
           "roofline": {"bound": "tensor", "achieved": round(tf, 1), "peak": peak, "unit": "TFLOP/s",
                        "frac": round(tf / peak, 4), "peak_source": kind, "kernel": "tc_gemm"},
           "cublas_bf16_out_tflops": round(2.0 * M * N * K / (ms_ref * 1e-3) / 1e12, 1), "gpu_launches": 1}
    del A, B, D, Dr
    torch.cuda.empty_cache()
    return out


def head_pipeline_lines(torch, flush, reps=5):
    """The head pipelines on the device, step by step: the student's (vl_head_kl: logits GEMM,
    one-pass CE + top-k KL in place, dx GEMM over the transposed weight plane) on 2048 rows of
    hidden size 4096 against a 32000 vocabulary, k 64; the teacher's (vl_teacher_topk: logits
    GEMM, streaming top-k) on 2048 rows against a 128256 vocabulary, k 256; chunks of 1024
    rows.  Each step timed alone after an L2 flush; `gemm_tflops` is the GEMMs' FLOPs over the
    whole step's time (the loss or top-k kernels included)."""
    from top_kl_distill_gb300 import vloss as vl
    g = torch.Generator(device="cuda").manual_seed(20261)
    n, hs = 2048, 4096

    def bf16(rows, cols, scale):
        return (torch.randn(rows, cols, device="cuda", generator=g) * scale).to(torch.bfloat16)

    def timed(fn):
        for _ in range(2):
            fn()
        ms = []
        for _ in range(reps):
            flush()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            ms.append(e0.elapsed_time(e1))
        return sorted(ms)[len(ms) // 2]

    out = {}
    hidden = bf16(n, hs, 1.0)
    V, k = 32000, 64
    w = bf16(V, hs, 3.0 / hs ** 0.5)
    wt = w.t().contiguous()
    lab = _dev(torch, W.random_labels(n, V, seed=31))
    tid, tp = W.random_teacher(n, V, k, seed=32)
    tid, tp = _dev(torch, tid), _dev(torch, tp)
    dx = torch.empty(n, hs, device="cuda")
    kl, ce, mean = (torch.empty(n, device="cuda"), torch.empty(n, device="cuda"), torch.empty(1, device="cuda"))
    ms = timed(lambda: vl.vl_head_kl(hidden, hs, w, wt, V, n, lab, tid, tp, k, 1.0 / n, 1.0 / n, 1.0, 0, n, dx, kl,
                                     ce, mean))
    out["head_kl"] = {"shape": f"{n} rows, hidden {hs}, V {V}, k {k}", "ms_per_step": round(ms, 4),
                      "rows_per_s": round(n / (ms * 1e-3), 1),
                      "gemm_tflops": round(2 * 2.0 * n * V * hs / (ms * 1e-3) / 1e12, 1), "gpu_launches": 9}
    del w, wt, lab, tid, tp, dx, kl, ce, mean
    torch.cuda.empty_cache()
    V, k = 128256, 256
    w = bf16(V, hs, 3.0 / hs ** 0.5)
    ids = torch.empty(n, k, dtype=torch.int32, device="cuda")
    probs = torch.empty(n, k, device="cuda")
    ms = timed(lambda: vl.vl_teacher_topk(hidden, hs, w, V, n, k, 0, n, ids, probs))
    out["teacher_topk"] = {"shape": f"{n} rows, hidden {hs}, V {V}, k {k}", "ms_per_step": round(ms, 4),
                           "rows_per_s": round(n / (ms * 1e-3), 1),
                           "gemm_tflops": round(2.0 * n * V * hs / (ms * 1e-3) / 1e12, 1), "gpu_launches": 6}
    del w, ids, probs, hidden
    torch.cuda.empty_cache()
    return out


# ------------------------------------------------------------------ clocks


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the loop runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.t is not None:
            self.t.join(timeout=5)

    def summary(self, t0: float, t1: float):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ts, line in self.lines:
            if not (t0 <= ts <= t1):
                continue
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ workloads


class Case:
    """One workload: pristine inputs on the device, R work buffers, step and kernel calls."""

    name = ""
    inplace = True
    launches_per_step = 1

    def rows(self) -> int:
        raise NotImplementedError

    def bytes_per_step(self) -> int:
        raise NotImplementedError


def _dev(torch, a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint32:
        return torch.from_numpy(a.view(np.int32)).cuda()
    return torch.from_numpy(a).cuda()


class CeFused(Case):
    def __init__(self, torch, w, nbuf):
        from top_kl_distill_gb300 import vloss as vl
        self.vl, self.w, self.torch = vl, w, torch
        self.name = w.name
        self.launches_per_step = 2          # fused kernel + windowed mean
        self.x_host = W.logits(w)
        self.lab_host = W.labels(w)
        self.pristine = _dev(torch, self.x_host)
        self.labels = _dev(torch, self.lab_host)
        self.bufs = [torch.empty_like(self.pristine) for _ in range(nbuf)]
        n = w.ntok
        self.loss = torch.zeros(n, device="cuda")
        self.lse = torch.zeros(n, device="cuda")
        self.mean = torch.zeros(1, device="cuda")

    def rows(self):
        return self.w.ntok

    def bytes_per_step(self):
        # per row: read and write V fp32, read the label, write loss and lse; plus the mean
        return self.w.ntok * (8 * self.w.V + 12) + (self.w.loss_end - self.w.loss_start) * 4 + 4

    def kernel_bytes(self):
        return self.w.ntok * (8 * self.w.V + 12)

    def restore(self, j):
        self.bufs[j].copy_(self.pristine)

    def step(self, j, mean=True):
        w = self.w
        self.vl.vl_ce_fused(self.bufs[j], w.V, w.ntok, w.V, self.labels, w.loss_start, w.loss_end, w.scale,
                            self.loss, self.lse, None, self.mean if mean else None, None)

    def kernel(self, j):
        self.step(j, mean=False)


class CeFusedShard(CeFused):
    """This rank's contiguous row shard of the fused CE batch (dist.window_shard): the fused
    kernel over its rows with its part of the loss window and the batch's gradient scale,
    then the one exchange step, an all-reduce of (mean x rows) that gives every rank the
    batch's mean over the window (dist.global_window_mean)."""

    def __init__(self, torch, w, nbuf, rank, ws):
        from top_kl_distill_gb300 import vloss as vl
        from top_kl_distill_gb300.dist import window_shard
        self.vl, self.torch = vl, torch
        self.batch = w
        r0, r1, ls, le = window_shard(w.ntok, rank, ws, w.loss_start, w.loss_end)
        self.r0, self.r1, self.ls, self.le = r0, r1, ls, le
        self.w = w
        self.name = w.name
        self.launches_per_step = 2
        self.x_host = W.logits(w, r0, r1)
        self.lab_host = W.labels(w, r0, r1)
        self.pristine = _dev(torch, self.x_host)
        self.labels = _dev(torch, self.lab_host)
        self.bufs = [torch.empty_like(self.pristine) for _ in range(nbuf)]
        n = r1 - r0
        self.loss = torch.zeros(max(n, 1), device="cuda")
        self.lse = torch.zeros(max(n, 1), device="cuda")
        self.mean = torch.zeros(1, device="cuda")
        self.global_mean = None

    def rows(self):
        return self.r1 - self.r0

    def bytes_per_step(self):
        return self.rows() * (8 * self.w.V + 12) + (self.le - self.ls) * 4 + 4

    def kernel_bytes(self):
        return self.rows() * (8 * self.w.V + 12)

    def step(self, j, mean=True):
        from top_kl_distill_gb300.dist import global_window_mean
        w, n = self.w, self.rows()
        self.vl.vl_ce_fused(self.bufs[j], w.V, n, w.V, self.labels, self.ls, self.le, w.scale,
                            self.loss, self.lse, None, self.mean if mean else None, None)
        if mean:
            self.global_mean = global_window_mean(self.mean, self.le - self.ls, w.loss_end - w.loss_start)


class CeFusedBf16(CeFused):
    """The fused CE step on bf16 logits (the same draws rounded to bf16): vl_ce_fused_bf16,
    2 bytes an element each way."""

    def __init__(self, torch, w, nbuf):
        super().__init__(torch, w, nbuf)
        self.name = w.name + "_bf16"
        self.pristine = self.pristine.to(torch.bfloat16)
        self.bufs = [torch.empty_like(self.pristine) for _ in range(nbuf)]

    def bytes_per_step(self):
        return self.w.ntok * (4 * self.w.V + 12) + (self.w.loss_end - self.w.loss_start) * 4 + 4

    def kernel_bytes(self):
        return self.w.ntok * (4 * self.w.V + 12)

    def step(self, j, mean=True):
        w = self.w
        self.vl.vl_ce_fused_bf16(self.bufs[j], w.V, w.ntok, w.V, self.labels, w.loss_start, w.loss_end, w.scale,
                                 self.loss, self.lse, None, self.mean if mean else None, None)


class Kl(Case):
    def __init__(self, torch, w, nbuf):
        from top_kl_distill_gb300 import vloss as vl
        self.vl, self.w = vl, w
        self.name = w.name
        self.pristine = _dev(torch, W.logits(w))
        tid, tp = W.teacher(w)
        self.tid, self.tp = _dev(torch, tid), _dev(torch, tp)
        self.bufs = [torch.empty_like(self.pristine) for _ in range(nbuf)]
        self.loss = torch.zeros(w.ntok, device="cuda")

    def rows(self):
        return self.w.ntok

    def bytes_per_step(self):
        return self.w.ntok * (8 * self.w.V + 8 * self.w.k + 4)

    kernel_bytes = bytes_per_step

    def restore(self, j):
        self.bufs[j].copy_(self.pristine)

    def step(self, j):
        w = self.w
        self.vl.vl_kl_topk_inplace(self.bufs[j], w.V, w.ntok, w.V, 0, w.V, self.tid, self.tp, w.k, w.coef,
                                   w.loss_start, w.loss_end, None, None, None, 0.0, self.loss, None)

    kernel = step


class TopK(Case):
    inplace = False
    _cache = {}

    def __init__(self, torch, w, nbuf, k):
        from top_kl_distill_gb300 import vloss as vl
        self.vl, self.w, self.k = vl, w, k
        self.name = f"{w.name}_k{k}"
        key = (w.name, w.ntok)
        if TopK._cache.get("key") != key:
            TopK._cache.clear()
            TopK._cache.update(key=key, x=_dev(torch, W.logits(w)))
        self.x = TopK._cache["x"]
        self.bufs = [self.x]
        self.ids = torch.zeros((w.ntok, k), dtype=torch.int32, device="cuda")
        self.probs = torch.zeros((w.ntok, k), device="cuda")
        self.launches_per_step = 2 if vl.vl_topk_workspace_bytes(w.ntok, w.V, k) else 1

    def rows(self):
        return self.w.ntok

    def bytes_per_step(self):
        return self.w.ntok * (4 * self.w.V + 8 * self.k)

    kernel_bytes = bytes_per_step

    def restore(self, j):
        pass

    def step(self, j):
        """One vl_topk_rows call: with the workspace, the streaming kernel (filter and
        finish warps) and the exact kernel for the rows it leaves (none on these rows)."""
        w = self.w
        self.vl.vl_topk_rows(self.x, w.V, w.ntok, w.V, self.k, 0, w.ntok, self.ids, self.probs)

    kernel = step


class LargeV(Case):
    """CE and top-k KL of 8192 rows x 128256 columns in one pass (vl_ce_kl_fused: each row
    read once and its combined gradient written once, a row per 3-CTA cluster), and the
    windowed CE mean."""

    def __init__(self, torch, w, nbuf):
        from top_kl_distill_gb300 import vloss as vl
        self.vl, self.w = vl, w
        self.name = w.name
        self.launches_per_step = 2
        self.pristine = _dev(torch, W.logits(w))
        self.labels = _dev(torch, W.labels(w))
        tid, tp = W.teacher(w)
        self.tid, self.tp = _dev(torch, tid), _dev(torch, tp)
        self.bufs = [torch.empty_like(self.pristine) for _ in range(nbuf)]
        n = w.ntok
        self.ce_loss = torch.zeros(n, device="cuda")
        self.kl_loss = torch.zeros(n, device="cuda")
        self.mean = torch.zeros(1, device="cuda")

    def rows(self):
        return self.w.ntok

    def bytes_per_step(self):
        w = self.w
        # per row: read and write V fp32, the teacher's ids and probabilities, the label,
        # both losses; plus the mean over the window
        return w.ntok * (8 * w.V + 8 * w.k + 4 + 8) + (w.loss_end - w.loss_start) * 4 + 4

    def kernel_bytes(self):
        w = self.w
        return w.ntok * (8 * w.V + 8 * w.k + 4 + 8)

    def restore(self, j):
        self.bufs[j].copy_(self.pristine)

    def step(self, j, mean=True):
        w = self.w
        self.vl.vl_ce_kl_fused(self.bufs[j], w.V, w.ntok, w.V, self.labels, self.tid, self.tp, w.k, w.coef,
                               w.ce_coef, w.loss_start, w.loss_end, self.kl_loss, self.ce_loss, None, None,
                               self.mean if mean else None, None)

    def kernel(self, j):
        self.step(j, mean=False)


class LargeVBf16(LargeV):
    """The one-pass large-vocabulary step on bf16 logits (vl_ce_kl_fused_bf16)."""

    def __init__(self, torch, w, nbuf):
        super().__init__(torch, w, nbuf)
        self.name = w.name + "_bf16"
        self.pristine = self.pristine.to(torch.bfloat16)
        self.bufs = [torch.empty_like(self.pristine) for _ in range(nbuf)]

    def bytes_per_step(self):
        w = self.w
        return w.ntok * (4 * w.V + 8 * w.k + 4 + 8) + (w.loss_end - w.loss_start) * 4 + 4

    def kernel_bytes(self):
        w = self.w
        return w.ntok * (4 * w.V + 8 * w.k + 4 + 8)

    def step(self, j, mean=True):
        w = self.w
        self.vl.vl_ce_kl_fused_bf16(self.bufs[j], w.V, w.ntok, w.V, self.labels, self.tid, self.tp, w.k, w.coef,
                                    w.ce_coef, w.loss_start, w.loss_end, self.kl_loss, self.ce_loss, None, None,
                                    self.mean if mean else None, None)


class LargeVSliced(Case):
    """The same step over two vocabulary slices of 64128 columns: CE forward over full
    rows (row statistics), then per slice the in-place KL + CE gradient from them, then
    acc_add of the slices' KL parts -- the slice API, 12 V bytes a row."""

    def __init__(self, torch, w, nbuf):
        from top_kl_distill_gb300 import vloss as vl
        self.vl, self.w = vl, w
        self.name = w.name + "_sliced"
        self.launches_per_step = 2 + w.slices
        self.pristine = _dev(torch, W.logits(w))
        self.labels = _dev(torch, W.labels(w))
        tid, tp = W.teacher(w)
        self.tid, self.tp = _dev(torch, tid), _dev(torch, tp)
        self.bufs = [torch.empty_like(self.pristine) for _ in range(nbuf)]
        n = w.ntok
        self.ce_loss = torch.zeros(n, device="cuda")
        self.lse = torch.zeros(n, device="cuda")
        self.stats = torch.zeros((n, 2), device="cuda")
        self.mean = torch.zeros(1, device="cuda")
        self.parts = [torch.zeros(n, device="cuda") for _ in range(w.slices)]
        self.kl_loss = self.parts[0]
        self.cuts = cuts_for_slices(w.V, w.slices)

    def rows(self):
        return self.w.ntok

    def bytes_per_step(self):
        w = self.w
        fwd = 4 * w.V + 4 + 4 + 4 + 8                     # row, label, loss, lse, stats
        per_slice = 8 * (w.V // w.slices) + 8 * w.k + 4 + 8 + 4   # slice rw, support, label, stats, part
        acc = 12 * (w.slices - 1)
        return w.ntok * (fwd + w.slices * per_slice + acc) + w.ntok * 4 + 4

    def kernel_bytes(self):
        w = self.w
        return w.ntok * (8 * self.cuts[0][1] + 8 * w.k + 4 + 8 + 4)

    def restore(self, j):
        self.bufs[j].copy_(self.pristine)

    def step(self, j):
        w, vl, x = self.w, self.vl, self.bufs[j]
        vl.vl_ce_fwd(x, w.V, w.ntok, w.V, self.labels, 0, w.ntok, self.ce_loss, self.lse, self.stats, self.mean,
                     None)
        for (c0, width), part in zip(self.cuts, self.parts):
            vl.vl_kl_topk_inplace(x, w.V, w.ntok, w.V, c0, width, self.tid, self.tp, w.k, w.coef, 0, w.ntok,
                                  None, self.stats, self.labels, w.ce_coef, part, None)
        for part in self.parts[1:]:
            vl.vl_acc_add(self.parts[0], part, w.ntok)

    def kernel(self, j):
        """The dominant kernel: the first vocabulary slice's KL + CE pass (statistics given)."""
        w, x = self.w, self.bufs[j]
        c0, width = self.cuts[0]
        self.vl.vl_kl_topk_inplace(x, w.V, w.ntok, w.V, c0, width, self.tid, self.tp, w.k, w.coef, 0, w.ntok,
                                   None, self.stats, self.labels, w.ce_coef, self.parts[0], None)


def nbuf_for(bytes_per_buf: int) -> int:
    """Work buffers per round: enough that a round streams well past L2, at most 16 GB."""
    return int(max(2, min(16, (16 << 30) // max(1, bytes_per_buf))))


def base_workload(name):
    if name.startswith("topk"):
        return W.WORKLOADS[name.split("_k")[0]]
    for suffix in ("_sliced", "_bf16"):
        if name.endswith(suffix):
            return W.WORKLOADS[name[:-len(suffix)]]
    return W.WORKLOADS[name]


def make_case(torch, name, ntok=None, nbuf=None):
    w = base_workload(name)
    if ntok:
        w = w.scaled(ntok)
    nb = nbuf or nbuf_for(w.ntok * w.V * 4)
    if w.kind == "ce":
        return CeFusedBf16(torch, w, nb) if name.endswith("_bf16") else CeFused(torch, w, nb)
    if w.kind == "kl":
        return Kl(torch, w, nb)
    if w.kind == "topk":
        k = int(name.split("_k")[1]) if "_k" in name else w.k
        return TopK(torch, w, 1, k)
    if w.kind == "ce_kl_sliced":
        if name.endswith("_sliced"):
            return LargeVSliced(torch, w, nb)
        return LargeVBf16(torch, w, nb) if name.endswith("_bf16") else LargeV(torch, w, nb)
    raise ValueError(name)


# ------------------------------------------------------------------ timing


def time_case(torch, case, steps, warmup, flush, kernel_only=False):
    """Times exactly `steps` steps; returns (total ms, per-round ms per step).

    Steps run in rounds over the R work buffers.  Before a round every buffer is
    restored from the pristine inputs and L2 is flushed (eager, untimed); the
    round's steps are then replayed from a captured CUDA graph between two
    events, so the device runs them back to back without waiting on the host.
    """
    fn = case.kernel if kernel_only else case.step
    R = len(case.bufs)
    for i in range(warmup):
        j = i % R
        case.restore(j)
        flush()
        fn(j)
    torch.cuda.synchronize()
    graphs = {}

    def graph_for(n):
        if n not in graphs:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                for j in range(n):
                    fn(j)
            graphs[n] = g
        return graphs[n]

    per = []
    total = 0.0
    done = 0
    while done < steps:
        n = min(R, steps - done)
        g = graph_for(n)
        for j in range(n):
            case.restore(j)
        flush()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record()
        g.replay()
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1)
        total += ms
        per.append(ms / n)
        done += n
    return total, per


CLOCK_WINDOW_S = 0.8


def soak(torch, case, flush, until):
    """Untimed rounds of the step (restore, flush, R steps) until wall time `until`."""
    R = len(case.bufs)
    n = 0
    while time.time() < until:
        for j in range(R):
            case.restore(j)
        flush()
        for j in range(R):
            case.step(j)
        torch.cuda.synchronize()
        n += 1
    return n


def e2e_ce(torch, case, steps, warmup, chunks=2):
    """The headline step end to end from pinned host buffers through the C ABI, run the way a
    training loop runs it: step after step, each step's logits and labels uploaded from
    pinned host memory, vl_ce_fused over them, then the gradient, loss, lse and the window
    mean downloaded.

    Three streams linked by events: copy-in (H2D), compute (vl_ce_fused a row chunk at a
    time, then vl_window_mean) and copy-out (D2H), so a chunk's download overlaps the next
    chunk's upload (2 chunks: 0.418 ms a step on a GB300, 1 chunk 0.419, 4 chunks 0.433, 8
    chunks 0.573; the host link moves about 330 GB/s with both directions busy).  Consecutive steps alternate between two sets of device buffers, so a
    step's uploads may start while the step before is still downloading, as a loader that
    prefetches the next batch does; a step's uploads wait for the downloads of the step two
    back, which used the same buffers.  Every step's copies and calls are in the timed
    region, which ends when the last step's mean is on the host.  Returns (ms per step, H2D
    bytes, D2H bytes, whether the last step's host gradient equals a device-only step's)."""
    w, vl = case.w, case.vl
    n, V = w.ntok, w.V
    hx = torch.from_numpy(case.x_host).pin_memory()
    hl = torch.from_numpy(case.lab_host.view(np.int32)).pin_memory()
    hg = torch.empty_like(hx).pin_memory()
    hloss = torch.empty(n).pin_memory()
    hlse = torch.empty(n).pin_memory()
    hmean = torch.empty(1).pin_memory()
    xs = [case.bufs[0], case.bufs[1]]
    labs = [case.labels, torch.empty_like(case.labels)]
    losses = [case.loss, torch.empty_like(case.loss)]
    lses = [case.lse, torch.empty_like(case.lse)]
    means = [case.mean, torch.empty_like(case.mean)]
    s_in, s_run, s_out = (torch.cuda.Stream() for _ in range(3))
    spans = [(i * n // chunks, (i + 1) * n // chunks) for i in range(chunks)]
    done = [None, None]          # per buffer set: the event after its last step's downloads

    def one(k):
        b = k % 2
        x, lab, loss, lse, mean = xs[b], labs[b], losses[b], lses[b], means[b]
        with torch.cuda.stream(s_in):
            if done[b] is not None:
                s_in.wait_event(done[b])
            lab.copy_(hl, non_blocking=True)
            ups = []
            for r0, r1 in spans:
                x[r0:r1].copy_(hx[r0:r1], non_blocking=True)
                ups.append(s_in.record_event())
        for (r0, r1), up in zip(spans, ups):
            s_run.wait_event(up)
            ls = min(max(w.loss_start - r0, 0), r1 - r0)
            le = min(max(w.loss_end - r0, 0), r1 - r0)
            vl.vl_ce_fused(x[r0:r1], V, r1 - r0, V, lab[r0:r1], ls, le, w.scale, loss[r0:r1], lse[r0:r1],
                           None, None, None, s_run)
            s_out.wait_event(s_run.record_event())
            with torch.cuda.stream(s_out):
                hg[r0:r1].copy_(x[r0:r1], non_blocking=True)
        vl.vl_window_mean(loss, n, w.loss_start, w.loss_end, mean, s_run)
        s_out.wait_event(s_run.record_event())
        with torch.cuda.stream(s_out):
            hloss.copy_(loss, non_blocking=True)
            hlse.copy_(lse, non_blocking=True)
            hmean.copy_(mean, non_blocking=True)
            done[b] = s_out.record_event()

    main = torch.cuda.current_stream()

    def run(k0, count):
        start = main.record_event()
        for st in (s_in, s_run, s_out):
            st.wait_event(start)
        for k in range(k0, k0 + count):
            one(k)
        for st in (s_in, s_run, s_out):
            main.wait_stream(st)

    run(0, warmup)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    run(warmup, steps)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    # the host copies hold the last step's results: check them against a device-only step
    last = xs[(warmup + steps - 1) % 2]
    ok = bool(torch.equal(hg.cuda(), last))
    for t in xs:
        t.copy_(case.pristine)
    h2d = hx.numel() * 4 + hl.numel() * 4
    d2h = hg.numel() * 4 + 2 * n * 4 + 4
    return ms, h2d, d2h, ok


# The sources each measured kernel is built from: its DRAM traffic in profiles/ncu_traffic.json
# stands only while these files are unchanged since the capture.
ROW_SOURCES = ("rows.cu", "vl_device.cuh", "vl_internal.h", "vloss_api.cu")
TOPK_SOURCES = ("topk_stream.cu", "topk.cu", "vl_topk.cuh", "vl_device.cuh", "vl_internal.h", "vloss_api.cu")
KERNEL_SOURCES = {"ce_fused": ROW_SOURCES, "ce_fused_tiny": ROW_SOURCES, "ce_fused_bf16": ROW_SOURCES,
                  "kl_resident": ROW_SOURCES, "ce_kl_fused": ROW_SOURCES, "ce_kl_fused_bf16": ROW_SOURCES,
                  "kl_sliced_stream": ROW_SOURCES, "topk_k256": TOPK_SOURCES, "topk_k2048": TOPK_SOURCES}


def kernel_traffic(kernel_tag: str):
    """DRAM bytes per launch from the committed ncu summary, if the kernel's sources still match."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p) or kernel_tag not in KERNEL_SOURCES:
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get("kernels", {}).get(kernel_tag)
    if e is None or e.get("sources_sha256") != sources_hash(KERNEL_SOURCES[kernel_tag]):
        return None
    return e.get("dram_bytes_per_launch")


def sources_hash(names) -> str:
    h = hashlib.sha256()
    d = os.path.join(ROOT, "top_kl_distill_gb300", "csrc")
    for f in sorted(names):
        with open(os.path.join(d, f), "rb") as fh:
            h.update(f.encode() + b"\0" + fh.read())
    return h.hexdigest()


def roofline(case, kernel_ms, peak, peak_kind, tag):
    achieved = case.kernel_bytes() / (kernel_ms * 1e-3) / 1e9
    return {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4), "peak_source": peak_kind,
            "traffic": kernel_traffic(tag), "kernel": tag,
            "algorithmic_bytes_per_launch": case.kernel_bytes()}


KERNEL_TAG = {"ce_lm": "ce_fused", "ce_tiny": "ce_fused_tiny", "kl": "kl_resident", "large_v": "ce_kl_fused",
              "large_v_sliced": "kl_sliced_stream", "ce_lm_bf16": "ce_fused_bf16", "large_v_bf16": "ce_kl_fused_bf16"}


# ------------------------------------------------------------------ CPU oracle baseline
#
# The oracle, as it stands (float64 numpy, one row at a time), timed on the host's
# cores: once in this process on one core, and on all cores with the rows split into
# contiguous slices, one spawned worker process per slice (spawned, never forked: a
# fork after the CUDA context exists can hang).  Inputs are drawn in the workers
# before the clock starts; only the oracle calls are timed.

def _oracle_inputs(name, r0, r1):
    w = base_workload(name)
    k = int(name.split("_k")[1]) if "_k" in name else w.k
    x = W.logits(w, r0, r1, threads=1)
    lab = W.labels(w, r0, r1)
    tid, tp = W.teacher(w, r0, r1) if w.k else (None, None)
    return w, k, x, lab, tid, tp


def _oracle_run(inp):
    from oracle import vloss_oracle as O
    w, k, x, lab, tid, tp = inp
    n = x.shape[0]
    if w.kind == "ce":
        ls, le = 0, n
        O.ce_fused(x, lab, ls, le, w.scale)
    elif w.kind == "kl":
        O.kl_topk(x, tid, tp, w.coef)
    elif w.kind == "topk":
        O.topk_rows(x, k)
    else:
        _, lse = O.ce_forward(x, lab, 0, n)
        for c0, width in cuts_for_slices(w.V, w.slices):
            O.kl_topk(x, tid, tp, w.coef, lse=lse, col0=c0, ncols=width, labels=lab, ce_coef=w.ce_coef)


_WORKER_INPUTS = {}


def _oracle_task(name, r0, r1, passes, barrier=None):
    """In a worker: the oracle over rows [r0, r1), `passes` times; returns (rows, t0, t1)."""
    key = (name, r0, r1)
    if key not in _WORKER_INPUTS:
        _WORKER_INPUTS.clear()
        _WORKER_INPUTS[key] = _oracle_inputs(name, r0, r1)
    inp = _WORKER_INPUTS[key]
    if barrier is not None:
        barrier.wait()
    t0 = time.time()
    for _ in range(passes):
        _oracle_run(inp)
    return (r1 - r0) * passes, t0, time.time()


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_one_core(name, budget_s=2.0):
    """Rows per second of the oracle on one core, over a bounded sample of the rows."""
    w = base_workload(name)
    chunk, r, n, spent = 8, 0, 0, 0.0
    while spent < budget_s and n < w.ntok:
        r1 = min(w.ntok, r + chunk)
        inp = _oracle_inputs(name, r, r1)
        t0 = time.perf_counter()
        _oracle_run(inp)
        spent += time.perf_counter() - t0
        n += r1 - r
        r = r1
    return n / max(1e-9, spent), n, spent


class OraclePool:
    """One spawned worker per host core, each always given the same row slice, so that
    its inputs are drawn once."""

    def __init__(self, cores=None):
        import concurrent.futures as cf
        import multiprocessing as mp
        self.cores = cores or host_cores()
        ctx = mp.get_context("spawn")
        self.ex = [cf.ProcessPoolExecutor(max_workers=1, mp_context=ctx) for _ in range(self.cores)]
        self.mgr = ctx.Manager()

    def slices(self, nrows):
        n = min(nrows, self.cores)
        return [(i * nrows // n, (i + 1) * nrows // n) for i in range(n)]

    def timed(self, name, nrows, passes):
        """All slices of rows [0, nrows), `passes` times each, started together; returns
        (rows done, wall seconds from the common start to the last finish)."""
        sl = self.slices(nrows)
        bar = self.mgr.Barrier(len(sl))
        futs = [self.ex[i].submit(_oracle_task, name, r0, r1, passes, bar) for i, (r0, r1) in enumerate(sl)]
        res = [f.result() for f in futs]
        rows = sum(r[0] for r in res)
        return rows, max(r[2] for r in res) - min(r[1] for r in res)

    def step(self, name, nrows):
        """One pass over rows [0, nrows) split over the workers; wall seconds of the call."""
        sl = self.slices(nrows)
        t0 = time.perf_counter()
        futs = [self.ex[i].submit(_oracle_task, name, r0, r1, 1) for i, (r0, r1) in enumerate(sl)]
        for f in futs:
            f.result()
        return time.perf_counter() - t0

    def close(self):
        for e in self.ex:
            e.shutdown(wait=True)
        self.mgr.shutdown()


def oracle_baseline(name, pool, work_s=1.5):
    """cpu_baseline: the oracle on all host cores (about work_s seconds of work a core)
    plus the one-core figure it is sized from."""
    w = base_workload(name)
    r1, n1, s1 = oracle_one_core(name)
    per_core = max(1, int(r1 * work_s))
    want = per_core * pool.cores
    nrows = min(w.ntok, want)
    passes = max(1, round(want / nrows)) if nrows == w.ntok else 1
    rows, wall = pool.timed(name, nrows, passes)
    sample = (f"{passes} passes over all {w.ntok} rows" if nrows == w.ntok else f"rows 0-{nrows - 1} of {w.ntok}")
    return {"value": round(rows / max(1e-9, wall), 2), "unit": UNIT, "cores": min(pool.cores, nrows), "kind": "oracle",
            "sample": f"{sample}, float64 numpy, one spawned process per core, {wall:.1f} s wall "
                      f"(input generation excluded)",
            "one_core": {"value": round(r1, 2), "unit": UNIT, "cores": 1,
                         "sample": f"{n1} rows, {s1:.1f} s on one core"}}


# ------------------------------------------------------------------ main


def dist_setup():
    return world()


def barrier_max(torch, ws, value: float) -> float:
    return max_over_ranks(value, "cuda") if ws > 1 else value


def run_reference(args, ws, rank):
    """The reference arm: the CPU oracle, as it stands, on all host cores; one step is
    one pass over the whole batch of the workload, its rows split over the cores."""
    if rank != 0:
        return
    name = args.workload
    w = base_workload(name)
    pool = OraclePool()
    try:
        for _ in range(args.warmup):               # workers draw their inputs here
            pool.step(name, w.ntok)
        total = 0.0
        for _ in range(args.steps):
            total += pool.step(name, w.ntok)
    finally:
        pool.close()
    v = w.ntok * args.steps / total
    cores = min(pool.cores, w.ntok)
    line = {
        "impl": "reference", "metric": METRIC, "value": round(v, 2), "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * total / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded numpy)",
        "config": {"workload": workload_desc(w), "step": f"all {w.ntok} rows, split over {cores} host cores"},
        "cpu_baseline": {"value": round(v, 2), "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"{args.steps} passes over the {w.ntok}-row batch, one spawned process per core"},
        "e2e": {"value": round(v, 2), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def workload_desc(w):
    if w.kind == "ce":
        return (f"{w.name}: fused CE, {w.ntok} x {w.V} fp32 logits, window [{w.loss_start}, {w.loss_end}), "
                f"scale 1/{round(1 / w.scale)}")
    return w.name


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--workload", default="ce_lm")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--sweep-steps", type=int, default=20)
    ap.add_argument("--sweep-only", default="", help="comma-separated sweep workloads (default: all)")
    ap.add_argument("--ntok", type=int, default=0, help="rows of a scaled-down workload (profiling only)")
    ap.add_argument("--bufs", type=int, default=0, help="work buffers per timing round (profiling only)")
    ap.add_argument("--no-oracle", action="store_true", help="skip the CPU baseline and the e2e leg")
    ap.add_argument("--shard", action="store_true",
                    help="split the fused CE batch into row shards over the N ranks (strong scaling) "
                         "instead of a batch per rank")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    ws, rank, local = dist_setup()

    if args.impl == "reference":
        run_reference(args, ws, rank)
        return

    import torch
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(local)
    from top_kl_distill_gb300 import vloss as vl
    vl.lib()                                  # fails loudly if the library is not built
    peak, peak_kind = peaks()
    flush_buf = torch.empty(L2_FLUSH_BYTES // 4, device="cuda")

    def flush():
        flush_buf.fill_(1.0)

    shard = args.shard and base_workload(args.workload).kind == "ce" and not args.workload.endswith("_bf16")
    if shard:
        w0 = base_workload(args.workload)
        w0 = w0.scaled(args.ntok) if args.ntok else w0
        case = CeFusedShard(torch, w0, args.bufs or nbuf_for(w0.ntok * w0.V * 4 // ws), rank, ws)
    else:
        case = make_case(torch, args.workload, args.ntok or None, args.bufs or None)
    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    time.sleep(0.3)
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    total_ms, per = time_case(torch, case, args.steps, args.warmup, flush)
    t_wall1 = time.time()
    total_ms = barrier_max(torch, ws, total_ms)
    k_ms_total, k_per = time_case(torch, case, args.steps, 2, flush, kernel_only=True)
    # nvidia-smi samples every 100 ms: a short timed region sees none, so the same step keeps
    # the GPU loaded (untimed rounds) until the sampled window spans CLOCK_WINDOW_S
    soak_rounds = soak(torch, case, flush, t_wall0 + CLOCK_WINDOW_S)
    t_wall2 = time.time()
    sampler.stop()
    clocks = sampler.summary(t_wall0, t_wall2)
    clocks["window_s"] = round(t_wall2 - t_wall0, 3)
    clocks["window"] = ("timed steps" if soak_rounds == 0 else
                        f"timed steps and {soak_rounds} further untimed rounds of the same step")

    ms_step = total_ms / args.steps
    rows_all = case.batch.ntok if shard else case.rows() * ws
    value = rows_all / (ms_step * 1e-3)
    kernel_ms = k_ms_total / args.steps
    e2e_ms, h2d, d2h, e2e_ok = (None, 0, 0, None)
    if isinstance(case, CeFused) and not shard and not args.no_oracle:
        e2e_ms, h2d, d2h, e2e_ok = e2e_ce(torch, case, max(30, args.steps), 3)

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": True,
        "scaling": "strong" if shard else "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded numpy, uploaded once)",
        "config": {"workload": workload_desc(case.w), "ntok": case.w.ntok, "V": case.w.V,
                   "parallelism": (f"row shards x{ws}, one all-reduce of the window mean a step" if shard
                                   else f"replicas x{ws}" if ws > 1 else "single GPU"),
                   "l2": "fresh input copy per step; a 512 MB write flushes L2 before each group of timed steps",
                   "work_buffers": len(case.bufs)},
        "hbm_gbs_step": round(case.bytes_per_step() / (ms_step * 1e-3) / 1e9, 1),
        "roofline": roofline(case, kernel_ms, peak, peak_kind, KERNEL_TAG.get(case.w.name, case.w.name)),
        "clocks": clocks,
        "gpu_launches": case.launches_per_step * args.steps,
    }
    if e2e_ms is not None:
        line["e2e"] = {"value": round(case.rows() * ws / (e2e_ms * 1e-3), 1), "unit": UNIT,
                       "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4),
                       "pipeline": "copy-in, compute and copy-out streams, 2 row chunks a step (one chunk's "
                                   "D2H overlaps the next one's H2D and vl_ce_fused); then vl_window_mean and "
                                   "D2H of loss, lse and mean; steps alternate between two device buffer sets, "
                                   "so a step's uploads overlap the previous step's downloads",
                       "host_gradient_matches_device": e2e_ok}
    pool = OraclePool() if rank == 0 and not args.no_oracle else None
    if pool is not None:
        line["cpu_baseline"] = oracle_baseline(args.workload, pool)
    del case
    torch.cuda.empty_cache()

    if not args.no_sweep:
        sweep = {}
        names = ["ce_tiny", "ce_lm_bf16", "kl", "topk_k256", "topk_k2048", "large_v", "large_v_bf16",
                 "large_v_sliced"]
        if args.sweep_only:
            names = [n for n in args.sweep_only.split(",") if n and n not in ("head_gemm", "head")]
        for name in names:
            c = make_case(torch, name, args.ntok or None, args.bufs or None)
            steps = args.sweep_steps
            tot, _ = time_case(torch, c, steps, 3, flush)
            ktot, _ = time_case(torch, c, steps, 2, flush, kernel_only=True)
            ms = barrier_max(torch, ws, tot) / steps
            entry = {
                "rows_per_s": round(c.rows() * ws / (ms * 1e-3), 1), "ms_per_step": round(ms, 4),
                "hbm_gbs_step": round(c.bytes_per_step() / (ms * 1e-3) / 1e9, 1),
                "algorithmic_bytes_per_step": c.bytes_per_step(), "steps": steps,
                "roofline": roofline(c, ktot / steps, peak, peak_kind, KERNEL_TAG.get(c.name, c.name)),
                "gpu_launches": c.launches_per_step * steps,
            }
            if pool is not None:
                entry["cpu_baseline"] = oracle_baseline(name, pool, work_s=0.5)
            sweep[name] = entry
            del c
            torch.cuda.empty_cache()
        if not args.sweep_only or "head_gemm" in args.sweep_only.split(","):
            sweep["head_gemm"] = head_gemm_line(torch, flush)
        if not args.sweep_only or "head" in args.sweep_only.split(","):
            sweep.update(head_pipeline_lines(torch, flush))
        line["sweep"] = sweep

    if pool is not None:
        pool.close()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
