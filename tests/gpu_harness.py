"""Shared helpers of the GPU parity tests: device buffers and the tolerances.

Tolerances (fp32 CUDA path against the float64 oracle):

* gradients: |dg| <= 1e-6 * c, with c the coefficient of the softmax term
  (scale for CE, coef + ce_coef for KL).  The kernels compute
  p = 2^(((s - m) - lnS) * log2 e); for large p the exponent is small and
  exact to a few ulp, so the relative error of p stays near 3e-7.
* per-row losses: |dl| <= 1e-5 * |l|, the stated bar.  Only rows whose loss is
  far below their lse (|l| < 0.01 |lse|) get a floor of 4 ulp(lse) on top: a
  loss is lse - s[label] (or a p-weighted sum of such terms), and lse carries a
  rounding error of about an ulp of itself whatever the size of the loss.
* lse: |d| <= 2 ulp(lse) + 64 * 2^-24 (same argument).
* mean: |d| <= 1e-6 * |mean| + 1e-7.
* top-k probabilities: |dp| <= 1e-5 * p + 1e-12; ids bit-exact.
"""
from __future__ import annotations

import numpy as np
import pytest

EPS = 2.0 ** -24


def torch_cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.fail("CUDA is not available but a GPU test was selected")
    return torch


def dev(x, torch=None, offset: int = 0):
    """Device copy of a numpy array; with offset > 0 the data starts `offset`
    elements into a larger allocation (a misaligned base pointer)."""
    torch = torch or torch_cuda()
    x = np.ascontiguousarray(x)
    if x.dtype == np.uint32:
        t = torch.from_numpy(x.view(np.int32)).cuda().view(torch.uint32) if offset == 0 else None
        if t is None:
            flat = torch.zeros(x.size + offset, dtype=torch.int32, device="cuda")
            flat[offset:] = torch.from_numpy(x.view(np.int32).ravel()).cuda()
            t = flat[offset:].view(x.shape).view(torch.uint32)
        return t
    if offset == 0:
        return torch.from_numpy(x).cuda()
    flat = torch.zeros(x.size + offset, dtype=torch.from_numpy(x[:0]).dtype, device="cuda")
    flat[offset:] = torch.from_numpy(x.ravel()).cuda()
    return flat[offset:].view(x.shape)


def strided(x: np.ndarray, ld: int, offset: int = 0, torch=None):
    """[n][V] logits placed in rows of stride ld (>= V), starting `offset` floats in."""
    torch = torch or torch_cuda()
    n, V = x.shape
    buf = torch.full((offset + n * ld + 8,), float("nan"), dtype=torch.float32, device="cuda")
    view = buf[offset:offset + n * ld].view(n, ld)
    view[:, :V] = torch.from_numpy(np.ascontiguousarray(x)).cuda()
    return buf, view


def host(t) -> np.ndarray:
    import torch
    if t.dtype == torch.uint32:
        return t.view(torch.int32).cpu().numpy().view(np.uint32)
    return t.detach().cpu().numpy()


def ulp(x):
    return np.spacing(np.abs(np.asarray(x, dtype=np.float32))).astype(np.float64)


def check_grad(got, want, c, what="gradient"):
    got = np.asarray(got, dtype=np.float64)
    err = np.abs(got - want)
    tol = 1e-6 * abs(c)
    bad = ~(err <= tol)
    assert not bad.any(), (f"{what}: {int(bad.sum())} elements off, max err {np.nanmax(err):.3e} "
                           f"(tol {tol:.3e}) at {np.unravel_index(np.nanargmax(err), err.shape)}")
    report(what, "max |dgrad|/c", float(err.max() / abs(c)) if err.size else 0.0)


def check_loss(got, want, lse, what="loss"):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    lse = np.broadcast_to(np.asarray(lse, dtype=np.float64), want.shape)
    small = np.abs(want) < 0.01 * np.abs(lse)
    floor = np.where(small, 4 * ulp(np.maximum(np.abs(lse), 1.0)), 0.0)
    tol = 1e-5 * np.abs(want) + floor
    err = np.abs(got - want)
    bad = ~(err <= tol)
    assert not bad.any(), f"{what}: rows {np.nonzero(bad)[0][:10]} off, max err {np.nanmax(err):.3e}"
    big = ~small & (want != 0)
    report(what, "max |dloss|/|loss|", float(np.max(err[big] / np.abs(want[big]))) if big.any() else 0.0)
    report(what, "rows under the lse floor", int(small.sum()))


def check_lse(got, want, what="lse"):
    got = np.asarray(got, dtype=np.float64)
    tol = 2 * ulp(want) + 64 * EPS
    err = np.abs(got - want)
    bad = ~(err <= tol)
    assert not bad.any(), f"{what}: rows {np.nonzero(bad)[0][:10]} off, max err {np.nanmax(err):.3e}"


def check_mean(got, want):
    assert abs(float(got) - want) <= 1e-6 * abs(want) + 1e-7, f"mean {float(got)!r} vs {want!r}"


def check_probs(got, want, what="probs"):
    got = np.asarray(got, dtype=np.float64)
    err = np.abs(got - want)
    tol = 1e-5 * np.abs(want) + 1e-12
    bad = ~(err <= tol)
    assert not bad.any(), f"{what}: {int(bad.sum())} off, max err {np.nanmax(err):.3e}"
    pos = want > 0
    report(what, "max |dp|/p", float(np.max(err[pos] / want[pos])) if pos.any() else 0.0)


def report(what, quantity, value):
    """Append an observed error to the file named by VL_PARITY_LOG (when set), one JSON
    line per check, so that a GPU run can record how far inside its tolerance each
    workload lands."""
    import json
    import os
    path = os.environ.get("VL_PARITY_LOG")
    if not path:
        return
    test = os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0]
    with open(path, "a") as f:
        f.write(json.dumps({"test": test, "check": what, "quantity": quantity, "value": value}) + "\n")
