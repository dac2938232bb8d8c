"""The vocabulary head pipelines through the C ABI against the oracle.

hidden and w are bf16 draws; the oracle takes their exact values and forms the logits
in float64, then applies its loss, gradient and top-k definitions.  The GPU forms the
logits with fp32 accumulation, so every logit may differ from the exact one by the
dot-product bound eps[r][n] = hs * 2^-24 * sum_k |h[r][k] w[n][k]|; the checks allow
exactly what that error, the stated loss/gradient tolerances and the bf16 rounding of
the gradient (2^-8 relative) can produce.
"""
import numpy as np
import pytest

from oracle import vloss_oracle as O
from tests import gpu_harness as H
from top_kl_distill_gb300 import workloads as W

pytestmark = pytest.mark.gpu

U24 = 2.0 ** -24


def bf16_bits(x):
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)


def bf16_value(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32)


def head_inputs(ntok, hs, V, seed):
    g = np.random.default_rng(seed)
    h = bf16_bits(g.standard_normal((ntok, hs)).astype(np.float32))
    w = bf16_bits((g.standard_normal((V, hs)) * (3.0 / np.sqrt(hs))).astype(np.float32))
    H64, W64 = bf16_value(h).astype(np.float64), bf16_value(w).astype(np.float64)
    L = H64 @ W64.T
    eps = hs * U24 * (np.abs(H64) @ np.abs(W64).T) * 1.01
    return h, w, H64, W64, L, eps


def dev_bf16(bits):
    torch = H.torch_cuda()
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def _vl():
    from top_kl_distill_gb300 import vloss
    return vloss


@pytest.mark.parametrize("ws_rows", [0, 7])
def test_teacher_topk_pipeline(ws_rows):
    """Rows [3, 37) of 40, V = 32000 (the streaming select), k = 64; with a workspace for 7
    rows the batch goes in chunks."""
    torch = H.torch_cuda()
    vl = _vl()
    ntok, hs, V, k, ls, le = 40, 256, 32000, 64, 3, 37
    h, w, H64, W64, L, eps = head_inputs(ntok, hs, V, seed=11)
    ids = torch.full((ntok, k), -1, dtype=torch.int32, device="cuda")
    probs = torch.full((ntok, k), -1.0, device="cuda")
    ws = "auto"
    if ws_rows:
        ws = torch.empty(vl.lib().vl_teacher_topk_workspace_bytes(ws_rows, V, k), dtype=torch.uint8, device="cuda")
    vl.vl_teacher_topk(dev_bf16(h), hs, dev_bf16(w), V, ntok, k, ls, le, ids, probs, None, ws)
    torch.cuda.synchronize()
    gid = H.host(ids).view(np.uint32).astype(np.int64)
    gp = H.host(probs).astype(np.float64)
    assert np.all(gid[:ls] == 0xFFFFFFFF) and np.all(gid[le:] == 0xFFFFFFFF), "rows outside the window written"
    for r in range(ls, le):
        e = 2 * eps[r].max()
        row = L[r]
        sel = gid[r]
        assert len(set(sel.tolist())) == k and sel.max() < V
        kth = np.sort(row)[::-1][k - 1]
        rest = np.setdiff1d(np.arange(V), sel)
        assert row[sel].min() >= kth - e and row[rest].max() <= kth + e, f"row {r}: not the top {k}"
        assert np.all(row[sel][1:] <= row[sel][:-1] + e), f"row {r}: not in descending order"
        v = row[sel]
        want = np.exp(v - v[0]) / np.exp(v - v[0]).sum()
        assert np.all(np.abs(gp[r] - want) <= (1e-5 + 4 * e) * want + 1e-12), f"row {r}: probabilities"


@pytest.mark.parametrize("ws_rows,with_wt", [(0, True), (5, True), (0, False)])
def test_head_kl_pipeline(ws_rows, with_wt):
    """The student's head step; with the transposed weight plane both GEMMs run on the
    tensor-core kernel, without it the dx GEMM goes through cuBLASLt."""
    torch = H.torch_cuda()
    vl = _vl()
    ntok, hs, V, k, ls, le = 24, 256, 8000, 32, 2, 21
    h, w, H64, W64, L, eps = head_inputs(ntok, hs, V, seed=12)
    lab = W.random_labels(ntok, V, seed=13)
    tid, tp = W.random_teacher(ntok, V, k, seed=14)
    coef, ce_coef, dx_scale = 1.0 / (le - ls), 0.5 / (le - ls), 0.25
    dx = torch.full((ntok, hs), -7.0, device="cuda")
    kl = torch.full((ntok,), -7.0, device="cuda")
    ce = torch.full((ntok,), -7.0, device="cuda")
    mean = torch.full((1,), -7.0, device="cuda")
    ws = "auto"
    if ws_rows:
        ws = torch.empty(vl.lib().vl_head_kl_workspace_bytes(ws_rows, V), dtype=torch.uint8, device="cuda")
    wt = dev_bf16(np.ascontiguousarray(w.T)) if with_wt else None
    vl.vl_head_kl(dev_bf16(h), hs, dev_bf16(w), wt, V, ntok, H.dev(lab), H.dev(tid), H.dev(tp), k, coef, ce_coef,
                  dx_scale, ls, le, dx, kl, ce, mean, None, ws)
    torch.cuda.synchronize()
    o_kl, og = O.kl_topk(L, tid, tp, coef, ls, le, labels=lab, ce_coef=ce_coef)
    o_ce, o_lse = O.ce_forward(L, lab, ls, le)
    e_row = 2 * eps.max(axis=1)
    # losses: the stated bar plus the logit error (lse and each logit move by at most eps)
    for got, want, what in [(H.host(kl), o_kl, "KL"), (H.host(ce), o_ce, "CE")]:
        err = np.abs(got - want)
        assert np.all(err <= 1e-5 * np.abs(want) + e_row), f"{what}: max err {err.max():.3e}"
    H.check_mean(H.host(mean)[0], O.ce_mean(H.host(ce).astype(np.float64), ls, le))
    # dx: bf16 rounding of the gradient (2^-8 relative), the stated 1e-6 c, the gradient's
    # change under the logit error (|dp| <= p * 2 eps), the GEMM's own accumulation error
    c = coef + ce_coef
    P = np.exp(L - o_lse[:, None])
    gamma = V * U24 * 1.01
    bound = abs(dx_scale) * ((2.0 ** -8 + gamma) * np.abs(og) + 1e-6 * c + c * P * e_row[:, None]) @ np.abs(W64)
    want = dx_scale * og @ W64
    got = H.host(dx).astype(np.float64)
    err = np.abs(got - want)
    assert np.all(err <= bound), f"dx: {int((err > bound).sum())} off, worst ratio {np.max(err / bound):.3f}"
    assert np.all(got[:ls] == 0.0) and np.all(got[le:] == 0.0), "rows outside the window"
    H.report("head dx", "max |ddx| / bound", float(np.max(err / bound)))
