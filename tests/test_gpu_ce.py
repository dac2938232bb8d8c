"""Cross-entropy through the C ABI against the oracle (fused, forward, sliced backward)."""
import zlib

import numpy as np
import pytest

from oracle import vloss_oracle as O
from tests import gpu_harness as H
from top_kl_distill_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _vl():
    from top_kl_distill_gb300 import vloss
    return vloss


def run_fused(x, lab, ls, le, scale, ld=None, off=0):
    torch = H.torch_cuda()
    vl = _vl()
    ntok, V = x.shape
    ld = ld or V
    buf, view = H.strided(x, ld, off)
    labels = H.dev(lab)
    loss = torch.full((max(ntok, 1),), -7.0, device="cuda")
    lse = torch.full((max(ntok, 1),), -7.0, device="cuda")
    stats = torch.full((max(ntok, 1), 2), -7.0, device="cuda")
    mean = torch.full((1,), -7.0, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    vl.vl_ce_fused(view.data_ptr() if ntok else buf.data_ptr(), ld, ntok, V, labels, ls, le, scale, loss, lse,
                   stats, mean, err)
    torch.cuda.synchronize()
    return buf, view, loss, lse, stats, mean, err


CASES = {
    # name: (ntok, V, ld, offset, ls, le, scale, sigma)
    "tiny_workload": None,
    "ragged_misaligned": (37, 5003, 5011, 1, 3, 30, 0.25, 3.0),
    "v1": (6, 1, 1, 0, 0, 6, 1.0, 1.0),
    "v3_offset2": (9, 3, 5, 2, 1, 8, 0.5, 2.0),
    "v7": (11, 7, 7, 3, 0, 11, 1.0, 2.0),
    "v8_ld9": (10, 8, 9, 0, 2, 10, 1.0, 2.0),
    "cluster_100003": (5, 100003, 100003, 0, 0, 5, 1.0 / 5, 3.0),
    "empty_window": (12, 777, 777, 0, 5, 5, 1.0, 2.0),
    "full_window_4tiles": (40, 8192, 8192, 0, 0, 40, 1.0 / 40, 2.0),
}


@pytest.mark.parametrize("name", list(CASES))
def test_ce_fused(name):
    if name == "tiny_workload":
        w = W.WORKLOADS["ce_tiny"]
        x, lab = W.logits(w), W.labels(w)
        ls, le, scale, ld, off = w.loss_start, w.loss_end, w.scale, w.V, 0
    else:
        ntok, V, ld, off, ls, le, scale, sigma = CASES[name]
        x = W.random_logits(ntok, V, seed=zlib.crc32(name.encode()), sigma=sigma)
        lab = W.random_labels(ntok, V, seed=zlib.crc32(name.encode()) + 1)
    ntok, V = x.shape
    buf, view, loss, lse, stats, mean, err = run_fused(x, lab, ls, le, scale, ld, off)
    oloss, olse, og, omean = O.ce_fused(x, lab, ls, le, scale)
    g = H.host(view)
    H.check_grad(g[:, :V], og, scale)
    if ld > V:
        assert np.isnan(g[:, V:]).all(), "columns past V were written"
    if off:
        assert np.isnan(H.host(buf)[:off]).all(), "memory before the first row was written"
    H.check_loss(H.host(loss)[:ntok], oloss, olse)
    H.check_lse(H.host(lse)[:ntok], olse)
    st = H.host(stats)[:ntok]
    assert np.array_equal(st[:, 0], x.max(axis=1)), "stats[:, 0] is the exact row max"
    H.check_lse(st[:, 0].astype(np.float64) + st[:, 1], olse, "m + lnS")
    H.check_mean(H.host(mean)[0], omean)
    assert int(H.host(err)[0]) == 0


# Past two rows a pair of SMs the fused CE runs on 2-CTA clusters: each CTA takes whole rows
# of its cluster's block, and an odd block's last row is split over the pair.  Bad labels
# sit on rows of both kinds (row 5 is split when the device holds 76 such clusters).
@pytest.mark.parametrize("ntok,V,ld,off,ls,le", [
    (160, 5003, 5011, 1, 3, 150),     # misaligned rows: every row its own head and tail
    (311, 4096, 4096, 0, 0, 311),     # aligned rows, 5 or 4 a cluster
    (200, 33, 37, 2, 10, 190),        # rows of a few chunks
])
def test_ce_fused_pairs(ntok, V, ld, off, ls, le):
    scale = 1.0 / (le - ls)
    x = W.random_logits(ntok, V, seed=ntok * 7 + V, sigma=3.0)
    lab = W.random_labels(ntok, V, seed=ntok * 7 + V + 1)
    bad = [5, 12, ntok - 2]
    lab[bad] = [V, V + 7, 0xFFFFFFFF]
    buf, view, loss, lse, stats, mean, err = run_fused(x, lab, ls, le, scale, ld, off)
    inwin = [t for t in bad if ls <= t < le]
    assert int(H.host(err)[0]) == len(inwin)
    fixed = np.where(lab < V, lab, 0).astype(np.uint32)
    oloss, olse, og, _ = O.ce_fused(x, fixed, ls, le, scale)
    ok = np.setdiff1d(np.arange(ntok), inwin)
    l = H.host(loss)
    H.check_loss(l[ok], oloss[ok], olse[ok])
    assert all(np.isnan(l[t]) for t in inwin)
    H.check_lse(H.host(lse), olse)
    st = H.host(stats)
    assert np.array_equal(st[:, 0], x.max(axis=1)), "stats[:, 0] is the exact row max"
    g = H.host(view)
    H.check_grad(g[ok, :V], og[ok], scale)
    for t in inwin:      # a bad label leaves the softmax part of the gradient
        H.check_grad(g[t, :V], scale * np.exp(x[t].astype(np.float64) - olse[t]), scale)
    if ld > V:
        assert np.isnan(g[:, V:]).all(), "columns past V were written"
    if off:
        assert np.isnan(H.host(buf)[:off]).all(), "memory before the first row was written"


def test_ce_lm_peaky_rows():
    w = W.WORKLOADS["ce_lm"].scaled(96)
    w = W.Workload(**{**w.__dict__, "window": (16, 96)})
    x, lab = W.logits(w), W.labels(w)
    _, view, loss, lse, _, mean, err = run_fused(x, lab, w.loss_start, w.loss_end, w.scale)
    oloss, olse, og, omean = O.ce_fused(x, lab, w.loss_start, w.loss_end, w.scale)
    H.check_grad(H.host(view), og, w.scale)
    H.check_loss(H.host(loss), oloss, olse)
    H.check_mean(H.host(mean)[0], omean)


def test_ce_zero_rows():
    torch = H.torch_cuda()
    vl = _vl()
    mean = torch.full((1,), 5.0, device="cuda")
    vl.vl_ce_fused(0, 10, 0, 10, 0, 0, 0, 1.0, 0, None, None, mean, None)
    torch.cuda.synchronize()
    assert float(mean[0]) == 0.0


def test_ce_bad_labels_counted():
    ntok, V, ls, le, scale = 20, 3000, 0, 16, 0.5
    x = W.random_logits(ntok, V, seed=5)
    lab = W.random_labels(ntok, V, seed=6)
    lab[[3, 7, 17]] = [V, V + 100, 0xFFFFFFFF]      # rows 3 and 7 in the window, row 17 outside
    _, view, loss, lse, _, _, err = run_fused(x, lab, ls, le, scale)
    assert int(H.host(err)[0]) == 2
    l = H.host(loss)
    assert np.isnan(l[3]) and np.isnan(l[7]) and l[17] == 0.0
    fixed = np.where(lab < V, lab, 0).astype(np.uint32)
    oloss, olse, og, _ = O.ce_fused(x, fixed, ls, le, scale)
    ok = np.setdiff1d(np.arange(ntok), [3, 7])
    H.check_loss(l[ok], oloss[ok], olse[ok])
    g = H.host(view)
    H.check_grad(g[ok], og[ok], scale)
    for t in (3, 7):   # a bad label leaves the softmax part of the gradient
        H.check_grad(g[t], scale * np.exp(x[t].astype(np.float64) - olse[t]), scale)


def test_ce_fwd_then_sliced_bwd():
    torch = H.torch_cuda()
    vl = _vl()
    ntok, V, ld, ls, le, scale = 19, 3001, 3007, 2, 17, 1.0 / 15
    x = W.random_logits(ntok, V, seed=8, sigma=3.0)
    lab = W.random_labels(ntok, V, seed=9)
    buf, view = H.strided(x, ld, 2)
    labels = H.dev(lab)
    loss = torch.zeros(ntok, device="cuda")
    lse = torch.zeros(ntok, device="cuda")
    stats = torch.zeros(ntok, 2, device="cuda")
    mean = torch.zeros(1, device="cuda")
    vl.vl_ce_fwd(view.data_ptr(), ld, ntok, V, labels, ls, le, loss, lse, stats, mean, None)
    parts = []
    for c0, w in [(0, 1000), (1000, 517), (1517, 1484)]:
        lp = torch.full((ntok,), -1.0, device="cuda")
        vl.vl_ce_bwd_inplace(view.data_ptr(), ld, ntok, V, c0, w, labels, None, stats, ls, le, scale, lp, None)
        parts.append(lp)
    torch.cuda.synchronize()
    oloss, olse = O.ce_forward(x, lab, ls, le)
    og, _ = O.ce_backward(x, lab, olse, ls, le, scale)
    H.check_loss(H.host(loss), oloss, olse)
    H.check_lse(H.host(lse), olse)
    H.check_mean(H.host(mean)[0], O.ce_mean(oloss, ls, le))
    H.check_grad(H.host(view)[:, :V], og, scale)
    assert np.isnan(H.host(view)[:, V:]).all()
    tot = sum(H.host(p).astype(np.float64) for p in parts)
    H.check_loss(tot, oloss, olse, "sum of slice loss parts")


def test_ce_bwd_with_lse_only():
    torch = H.torch_cuda()
    vl = _vl()
    ntok, V, scale = 8, 2500, 0.125
    x = W.random_logits(ntok, V, seed=10, sigma=1.0)
    lab = W.random_labels(ntok, V, seed=11)
    _, olse = O.ce_forward(x, lab, 0, ntok)
    lse32 = olse.astype(np.float32)
    xt = H.dev(x)
    vl.vl_ce_bwd_inplace(xt, V, ntok, V, 0, V, H.dev(lab), H.dev(lse32), None, 0, ntok, scale, None, None)
    torch.cuda.synchronize()
    # the oracle given the same fp32 lse (an input of both sides)
    og, _ = O.ce_backward(x, lab, lse32.astype(np.float64), 0, ntok, scale)
    H.check_grad(H.host(xt), og, scale)


def test_ce_fused_beyond_on_chip_rows():
    """V past 8 CTAs of staged row: statistics pass + in-place pass through the stats buffer."""
    ntok, V, scale = 3, 8 * 2048 * 24 + 5, 1.0 / 3
    x = W.random_logits(ntok, V, seed=12, sigma=2.0)
    lab = W.random_labels(ntok, V, seed=13)
    _, view, loss, lse, stats, mean, err = run_fused(x, lab, 0, ntok, scale)
    oloss, olse, og, omean = O.ce_fused(x, lab, 0, ntok, scale)
    H.check_grad(H.host(view), og, scale)
    H.check_loss(H.host(loss), oloss, olse)
    H.check_mean(H.host(mean)[0], omean)


@pytest.mark.parametrize("ntok,V,ld,off", [
    (1, 4000, 4000, 0),          # one row over every SM
    (151, 3000, 3001, 1),        # one row short of a wave: ragged stride, misaligned base
    (152, 3000, 3000, 0),        # exactly one wave per SM count of a GB300 (no tail)
    (153, 2999, 3003, 3),        # one row past a wave
    (300, 1003, 1003, 2),
    (457, 7, 9, 1),              # rows shorter than a float4 run
    (512, 32000, 32000, 0),      # the LM workload's shape
])
def test_ce_fused_row_counts(ntok, V, ld, off):
    """Row counts around a wave of SMs, ragged strides and misaligned bases: every row, its
    lse, loss and gradient; two calls in a row both match."""
    seed = ntok * 7919 + V
    x = W.random_logits(ntok, V, seed=seed, sigma=3.0)
    lab = W.random_labels(ntok, V, seed=seed + 1)
    ls, le, scale = ntok // 5, ntok, 1.0 / max(1, ntok - ntok // 5)
    oloss, olse, og, omean = O.ce_fused(x, lab, ls, le, scale)
    for _ in range(2):
        buf, view, loss, lse, stats, mean, err = run_fused(x, lab, ls, le, scale, ld, off)
        g = H.host(view)
        H.check_grad(g[:, :V], og, scale, "gradient")
        if ld > V:
            assert np.isnan(g[:, V:]).all()
        if off:
            assert np.isnan(H.host(buf)[:off]).all()
        H.check_loss(H.host(loss), oloss, olse, "loss")
        H.check_lse(H.host(lse), olse, "lse")
        st = H.host(stats)
        assert np.array_equal(st[:, 0], x.max(axis=1))
        H.check_mean(H.host(mean)[0], omean)
        assert int(H.host(err)[0]) == 0


def test_ce_fused_bad_labels_counted_once_per_row():
    """A bad label in a row split over a cluster of CTAs is counted once and gives a NaN loss."""
    ntok, V = 40, 20000
    x = W.random_logits(ntok, V, seed=71)
    lab = W.random_labels(ntok, V, seed=72)
    lab[[0, 17, 39]] = [V, V + 5, 0xFFFFFFFF]
    _, view, loss, _, _, _, err = run_fused(x, lab, 0, ntok, 0.5)
    assert int(H.host(err)[0]) == 3
    l = H.host(loss)
    assert np.isnan(l[[0, 17, 39]]).all()
    ok = np.setdiff1d(np.arange(ntok), [0, 17, 39])
    oloss, olse, og, _ = O.ce_fused(x, np.where(lab < V, lab, 0).astype(np.uint32), 0, ntok, 0.5)
    H.check_loss(l[ok], oloss[ok], olse[ok])
    H.check_grad(H.host(view)[ok], og[ok], 0.5)


def test_ce_fused_long_rows_on_clusters():
    """Rows of 128256 fp32 columns: the fused CE splits each row over a cluster of CTAs, every
    warp sending its pass A partial to every rank; a window, a ragged stride, a misaligned base,
    two calls in a row."""
    ntok, V, ld, off = 41, 128256, 128263, 3
    x = W.random_logits(ntok, V, seed=777, sigma=2.0)
    lab = W.random_labels(ntok, V, seed=778)
    ls, le, scale = 5, 37, 1.0 / 32
    oloss, olse, og, omean = O.ce_fused(x, lab, ls, le, scale)
    for _ in range(2):
        buf, view, loss, lse, stats, mean, err = run_fused(x, lab, ls, le, scale, ld, off)
        g = H.host(view)
        H.check_grad(g[:, :V], og, scale, "long-row gradient")
        assert np.isnan(g[:, V:]).all()
        assert np.isnan(H.host(buf)[:off]).all()
        H.check_loss(H.host(loss), oloss, olse, "long-row loss")
        H.check_lse(H.host(lse), olse, "long-row lse")
        assert np.array_equal(H.host(stats)[:, 0], x.max(axis=1))
        H.check_mean(H.host(mean)[0], omean)
        assert int(H.host(err)[0]) == 0


@pytest.mark.parametrize("jump", [30.0, 62.0, 66.0, 89.5, 90.5, 120.0, 300.0])
def test_ce_fused_running_max_jumps(jump):
    """A value far above everything before it in its row, in a later tile: the thread that
    meets it raises its running max by about `jump` - 2 (its earlier values are N(0, 1)), so
    the pass-A sum is rescaled (a small rise) or summed again against the new max (a rise of
    64 or more, where the rescale factor would leave the normal range).  lse, loss and
    gradient against the oracle."""
    ntok, V, scale = 8, 20000, 0.125
    x = W.random_logits(ntok, V, seed=int(jump * 10), sigma=1.0)
    x[np.arange(ntok), 15000 + 7 * np.arange(ntok)] = np.float32(jump)
    lab = W.random_labels(ntok, V, seed=int(jump * 10) + 1)
    _, view, loss, lse, _, _, err = run_fused(x, lab, 0, ntok, scale)
    oloss, olse, og, _ = O.ce_fused(x, lab, 0, ntok, scale)
    H.check_grad(H.host(view), og, scale, f"gradient, jump {jump}")
    H.check_loss(H.host(loss), oloss, olse, f"loss, jump {jump}")
    H.check_lse(H.host(lse), olse, f"lse, jump {jump}")
    assert int(H.host(err)[0]) == 0
