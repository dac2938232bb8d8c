"""Top-k distillation KL through the C ABI against the oracle (self-contained, sliced, CE fold)."""
import numpy as np
import pytest

from oracle import vloss_oracle as O
from tests import gpu_harness as H
from top_kl_distill_gb300 import workloads as W
from top_kl_distill_gb300.slicing import cuts_for_slices

pytestmark = pytest.mark.gpu


def _vl():
    from top_kl_distill_gb300 import vloss
    return vloss


def run_kl(x, tid, tp, coef, ls, le, ld=None, off=0, labels=None, ce_coef=0.0):
    torch = H.torch_cuda()
    vl = _vl()
    ntok, V = x.shape
    k = tid.shape[1]
    ld = ld or V
    buf, view = H.strided(x, ld, off)
    loss = torch.full((ntok,), -7.0, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    vl.vl_kl_topk_inplace(view.data_ptr(), ld, ntok, V, 0, V, H.dev(tid), H.dev(tp), k, coef, ls, le,
                          None, None, None if labels is None else H.dev(labels), ce_coef, loss, err)
    torch.cuda.synchronize()
    return buf, view, loss, err


def _lse(x):
    _, lse = O.ce_forward(x, np.zeros(x.shape[0], dtype=np.uint32), 0, x.shape[0])
    return lse


def test_kl_workload_rows():
    w = W.WORKLOADS["kl"].scaled(48)
    x = W.logits(w)
    tid, tp = W.teacher(w)
    _, view, loss, err = run_kl(x, tid, tp, w.coef, 0, w.ntok)
    oloss, og = O.kl_topk(x, tid, tp, w.coef)
    H.check_grad(H.host(view), og, w.coef)
    H.check_loss(H.host(loss), oloss, _lse(x), "KL")
    assert int(H.host(err)[0]) == 0


@pytest.mark.parametrize("ntok,V,ld,off,k,ls,le", [
    (23, 4099, 4103, 3, 37, 2, 20),        # ragged rows, misaligned base, a window
    (9, 2048, 2048, 0, 1024, 0, 9),         # the largest support
    (4, 100003, 100003, 1, 128, 0, 4),     # a cluster of CTAs per row
    (30, 13, 13, 0, 5, 0, 30),              # rows shorter than a float4 run
])
def test_kl_shapes(ntok, V, ld, off, k, ls, le):
    x = W.random_logits(ntok, V, seed=V + k, sigma=2.0)
    tid, tp = W.random_teacher(ntok, V, k, seed=V + 2 * k)
    coef = 1.0 / max(1, le - ls)
    buf, view, loss, err = run_kl(x, tid, tp, coef, ls, le, ld, off)
    oloss, og = O.kl_topk(x, tid, tp, coef, ls, le)
    g = H.host(view)
    H.check_grad(g[:, :V], og, coef)
    if ld > V:
        assert np.isnan(g[:, V:]).all()
    if off:
        assert np.isnan(H.host(buf)[:off]).all()
    H.check_loss(H.host(loss), oloss, _lse(x), "KL")


def test_kl_duplicates_zeros_and_bad_ids():
    ntok, V, k, coef = 16, 3000, 40, 0.25
    x = W.random_logits(ntok, V, seed=21, sigma=2.0)
    tid, tp = W.random_teacher(ntok, V, k, seed=22)
    tid[:, 5] = tid[:, 9]                  # a repeated id in every row
    tp[:, 11] = 0.0                        # zero teacher probability
    tid[2, 3] = V + 7                      # bad ids in two rows
    tid[9, 0] = 0xFFFFFFFF
    _, view, loss, err = run_kl(x, tid, tp, coef, 0, ntok)
    assert int(H.host(err)[0]) == 2
    keep = tid < V
    tp_o = np.where(keep, tp, 0.0)          # a bad id contributes nothing
    tid_o = np.where(keep, tid, 0).astype(np.uint32)
    oloss, og = O.kl_topk(x, tid_o, tp_o, coef)
    H.check_grad(H.host(view), og, coef)
    H.check_loss(H.host(loss), oloss, _lse(x), "KL")


def test_kl_with_ce_fold_self_contained():
    ntok, V, k, coef, ce_coef = 12, 5000, 64, 0.5, 0.25
    x = W.random_logits(ntok, V, seed=31, sigma=2.0)
    tid, tp = W.random_teacher(ntok, V, k, seed=32)
    lab = W.random_labels(ntok, V, seed=33)
    _, view, loss, err = run_kl(x, tid, tp, coef, 1, 11, labels=lab, ce_coef=ce_coef)
    oloss, og = O.kl_topk(x, tid, tp, coef, 1, 11, labels=lab, ce_coef=ce_coef)
    H.check_grad(H.host(view), og, coef + ce_coef)
    H.check_loss(H.host(loss), oloss, _lse(x), "KL")


def test_kl_many_rows_a_cta():
    """Rows of four tiles and more, more rows than SMs: the self-contained KL runs without a
    CTA barrier per row (partials and pass-B completion on mbarriers, one warp in turn
    combining).  Repeated ids, zero probabilities, bad ids and folded labels, misaligned."""
    ntok, V, ld, off, k = 400, 32003, 32009, 1, 64
    x = W.random_logits(ntok, V, seed=41, sigma=2.5)
    tid, tp = W.random_teacher(ntok, V, k, seed=42)
    lab = W.random_labels(ntok, V, seed=43)
    tid[:, 5] = tid[:, 9]
    tid[:, 6] = lab
    tp[:, 11] = 0.0
    tid[7, 3] = V + 1
    tid[250, 0] = 0xFFFFFFFF
    coef, ce_coef = 1.0 / ntok, 0.5 / ntok
    buf, view, loss, err = run_kl(x, tid, tp, coef, 0, ntok, ld, off, labels=lab, ce_coef=ce_coef)
    assert int(H.host(err)[0]) == 2
    keep = tid < V
    tp_o = np.where(keep, tp, 0.0)
    tid_o = np.where(keep, tid, 0).astype(np.uint32)
    oloss, og = O.kl_topk(x, tid_o, tp_o, coef, labels=lab, ce_coef=ce_coef)
    g = H.host(view)
    H.check_grad(g[:, :V], og, coef + ce_coef)
    assert np.isnan(g[:, V:]).all()
    assert np.isnan(H.host(buf)[:off]).all()
    H.check_loss(H.host(loss), oloss, _lse(x), "KL")


@pytest.mark.parametrize("use_stats", [True, False])
def test_large_vocab_sliced_step(use_stats):
    """The large-vocabulary step at 16 rows: CE forward over full rows, then per vocabulary
    slice the in-place KL + CE gradient from the row statistics, then acc_add of the
    slices' KL parts."""
    torch = H.torch_cuda()
    vl = _vl()
    w = W.WORKLOADS["large_v"].scaled(16)
    x, lab = W.logits(w), W.labels(w)
    tid, tp = W.teacher(w)
    ntok, V, k = w.ntok, w.V, w.k
    xt = H.dev(x)
    labels, tidd, tpd = H.dev(lab), H.dev(tid), H.dev(tp)
    ce_loss = torch.zeros(ntok, device="cuda")
    lse = torch.zeros(ntok, device="cuda")
    stats = torch.zeros(ntok, 2, device="cuda")
    vl.vl_ce_fwd(xt, V, ntok, V, labels, 0, ntok, ce_loss, lse, stats, None, None)
    parts = [torch.zeros(ntok, device="cuda") for _ in range(w.slices)]
    for (c0, width), lp in zip(cuts_for_slices(V, w.slices), parts):
        vl.vl_kl_topk_inplace(xt, V, ntok, V, c0, width, tidd, tpd, k, w.coef, 0, ntok,
                              None if use_stats else lse, stats if use_stats else None,
                              labels, w.ce_coef, lp, None)
    for lp in parts[1:]:
        vl.vl_acc_add(parts[0], lp, ntok)
    torch.cuda.synchronize()
    o_ce, o_lse = O.ce_forward(x, lab, 0, ntok)
    if use_stats:
        o_kl, og = O.kl_topk(x, tid, tp, w.coef, labels=lab, ce_coef=w.ce_coef)
    else:   # both sides take the same fp32 lse as an input
        o_kl, og = O.kl_topk(x, tid, tp, w.coef, lse=o_lse.astype(np.float32).astype(np.float64),
                             labels=lab, ce_coef=w.ce_coef)
    H.check_loss(H.host(ce_loss), o_ce, o_lse, "CE")
    H.check_lse(H.host(lse), o_lse)
    H.check_grad(H.host(xt), og, w.coef + w.ce_coef)
    H.check_loss(H.host(parts[0]), o_kl, o_lse, "KL summed over slices")


def run_ce_kl(x, lab, tid, tp, coef, ce_coef, ls, le, ld=None, off=0):
    torch = H.torch_cuda()
    vl = _vl()
    ntok, V = x.shape
    k = tid.shape[1]
    ld = ld or V
    buf, view = H.strided(x, ld, off)
    kl = torch.full((ntok,), -7.0, device="cuda")
    ce = torch.full((ntok,), -7.0, device="cuda")
    lse = torch.full((ntok,), -7.0, device="cuda")
    stats = torch.full((ntok, 2), -7.0, device="cuda")
    mean = torch.full((1,), -7.0, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    vl.vl_ce_kl_fused(view.data_ptr(), ld, ntok, V, H.dev(lab), H.dev(tid), H.dev(tp), k, coef, ce_coef, ls, le,
                      kl, ce, lse, stats, mean, err)
    torch.cuda.synchronize()
    return buf, view, kl, ce, lse, stats, mean, err


def check_ce_kl(x, lab, tid, tp, coef, ce_coef, ls, le, ld=None, off=0, what="CE+KL"):
    ntok, V = x.shape
    buf, view, kl, ce, lse, stats, mean, err = run_ce_kl(x, lab, tid, tp, coef, ce_coef, ls, le, ld, off)
    o_kl, og = O.kl_topk(x, tid, tp, coef, ls, le, labels=lab, ce_coef=ce_coef)
    o_ce, o_lse = O.ce_forward(x, lab, ls, le)
    g = H.host(view)
    H.check_grad(g[:, :V], og, coef + ce_coef, f"{what} gradient")
    if ld and ld > V:
        assert np.isnan(g[:, V:]).all(), "columns past V were written"
    if off:
        assert np.isnan(H.host(buf)[:off]).all(), "memory before the first row was written"
    H.check_loss(H.host(kl), o_kl, o_lse, f"{what} KL")
    H.check_loss(H.host(ce), o_ce, o_lse, f"{what} CE")
    win = slice(ls, le)
    H.check_lse(H.host(lse)[win], o_lse[win], f"{what} lse")
    assert np.all(H.host(lse)[:ls] == -7.0) and np.all(H.host(lse)[le:] == -7.0), "lse outside the window written"
    st = H.host(stats)[win]
    assert np.array_equal(st[:, 0], x[win].max(axis=1))
    H.check_mean(H.host(mean)[0], O.ce_mean(o_ce, ls, le))
    return int(H.host(err)[0])


def test_ce_kl_fused_large_vocab_rows():
    """The large-vocabulary workload's rows (128256 columns: a row per 4-CTA cluster)."""
    w = W.WORKLOADS["large_v"].scaled(24)
    x, lab = W.logits(w), W.labels(w)
    tid, tp = W.teacher(w)
    assert check_ce_kl(x, lab, tid, tp, w.coef, w.ce_coef, 0, w.ntok) == 0


@pytest.mark.parametrize("ntok,V,ld,off,k,ls,le", [
    (9, 100003, 100007, 3, 128, 2, 8),     # clusters, ragged rows, misaligned base, a window
    (23, 4099, 4103, 1, 37, 2, 20),        # one CTA per row
    (6, 2048, 2048, 0, 1024, 0, 6),        # the largest support
    (30, 13, 13, 0, 5, 0, 30),             # rows shorter than a float4 run
    (3, 300007, 300007, 2, 64, 0, 3),      # rows past 8 CTAs of tiles
])
def test_ce_kl_fused_shapes(ntok, V, ld, off, k, ls, le):
    x = W.random_logits(ntok, V, seed=V + k + 1, sigma=2.5)
    lab = W.random_labels(ntok, V, seed=V + 3)
    tid, tp = W.random_teacher(ntok, V, k, seed=V + 5)
    coef, ce_coef = 1.0 / max(1, le - ls), 0.5 / max(1, le - ls)
    assert check_ce_kl(x, lab, tid, tp, coef, ce_coef, ls, le, ld, off) == 0


def test_ce_kl_fused_duplicates_zeros_bad_ids_and_labels():
    ntok, V, k = 12, 140000, 40
    x = W.random_logits(ntok, V, seed=81, sigma=2.0)
    lab = W.random_labels(ntok, V, seed=82)
    tid, tp = W.random_teacher(ntok, V, k, seed=83)
    tid[:, 5] = tid[:, 9]                  # a repeated id in every row
    tp[:, 11] = 0.0                        # zero teacher probability
    tid[2, 3] = V + 7                      # a bad id
    lab[4] = V                             # a bad label
    buf, view, kl, ce, lse, stats, mean, err = run_ce_kl(x, lab, tid, tp, 0.25, 0.125, 0, ntok)
    assert int(H.host(err)[0]) == 2
    assert np.isnan(H.host(ce)[4])
    keep = tid < V
    tp_o = np.where(keep, tp, 0.0)
    tid_o = np.where(keep, tid, 0).astype(np.uint32)
    lab_o = np.where(lab < V, lab, 0).astype(np.uint32)
    o_kl, og = O.kl_topk(x, tid_o, tp_o, 0.25, labels=lab_o, ce_coef=0.125)
    o_ce, o_lse = O.ce_forward(x, lab_o, 0, ntok)
    ok = np.setdiff1d(np.arange(ntok), [4])
    g = H.host(view)
    H.check_grad(g[ok], og[ok], 0.375)
    # a bad label leaves the softmax and teacher parts of the gradient
    o_kl4, og4 = O.kl_topk(x[4:5], tid_o[4:5], tp_o[4:5], 0.25)
    H.check_grad(g[4:5], og4 + 0.125 * np.exp(x[4:5].astype(np.float64) - o_lse[4]), 0.375)
    H.check_loss(H.host(kl), o_kl, o_lse, "KL")
    H.check_loss(H.host(ce)[ok], o_ce[ok], o_lse[ok], "CE")
