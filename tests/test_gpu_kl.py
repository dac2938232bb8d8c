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
