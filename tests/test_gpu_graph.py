"""The C-ABI calls capture into a CUDA graph: the replayed step matches the oracle."""
import numpy as np
import pytest

from oracle import vloss_oracle as O
from tests import gpu_harness as H
from top_kl_distill_gb300 import workloads as W
from top_kl_distill_gb300.slicing import cuts_for_slices

pytestmark = pytest.mark.gpu


def test_ce_fused_in_a_graph():
    torch = H.torch_cuda()
    from top_kl_distill_gb300 import vloss as vl
    w = W.WORKLOADS["ce_lm"].scaled(64)
    w = W.Workload(**{**w.__dict__, "window": (8, 64)})
    x, lab = W.logits(w), W.labels(w)
    pristine = H.dev(x)
    xt = pristine.clone()
    labels = H.dev(lab)
    loss = torch.zeros(w.ntok, device="cuda")
    lse = torch.zeros(w.ntok, device="cuda")
    mean = torch.zeros(1, device="cuda")

    def step():
        vl.vl_ce_fused(xt, w.V, w.ntok, w.V, labels, w.loss_start, w.loss_end, w.scale, loss, lse, None, mean, None)

    step()                                    # eager first: attributes and caches set outside capture
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for _ in range(2):
        xt.copy_(pristine)
        loss.zero_()
        mean.zero_()
        g.replay()
    torch.cuda.synchronize()
    oloss, olse, og, omean = O.ce_fused(x, lab, w.loss_start, w.loss_end, w.scale)
    H.check_grad(H.host(xt), og, w.scale)
    H.check_loss(H.host(loss), oloss, olse)
    H.check_mean(H.host(mean)[0], omean)


def test_large_vocab_step_in_a_graph():
    torch = H.torch_cuda()
    from top_kl_distill_gb300 import vloss as vl
    w = W.WORKLOADS["large_v"].scaled(8)
    x, lab = W.logits(w), W.labels(w)
    tid, tp = W.teacher(w)
    pristine = H.dev(x)
    xt = pristine.clone()
    labels, tidd, tpd = H.dev(lab), H.dev(tid), H.dev(tp)
    n = w.ntok
    ce = torch.zeros(n, device="cuda")
    stats = torch.zeros((n, 2), device="cuda")
    parts = [torch.zeros(n, device="cuda") for _ in range(w.slices)]
    cuts = cuts_for_slices(w.V, w.slices)

    def step():
        vl.vl_ce_fwd(xt, w.V, n, w.V, labels, 0, n, ce, None, stats, None, None)
        for (c0, width), part in zip(cuts, parts):
            vl.vl_kl_topk_inplace(xt, w.V, n, w.V, c0, width, tidd, tpd, w.k, w.coef, 0, n, None, stats,
                                  labels, w.ce_coef, part, None)
        vl.vl_acc_add(parts[0], parts[1], n)

    step()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    xt.copy_(pristine)
    g.replay()
    torch.cuda.synchronize()
    o_ce, o_lse = O.ce_forward(x, lab, 0, n)
    o_kl, og = O.kl_topk(x, tid, tp, w.coef, labels=lab, ce_coef=w.ce_coef)
    H.check_loss(H.host(ce), o_ce, o_lse, "CE")
    H.check_grad(H.host(xt), og, w.coef + w.ce_coef)
    H.check_loss(H.host(parts[0]), o_kl, o_lse, "KL")
