"""bf16 logits through the C ABI against the oracle.

The inputs are fp32 draws rounded to bf16; both sides take those bf16 values (as exact
fp32 / float64 numbers).  Losses, lse and stats are fp32 and keep the fp32 tolerances.
Each gradient element is the kernel's fp32 value (within 1e-6 c of the exact one, c the
softmax coefficient) rounded once to bf16, nearest even: so it must lie between the bf16
roundings of exact - 1e-6 c and exact + 1e-6 c.
"""
import numpy as np
import pytest

from oracle import vloss_oracle as O
from tests import gpu_harness as H
from top_kl_distill_gb300 import workloads as W
from top_kl_distill_gb300.slicing import cuts_for_slices

pytestmark = pytest.mark.gpu


def bf16_bits(x):
    """Round float32 values to bf16 (nearest even) and return the 16-bit patterns."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def bf16_value(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32)


def rne_bf16(v):
    """float64 -> nearest bf16 value (through fp32; the interval below is widened by an fp32 ulp)."""
    return bf16_value(bf16_bits(np.asarray(v, dtype=np.float64).astype(np.float32))).astype(np.float64)


def check_grad_bf16(got_bits, exact, c, what="bf16 gradient"):
    got = bf16_value(got_bits).astype(np.float64)
    d = 1e-6 * abs(c) + np.spacing(np.abs(exact).astype(np.float32)).astype(np.float64)
    lo, hi = rne_bf16(exact - d), rne_bf16(exact + d)
    bad = ~((got >= lo) & (got <= hi))
    assert not bad.any(), (f"{what}: {int(bad.sum())} elements off; first at "
                           f"{np.unravel_index(np.argmax(bad), bad.shape)}: got {got[bad][0]!r}, "
                           f"exact {exact[bad][0]!r}")
    H.report(what, "max |dgrad|/(c + 2^-8 |g|)",
             float(np.max(np.abs(got - exact) / (abs(c) + 2.0 ** -8 * np.abs(exact)))) if got.size else 0.0)


def dev_bf16(bits, ld=None, off=0):
    """[n][V] bf16 rows placed in rows of stride ld, starting `off` elements in (NaN-filled gaps)."""
    torch = H.torch_cuda()
    n, V = bits.shape
    ld = ld or V
    buf = torch.full((off + n * ld + 16,), float("nan"), dtype=torch.bfloat16, device="cuda")
    view = buf[off:off + n * ld].view(n, ld)
    view[:, :V] = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)
    return buf, view


def host_bits(t):
    torch = H.torch_cuda()
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _vl():
    from top_kl_distill_gb300 import vloss
    return vloss


@pytest.mark.parametrize("ntok,V,ld,off,ls,le,sigma", [
    (96, 32000, 32000, 0, 16, 96, 3.0),     # the LM shape, a window
    (37, 5003, 5011, 1, 3, 30, 3.0),        # ragged stride, base 2 bytes past a 16-byte boundary
    (23, 4099, 4103, 7, 0, 23, 2.0),        # base 14 bytes past: a 1-element head
    (11, 15, 15, 3, 0, 11, 2.0),            # a head and a tail, one chunk of body at most
    (9, 7, 9, 2, 1, 8, 2.0),                # rows shorter than a 16-byte chunk
    (6, 1, 1, 0, 0, 6, 1.0),
    (5, 100003, 100003, 0, 0, 5, 3.0),      # a cluster of CTAs per row
    (160, 5003, 5011, 1, 3, 150, 3.0),      # 2-CTA clusters, whole rows and split odd rows
    (200, 33, 37, 3, 10, 190, 2.0),         # the same with rows of a few chunks
])
def test_ce_fused_bf16(ntok, V, ld, off, ls, le, sigma):
    torch = H.torch_cuda()
    vl = _vl()
    seed = ntok * 131 + V
    x = W.random_logits(ntok, V, seed=seed, sigma=sigma)
    lab = W.random_labels(ntok, V, seed=seed + 1)
    bits = bf16_bits(x)
    xb = bf16_value(bits)
    scale = 1.0 / max(1, le - ls)
    buf, view = dev_bf16(bits, ld, off)
    loss = torch.full((ntok,), -7.0, device="cuda")
    lse = torch.full((ntok,), -7.0, device="cuda")
    stats = torch.full((ntok, 2), -7.0, device="cuda")
    mean = torch.full((1,), -7.0, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    vl.vl_ce_fused_bf16(view.data_ptr(), ld, ntok, V, H.dev(lab), ls, le, scale, loss, lse, stats, mean, err)
    torch.cuda.synchronize()
    oloss, olse, og, omean = O.ce_fused(xb, lab, ls, le, scale)
    g = host_bits(view)
    check_grad_bf16(g[:, :V], og, scale)
    if ld > V:
        assert np.isnan(bf16_value(g[:, V:])).all(), "columns past V were written"
    if off:
        assert np.isnan(bf16_value(host_bits(buf)[:off])).all(), "memory before the first row was written"
    H.check_loss(H.host(loss), oloss, olse, "bf16 CE loss")
    H.check_lse(H.host(lse), olse, "bf16 lse")
    assert np.array_equal(H.host(stats)[:, 0], xb.max(axis=1))
    H.check_mean(H.host(mean)[0], omean)
    assert int(H.host(err)[0]) == 0


def test_ce_fwd_then_sliced_bwd_bf16():
    torch = H.torch_cuda()
    vl = _vl()
    ntok, V, ld, ls, le, scale = 19, 3001, 3009, 2, 17, 1.0 / 15
    x = W.random_logits(ntok, V, seed=8, sigma=3.0)
    lab = W.random_labels(ntok, V, seed=9)
    bits = bf16_bits(x)
    xb = bf16_value(bits)
    buf, view = dev_bf16(bits, ld, 3)
    labels = H.dev(lab)
    loss = torch.zeros(ntok, device="cuda")
    lse = torch.zeros(ntok, device="cuda")
    stats = torch.zeros(ntok, 2, device="cuda")
    vl.vl_ce_fwd_bf16(view.data_ptr(), ld, ntok, V, labels, ls, le, loss, lse, stats, None, None)
    parts = []
    for c0, w in [(0, 1000), (1000, 517), (1517, 1484)]:
        lp = torch.full((ntok,), -1.0, device="cuda")
        vl.vl_ce_bwd_inplace_bf16(view.data_ptr(), ld, ntok, V, c0, w, labels, None, stats, ls, le, scale, lp, None)
        parts.append(lp)
    torch.cuda.synchronize()
    oloss, olse = O.ce_forward(xb, lab, ls, le)
    og, _ = O.ce_backward(xb, lab, olse, ls, le, scale)
    H.check_loss(H.host(loss), oloss, olse, "bf16 CE forward loss")
    H.check_lse(H.host(lse), olse, "bf16 lse")
    check_grad_bf16(host_bits(view)[:, :V], og, scale, "bf16 sliced CE gradient")
    tot = sum(H.host(p).astype(np.float64) for p in parts)
    H.check_loss(tot, oloss, olse, "bf16 sum of slice loss parts")


@pytest.mark.parametrize("ntok,V,ld,off,k,dup", [
    (48, 32000, 32000, 0, 64, False),       # the KL workload's shape
    (23, 4099, 4103, 5, 37, True),          # repeated ids, a misaligned base
    (6, 2048, 2048, 0, 1024, False),        # the largest support
    (4, 100003, 100003, 1, 128, True),      # a cluster of CTAs per row
    (300, 70001, 70009, 3, 64, True),       # rows of four tiles and more, more rows than SMs
])
def test_kl_self_contained_bf16(ntok, V, ld, off, k, dup):
    torch = H.torch_cuda()
    vl = _vl()
    x = W.random_logits(ntok, V, seed=V + k, sigma=2.0)
    tid, tp = W.random_teacher(ntok, V, k, seed=V + 2 * k)
    lab = W.random_labels(ntok, V, seed=V + 3)
    if dup:
        tid[:, 3] = tid[:, 7]
        tid[:, 5] = lab                     # the label inside the support
        tp[:, 2] = 0.0
    bits = bf16_bits(x)
    xb = bf16_value(bits)
    coef, ce_coef = 1.0 / ntok, 0.5 / ntok
    buf, view = dev_bf16(bits, ld, off)
    loss = torch.full((ntok,), -7.0, device="cuda")
    vl.vl_kl_topk_inplace_bf16(view.data_ptr(), ld, ntok, V, 0, V, H.dev(tid), H.dev(tp), k, coef, 0, ntok, None,
                               None, H.dev(lab), ce_coef, loss, None)
    torch.cuda.synchronize()
    oloss, og = O.kl_topk(xb, tid, tp, coef, labels=lab, ce_coef=ce_coef)
    _, olse = O.ce_forward(xb, lab, 0, ntok)
    check_grad_bf16(host_bits(view)[:, :V], og, coef + ce_coef, "bf16 KL + CE gradient")
    H.check_loss(H.host(loss), oloss, olse, "bf16 KL")


def test_large_vocab_bf16_fused_and_sliced():
    """The large-vocabulary rows in bf16: one pass (vl_ce_kl_fused_bf16) and the slice API
    (CE forward, two slices of KL + CE gradient from the row statistics, acc_add)."""
    torch = H.torch_cuda()
    vl = _vl()
    w = W.WORKLOADS["large_v"].scaled(12)
    x, lab = W.logits(w), W.labels(w)
    tid, tp = W.teacher(w)
    bits = bf16_bits(x)
    xb = bf16_value(bits)
    n, V, k = w.ntok, w.V, w.k
    o_ce, o_lse = O.ce_forward(xb, lab, 0, n)
    o_kl, og = O.kl_topk(xb, tid, tp, w.coef, labels=lab, ce_coef=w.ce_coef)
    labels, tidd, tpd = H.dev(lab), H.dev(tid), H.dev(tp)
    # one pass
    _, view = dev_bf16(bits)
    kl, ce = torch.zeros(n, device="cuda"), torch.zeros(n, device="cuda")
    mean = torch.zeros(1, device="cuda")
    vl.vl_ce_kl_fused_bf16(view.data_ptr(), V, n, V, labels, tidd, tpd, k, w.coef, w.ce_coef, 0, n, kl, ce, None,
                           None, mean, None)
    torch.cuda.synchronize()
    check_grad_bf16(host_bits(view), og, w.coef + w.ce_coef, "bf16 CE+KL one pass")
    H.check_loss(H.host(kl), o_kl, o_lse, "bf16 one-pass KL")
    H.check_loss(H.host(ce), o_ce, o_lse, "bf16 one-pass CE")
    H.check_mean(H.host(mean)[0], O.ce_mean(o_ce, 0, n))
    # the slice API
    _, view = dev_bf16(bits)
    ce2 = torch.zeros(n, device="cuda")
    stats = torch.zeros((n, 2), device="cuda")
    vl.vl_ce_fwd_bf16(view.data_ptr(), V, n, V, labels, 0, n, ce2, None, stats, None, None)
    parts = [torch.zeros(n, device="cuda") for _ in range(w.slices)]
    for (c0, width), part in zip(cuts_for_slices(V, w.slices), parts):
        vl.vl_kl_topk_inplace_bf16(view.data_ptr(), V, n, V, c0, width, tidd, tpd, k, w.coef, 0, n, None, stats,
                                   labels, w.ce_coef, part, None)
    vl.vl_acc_add(parts[0], parts[1], n)
    torch.cuda.synchronize()
    check_grad_bf16(host_bits(view), og, w.coef + w.ce_coef, "bf16 CE+KL slices")
    H.check_loss(H.host(parts[0]), o_kl, o_lse, "bf16 sliced KL")
    H.check_loss(H.host(ce2), o_ce, o_lse, "bf16 CE forward")
