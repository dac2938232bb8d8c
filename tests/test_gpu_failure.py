"""The failure path of the kernels' bounded waits, provoked without a fault.

The test hook makes CTA 0 of one launch stop issuing its row tiles, so that its
consumers wait for a tile that never comes, with a wait limit of about a millisecond.
The wait runs out, the kernel raises the watchdog flag, lets the copies it issued
land and returns; the other CTAs' rows are still right, and the next launch on the
same context is correct again.
"""
import time

import numpy as np
import pytest

from oracle import vloss_oracle as O
from tests import gpu_harness as H
from top_kl_distill_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def test_withheld_tile_times_out_and_the_context_stays_usable():
    torch = H.torch_cuda()
    from top_kl_distill_gb300 import vloss as vl
    ntok, V, scale = 4, 40000, 0.25               # streaming backward: one CTA per row, ~10 tiles a row
    x = W.random_logits(ntok, V, seed=61, sigma=2.0)
    lab = W.random_labels(ntok, V, seed=62)
    _, olse = O.ce_forward(x, lab, 0, ntok)
    lse32 = olse.astype(np.float32)
    og, _ = O.ce_backward(x, lab, lse32.astype(np.float64), 0, ntok, scale)
    labels, lse = H.dev(lab), H.dev(lse32)
    dev = torch.cuda.current_device()
    assert vl.vl_watchdog_flag(dev, True) == 0

    xt = H.dev(x)
    vl.vl_test_inject_wait_timeout(3, 2_000_000)  # CTA 0 withholds its 4th tile; waits give up after 2e6 cycles
    t0 = time.time()
    vl.vl_ce_bwd_inplace(xt, V, ntok, V, 0, V, labels, lse, None, 0, ntok, scale, None, None)
    torch.cuda.synchronize()
    assert time.time() - t0 < 10.0
    assert vl.vl_watchdog_flag(dev, True) == 1, "the timed-out wait was not reported"
    H.check_grad(H.host(xt)[1:], og[1:], scale, "rows of the CTAs that were not stopped")

    # the hook is used once: the same call again is complete and correct on every row
    xt = H.dev(x)
    vl.vl_ce_bwd_inplace(xt, V, ntok, V, 0, V, labels, lse, None, 0, ntok, scale, None, None)
    torch.cuda.synchronize()
    assert vl.vl_watchdog_flag(dev, True) == 0
    H.check_grad(H.host(xt), og, scale)

