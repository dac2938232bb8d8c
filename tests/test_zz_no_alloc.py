"""vl_topk_rows_noalloc: the top-k for callers that cannot allocate device memory where they
call it (an allocator hook that must not re-enter the allocator, a path that may not risk an
allocation, a runtime without a device allocator).  Its scratch is one fixed array in the
library instead of a workspace from the caller.

Two calls in a row share that array: each must match vl_topk_rows (the workspace entry
point) on its own input -- ids bit-exact, probabilities within the top-k tolerance -- so
nothing the first call left in the array can leak into the second.  This file is collected
last on purpose, and passes alone in a fresh process as well.
"""
import re

import numpy as np
import pytest

from tests import gpu_harness as H
from top_kl_distill_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _topk(fn, x, k, ls, le, ld, off):
    torch = H.torch_cuda()
    ntok, V = x.shape
    _, view = H.strided(x, ld, off)
    ids = torch.full((ntok, k), -1, dtype=torch.int32, device="cuda")
    probs = torch.full((ntok, k), -1.0, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    fn(view.data_ptr(), ld, ntok, V, k, ls, le, ids, probs, err)
    torch.cuda.synchronize()
    return H.host(ids).view(np.uint32), H.host(probs), int(H.host(err)[0])


@pytest.mark.parametrize("k", [256, 2048])
def test_noalloc_matches_the_workspace_entry_point_twice(k):
    from top_kl_distill_gb300 import vloss as vl
    w = W.WORKLOADS["topk"].scaled(40)
    inputs = [
        (W.logits(w), 0, 40, w.V, 0),                                   # the teacher workload's rows
        (W.random_logits(37, 60011, seed=k, sigma=3.0), 3, 35, 60013, 1),  # other rows, a window, misaligned
    ]
    for x, ls, le, ld, off in inputs:                                   # two calls in a row on the one array
        ref_ids, ref_probs, ref_err = _topk(vl.vl_topk_rows, x, k, ls, le, ld, off)
        ids, probs, err = _topk(vl.vl_topk_rows_noalloc, x, k, ls, le, ld, off)
        assert err == ref_err == 0
        assert np.array_equal(ids, ref_ids), "ids differ from vl_topk_rows"
        win = slice(ls, le)
        H.check_probs(probs[win], ref_probs[win].astype(np.float64), "no-alloc top-k probs")
        assert np.all(ids[:ls] == 0xFFFFFFFF) and np.all(ids[le:] == 0xFFFFFFFF), "rows outside the window written"


def test_noalloc_rejects_more_rows_than_its_scratch_holds_and_takes_the_limit():
    """A window larger than the fixed array holds is rejected before anything runs, with the
    limit in the message; one row more than the limit is rejected too, and exactly the limit
    (rows of 2^20 columns, k = 2048: the regions of about a hundred CTAs) runs and matches
    vl_topk_rows."""
    torch = H.torch_cuda()
    from top_kl_distill_gb300 import vloss as vl
    V, k = 1 << 20, 2048
    P = 1 << 20                                   # never dereferenced: the host rejects the call first
    with pytest.raises(vl.VlossError) as e:
        vl.vl_topk_rows_noalloc(P, V, 10 ** 6, V, k, 0, 10 ** 6, P, P, None, 0)
    assert e.value.status == vl.VL_EUNSUPPORTED
    most = int(re.search(r"at most (\d+) rows", str(e.value)).group(1))
    assert 10 < most < 10 ** 6
    with pytest.raises(vl.VlossError) as e:
        vl.vl_topk_rows_noalloc(P, V, most + 1, V, k, 0, most + 1, P, P, None, 0)
    assert e.value.status == vl.VL_EUNSUPPORTED
    g = torch.Generator(device="cuda").manual_seed(2024)
    x = torch.randn(most, V, device="cuda", generator=g) * 3.0
    outs = []
    for fn in (vl.vl_topk_rows, vl.vl_topk_rows_noalloc):
        ids = torch.full((most, k), -1, dtype=torch.int32, device="cuda")
        probs = torch.full((most, k), -1.0, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        fn(x, V, most, V, k, 0, most, ids, probs, err)
        torch.cuda.synchronize()
        outs.append((H.host(ids), H.host(probs), int(H.host(err)[0])))
    (ri, rp, re_), (ni, np_, ne) = outs
    assert re_ == ne == 0
    assert np.array_equal(ni, ri), "ids differ from vl_topk_rows"
    H.check_probs(np_, rp.astype(np.float64), "no-alloc top-k probs at the row limit")
