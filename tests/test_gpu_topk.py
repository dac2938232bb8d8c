"""Teacher top-k through the C ABI against the oracle's full stable sort."""
import numpy as np
import pytest

from oracle import vloss_oracle as O
from tests import gpu_harness as H
from top_kl_distill_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def run_topk(x, k, ls=0, le=None, ld=None, off=0, with_err=False, workspace="auto"):
    torch = H.torch_cuda()
    from top_kl_distill_gb300 import vloss as vl
    ntok, V = x.shape
    le = ntok if le is None else le
    ld = ld or V
    _, view = H.strided(x, ld, off)
    ids = torch.full((ntok, k), -1, dtype=torch.int32, device="cuda")
    probs = torch.full((ntok, k), -1.0, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    vl.vl_topk_rows(view.data_ptr(), ld, ntok, V, k, ls, le, ids, probs, err, workspace)
    torch.cuda.synchronize()
    out = H.host(ids).view(np.uint32), H.host(probs)
    return out + (int(H.host(err)[0]),) if with_err else out


def check(x, k, ls=0, le=None, **kw):
    """Exact against the oracle; rows of 30720 columns or more go through the streaming
    kernel (the default workspace) and, with workspace=None, the single kernel."""
    ntok = x.shape[0]
    le = ntok if le is None else le
    ids, probs, err = run_topk(x, k, ls, le, with_err=True, **kw)
    assert err == 0
    oids, oprobs, valid = O.topk_rows(x, k, ls, le)
    assert np.array_equal(ids[valid].astype(np.int64), oids[valid]), "top-k ids differ"
    H.check_probs(probs[valid], oprobs[valid])
    assert np.all(ids[~valid] == 0xFFFFFFFF) and np.all(probs[~valid] == -1.0), "rows outside the window written"


@pytest.mark.parametrize("path", ["stream", "single_kernel"])
@pytest.mark.parametrize("k", [256, 2048])
def test_topk_workload_rows(k, path):
    w = W.WORKLOADS["topk"].scaled(6)
    check(W.logits(w), k, workspace="auto" if path == "stream" else None)


def test_topk_stream_few_ctas_with_fallback_rows():
    """A workspace with candidate regions for three CTAs only: 11 rows on 3 CTAs, each
    alternating its two region sets over four rows, with monotone rows (threshold check
    fails, or the regions overflow) mixed in for the exact kernel."""
    torch = H.torch_cuda()
    from top_kl_distill_gb300 import vloss as vl
    V, k = 40000, 300
    x = W.random_logits(11, V, seed=51, sigma=3.0)
    up = np.arange(V, dtype=np.float32) * np.float32(1e-3)
    x[2], x[7] = up, up[::-1]
    f = vl.vl_topk_workspace_bytes
    cta = f(2, V, k) - f(1, V, k)
    ws = torch.empty(f(11, V, k) - 8 * cta, dtype=torch.uint8, device="cuda")
    assert cta > 0
    check(x, k, workspace=ws)
    check(x, k, ls=3, le=10, workspace=ws)


@pytest.mark.parametrize("k", [1, 7, 100, 700])
def test_topk_tie_heavy(k):
    check(W.tie_heavy_logits(16, 3000, seed=k), k)


def test_topk_all_equal_and_signed_zeros():
    x = np.zeros((3, 5000), dtype=np.float32)
    x[1, ::2] = -0.0
    x[2] = 1.5
    check(x, 50)
    check(x, 2048)


@pytest.mark.parametrize("ws", ["auto", None])
def test_topk_monotone_rows(ws):
    """Ascending rows admit every new column (the most compactions, or a list overflow);
    descending rows almost none (the threshold check fails): the exact kernel's rows."""
    V = 50000
    up = np.arange(V, dtype=np.float32)[None, :] * np.float32(1e-3)
    x = np.concatenate([up, up[:, ::-1].copy(), -up], axis=0)
    for k in (1, 256, 2048):
        check(x, k, workspace=ws)


def test_topk_k_equals_v_and_misaligned():
    x = W.random_logits(5, 1500, seed=3)
    check(x, 1500)
    x = W.random_logits(11, 6007, seed=4)
    check(x, 333, ls=2, le=9, ld=6011, off=1)


def test_topk_window_only():
    x = W.random_logits(10, 4000, seed=5)
    check(x, 64, ls=3, le=7)


@pytest.mark.parametrize("k", [1, 256, 2048])
def test_topk_tie_heavy_long_rows(k):
    """Rows long enough for the speculative threshold, with many exact ties at it."""
    x = W.tie_heavy_logits(6, 40000, seed=100 + k, step=0.25, sigma=1.5)
    x[5] = np.float32(0.5)                     # one row all equal: every value ties
    check(x, k)


def test_topk_long_rows_misaligned_and_windowed():
    """The speculative path with head and tail columns (odd row stride and offset) and a
    loss window (rows outside it are left alone)."""
    x = W.random_logits(9, 40007, seed=21, sigma=3.0)
    check(x, 300, ls=1, le=8, ld=40011, off=3)
    check(x, 2048, ls=2, le=9, ld=40011, off=1)


@pytest.mark.parametrize("V", [1, 2, 3, 4, 5, 6, 7, 8, 9])
def test_topk_tiny_rows(V):
    """Rows shorter than one float4 run: only head and tail columns (no bulk copy), at
    every base misalignment and with k = V, k = 1 and a middle k."""
    x = W.tie_heavy_logits(7, V, seed=300 + V, step=0.5, sigma=1.0)
    for off in range(4):
        for k in sorted({1, max(1, V // 2), V}):
            check(x, k, ld=V + (off & 1), off=off)


def test_topk_nan_rows_counted():
    """NaN is a data error: never selected, one count per row in the window that holds
    one.  Rows with at least k other values get the top k of those values."""
    x = W.random_logits(7, 5000, seed=41, sigma=2.0)
    x[1, [7, 100, 4999]] = np.nan
    x[4, 0] = np.nan                          # a head column (offset 1 below)
    x[6, 2] = np.nan                          # outside the window: not counted
    ids, probs, err = run_topk(x, 64, 0, 6, off=1, with_err=True)
    assert err == 2
    xo = np.where(np.isnan(x), -np.inf, x).astype(np.float32)
    oids, oprobs, valid = O.topk_rows(xo, 64, 0, 6)
    assert np.array_equal(ids[valid].astype(np.int64), oids[valid])
    H.check_probs(probs[valid], oprobs[valid])
    # a long row (speculative threshold) with a NaN in its body
    y = W.random_logits(3, 40000, seed=42, sigma=3.0)
    y[2, 12345] = np.nan
    ids, probs, err = run_topk(y, 256, with_err=True)
    assert err == 1
    oids, oprobs, _ = O.topk_rows(np.where(np.isnan(y), -np.inf, y).astype(np.float32), 256)
    assert np.array_equal(ids.astype(np.int64), oids)


def test_topk_row_with_fewer_values_than_k():
    x = W.random_logits(2, 50, seed=43)
    x[1, 5:] = np.nan                          # five values left in row 1
    ids, probs, err = run_topk(x, 10, with_err=True)
    assert err == 1
    oids, oprobs, _ = O.topk_rows(x[:1], 10)
    assert np.array_equal(ids[0].astype(np.int64), oids[0])
    o5, p5, _ = O.topk_rows(x[1:, :5], 5)
    assert np.array_equal(ids[1, :5].astype(np.int64), o5[0])
    H.check_probs(probs[1, :5], p5[0])
    assert np.all(ids[1, 5:] == 0xFFFFFFFF) and np.all(probs[1, 5:] == 0.0)
