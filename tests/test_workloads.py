"""Host logic: seeded input generators and vocabulary slicing (no GPU)."""
import numpy as np

from top_kl_distill_gb300 import workloads as W
from top_kl_distill_gb300.slicing import cuts_for_slices, vocab_cuts


def test_rows_regenerate_independently():
    w = W.WORKLOADS["ce_lm"].scaled(200)
    full = W.logits(w, threads=4)
    part = W.logits(w, 70, 141, threads=1)
    assert np.array_equal(full[70:141], part)
    assert np.array_equal(W.labels(w)[70:141], W.labels(w, 70, 141))
    ids, tp = W.teacher(W.WORKLOADS["kl"].scaled(130))
    ids2, tp2 = W.teacher(W.WORKLOADS["kl"].scaled(130), 65, 130)
    assert np.array_equal(ids[65:], ids2) and np.array_equal(tp[65:], tp2)


def test_ce_lm_peaks_at_labels():
    w = W.WORKLOADS["ce_lm"].scaled(256)
    x = W.logits(w)
    lab = W.labels(w)
    at = x[np.arange(256), lab]
    assert 0.2 < np.mean(at > 6.0) < 0.45          # about 30% of the rows carry the +8 peak
    assert abs(x.std() - 3.0) < 0.05


def test_teacher_support():
    w = W.WORKLOADS["kl"].scaled(64)
    ids, tp = W.teacher(w)
    assert ids.shape == (64, 64) and ids.dtype == np.uint32
    assert all(len(set(r.tolist())) == 64 for r in ids)
    assert np.all(ids < w.V)
    assert np.all(tp > 0) and np.allclose(tp.astype(np.float64).sum(1), 1.0, atol=1e-6)


def test_topk_rows_are_distinct():
    w = W.WORKLOADS["topk"].scaled(3)
    x = W.logits(w)
    for r in x:
        assert np.unique(r).size == r.size


def test_large_v_heavy_tails():
    w = W.WORKLOADS["large_v"].scaled(2)
    x = W.logits(w)
    assert x.shape == (2, 128256)
    assert np.abs(x).max() > 20.0          # 2 * t_4 reaches far past a Gaussian of the same scale


def test_make_distinct():
    r = np.array([1.0, 1.0, 1.0, 2.0, np.nextafter(np.float32(1.0), np.float32(2.0))], dtype=np.float32)
    W.make_distinct(r)
    assert np.unique(r).size == r.size and r[0] == 1.0


def test_page_slice_rule():
    # the page's own test asserts three slices for v = 1024 with at most 384 rows
    assert vocab_cuts(1024, max_rows=384) == [(0, 384), (384, 384), (768, 256)]
    # the large-vocabulary workload: two slices of 64128 (= 501 * 128)
    assert cuts_for_slices(128256, 2) == [(0, 64128), (64128, 64128)]
    # default cap: 2 GiB of f16 weights, e.g. a 248k x 5120 head needs two slices
    cuts = vocab_cuts(248000, hs=5120)
    assert len(cuts) == 2 and sum(w for _, w in cuts) == 248000
    assert all(w % 128 == 0 for _, w in cuts[:-1])
