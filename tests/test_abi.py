"""The C-ABI library without a GPU: it loads, exports what include/vloss.h declares,
and rejects bad arguments on the host before any CUDA call."""
import pytest

from top_kl_distill_gb300 import vloss as vl


def test_library_exports_every_declared_symbol():
    L = vl.lib()
    names = vl.declared_symbols()
    assert {"vl_ce_fwd", "vl_ce_bwd_inplace", "vl_ce_fused", "vl_kl_topk_inplace", "vl_topk_rows",
            "vl_acc_add"} <= set(names)
    missing = [n for n in names if not hasattr(L, n)]
    assert not missing, f"declared but not exported: {missing}"
    assert vl.vl_version() >= 100
    assert L.vl_status_string(1) == b"invalid argument"


def _status(fn, *args):
    with pytest.raises(vl.VlossError) as e:
        fn(*args)
    return e.value.status


# raw addresses never dereferenced: the host checks reject the call first
P = 1 << 20


def test_rejects_bad_rows():
    assert _status(vl.vl_ce_fused, P, 10, 4, 11, P, 0, 4, 1.0, P, None, None, None, None, 0) == vl.VL_EINVAL
    assert _status(vl.vl_ce_fused, P, 10, 4, 0, P, 0, 4, 1.0, P, None, None, None, None, 0) == vl.VL_EINVAL
    assert _status(vl.vl_ce_fused, P, 10, -1, 10, P, 0, 0, 1.0, P, None, None, None, None, 0) == vl.VL_EINVAL
    assert _status(vl.vl_ce_fused, None, 10, 4, 10, P, 0, 4, 1.0, P, None, None, None, None, 0) == vl.VL_EINVAL


def test_rejects_bad_windows():
    assert _status(vl.vl_ce_fwd, P, 10, 4, 10, P, 3, 2, P, None, None, None, None, 0) == vl.VL_EINVAL
    assert _status(vl.vl_ce_fwd, P, 10, 4, 10, P, 0, 5, P, None, None, None, None, 0) == vl.VL_EINVAL
    assert _status(vl.vl_ce_fwd, P, 10, 4, 10, P, -1, 2, P, None, None, None, None, 0) == vl.VL_EINVAL
    assert "window" in vl.lib().vl_last_error_string().decode()


def test_rejects_bad_slices_and_missing_statistics():
    assert _status(vl.vl_ce_bwd_inplace, P, 10, 4, 10, 6, 5, P, P, None, 0, 4, 1.0, None, None, 0) == vl.VL_EINVAL
    assert _status(vl.vl_ce_bwd_inplace, P, 10, 4, 10, 0, 5, P, None, None, 0, 4, 1.0, None, None, 0) == vl.VL_EINVAL
    # a KL slice needs the full-row statistics
    assert _status(vl.vl_kl_topk_inplace, P, 10, 4, 10, 2, 5, P, P, 3, 1.0, 0, 4,
                   None, None, None, 0.0, P, None, 0) == vl.VL_EINVAL


def test_rejects_k_out_of_range():
    assert _status(vl.vl_kl_topk_inplace, P, 10, 4, 10, 0, 10, P, P, 0, 1.0, 0, 4,
                   None, None, None, 0.0, P, None, 0) == vl.VL_EINVAL
    assert _status(vl.vl_kl_topk_inplace, P, 5000, 4, 5000, 0, 5000, P, P, vl.VL_KL_KMAX + 1, 1.0, 0, 4,
                   None, None, None, 0.0, P, None, 0) == vl.VL_EUNSUPPORTED
    assert _status(vl.vl_topk_rows, P, 10, 4, 10, 11, 0, 4, P, P, None, None, 0, 0) == vl.VL_EINVAL
    assert _status(vl.vl_topk_rows, P, 5000, 4, 5000, vl.VL_TOPK_KMAX + 1, 0, 4, P, P, None, None, 0, 0) == vl.VL_EUNSUPPORTED


def test_acc_add_host_checks():
    assert _status(vl.vl_acc_add, P, P + 16, -1, 0) == vl.VL_EINVAL
    assert _status(vl.vl_acc_add, P, P + 16, 8, 0) == vl.VL_EINVAL      # overlap: b starts 4 floats into a
    assert _status(vl.vl_acc_add, None, P, 8, 0) == vl.VL_EINVAL
    vl.vl_acc_add(P, P + 64, 0, 0)                                     # n = 0 is a no-op


def test_empty_calls_launch_nothing():
    vl.vl_ce_bwd_inplace(P, 10, 0, 10, 0, 10, None, None, None, 0, 0, 1.0, None, None, 0)
    vl.vl_kl_topk_inplace(P, 10, 0, 10, 0, 10, None, None, 3, 1.0, 0, 0, None, None, None, 0.0, None, None, 0)
    vl.vl_topk_rows(P, 10, 4, 10, 3, 2, 2, None, None, None, None, 0, 0)


def test_rejects_missing_outputs_and_huge_rows():
    # KL without its teacher or loss pointer, top-k without its outputs
    assert _status(vl.vl_kl_topk_inplace, P, 10, 4, 10, 0, 10, None, P, 3, 1.0, 0, 4,
                   None, None, None, 0.0, P, None, 0) == vl.VL_EINVAL
    assert _status(vl.vl_kl_topk_inplace, P, 10, 4, 10, 0, 10, P, P, 3, 1.0, 0, 4,
                   None, None, None, 0.0, None, None, 0) == vl.VL_EINVAL
    assert _status(vl.vl_topk_rows, P, 10, 4, 10, 3, 0, 4, None, P, None, None, 0, 0) == vl.VL_EINVAL
    # CE backward without labels; rows of 2^31 columns or more
    assert _status(vl.vl_ce_bwd_inplace, P, 10, 4, 10, 0, 10, None, P, None, 0, 4, 1.0, None, None, 0) == vl.VL_EINVAL
    assert _status(vl.vl_ce_fwd, P, 1 << 31, 2, 1 << 31, P, 0, 2, P, None, None, None, None, 0) == vl.VL_EINVAL
    # every failure leaves a message naming the entry point
    assert "vl_ce_fwd" in vl.lib().vl_last_error_string().decode()


def test_row_length_limit():
    """Rows are indexed with 32-bit ints: the longest accepted row is VL_MAX_COLS
    (2^31 - 2^16) columns, checked on the host before anything is launched."""
    big = vl.VL_MAX_COLS
    assert _status(vl.vl_ce_fwd, P, big + 1, 2, big + 1, P, 0, 2, P, None, None, None, None, 0) == vl.VL_EINVAL
    assert str(big) in vl.lib().vl_last_error_string().decode()
    for fn, args in [
        (vl.vl_ce_fused, (P, big + 1, 3, big + 1, P, 0, 3, 1.0, P, None, None, None, None, 0)),
        (vl.vl_ce_bwd_inplace, (P, big + 1, 3, big + 1, 0, 8, P, P, None, 0, 3, 1.0, None, None, 0)),
        (vl.vl_kl_topk_inplace, (P, big + 1, 3, big + 1, 0, big + 1, P, P, 3, 1.0, 0, 3,
                                 None, None, None, 0.0, P, None, 0)),
        (vl.vl_topk_rows, (P, big + 1, 3, big + 1, 3, 0, 3, P, P, None, None, 0, 0)),
    ]:
        assert _status(fn, *args) == vl.VL_EINVAL, fn.__name__
    # exactly VL_MAX_COLS passes the checks (no rows: nothing is launched)
    vl.vl_ce_fwd(P, big, 0, big, None, 0, 0, None, None, None, None, None, 0)


def test_wait_timeout_hook_rejects_bad_settings():
    for args in [(-1, 10_000), (0, 10), (0, 5_000_000_000)]:
        assert _status(vl.vl_test_inject_wait_timeout, *args) == vl.VL_EINVAL


def test_window_mean_host_checks():
    assert _status(vl.vl_window_mean, P, 10, 3, 2, P, 0) == vl.VL_EINVAL       # window reversed
    assert _status(vl.vl_window_mean, P, 10, 0, 11, P, 0) == vl.VL_EINVAL      # past ntok
    assert _status(vl.vl_window_mean, P, 10, 0, 4, None, 0) == vl.VL_EINVAL    # no output
    assert _status(vl.vl_window_mean, None, 10, 0, 4, P, 0) == vl.VL_EINVAL    # no losses


def test_topk_workspace_size():
    """The streaming top-k takes rows of 30720 to 2^20 columns with k up to about 6% of V.
    Its workspace holds two sets of 15 candidate regions per CTA (one CTA per SM of the
    current device, at most one per row) and 4 bytes a row for the list of rows left to
    the exact kernel."""
    f = vl.vl_topk_workspace_bytes
    assert f(4096, 128256, 256) > 0 and f(4096, 128256, 2048) > 0
    for k, expect in [(256, 3 * 128256 / 256 / 15), (2048, 8 * 128256 / 256 / 15)]:
        cta = f(2, 128256, k) - f(1, 128256, k)      # one more CTA's regions
        slots = cta / (2 * 15 * 8)
        assert expect * 1.5 < slots < expect * 2.5 + 64, (k, slots)
    big = f(100_000, 128256, 2048)
    assert 0 <= f(100_001, 128256, 2048) - big <= 256  # past one CTA per SM only the list grows
    assert f(10, 30719, 16) == 0                  # too short to estimate from the first tile
    assert f(10, (1 << 20) + 1, 16) == 0          # longer than the stream kernel takes
    assert f(10, 40000, 5000) == 0                # k too large a share of the row
    assert f(0, 128256, 256) == 0 and f(10, 128256, 0) == 0 and f(10, 100, 101) == 0
    # a misaligned workspace is rejected before anything is launched
    assert _status(vl.vl_topk_rows, P, 40000, 4, 40000, 8, 0, 4, P, P, None, P + 8, 1 << 20, 0) == vl.VL_EINVAL


def test_gemm_host_checks():
    assert _status(vl.vl_gemm_bf16_tn, P, P + 1024, P + 4096, 4, 4, 12, 4, 1.0, 0) == vl.VL_EINVAL   # K % 8
    assert _status(vl.vl_gemm_bf16_tn, P, P + 1024, P + 4096, 4, 4, 16, 3, 1.0, 0) == vl.VL_EINVAL   # ldd < N
    assert _status(vl.vl_gemm_bf16_tn, P + 2, P + 1024, P + 4096, 4, 4, 16, 4, 1.0, 0) == vl.VL_EINVAL  # alignment
    assert _status(vl.vl_gemm_bf16_tn, None, P, P, 4, 4, 16, 4, 1.0, 0) == vl.VL_EINVAL
    vl.vl_gemm_bf16_tn(P, P, P, 0, 4, 16, 4, 1.0, 0)          # an empty product launches nothing


def test_head_host_checks():
    f = vl.lib()
    assert f.vl_teacher_topk_workspace_bytes(1, 128256, 256) > (32 << 20)
    assert f.vl_head_kl_workspace_bytes(2, 1000) - f.vl_head_kl_workspace_bytes(1, 1000) >= 6 * 1000
    ws = (P, 1 << 30)
    assert _status(vl.vl_teacher_topk, P, 12, P, 1000, 4, 8, 0, 4, P, P, None, ws, 0) == vl.VL_EINVAL     # hs % 8
    assert _status(vl.vl_head_kl, P, 16, P, None, 1000, 4, P, P, P, 8, 1.0, 1.0, 1.0, 0, 4, P + 4, P, P, None,
                   None, ws, 0) == vl.VL_EINVAL                                                         # dx alignment
