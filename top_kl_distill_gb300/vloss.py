"""Python binding of libvloss: the C entry points under the same names.

Argument marshalling only: every step runs in the CUDA library.  Each pointer
parameter accepts a torch tensor (its data pointer is passed after a dtype
and device check), a raw integer device address, or None for NULL.  ``stream``
accepts a torch.cuda.Stream, a raw cudaStream_t integer, or None for torch's
current stream on the current device.  A status other than VL_OK raises
VlossError with the library's message.

The library must have been built in-tree (``python -m top_kl_distill_gb300.build``
or ``__graft_entry__.build()``); there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import re

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libvloss.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "vloss.h")

VL_OK, VL_EINVAL, VL_ELAUNCH, VL_EUNSUPPORTED = 0, 1, 2, 3
VL_KL_KMAX = 1024
VL_TOPK_KMAX = 2048
VL_MAX_COLS = 0x7FFF0000

_P = ctypes.c_void_p
_I = ctypes.c_int64
_F = ctypes.c_float

_SIGS = {
    "vl_ce_fwd": [_P, _I, _I, _I, _P, _I, _I, _P, _P, _P, _P, _P, _P],
    "vl_ce_bwd_inplace": [_P, _I, _I, _I, _I, _I, _P, _P, _P, _I, _I, _F, _P, _P, _P],
    "vl_ce_fused": [_P, _I, _I, _I, _P, _I, _I, _F, _P, _P, _P, _P, _P, _P],
    "vl_kl_topk_inplace": [_P, _I, _I, _I, _I, _I, _P, _P, _I, _F, _I, _I, _P, _P, _P, _F, _P, _P, _P],
    "vl_topk_rows": [_P, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P, _I, _P],
    "vl_ce_kl_fused": [_P, _I, _I, _I, _P, _P, _P, _I, _F, _F, _I, _I, _P, _P, _P, _P, _P, _P, _P],
    "vl_teacher_topk": [_P, _I, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _I, _P],
    "vl_gemm_bf16_tn": [_P, _P, _P, _I, _I, _I, _I, _F, _P],
    "vl_topk_rows_noalloc": [_P, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P],
    "vl_head_kl": [_P, _I, _P, _P, _I, _I, _P, _P, _P, _I, _F, _F, _F, _I, _I, _P, _P, _P, _P, _P, _P, _I, _P],
    "vl_ce_fwd_bf16": [_P, _I, _I, _I, _P, _I, _I, _P, _P, _P, _P, _P, _P],
    "vl_ce_bwd_inplace_bf16": [_P, _I, _I, _I, _I, _I, _P, _P, _P, _I, _I, _F, _P, _P, _P],
    "vl_ce_fused_bf16": [_P, _I, _I, _I, _P, _I, _I, _F, _P, _P, _P, _P, _P, _P],
    "vl_kl_topk_inplace_bf16": [_P, _I, _I, _I, _I, _I, _P, _P, _I, _F, _I, _I, _P, _P, _P, _F, _P, _P, _P],
    "vl_ce_kl_fused_bf16": [_P, _I, _I, _I, _P, _P, _P, _I, _F, _F, _I, _I, _P, _P, _P, _P, _P, _P, _P],
    "vl_acc_add": [_P, _P, _I, _P],
    "vl_test_inject_wait_timeout": [_I, _I],
    "vl_window_mean": [_P, _I, _I, _I, _P, _P],
}

_lib = None


class VlossError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn} -> status {status}: {msg}")
        self.status = status


def lib() -> ctypes.CDLL:
    """Load libvloss.so (once).  Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -m top_kl_distill_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        for name, args in _SIGS.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = ctypes.c_int
        L.vl_version.restype = ctypes.c_int
        L.vl_status_string.restype = ctypes.c_char_p
        L.vl_status_string.argtypes = [ctypes.c_int]
        L.vl_last_error_string.restype = ctypes.c_char_p
        L.vl_watchdog_flag.argtypes = [ctypes.c_int, ctypes.c_int]
        L.vl_watchdog_flag.restype = ctypes.c_int
        L.vl_topk_workspace_bytes.argtypes = [_I, _I, _I]
        L.vl_topk_workspace_bytes.restype = ctypes.c_int64
        L.vl_teacher_topk_workspace_bytes.argtypes = [_I, _I, _I]
        L.vl_teacher_topk_workspace_bytes.restype = ctypes.c_int64
        L.vl_head_kl_workspace_bytes.argtypes = [_I, _I]
        L.vl_head_kl_workspace_bytes.restype = ctypes.c_int64
        _lib = L
    return _lib


def declared_symbols() -> list[str]:
    """Names of the functions include/vloss.h declares."""
    txt = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:[\w\s\*]+?)\b(vl_\w+)\s*\(", txt, flags=re.M)))


_DT = {"f32": "torch.float32", "u32": "torch.uint32", "i32": "torch.int32", "bf16": "torch.bfloat16"}


def _ptr(x, kind: str, name: str):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    import torch
    if not isinstance(x, torch.Tensor):
        raise TypeError(f"{name}: expected a tensor, an int address or None")
    if not x.is_cuda:
        raise ValueError(f"{name}: tensor must live on a CUDA device")
    want = {"f32": (torch.float32,), "u32": (torch.uint32, torch.int32), "i32": (torch.int32,),
            "bf16": (torch.bfloat16,)}[kind]
    if x.dtype not in want:
        raise TypeError(f"{name}: dtype {x.dtype}, expected {_DT[kind]}")
    return x.data_ptr()


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(fn: str, status: int):
    if status != VL_OK:
        msg = lib().vl_last_error_string().decode()
        raise VlossError(fn, status, msg)


def vl_version() -> int:
    return lib().vl_version()


def vl_ce_fwd(logits, ld, ntok, V, labels, loss_start, loss_end, loss, lse=None, stats=None, mean=None,
              err=None, stream=None):
    _check("vl_ce_fwd", lib().vl_ce_fwd(
        _ptr(logits, "f32", "logits"), ld, ntok, V, _ptr(labels, "u32", "labels"), loss_start, loss_end,
        _ptr(loss, "f32", "loss"), _ptr(lse, "f32", "lse"), _ptr(stats, "f32", "stats"),
        _ptr(mean, "f32", "mean"), _ptr(err, "i32", "err"), _stream(stream)))


def vl_ce_bwd_inplace(logits, ld, ntok, V, col0, ncols, labels, lse, stats, loss_start, loss_end, scale,
                      loss_part=None, err=None, stream=None):
    _check("vl_ce_bwd_inplace", lib().vl_ce_bwd_inplace(
        _ptr(logits, "f32", "logits"), ld, ntok, V, col0, ncols, _ptr(labels, "u32", "labels"),
        _ptr(lse, "f32", "lse"), _ptr(stats, "f32", "stats"), loss_start, loss_end, float(scale),
        _ptr(loss_part, "f32", "loss_part"), _ptr(err, "i32", "err"), _stream(stream)))


def vl_ce_fused(logits, ld, ntok, V, labels, loss_start, loss_end, scale, loss, lse=None, stats=None,
                mean=None, err=None, stream=None):
    _check("vl_ce_fused", lib().vl_ce_fused(
        _ptr(logits, "f32", "logits"), ld, ntok, V, _ptr(labels, "u32", "labels"), loss_start, loss_end,
        float(scale), _ptr(loss, "f32", "loss"), _ptr(lse, "f32", "lse"), _ptr(stats, "f32", "stats"),
        _ptr(mean, "f32", "mean"), _ptr(err, "i32", "err"), _stream(stream)))


def vl_kl_topk_inplace(logits, ld, ntok, V, col0, ncols, tid, tp, k, coef, loss_start, loss_end,
                       lse_in=None, stats_in=None, labels=None, ce_coef=0.0, loss=None, err=None, stream=None):
    _check("vl_kl_topk_inplace", lib().vl_kl_topk_inplace(
        _ptr(logits, "f32", "logits"), ld, ntok, V, col0, ncols, _ptr(tid, "u32", "tid"), _ptr(tp, "f32", "tp"),
        k, float(coef), loss_start, loss_end, _ptr(lse_in, "f32", "lse_in"), _ptr(stats_in, "f32", "stats_in"),
        _ptr(labels, "u32", "labels"), float(ce_coef), _ptr(loss, "f32", "loss"), _ptr(err, "i32", "err"),
        _stream(stream)))


def vl_ce_kl_fused(logits, ld, ntok, V, labels, tid, tp, k, coef, ce_coef, loss_start, loss_end, kl_loss,
                   ce_loss, lse=None, stats=None, ce_mean=None, err=None, stream=None):
    _check("vl_ce_kl_fused", lib().vl_ce_kl_fused(
        _ptr(logits, "f32", "logits"), ld, ntok, V, _ptr(labels, "u32", "labels"), _ptr(tid, "u32", "tid"),
        _ptr(tp, "f32", "tp"), k, float(coef), float(ce_coef), loss_start, loss_end,
        _ptr(kl_loss, "f32", "kl_loss"), _ptr(ce_loss, "f32", "ce_loss"), _ptr(lse, "f32", "lse"),
        _ptr(stats, "f32", "stats"), _ptr(ce_mean, "f32", "ce_mean"), _ptr(err, "i32", "err"),
        _stream(stream)))


# bf16 logits: the same calls; `logits` a torch.bfloat16 tensor (or an int address of bf16 data)


def vl_ce_fwd_bf16(logits, ld, ntok, V, labels, loss_start, loss_end, loss, lse=None, stats=None, mean=None,
                   err=None, stream=None):
    _check("vl_ce_fwd_bf16", lib().vl_ce_fwd_bf16(
        _ptr(logits, "bf16", "logits"), ld, ntok, V, _ptr(labels, "u32", "labels"), loss_start, loss_end,
        _ptr(loss, "f32", "loss"), _ptr(lse, "f32", "lse"), _ptr(stats, "f32", "stats"),
        _ptr(mean, "f32", "mean"), _ptr(err, "i32", "err"), _stream(stream)))


def vl_ce_bwd_inplace_bf16(logits, ld, ntok, V, col0, ncols, labels, lse, stats, loss_start, loss_end, scale,
                           loss_part=None, err=None, stream=None):
    _check("vl_ce_bwd_inplace_bf16", lib().vl_ce_bwd_inplace_bf16(
        _ptr(logits, "bf16", "logits"), ld, ntok, V, col0, ncols, _ptr(labels, "u32", "labels"),
        _ptr(lse, "f32", "lse"), _ptr(stats, "f32", "stats"), loss_start, loss_end, float(scale),
        _ptr(loss_part, "f32", "loss_part"), _ptr(err, "i32", "err"), _stream(stream)))


def vl_ce_fused_bf16(logits, ld, ntok, V, labels, loss_start, loss_end, scale, loss, lse=None, stats=None,
                     mean=None, err=None, stream=None):
    _check("vl_ce_fused_bf16", lib().vl_ce_fused_bf16(
        _ptr(logits, "bf16", "logits"), ld, ntok, V, _ptr(labels, "u32", "labels"), loss_start, loss_end,
        float(scale), _ptr(loss, "f32", "loss"), _ptr(lse, "f32", "lse"), _ptr(stats, "f32", "stats"),
        _ptr(mean, "f32", "mean"), _ptr(err, "i32", "err"), _stream(stream)))


def vl_kl_topk_inplace_bf16(logits, ld, ntok, V, col0, ncols, tid, tp, k, coef, loss_start, loss_end,
                            lse_in=None, stats_in=None, labels=None, ce_coef=0.0, loss=None, err=None, stream=None):
    _check("vl_kl_topk_inplace_bf16", lib().vl_kl_topk_inplace_bf16(
        _ptr(logits, "bf16", "logits"), ld, ntok, V, col0, ncols, _ptr(tid, "u32", "tid"), _ptr(tp, "f32", "tp"),
        k, float(coef), loss_start, loss_end, _ptr(lse_in, "f32", "lse_in"), _ptr(stats_in, "f32", "stats_in"),
        _ptr(labels, "u32", "labels"), float(ce_coef), _ptr(loss, "f32", "loss"), _ptr(err, "i32", "err"),
        _stream(stream)))


def vl_ce_kl_fused_bf16(logits, ld, ntok, V, labels, tid, tp, k, coef, ce_coef, loss_start, loss_end, kl_loss,
                        ce_loss, lse=None, stats=None, ce_mean=None, err=None, stream=None):
    _check("vl_ce_kl_fused_bf16", lib().vl_ce_kl_fused_bf16(
        _ptr(logits, "bf16", "logits"), ld, ntok, V, _ptr(labels, "u32", "labels"), _ptr(tid, "u32", "tid"),
        _ptr(tp, "f32", "tp"), k, float(coef), float(ce_coef), loss_start, loss_end,
        _ptr(kl_loss, "f32", "kl_loss"), _ptr(ce_loss, "f32", "ce_loss"), _ptr(lse, "f32", "lse"),
        _ptr(stats, "f32", "stats"), _ptr(ce_mean, "f32", "ce_mean"), _ptr(err, "i32", "err"),
        _stream(stream)))


def vl_topk_workspace_bytes(ntok, V, k) -> int:
    return int(lib().vl_topk_workspace_bytes(ntok, V, k))


_topk_ws = {}


def topk_workspace(nbytes, device=None):
    """A cached device buffer of at least `nbytes` for vl_topk_rows on `device` (grown on
    demand).  One per device: calls that use it must not overlap on the GPU."""
    import torch
    dev = torch.cuda.current_device() if device is None else int(device)
    ws = _topk_ws.get(dev)
    if ws is None or ws.numel() < nbytes:
        ws = torch.empty(int(nbytes), dtype=torch.uint8, device=f"cuda:{dev}")
        _topk_ws[dev] = ws
    return ws


def vl_topk_rows(logits, ld, ntok, V, k, loss_start, loss_end, ids, probs, err=None, workspace="auto",
                 workspace_bytes=0, stream=None):
    """workspace: 'auto' (a cached buffer sized by vl_topk_workspace_bytes for the rows of
    the window), a tensor, an int address (with workspace_bytes) or None."""
    if isinstance(workspace, str):
        if workspace != "auto":
            raise ValueError("workspace: a tensor, an int address, None or 'auto'")
        need = vl_topk_workspace_bytes(max(1, loss_end - loss_start), V, k) if loss_end > loss_start else 0
        if need:
            import torch
            dev = logits.device.index if isinstance(logits, torch.Tensor) else None
            w = topk_workspace(need, dev)
            workspace, workspace_bytes = w.data_ptr(), need
        else:
            workspace, workspace_bytes = None, 0
    elif workspace is not None and not isinstance(workspace, int):
        workspace_bytes = workspace.numel() * workspace.element_size()
        workspace = workspace.data_ptr()
    _check("vl_topk_rows", lib().vl_topk_rows(
        _ptr(logits, "f32", "logits"), ld, ntok, V, k, loss_start, loss_end, _ptr(ids, "u32", "ids"),
        _ptr(probs, "f32", "probs"), _ptr(err, "i32", "err"), workspace, int(workspace_bytes), _stream(stream)))


def vl_window_mean(loss, ntok, loss_start, loss_end, mean, stream=None):
    _check("vl_window_mean", lib().vl_window_mean(_ptr(loss, "f32", "loss"), ntok, loss_start, loss_end,
                                                  _ptr(mean, "f32", "mean"), _stream(stream)))


def vl_acc_add(a, b, n, stream=None):
    _check("vl_acc_add", lib().vl_acc_add(_ptr(a, "f32", "a"), _ptr(b, "f32", "b"), n, _stream(stream)))


def vl_test_inject_wait_timeout(withhold_tile: int, wait_cycles: int):
    _check("vl_test_inject_wait_timeout", lib().vl_test_inject_wait_timeout(withhold_tile, wait_cycles))


def vl_watchdog_flag(device: int = 0, clear: bool = True) -> int:
    return lib().vl_watchdog_flag(device, 1 if clear else 0)


# ---------------------------------------------------------------- the vocabulary head


def _buf(ws, nbytes_auto, logits_like):
    """(address, bytes) of a workspace argument: 'auto' (a cached buffer of nbytes_auto), a tensor,
    or (address, bytes)."""
    if isinstance(ws, str):
        if ws != "auto":
            raise ValueError("workspace: a tensor, an int address or 'auto'")
        import torch
        dev = logits_like.device.index if isinstance(logits_like, torch.Tensor) else None
        w = topk_workspace(nbytes_auto, dev)
        return w.data_ptr(), int(nbytes_auto)
    if isinstance(ws, tuple):
        return int(ws[0]), int(ws[1])
    if isinstance(ws, int):
        raise ValueError("give a raw workspace as (address, bytes)")
    return ws.data_ptr(), ws.numel() * ws.element_size()


def vl_teacher_topk(hidden, hs, w, V, ntok, k, loss_start, loss_end, ids, probs, err=None, workspace="auto",
                    stream=None, chunk=1024):
    """hidden [ntok][hs] and w [V][hs]: torch.bfloat16 tensors (or int addresses).  With
    workspace='auto' a cached buffer for chunks of `chunk` rows."""
    rows = max(1, min(chunk, max(1, loss_end - loss_start)))
    ws, nb = _buf(workspace, int(lib().vl_teacher_topk_workspace_bytes(rows, V, k)), hidden)
    _check("vl_teacher_topk", lib().vl_teacher_topk(
        _ptr(hidden, "bf16", "hidden"), hs, _ptr(w, "bf16", "w"), V, ntok, k, loss_start, loss_end,
        _ptr(ids, "u32", "ids"), _ptr(probs, "f32", "probs"), _ptr(err, "i32", "err"), ws, nb, _stream(stream)))


def vl_head_kl(hidden, hs, w, wt, V, ntok, labels, tid, tp, k, coef, ce_coef, dx_scale, loss_start, loss_end, dx,
               kl_loss, ce_loss, ce_mean=None, err=None, workspace="auto", stream=None, chunk=1024):
    """The student's head step; hidden, w (and the transposed plane wt, or None) bf16
    tensors, dx fp32 [ntok][hs]."""
    rows = max(1, min(chunk, max(1, ntok)))
    ws, nb = _buf(workspace, int(lib().vl_head_kl_workspace_bytes(rows, V)), hidden)
    _check("vl_head_kl", lib().vl_head_kl(
        _ptr(hidden, "bf16", "hidden"), hs, _ptr(w, "bf16", "w"), _ptr(wt, "bf16", "wt"), V, ntok,
        _ptr(labels, "u32", "labels"),
        _ptr(tid, "u32", "tid"), _ptr(tp, "f32", "tp"), k, float(coef), float(ce_coef), float(dx_scale),
        loss_start, loss_end, _ptr(dx, "f32", "dx"), _ptr(kl_loss, "f32", "kl_loss"),
        _ptr(ce_loss, "f32", "ce_loss"), _ptr(ce_mean, "f32", "ce_mean"), _ptr(err, "i32", "err"), ws, nb,
        _stream(stream)))


def vl_gemm_bf16_tn(A, B, D, M, N, K, ldd, alpha=1.0, stream=None):
    """D[M][N] = alpha * A[M][K] . B[N][K]^T on the tensor cores; A, B bf16, D fp32."""
    _check("vl_gemm_bf16_tn", lib().vl_gemm_bf16_tn(_ptr(A, "bf16", "A"), _ptr(B, "bf16", "B"), _ptr(D, "f32", "D"),
                                                    M, N, K, ldd, float(alpha), _stream(stream)))


def vl_topk_rows_noalloc(logits, ld, ntok, V, k, loss_start, loss_end, ids, probs, err=None, stream=None):
    """vl_topk_rows with the library's fixed scratch array instead of a workspace: for callers
    that cannot allocate device memory at the point of the call (see include/vloss.h)."""
    _check("vl_topk_rows_noalloc", lib().vl_topk_rows_noalloc(
        _ptr(logits, "f32", "logits"), ld, ntok, V, k, loss_start, loss_end, _ptr(ids, "u32", "ids"),
        _ptr(probs, "f32", "probs"), _ptr(err, "i32", "err"), _stream(stream)))
