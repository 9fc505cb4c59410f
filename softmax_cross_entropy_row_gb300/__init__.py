"""Fused softmax cross-entropy forward + gradient on one GB300 GPU.

A thin binding over the C-ABI library ``libce.so`` (declared in
``include/ce.h``): each function marshals torch tensors into the pointers,
sizes and stream of the C call of the same name and turns a non-zero status
into an exception.  Every step of the computation runs in the library's
CUDA kernels; there is no CPU fallback: every call raises ImportError when
the library has not been built (``build()``).

The operation (the rumus project page, milestone M7a; the per-row steps of
Pass 1 and the reduction of Pass 2 of rumus 0.1.1's cross_entropy.wgsl):

    loss = (1/B) * sum_b (logsumexp(z_b) - z_b[t_b])
    grad = (softmax(z_b) - onehot(t_b)) / B

and, through ce_fwd_bwd_ex / ce_forward, the sum and per-row reductions, an
upstream gradient fused into the gradient's write, and the loss alone.
"""

from __future__ import annotations

import ctypes
import os

from .build import LIB, build  # noqa: F401

CE_F32 = 0
CE_BF16 = 1
CE_F16 = 2

CE_PATH_AUTO = 0
CE_PATH_ROWS_WARP = 1
CE_PATH_ROW_SPLIT = 2
CE_PATH_STREAM = 3
CE_PATH_ROW_TWOPASS = 4
CE_PATH_ROWS_ONLINE = 5

CE_REDUCE_MEAN = 0
CE_REDUCE_SUM = 1
CE_REDUCE_NONE = 2

PATH_NAMES = {CE_PATH_ROWS_WARP: "rows_warp", CE_PATH_ROW_SPLIT: "row_split",
              CE_PATH_STREAM: "stream", CE_PATH_ROW_TWOPASS: "row_twopass",
              CE_PATH_ROWS_ONLINE: "rows_online"}

STATUS = {0: "CE_OK", 1: "CE_ERR_NULL", 2: "CE_ERR_SHAPE", 3: "CE_ERR_DTYPE",
          4: "CE_ERR_ALIGN", 5: "CE_ERR_CUDA", 6: "CE_ERR_OVERLAP", 7: "CE_ERR_POINTER",
          8: "CE_ERR_CAPTURE", 9: "CE_ERR_PATH", 10: "CE_ERR_SCRATCH", 11: "CE_ERR_REDUCTION"}

# Symbols declared in include/ce.h.
EXPORTS = ("ce_fwd_bwd", "ce_fwd_bwd_path", "ce_query_plan", "ce_get_device_errors",
           "ce_release_workspaces", "ce_status_string", "ce_last_cuda_error",
           "ce_fwd_bwd_noalloc", "ce_fwd_bwd_ex", "ce_fwd_bwd_ex_path", "ce_forward",
           "ce_softmax_fwd", "ce_softmax_fwd_path", "ce_softmax_bwd", "ce_fwd_bwd_host",
           "ce_fwd_bwd_host_grad")
# Symbols declared in include/ce_testing.h (test hooks).
TEST_EXPORTS = ("ce_fwd_bwd_test",)


class TestHooks(ctypes.Structure):
    """ce_test_hooks of include/ce_testing.h."""

    _fields_ = [("skip_copy_row", ctypes.c_int64), ("wait_limit_cycles", ctypes.c_int64),
                ("grad_f32_out", ctypes.c_void_p)]


class CEError(RuntimeError):
    """A non-zero ce_status from the library."""

    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


_lib = None


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Load libce.so (no CUDA call is made by loading it)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB
    if not os.path.exists(p):
        raise ImportError(f"{p} is missing: build it with softmax_cross_entropy_row_gb300.build()")
    lib = ctypes.CDLL(p)
    i64, vp, ci = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
    pi = ctypes.POINTER(ctypes.c_int)
    lib.ce_fwd_bwd.argtypes = [vp, vp, i64, i64, ci, vp, vp, vp]
    lib.ce_fwd_bwd.restype = ci
    lib.ce_fwd_bwd_path.argtypes = [vp, vp, i64, i64, ci, vp, vp, vp, ci, ci]
    lib.ce_fwd_bwd_path.restype = ci
    lib.ce_query_plan.argtypes = [i64, i64, ci, pi, pi, pi, pi, pi, pi]
    lib.ce_query_plan.restype = ci
    lib.ce_get_device_errors.argtypes = [vp, ctypes.POINTER(ctypes.c_int32),
                                         ctypes.POINTER(ctypes.c_int32)]
    lib.ce_get_device_errors.restype = ci
    lib.ce_release_workspaces.argtypes = []
    lib.ce_release_workspaces.restype = ci
    lib.ce_status_string.argtypes = [ci]
    lib.ce_status_string.restype = ctypes.c_char_p
    lib.ce_last_cuda_error.argtypes = []
    lib.ce_last_cuda_error.restype = ctypes.c_char_p
    lib.ce_fwd_bwd_noalloc.argtypes = [vp, vp, i64, i64, ci, vp, vp, vp]
    lib.ce_fwd_bwd_noalloc.restype = ci
    lib.ce_fwd_bwd_ex.argtypes = [vp, vp, i64, i64, ci, ci, vp, vp, vp, vp]
    lib.ce_fwd_bwd_ex.restype = ci
    lib.ce_fwd_bwd_ex_path.argtypes = [vp, vp, i64, i64, ci, ci, vp, vp, vp, vp, ci, ci]
    lib.ce_fwd_bwd_ex_path.restype = ci
    lib.ce_forward.argtypes = [vp, vp, i64, i64, ci, ci, vp, vp]
    lib.ce_forward.restype = ci
    lib.ce_softmax_fwd.argtypes = [vp, i64, i64, ci, vp, vp]
    lib.ce_softmax_fwd.restype = ci
    lib.ce_fwd_bwd_host.argtypes = [vp, vp, i64, i64, ci, vp, vp, vp]
    lib.ce_fwd_bwd_host.restype = ci
    lib.ce_fwd_bwd_host_grad.argtypes = [vp, vp, i64, i64, ci, vp, vp, vp]
    lib.ce_fwd_bwd_host_grad.restype = ci
    lib.ce_softmax_fwd_path.argtypes = [vp, i64, i64, ci, vp, vp, ci, ci]
    lib.ce_softmax_fwd_path.restype = ci
    lib.ce_softmax_bwd.argtypes = [vp, vp, i64, i64, ci, vp, vp]
    lib.ce_softmax_bwd.restype = ci
    lib.ce_fwd_bwd_test.argtypes = [vp, vp, i64, i64, ci, vp, vp, vp, ci, ci,
                                    ctypes.POINTER(TestHooks)]
    lib.ce_fwd_bwd_test.restype = ci
    if path is None:
        _lib = lib
    return lib


def _check(rc: int) -> None:
    if rc != 0:
        lib = load_library()
        msg = lib.ce_status_string(rc).decode()
        if rc == 5:
            msg += ": " + lib.ce_last_cuda_error().decode()
        raise CEError(rc, msg)


def _dtype_code(t) -> int:
    import torch

    if t.dtype == torch.float32:
        return CE_F32
    if t.dtype == torch.bfloat16:
        return CE_BF16
    if t.dtype == torch.float16:
        return CE_F16
    raise TypeError(f"logits must be float32, bfloat16 or float16, got {t.dtype}")


def _stream_handle(stream) -> int:
    import torch

    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _ptr(t) -> int:
    return 0 if t is None else t.data_ptr()


def _check_io(logits, targets, loss_out, reduction=CE_REDUCE_MEAN, grad_scale=None,
              device="cuda") -> None:
    """Types, sizes and placement of the tensors a call reads or writes: the
    C layer receives plain pointers and cannot check how large they are."""
    import torch

    B = logits.shape[0]
    n = B if reduction == CE_REDUCE_NONE else 1
    for name, t in (("logits", logits), ("targets", targets), ("loss_out", loss_out),
                    ("grad_scale", grad_scale)):
        if t is not None and t.device.type != device:
            raise ValueError(f"{name} must be a {device.upper()} tensor")
    if (targets is None or targets.dtype != torch.int32 or targets.dim() != 1
            or targets.numel() != B or not targets.is_contiguous()):
        raise ValueError("targets must be a contiguous [B] int32 tensor")
    if (loss_out is None or loss_out.dtype != torch.float32 or loss_out.numel() < n
            or not loss_out.is_contiguous()):
        raise ValueError(f"loss_out must be a contiguous float32 tensor of at least {n} element(s)")
    if grad_scale is not None and (grad_scale.dtype != torch.float32 or grad_scale.numel() != n
                                   or not grad_scale.is_contiguous()):
        raise ValueError(f"grad_scale must be a contiguous float32 tensor of {n} element(s)")


def ce_fwd_bwd(logits, targets, loss_out, grad_out, stream=None) -> None:
    """Loss (one fp32 on the device) and gradient of softmax cross-entropy.

    logits   [B, C] float32, bfloat16 or float16 CUDA tensor, contiguous
    targets  [B] int32 CUDA tensor
    loss_out one-element float32 CUDA tensor
    grad_out [B, C] CUDA tensor of the logits' dtype, contiguous
    stream   torch.cuda.Stream, raw cudaStream_t int, or None (current stream)
    """
    ce_fwd_bwd_path(logits, targets, loss_out, grad_out, stream, CE_PATH_AUTO, 0)


def ce_fwd_bwd_path(logits, targets, loss_out, grad_out, stream=None, path=CE_PATH_AUTO,
                    split=0) -> None:
    """ce_fwd_bwd with the kernel path (and split) forced."""
    lib = load_library()
    if logits.dim() != 2 or not logits.is_contiguous():
        raise ValueError("logits must be a contiguous [B, C] tensor")
    if grad_out.shape != logits.shape or grad_out.dtype != logits.dtype or not grad_out.is_contiguous():
        raise ValueError("grad_out must be a contiguous tensor of the logits' shape and dtype")
    _check_io(logits, targets, loss_out)
    B, C = logits.shape
    _check(lib.ce_fwd_bwd_path(_ptr(logits), _ptr(targets), B, C, _dtype_code(logits),
                               _ptr(loss_out), _ptr(grad_out), _stream_handle(stream),
                               int(path), int(split)))


def ce_fwd_bwd_ex(logits, targets, loss_out, grad_out=None, reduction=CE_REDUCE_MEAN,
                  grad_scale=None, stream=None, path=CE_PATH_AUTO, split=0) -> None:
    """ce_fwd_bwd with a reduction (CE_REDUCE_MEAN / SUM / NONE), an optional
    upstream gradient ``grad_scale`` (a one-element fp32 CUDA tensor for the
    mean and sum, a [B] one for NONE) and an optional ``grad_out`` (None: the
    loss alone).  ``loss_out`` holds one fp32 (mean, sum) or B (none)."""
    lib = load_library()
    if logits.dim() != 2 or not logits.is_contiguous():
        raise ValueError("logits must be a contiguous [B, C] tensor")
    if grad_out is not None and (grad_out.shape != logits.shape or grad_out.dtype != logits.dtype
                                 or not grad_out.is_contiguous()):
        raise ValueError("grad_out must be a contiguous tensor of the logits' shape and dtype")
    _check_io(logits, targets, loss_out, reduction, grad_scale)
    B, C = logits.shape
    _check(lib.ce_fwd_bwd_ex_path(_ptr(logits), _ptr(targets), B, C, _dtype_code(logits),
                                  int(reduction), _ptr(grad_scale), _ptr(loss_out),
                                  _ptr(grad_out), _stream_handle(stream), int(path), int(split)))


def ce_forward(logits, targets, loss_out, reduction=CE_REDUCE_MEAN, stream=None) -> None:
    """The loss alone (no gradient): one fp32 (mean, sum) or [B] (none)."""
    lib = load_library()
    if logits.dim() != 2 or not logits.is_contiguous():
        raise ValueError("logits must be a contiguous [B, C] tensor")
    _check_io(logits, targets, loss_out, reduction)
    B, C = logits.shape
    _check(lib.ce_forward(_ptr(logits), _ptr(targets), B, C, _dtype_code(logits),
                          int(reduction), _ptr(loss_out), _stream_handle(stream)))


def ce_fwd_bwd_host(logits_host, targets_host, loss_host, grad_out, stream=None) -> None:
    """ce_fwd_bwd with the logits, targets and loss in host memory (CPU
    tensors, page-locked for asynchronous copies); the gradient goes to the CUDA
    tensor ``grad_out``.  ``loss_host`` is written when ``stream`` reaches the
    end of the call."""
    lib = load_library()
    if logits_host.dim() != 2 or not logits_host.is_contiguous():
        raise ValueError("logits_host must be a contiguous [B, C] tensor")
    if grad_out.shape != logits_host.shape or grad_out.dtype != logits_host.dtype or \
            not grad_out.is_contiguous():
        raise ValueError("grad_out must be a contiguous tensor of the logits' shape and dtype")
    _check_io(logits_host, targets_host, loss_host, device="cpu")
    if grad_out.device.type != "cuda":
        raise ValueError("grad_out must be a CUDA tensor")
    B, C = logits_host.shape
    _check(lib.ce_fwd_bwd_host(_ptr(logits_host), _ptr(targets_host), B, C,
                               _dtype_code(logits_host), _ptr(loss_host), _ptr(grad_out),
                               _stream_handle(stream)))


def ce_fwd_bwd_host_grad(logits_host, targets_host, loss_host, grad_host, stream=None) -> None:
    """ce_fwd_bwd with the logits, targets, loss and gradient all in host memory
    (CPU tensors, page-locked for asynchronous copies).  The outputs are
    written when ``stream`` reaches the end of the call."""
    lib = load_library()
    if logits_host.dim() != 2 or not logits_host.is_contiguous():
        raise ValueError("logits_host must be a contiguous [B, C] tensor")
    if grad_host.shape != logits_host.shape or grad_host.dtype != logits_host.dtype or \
            not grad_host.is_contiguous():
        raise ValueError("grad_host must be a contiguous tensor of the logits' shape and dtype")
    _check_io(logits_host, targets_host, loss_host, device="cpu")
    if grad_host.device.type != "cpu":
        raise ValueError("grad_host must be a CPU tensor")
    B, C = logits_host.shape
    _check(lib.ce_fwd_bwd_host_grad(_ptr(logits_host), _ptr(targets_host), B, C,
                                    _dtype_code(logits_host), _ptr(loss_host), _ptr(grad_host),
                                    _stream_handle(stream)))


def ce_softmax_fwd(logits, probs_out, stream=None, path=CE_PATH_AUTO, split=0) -> None:
    """Row-wise softmax of a contiguous [B, C] tensor into ``probs_out`` (same
    shape and dtype); ``path`` / ``split`` force a kernel as for ce_fwd_bwd_path."""
    lib = load_library()
    if logits.dim() != 2 or not logits.is_contiguous():
        raise ValueError("logits must be a contiguous [B, C] tensor")
    if probs_out.shape != logits.shape or probs_out.dtype != logits.dtype or not probs_out.is_contiguous():
        raise ValueError("probs_out must be a contiguous tensor of the logits' shape and dtype")
    B, C = logits.shape
    _check(lib.ce_softmax_fwd_path(_ptr(logits), B, C, _dtype_code(logits), _ptr(probs_out),
                                   _stream_handle(stream), int(path), int(split)))


def ce_softmax_bwd(probs, dy, dx_out, stream=None) -> None:
    """dx = p * (dy - sum(p * dy, row)) for contiguous [B, C] tensors of one dtype."""
    lib = load_library()
    for name, t in (("probs", probs), ("dy", dy), ("dx_out", dx_out)):
        if t.dim() != 2 or not t.is_contiguous() or t.shape != probs.shape or t.dtype != probs.dtype:
            raise ValueError(f"{name} must be a contiguous tensor of the probabilities' shape and dtype")
    B, C = probs.shape
    _check(lib.ce_softmax_bwd(_ptr(probs), _ptr(dy), B, C, _dtype_code(probs), _ptr(dx_out),
                              _stream_handle(stream)))


def ce_fwd_bwd_raw(logits_ptr: int, targets_ptr: int, B: int, C: int, dtype: int,
                   loss_ptr: int, grad_ptr: int, stream: int = 0, path: int = CE_PATH_AUTO,
                   split: int = 0) -> int:
    """The C call with raw integer pointers; returns the ce_status (no raise)."""
    return load_library().ce_fwd_bwd_path(logits_ptr, targets_ptr, B, C, dtype, loss_ptr,
                                          grad_ptr, stream, path, split)


def ce_fwd_bwd_noalloc(logits, targets, loss_out, grad_out, stream=None) -> None:
    """ce_fwd_bwd without any device allocation, for callers that cannot call
    cudaMalloc (a memory manager owns the device, a fixed memory budget, or no
    tolerance for the synchronisation an allocation can cause).  Its scratch
    is a static device array of the library (B <= 262144); calls that overlap
    on the GPU share it and race.  Make the first call on a device before any
    stream capture."""
    lib = load_library()
    if logits.dim() != 2 or not logits.is_contiguous():
        raise ValueError("logits must be a contiguous [B, C] tensor")
    if grad_out.shape != logits.shape or grad_out.dtype != logits.dtype or not grad_out.is_contiguous():
        raise ValueError("grad_out must be a contiguous tensor of the logits' shape and dtype")
    _check_io(logits, targets, loss_out)
    B, C = logits.shape
    _check(lib.ce_fwd_bwd_noalloc(_ptr(logits), _ptr(targets), B, C, _dtype_code(logits),
                                  _ptr(loss_out), _ptr(grad_out), _stream_handle(stream)))


def ce_fwd_bwd_test(logits, targets, loss_out, grad_out, stream=None, path=CE_PATH_AUTO, split=0,
                    skip_copy_row=-1, wait_limit_cycles=0, grad_f32_out=None) -> None:
    """ce_fwd_bwd_path with the test hooks of include/ce_testing.h: leave out
    the copy of one row (its bounded wait must give up), shorten the copy
    waits, or record the fp32 gradient before rounding (``grad_f32_out``, a
    contiguous float32 CUDA tensor of the logits' shape).  Tests only."""
    lib = load_library()
    if logits.dim() != 2 or not logits.is_contiguous():
        raise ValueError("logits must be a contiguous [B, C] tensor")
    if grad_out.shape != logits.shape or grad_out.dtype != logits.dtype or not grad_out.is_contiguous():
        raise ValueError("grad_out must be a contiguous tensor of the logits' shape and dtype")
    _check_io(logits, targets, loss_out)
    import torch

    if grad_f32_out is not None and (grad_f32_out.shape != logits.shape or not
                                     grad_f32_out.is_contiguous() or
                                     grad_f32_out.dtype != torch.float32):
        raise ValueError("grad_f32_out must be a contiguous float32 tensor of the logits' shape")
    hooks = TestHooks(int(skip_copy_row), int(wait_limit_cycles), _ptr(grad_f32_out) or None)
    B, C = logits.shape
    _check(lib.ce_fwd_bwd_test(_ptr(logits), _ptr(targets), B, C, _dtype_code(logits),
                               _ptr(loss_out), _ptr(grad_out), _stream_handle(stream), int(path),
                               int(split), ctypes.byref(hooks)))


def ce_query_plan(B: int, C: int, dtype: int) -> dict:
    lib = load_library()
    vals = [ctypes.c_int(0) for _ in range(6)]
    _check(lib.ce_query_plan(B, C, dtype, *[ctypes.byref(v) for v in vals]))
    path, split, ctas, threads, smem, launches = (v.value for v in vals)
    return {"path": path, "path_name": PATH_NAMES.get(path, "?"), "split": split, "ctas": ctas,
            "threads": threads, "smem_bytes": smem, "launches": launches}


def ce_get_device_errors(stream=None) -> tuple[int, int]:
    """(rows with an out-of-range target, waits that gave up) since the last read."""
    lib = load_library()
    bad, tmo = ctypes.c_int32(0), ctypes.c_int32(0)
    _check(lib.ce_get_device_errors(_stream_handle(stream), ctypes.byref(bad), ctypes.byref(tmo)))
    return bad.value, tmo.value


def ce_release_workspaces() -> None:
    _check(load_library().ce_release_workspaces())


def cross_entropy_fwd_bwd(logits, targets, stream=None):
    """Allocate the outputs and run ce_fwd_bwd; returns (loss [1] fp32, grad)."""
    import torch

    loss = torch.empty(1, dtype=torch.float32, device=logits.device)
    grad = torch.empty_like(logits)
    ce_fwd_bwd(logits, targets, loss, grad, stream)
    return loss, grad
