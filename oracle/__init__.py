"""fp64 CPU oracle of the fused softmax cross-entropy forward + gradient.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers.  The product path (the
``softmax_cross_entropy_row_gb300`` package and its CUDA library) never
imports, links or runs anything here, and nothing here imports it.

The arithmetic lives in ``ce_oracle.c`` (plain C, double precision, one loop
per step of the rumus ``cross_entropy.wgsl`` Pass 1 and Pass 2); this module
compiles it with gcc and marshals numpy arrays through ctypes.

Pinned by ``tests/test_oracle.py`` against closed forms, invariants, an
independent multi-precision restatement and finite differences; no function
here is "parity unpinned".
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ce_oracle.c")
_LIB = os.path.join(_HERE, "libce_oracle.so")
_lock = threading.Lock()
_lib = None

F32 = 0
BF16 = 1
F16 = 2


def build(force: bool = False) -> str:
    """Compile ce_oracle.c into libce_oracle.so next to it (gcc, -O2, OpenMP)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True, text=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, vp = ctypes.c_int64, ctypes.c_void_p
            lib.ce_oracle_rows.argtypes = [vp, ctypes.c_int, vp, i64, i64, vp, i64, vp, vp]
            lib.ce_oracle_rows.restype = ctypes.c_int
            lib.ce_oracle_batch_loss.argtypes = [vp, i64]
            lib.ce_oracle_rows_ex.argtypes = [vp, ctypes.c_int, vp, i64, i64, ctypes.c_int, vp,
                                              vp, i64, vp, vp]
            lib.ce_oracle_rows_ex.restype = ctypes.c_int
            lib.ce_oracle_reduce.argtypes = [vp, i64, ctypes.c_int]
            lib.ce_oracle_reduce.restype = ctypes.c_double
            lib.ce_oracle_softmax.argtypes = [vp, ctypes.c_int, i64, i64, vp, i64, vp]
            lib.ce_oracle_softmax.restype = ctypes.c_int
            lib.ce_oracle_softmax_bwd.argtypes = [vp, vp, ctypes.c_int, i64, i64, vp, i64, vp]
            lib.ce_oracle_softmax_bwd.restype = ctypes.c_int
            lib.ce_oracle_batch_loss.restype = ctypes.c_double
            lib.ce_oracle_fwd_bwd.argtypes = [vp, ctypes.c_int, vp, i64, i64, vp, vp, vp]
            lib.ce_oracle_fwd_bwd.restype = ctypes.c_int
            lib.ce_oracle_threads.argtypes = []
            lib.ce_oracle_threads.restype = ctypes.c_int
            lib.ce_oracle_set_threads.argtypes = [ctypes.c_int]
            lib.ce_oracle_set_threads.restype = None
            _lib = lib
    return _lib


def _dtype_code(logits: np.ndarray) -> int:
    if logits.dtype == np.float32:
        return F32
    if logits.dtype == np.uint16:  # bf16 bit patterns
        return BF16
    if logits.dtype == np.float16:
        return F16
    raise TypeError(f"oracle logits must be float32, uint16 (bf16 bits) or float16, got {logits.dtype}")


def rows(logits: np.ndarray, targets: np.ndarray, row_ids=None, grad: bool = True):
    """Per-row losses l_b (fp64) and, if ``grad``, fp64 gradient rows.

    ``logits`` is ``[B, C]`` float32 or uint16 bf16 bits, C-contiguous;
    ``targets`` is int32 ``[B]``; ``row_ids`` selects rows (default: all).
    The gradient rows carry the 1/B factor of the full batch of B rows.
    """
    lib = _load()
    logits = np.ascontiguousarray(logits)
    targets = np.ascontiguousarray(targets, dtype=np.int32)
    B, C = logits.shape
    if targets.shape != (B,):
        raise ValueError("targets must have shape [B]")
    if row_ids is None:
        ids_ptr, n = None, B
    else:
        ids = np.ascontiguousarray(row_ids, dtype=np.int64)
        ids_ptr, n = ids.ctypes.data, ids.size
    loss = np.empty(n, dtype=np.float64)
    g = np.empty((n, C), dtype=np.float64) if grad else None
    rc = lib.ce_oracle_rows(logits.ctypes.data, _dtype_code(logits), targets.ctypes.data,
                            B, C, ids_ptr, n, loss.ctypes.data,
                            None if g is None else g.ctypes.data)
    if rc != 0:
        raise ValueError("ce_oracle_rows rejected its arguments")
    return (loss, g) if grad else loss


MEAN, SUM, NONE = 0, 1, 2


def rows_ex(logits: np.ndarray, targets: np.ndarray, reduction: int, upstream=None,
            row_ids=None, grad: bool = True):
    """Per-row losses and fp64 gradient rows for a reduction (MEAN, SUM, NONE)
    and an upstream gradient ``upstream`` (None = 1; one value for MEAN and
    SUM, [B] values for NONE): the gradient is upstream * dL/dz."""
    lib = _load()
    logits = np.ascontiguousarray(logits)
    targets = np.ascontiguousarray(targets, dtype=np.int32)
    B, C = logits.shape
    if targets.shape != (B,):
        raise ValueError("targets must have shape [B]")
    up = None
    if upstream is not None:
        up = np.ascontiguousarray(np.atleast_1d(np.asarray(upstream, dtype=np.float64)))
        if up.size != (B if reduction == NONE else 1):
            raise ValueError("upstream must hold one value (mean, sum) or B values (none)")
    if row_ids is None:
        ids_ptr, n = None, B
    else:
        ids = np.ascontiguousarray(row_ids, dtype=np.int64)
        ids_ptr, n = ids.ctypes.data, ids.size
    loss = np.empty(n, dtype=np.float64)
    g = np.empty((n, C), dtype=np.float64) if grad else None
    rc = lib.ce_oracle_rows_ex(logits.ctypes.data, _dtype_code(logits), targets.ctypes.data,
                               B, C, int(reduction), None if up is None else up.ctypes.data,
                               ids_ptr, n, loss.ctypes.data, None if g is None else g.ctypes.data)
    if rc != 0:
        raise ValueError("ce_oracle_rows_ex rejected its arguments")
    return (loss, g) if grad else loss


def reduce(loss_rows: np.ndarray, reduction: int) -> float:
    """Pass 2 for MEAN ((sum l_b) / B) or SUM (sum l_b), in row order, fp64."""
    lr = np.ascontiguousarray(loss_rows, dtype=np.float64)
    return float(_load().ce_oracle_reduce(lr.ctypes.data, lr.size, int(reduction)))


def _row_ids(B, row_ids):
    if row_ids is None:
        return None, B, None
    ids = np.ascontiguousarray(row_ids, dtype=np.int64)
    return ids.ctypes.data, ids.size, ids


def softmax(logits: np.ndarray, row_ids=None) -> np.ndarray:
    """Row-wise softmax in fp64 ([B, C] or the listed rows)."""
    lib = _load()
    logits = np.ascontiguousarray(logits)
    B, C = logits.shape
    ptr, n, keep = _row_ids(B, row_ids)
    out = np.empty((n, C), dtype=np.float64)
    if lib.ce_oracle_softmax(logits.ctypes.data, _dtype_code(logits), B, C, ptr, n,
                             out.ctypes.data) != 0:
        raise ValueError("ce_oracle_softmax rejected its arguments")
    return out


def softmax_bwd(probs: np.ndarray, dy: np.ndarray, row_ids=None) -> np.ndarray:
    """dx = p * (dy - sum(p * dy)) per row in fp64; p and dy of one element type."""
    lib = _load()
    probs = np.ascontiguousarray(probs)
    dy = np.ascontiguousarray(dy)
    if probs.shape != dy.shape or probs.dtype != dy.dtype:
        raise ValueError("probs and dy must have one shape and element type")
    B, C = probs.shape
    ptr, n, keep = _row_ids(B, row_ids)
    out = np.empty((n, C), dtype=np.float64)
    if lib.ce_oracle_softmax_bwd(probs.ctypes.data, dy.ctypes.data, _dtype_code(probs), B, C,
                                 ptr, n, out.ctypes.data) != 0:
        raise ValueError("ce_oracle_softmax_bwd rejected its arguments")
    return out


def batch_loss(loss_rows: np.ndarray) -> float:
    """L = (sum_b l_b) / B, summed in row order in fp64."""
    lr = np.ascontiguousarray(loss_rows, dtype=np.float64)
    return float(_load().ce_oracle_batch_loss(lr.ctypes.data, lr.size))


def loss_and_grad(logits: np.ndarray, targets: np.ndarray):
    """(L, l [B], g [B, C]) in fp64 for a whole (small) batch."""
    l, g = rows(logits, targets)
    return batch_loss(l), l, g


def fwd_bwd(logits: np.ndarray, targets: np.ndarray, grad_out: np.ndarray,
            row_scratch: np.ndarray) -> float:
    """Forward + gradient with the gradient narrowed to the logits' type.

    ``grad_out`` has the logits' shape and type; ``row_scratch`` holds B
    doubles.  Returns L.  This is the call the CPU baseline times.
    """
    lib = _load()
    B, C = logits.shape
    out = ctypes.c_double(0.0)
    rc = lib.ce_oracle_fwd_bwd(logits.ctypes.data, _dtype_code(logits), targets.ctypes.data,
                               B, C, ctypes.addressof(out), grad_out.ctypes.data,
                               row_scratch.ctypes.data)
    if rc != 0:
        raise ValueError("ce_oracle_fwd_bwd rejected its arguments")
    return out.value


def threads() -> int:
    return int(_load().ce_oracle_threads())


def set_threads(n: int) -> None:
    _load().ce_oracle_set_threads(int(n))
