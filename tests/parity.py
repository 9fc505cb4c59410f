"""Shared helpers of the GPU parity tests: move seeded inputs to the device,
call the library through its C-ABI binding, and compare with the fp64 oracle
at the tolerances the method's targets state:

  fp32 logits:  |L - L_ref| <= 1e-5 |L_ref| (+1e-7 for L near 0)
                |g - g_ref| <= 1e-6 / B per element
                |sum_c g|   <= 1e-6 / B per row
  bf16 / f16 logits:  the same loss bound, against the oracle run on the
                16-bit values;
                |g - g_ref| <= 1 ulp of g_ref in the logits' type (0 allowed for
                |g_ref| < 2^-126, the kernels flush subnormal fp32 results)
                |sum_c g|   <= 1e-6 / B + sum_c ulp(g_c) / 2 per row (the bf16
                rounding of each element; checked on the fp32 path exactly)
"""

from __future__ import annotations

import numpy as np

import oracle

LOSS_RTOL = 1e-5
LOSS_ATOL = 1e-7
GRAD_ATOL_TIMES_B = 1e-6
ROWSUM_ATOL_TIMES_B = 1e-6


def device_inputs(inp, device="cuda"):
    import torch

    if inp.workload.dtype == "bf16":
        z = torch.from_numpy(inp.logits.view(np.int16)).view(torch.bfloat16).to(device)
    else:
        z = torch.from_numpy(inp.logits).to(device)
    t = torch.from_numpy(inp.targets).to(device)
    return z, t


def run(z, t, path=0, split=0, stream=None):
    import torch

    import softmax_cross_entropy_row_gb300 as ce

    loss = torch.full((1,), float("nan"), dtype=torch.float32, device=z.device)
    grad = torch.empty_like(z)
    ce.ce_fwd_bwd_path(z, t, loss, grad, stream, path, split)
    return loss, grad


def grad_rows_host(grad, rows=None) -> np.ndarray:
    """fp64 copy of gradient rows (all rows when rows is None)."""
    import torch

    g = grad if rows is None else grad.index_select(
        0, torch.as_tensor(np.asarray(rows), dtype=torch.int64, device=grad.device))
    return g.float().cpu().numpy().astype(np.float64)


def ulp_bf16(x: np.ndarray) -> np.ndarray:
    ax = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(ax, 2.0 ** -126)))
    return np.exp2(e - 7)


def ulp_f16(x: np.ndarray) -> np.ndarray:
    """Spacing of IEEE binary16 values in x's binade (2^-24 below 2^-14)."""
    ax = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(ax, 2.0 ** -14)))
    return np.exp2(e - 10)


def check_loss(L: float, L_ref: float) -> None:
    if np.isnan(L_ref):
        assert np.isnan(L), f"loss {L}, expected NaN"
        return
    err = abs(L - L_ref)
    assert err <= LOSS_RTOL * abs(L_ref) + LOSS_ATOL, f"loss {L!r} vs oracle {L_ref!r} (err {err:.3g})"


def check_grad(g: np.ndarray, g_ref: np.ndarray, B: int, dtype: str, what: str = "",
               valid=None) -> None:
    """``valid`` marks rows whose target is in range (default: all); a row with
    an out-of-range target has no one-hot term, so it sums to 1/B instead of 0."""
    assert g.shape == g_ref.shape
    valid = np.ones(g.shape[0], dtype=bool) if valid is None else np.asarray(valid, dtype=bool)
    target_sum = np.where(valid, 0.0, 1.0 / B)
    if dtype == "f32":
        err = np.abs(g - g_ref)
        worst = float(err.max()) * B if err.size else 0.0
        assert worst <= GRAD_ATOL_TIMES_B, f"{what}: max |g - g_ref| = {worst:.3g}/B"
        rs = np.abs(g.sum(axis=1) - target_sum) * B
        assert float(rs.max()) <= ROWSUM_ATOL_TIMES_B, f"{what}: row sum {float(rs.max()):.3g}/B"
    else:
        ulp = ulp_f16 if dtype == "f16" else ulp_bf16
        tol = ulp(g_ref)
        flushed = (g == 0) & (np.abs(g_ref) < 2.0 ** -126)
        bad = (np.abs(g - g_ref) > tol) & ~flushed
        if bad.any():
            i = np.argwhere(bad)[0]
            raise AssertionError(f"{what}: {int(bad.sum())} bf16 grads beyond 1 ulp, first at "
                                 f"{tuple(i)}: {g[tuple(i)]!r} vs {g_ref[tuple(i)]!r}")
        rs = np.abs(g.sum(axis=1) - target_sum)
        bound = ROWSUM_ATOL_TIMES_B / B + 0.5 * ulp(g).sum(axis=1)
        assert np.all(rs <= bound), f"{what}: {dtype} row sum beyond its rounding bound"


def check_full(inp, loss, grad, what: str = "") -> None:
    """Element-by-element comparison of a whole (small) batch."""
    L_ref, _, g_ref = oracle.loss_and_grad(inp.logits, inp.targets)
    check_loss(float(loss.item()), L_ref)
    valid = (inp.targets >= 0) & (inp.targets < inp.workload.C)
    check_grad(grad_rows_host(grad), g_ref, inp.workload.B, inp.workload.dtype, what, valid)


def check_all_rows(inp, loss, grad, what: str = "", block: int = 256) -> None:
    """Full-size check of every element: L against the oracle over every row,
    then the gradient compared element by element with the oracle's, streamed
    through the oracle in blocks of rows (an fp64 [B, C] of the largest
    workloads would not fit in host memory at once)."""
    B, C = inp.workload.B, inp.workload.C
    l_all = oracle.rows(inp.logits, inp.targets, grad=False)
    check_loss(float(loss.item()), oracle.batch_loss(l_all))
    valid = (inp.targets >= 0) & (inp.targets < C)
    for r0 in range(0, B, block):
        r1 = min(B, r0 + block)
        _, g_ref = oracle.rows(inp.logits, inp.targets, row_ids=np.arange(r0, r1))
        g = grad[r0:r1].float().cpu().numpy().astype(np.float64)
        check_grad(g, g_ref, B, inp.workload.dtype, f"{what} rows {r0}..{r1 - 1}", valid[r0:r1])
