"""The allocation-free entry point, ce_fwd_bwd_noalloc.

Some callers cannot call cudaMalloc: a memory manager owns the whole device,
the device memory budget is fixed at start-up, or the caller must never stall
on the synchronisation an allocation can cause.  ce_fwd_bwd_noalloc serves
them with a statically sized scratch array inside the library.  This file is
collected last, so a run that stops at the first failure has run every other
test before it; it passes on its own in a fresh process as well.
"""

import numpy as np
import pytest

import workloads as wl

from parity import GRAD_ATOL_TIMES_B, check_loss, device_inputs, ulp_bf16

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU-only machines
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import softmax_cross_entropy_row_gb300 as ce  # noqa: E402

CE_ERR_SCRATCH = 10


@pytest.fixture(scope="module", autouse=True)
def _built():
    ce.build()
    ce.load_library()


def _both(inp):
    z, t = device_inputs(inp)
    ref_loss = torch.empty(1, dtype=torch.float32, device="cuda")
    ref_grad = torch.empty_like(z)
    ce.ce_fwd_bwd(z, t, ref_loss, ref_grad)
    loss = torch.full((1,), float("nan"), dtype=torch.float32, device="cuda")
    grad = torch.full_like(z, float("nan"))
    ce.ce_fwd_bwd_noalloc(z, t, loss, grad)
    torch.cuda.synchronize()
    return ref_loss, ref_grad, loss, grad


def _agree(inp, ref_loss, ref_grad, loss, grad):
    B = inp.workload.B
    check_loss(float(loss.item()), float(ref_loss.item()))
    g = grad.float().cpu().numpy().astype(np.float64)
    r = ref_grad.float().cpu().numpy().astype(np.float64)
    if inp.workload.dtype == "f32":
        assert np.max(np.abs(g - r)) * B <= GRAD_ATOL_TIMES_B
    else:
        assert np.all(np.abs(g - r) <= ulp_bf16(r))


def test_noalloc_matches_ce_fwd_bwd_on_two_calls_in_a_row():
    """Two consecutive calls (different shapes, paths and dtypes) share the
    static scratch; each matches the allocating entry point."""
    first = wl.random_case(300, 1000, "f32", seed=11, sigma=2.0)     # warp-per-row path
    second = wl.random_case(97, 40000, "bf16", seed=12, sigma=3.0)   # split-row path
    for inp in (first, second):
        _agree(inp, *_both(inp))


def test_noalloc_rejects_shapes_beyond_its_scratch():
    z = torch.zeros(262145, 4, device="cuda")
    t = torch.zeros(262145, dtype=torch.int32, device="cuda")
    loss = torch.empty(1, device="cuda")
    grad = torch.empty_like(z)
    with pytest.raises(ce.CEError) as ei:
        ce.ce_fwd_bwd_noalloc(z, t, loss, grad)
    assert ei.value.status == CE_ERR_SCRATCH
    z2 = torch.zeros(2, 300000, device="cuda")  # needs the streaming path
    t2 = torch.zeros(2, dtype=torch.int32, device="cuda")
    with pytest.raises(ce.CEError) as ei:
        ce.ce_fwd_bwd_noalloc(z2, t2, loss, torch.empty_like(z2))
    assert ei.value.status == CE_ERR_SCRATCH
