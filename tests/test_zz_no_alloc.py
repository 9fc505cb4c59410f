"""The allocation-free entry point, ce_fwd_bwd_noalloc.

Some callers cannot call cudaMalloc: a memory manager owns the whole device,
the device memory budget is fixed at start-up, or the caller must never stall
on the synchronisation an allocation can cause.  ce_fwd_bwd_noalloc serves
them with a statically sized scratch array inside the library.  It runs the
kernels of ce_fwd_bwd, so its loss and gradient must be the same bits.  This
file is collected last, so a run that stops at the first failure has run every
other test before it; it passes on its own in a fresh process as well.
"""

import pytest

import workloads as wl

from parity import device_inputs

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU-only machines
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import softmax_cross_entropy_row_gb300 as ce  # noqa: E402

CE_ERR_OVERLAP = 6
CE_ERR_SCRATCH = 10
MAX_ROWS = 262144


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


def _same_bits(a, b):
    if a.dtype in (torch.bfloat16, torch.float16):
        return torch.equal(a.view(torch.int16), b.view(torch.int16))
    return torch.equal(a.view(torch.int32), b.view(torch.int32))


# (B, C, dtype): the warp-per-row kernel (rows in registers, and 18 KB rows
# swept in shared memory), the split kernel (one CTA per row),
# the two-pass kernel (fp32 C = 200000), and B at the scratch's limit (the last
# row losses sit at the end of the static array)
CASES = [(300, 1000, "f32"), (300, 9001, "bf16"), (97, 32000, "bf16"), (40, 200000, "f32"),
         (MAX_ROWS, 8, "f32")]


def test_noalloc_matches_ce_fwd_bwd_on_two_calls_in_a_row():
    """Consecutive calls (different shapes, kernels and dtypes) share the static
    scratch; each gives the allocating entry point's loss and gradient bits."""
    for B, C, dtype in CASES:
        inp = wl.random_case(B, C, dtype, seed=B + C, sigma=2.0)
        ref_loss, ref_grad, loss, grad = _both(inp)
        assert _same_bits(loss, ref_loss), (B, C, dtype, loss.item(), ref_loss.item())
        assert _same_bits(grad, ref_grad), (B, C, dtype)


def test_noalloc_rejects_what_it_cannot_hold():
    z = torch.zeros(MAX_ROWS + 1, 4, device="cuda")
    t = torch.zeros(MAX_ROWS + 1, dtype=torch.int32, device="cuda")
    loss = torch.empty(1, device="cuda")
    grad = torch.empty_like(z)
    with pytest.raises(ce.CEError) as ei:
        ce.ce_fwd_bwd_noalloc(z, t, loss, grad)
    assert ei.value.status == CE_ERR_SCRATCH
    # the loss may not alias an input (checked like ce_fwd_bwd's)
    z2 = torch.zeros(8, 16, device="cuda")
    t2 = torch.zeros(8, dtype=torch.int32, device="cuda")
    for alias in (z2.view(-1)[3:4], t2.view(torch.float32)[5:6]):
        with pytest.raises(ce.CEError) as ei:
            ce.ce_fwd_bwd_noalloc(z2, t2, alias, torch.empty_like(z2))
        assert ei.value.status == CE_ERR_OVERLAP
