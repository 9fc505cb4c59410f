"""GPU parity of the host-buffer entry points ce_fwd_bwd_host (gradient on the
device) and ce_fwd_bwd_host_grad (gradient back in host memory): the same loss
bits and gradient as ce_fwd_bwd on the same inputs (the same kernels on
library-owned device copies, chunk by chunk), on every path, and the oracle's
values on the small cases."""

import numpy as np
import pytest

import workloads as wl

from parity import check_full, device_inputs

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU-only machines
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import softmax_cross_entropy_row_gb300 as ce  # noqa: E402
import oracle  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    ce.build()
    ce.load_library()
    oracle.build()
    yield
    torch.cuda.synchronize()


def _host_inputs(inp, pinned):
    if inp.workload.dtype == "bf16":
        z = torch.from_numpy(inp.logits.view(np.int16)).view(torch.bfloat16)
    else:
        z = torch.from_numpy(inp.logits)
    t = torch.from_numpy(inp.targets)
    loss = torch.full((1,), float("nan"), dtype=torch.float32)
    if pinned:
        z, t, loss = z.pin_memory(), t.pin_memory(), loss.pin_memory()
    return z, t, loss


def _both(inp, pinned=True, stream=None, grad_to_host=False):
    zh, th, lh = _host_inputs(inp, pinned)
    if grad_to_host:
        grad_h = torch.empty(zh.shape, dtype=zh.dtype)
        if pinned:
            grad_h = grad_h.pin_memory()
        ce.ce_fwd_bwd_host_grad(zh, th, lh, grad_h, stream)
    else:
        grad_h = torch.empty(zh.shape, dtype=zh.dtype, device="cuda")
        ce.ce_fwd_bwd_host(zh, th, lh, grad_h, stream)
    z, t = device_inputs(inp)
    loss_d = torch.empty(1, device="cuda")
    grad_d = torch.empty_like(z)
    ce.ce_fwd_bwd(z, t, loss_d, grad_d, stream)
    torch.cuda.synchronize()
    return lh, grad_h, loss_d, grad_d


# (B, C, dtype): the warp kernel (rows in registers and swept in shared
# memory), the split and two-pass kernels, f16, ragged rows, and
# batches of several 64 MiB chunks (a last chunk of fewer rows included)
CASES = [(8, 10, "f32"), (3, 200000, "f32"), (4096, 1000, "f32"), (600, 9001, "bf16"),
         (1024, 32000, "bf16"),
         (512, 32000, "f16"), (7, 3001, "f32"), (40000, 1000, "f32"), (4096, 32000, "bf16"),
         (110, 600000, "bf16"), (1500, 50257, "f32"), (1100, 128256, "bf16")]


@pytest.mark.parametrize("B,C,dtype", CASES)
@pytest.mark.parametrize("pinned", [True, False])
@pytest.mark.parametrize("grad_to_host", [False, True])
def test_host_entry_matches_the_device_entry(B, C, dtype, pinned, grad_to_host):
    inp = wl.random_case(B, C, dtype, seed=B + C, sigma=3.0)
    lh, grad_h, loss_d, grad_d = _both(inp, pinned, grad_to_host=grad_to_host)
    assert lh.item() == loss_d.item(), (lh.item(), loss_d.item())
    assert torch.equal(grad_h.cuda() if grad_to_host else grad_h, grad_d)
    if B * C <= 5_000_000:
        check_full(inp, lh, grad_h.cuda() if grad_to_host else grad_h, f"host entry {B}x{C} {dtype}")


def test_back_to_back_calls_on_one_stream():
    """Two calls in a row on one stream share its staging buffers: the second
    call's copies are ordered after the first call's kernel."""
    s = torch.cuda.Stream()
    a = wl.random_case(2048, 2000, "f32", seed=1)
    b = wl.random_case(2048, 2000, "f32", seed=2)
    za, ta, la = _host_inputs(a, True)
    zb, tb, lb = _host_inputs(b, True)
    ga = torch.empty(za.shape, device="cuda")
    gb = torch.empty(zb.shape, device="cuda")
    with torch.cuda.stream(s):
        ce.ce_fwd_bwd_host(za, ta, la, ga, s)
        ce.ce_fwd_bwd_host(zb, tb, lb, gb, s)
    s.synchronize()
    check_full(a, la, ga, "first of two calls")
    check_full(b, lb, gb, "second of two calls")


def test_back_to_back_calls_with_the_gradient_to_the_host():
    """Consecutive calls of different sizes on one stream, gradients to the
    host: the staging grows between them, the results are those of the device
    entry point."""
    s = torch.cuda.Stream()
    cases = [wl.random_case(700, 50257, "f32", seed=5), wl.random_case(4096, 1000, "f32", seed=6),
             wl.random_case(1400, 50257, "f32", seed=7)]
    outs = []
    with torch.cuda.stream(s):
        for inp in cases:
            zh, th, lh = _host_inputs(inp, True)
            gh = torch.empty(zh.shape, dtype=zh.dtype).pin_memory()
            ce.ce_fwd_bwd_host_grad(zh, th, lh, gh, s)
            outs.append((lh, gh))
    s.synchronize()
    for inp, (lh, gh) in zip(cases, outs):
        z, t = device_inputs(inp)
        loss_d = torch.empty(1, device="cuda")
        grad_d = torch.empty_like(z)
        ce.ce_fwd_bwd(z, t, loss_d, grad_d)
        torch.cuda.synchronize()
        assert lh.item() == loss_d.item() and torch.equal(gh.cuda(), grad_d)


def test_capture_is_refused_and_bad_targets_are_counted():
    inp = wl.random_case(6, 100, "f32", seed=3)
    inp.targets[2] = 100
    zh, th, lh = _host_inputs(inp, True)
    grad = torch.empty(zh.shape, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        ce.ce_get_device_errors(s)
        ce.ce_fwd_bwd_host(zh, th, lh, grad, s)
        assert ce.ce_get_device_errors(s) == (1, 0)
    assert np.isnan(lh.item())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with pytest.raises(ce.CEError) as ei:
            with torch.cuda.graph(graph, stream=s):
                ce.ce_fwd_bwd_host(zh, th, lh, grad, s)
    assert ei.value.status == 8
