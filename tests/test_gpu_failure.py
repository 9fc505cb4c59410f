"""Bounded waits on the GPU: a row copy that never lands.

Every kernel waits for its TMA copies with a bounded wait.  The test entry
point (include/ce_testing.h) leaves out the copy of one row, so that wait can
only give up, and shortens the copy waits to about half a millisecond.  The
kernel must then count a timeout, make the loss NaN (the caller's signal when
it cannot read the counters), wait for the copies it did issue and return;
the next call on the same stream must be correct again.  Nothing here faults,
traps or hangs the GPU: the skipped copy is never issued, so no copy is ever
in flight to the slot whose wait gives up, and every wait is bounded.
"""

import math

import pytest

import workloads as wl

from parity import check_full, device_inputs, run

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU-only machines
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import softmax_cross_entropy_row_gb300 as ce  # noqa: E402
import oracle  # noqa: E402

WARP, SPLIT, TWOPASS = ce.CE_PATH_ROWS_WARP, ce.CE_PATH_ROW_SPLIT, ce.CE_PATH_ROW_TWOPASS
SHORT_WAIT_CYCLES = 1_000_000  # about half a millisecond

# (path, split, B, C, dtype): the warp kernel; the barrier-per-row split
# kernel alone (K = 1) and in a cluster of two (100 KB slices, so not the
# pipelined kernel); the pipelined split kernel (K = 2, 9 KB slices); the
# two-pass kernel
CASES = [(WARP, 0, 40, 1000, "f32"), (WARP, 0, 40, 9001, "bf16"), (SPLIT, 1, 6, 7000, "f32"), (SPLIT, 1, 6, 20000, "f32"), (SPLIT, 2, 6, 50257, "f32"),
         (SPLIT, 2, 6, 9000, "bf16"), (TWOPASS, 0, 6, 50257, "f32"), (TWOPASS, 0, 5, 9000, "bf16")]


@pytest.fixture(scope="module", autouse=True)
def _built():
    ce.build()
    ce.load_library()
    oracle.build()
    yield
    torch.cuda.synchronize()


@pytest.mark.parametrize("path,split,B,C,dtype", CASES)
def test_a_copy_that_never_lands(path, split, B, C, dtype):
    inp = wl.random_case(B, C, dtype, seed=B + C, sigma=2.0)
    z, t = device_inputs(inp)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        run(z, t, path, split, s)  # sizes the stream's workspace
        assert ce.ce_get_device_errors(s) == (0, 0)
        loss = torch.full((1,), 0.0, dtype=torch.float32, device="cuda")
        grad = torch.empty_like(z)
        ce.ce_fwd_bwd_test(z, t, loss, grad, s, path, split, skip_copy_row=B // 2,
                           wait_limit_cycles=SHORT_WAIT_CYCLES)
        bad, timeouts = ce.ce_get_device_errors(s)
    assert bad == 0
    assert timeouts >= 1, "the wait for the copy that was never issued did not give up"
    assert math.isnan(loss.item()), f"the loss of a call that gave up is {loss.item()}, not NaN"
    # the kernel returned, the context is usable, the stream's workspace is
    # ready for the next call, which is correct
    with torch.cuda.stream(s):
        loss2, grad2 = run(z, t, path, split, s)
        s.synchronize()
        assert ce.ce_get_device_errors(s) == (0, 0)
    check_full(inp, loss2, grad2, f"after a timeout, path {path} K={split}")


def test_hooks_off_change_nothing():
    """The test entry point with no hook set gives the plain call's bits."""
    inp = wl.random_case(64, 50257, "f32", seed=3, sigma=2.0)
    z, t = device_inputs(inp)
    for path, split in [(WARP, 0), (SPLIT, 2), (TWOPASS, 0)]:
        if path == WARP:
            inp = wl.random_case(64, 1000, "f32", seed=3, sigma=2.0)
            z, t = device_inputs(inp)
        l0, g0 = run(z, t, path, split)
        l1 = torch.empty(1, device="cuda")
        g1 = torch.empty_like(z)
        ce.ce_fwd_bwd_test(z, t, l1, g1, None, path, split)
        torch.cuda.synchronize()
        assert torch.equal(l0, l1) and torch.equal(g0, g1), (path, split)
