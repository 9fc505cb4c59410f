"""GPU parity of the reductions, the upstream gradient and the loss-only
forward (ce_fwd_bwd_ex, ce_forward) against the fp64 oracle, on every kernel
path.

Tolerances are those of the mean, with the gradient bound taken relative to
the gradient's row factor: 1e-6 x |u| / B for the mean and 1e-6 x |u| for the
sum and the per-row losses (whose gradients carry no 1/B), u the upstream
gradient; bf16 gradients within 1 ulp.  Per-row losses are held to the batch
loss's bound each.
"""

import numpy as np
import pytest

import workloads as wl

from parity import check_grad, check_loss, device_inputs, grad_rows_host

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU-only machines
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import softmax_cross_entropy_row_gb300 as ce  # noqa: E402
import oracle  # noqa: E402

WARP, SPLIT, STREAM = ce.CE_PATH_ROWS_WARP, ce.CE_PATH_ROW_SPLIT, ce.CE_PATH_STREAM
TWOPASS = ce.CE_PATH_ROW_TWOPASS
MEAN, SUM, NONE = ce.CE_REDUCE_MEAN, ce.CE_REDUCE_SUM, ce.CE_REDUCE_NONE

# (path, split, B, C): the warp kernel, the barrier-per-row split kernel at
# K = 1 and with 100 KB fp32 slices, the pipelined split kernel, the streaming
# path, the two-pass path
PATHS = [(WARP, 0, 300, 1000), (WARP, 0, 7, 9001), (SPLIT, 1, 5, 20000), (SPLIT, 4, 6, 40000),
         (SPLIT, 2, 3, 50257), (STREAM, 0, 3, 10000), (TWOPASS, 0, 5, 50257)]


@pytest.fixture(scope="module", autouse=True)
def _built():
    ce.build()
    ce.load_library()
    oracle.build()
    yield
    torch.cuda.synchronize()


def _upstream(reduction, B, seed):
    """A scalar for the mean and the sum, one value per row for none (kept
    away from 0 so that the gradient bound can be taken relative to it)."""
    g = np.random.default_rng(seed)
    if reduction == NONE:
        return (g.uniform(0.5, 2.0, B) * g.choice([-1.0, 1.0], B)).astype(np.float32)
    return np.array([-1.75], dtype=np.float32)


def _check(inp, reduction, loss, grad, u, what):
    B = inp.workload.B
    ref = oracle.rows_ex(inp.logits, inp.targets, reduction,
                         upstream=None if u is None else u.astype(np.float64),
                         grad=grad is not None)
    l_ref, g_ref = ref if grad is not None else (ref, None)
    if reduction == NONE:
        got = loss.cpu().numpy().astype(np.float64)
        for b in range(B):
            check_loss(float(got[b]), float(l_ref[b]))
    else:
        check_loss(float(loss.item()), oracle.reduce(l_ref, reduction))
    if grad is None:
        return
    g = grad_rows_host(grad)
    # the gradient bound relative to the row factor: divide the factor out
    scale = np.ones(B) if u is None else (u.astype(np.float64) if reduction == NONE
                                          else np.full(B, float(u[0])))
    if inp.workload.dtype == "f32":
        eff_b = B if reduction == MEAN else 1
        check_grad(g / scale[:, None], g_ref / scale[:, None], eff_b, "f32", what)
    else:
        check_grad(g, g_ref, B, inp.workload.dtype, what)


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("reduction", [MEAN, SUM, NONE])
@pytest.mark.parametrize("path,split,B,C", PATHS)
@pytest.mark.parametrize("with_grad", [True, False])
def test_reductions_on_every_path(path, split, B, C, dtype, reduction, with_grad):
    inp = wl.random_case(B, C, dtype, seed=B * 31 + C + reduction, sigma=3.0)
    z, t = device_inputs(inp)
    u = _upstream(reduction, B, seed=C) if with_grad else None
    u_dev = None if u is None else torch.from_numpy(u).cuda()
    loss = torch.full((B if reduction == NONE else 1,), float("nan"), device="cuda")
    grad = torch.empty_like(z) if with_grad else None
    ce.ce_fwd_bwd_ex(z, t, loss, grad, reduction, u_dev, None, path, split)
    torch.cuda.synchronize()
    _check(inp, reduction, loss, grad, u, f"path {path} K={split} {dtype} red={reduction}")


def test_loss_only_matches_the_full_call_bitwise():
    """Where the loss alone runs the full call's kernel (rows of at most 8 KB,
    or batches of fewer than 8 rows per SM), ce_forward, ce_fwd_bwd_ex
    without a gradient and the full call give the same loss bits (same row
    arithmetic, same fixed-order sum).  Larger loss-only batches take the
    online kernel, whose sums are formed in another order
    (test_gpu_online.py)."""
    for B, C, dtype in [(512, 3000, "f32"), (64, 32000, "bf16"), (24, 128256, "bf16")]:
        inp = wl.random_case(B, C, dtype, seed=4)
        z, t = device_inputs(inp)
        l_fwd = torch.empty(1, device="cuda")
        ce.ce_forward(z, t, l_fwd)
        l_full = torch.empty(1, device="cuda")
        ce.ce_fwd_bwd_ex(z, t, l_full, torch.empty_like(z))
        l_none = torch.empty(1, device="cuda")
        ce.ce_fwd_bwd_ex(z, t, l_none, None)
        torch.cuda.synchronize()
        assert l_fwd.item() == l_full.item() == l_none.item(), (B, C, dtype)


@pytest.mark.parametrize("name", ["classifier_4096x1000_f32", "lm_head_8192x32000_bf16",
                                  "lm_head_4096x128256_bf16_peaked", "stress_16384x50257_f32"])
def test_full_size_loss_only_and_per_row(name):
    """The benchmark workloads: the loss alone (mean) and every row's loss."""
    w = wl.WORKLOADS_BY_NAME[name]
    inp = wl.make_inputs(w)
    z, t = device_inputs(inp)
    l_ref = oracle.rows(inp.logits, inp.targets, grad=False)
    loss = torch.empty(1, device="cuda")
    ce.ce_forward(z, t, loss)
    rows = torch.empty(w.B, device="cuda")
    ce.ce_forward(z, t, rows, ce.CE_REDUCE_NONE)
    torch.cuda.synchronize()
    check_loss(float(loss.item()), oracle.batch_loss(l_ref))
    got = rows.cpu().numpy().astype(np.float64)
    err = np.abs(got - l_ref) - (1e-5 * np.abs(l_ref) + 1e-7)
    assert float(err.max()) <= 0.0, f"{name}: worst per-row loss excess {float(err.max()):.3g}"
