"""GPU parity of the loss-only warp-per-row path (CE_PATH_ROWS_ONLINE) against
the fp64 oracle: every build, reduction and element type; rows that do not
start on a 16-byte boundary; the target in a row's head, vectors and tail;
rows whose maximum grows at every step (a rescale each time); out-of-range
targets; determinism; and which calls the planner sends there.

Tolerances are the loss's: |l - l_ref| <= 1e-5 |l_ref| + 1e-7 per row and for
the reduced loss.
"""

import numpy as np
import pytest

import workloads as wl

from parity import check_loss, device_inputs

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU-only machines
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import softmax_cross_entropy_row_gb300 as ce  # noqa: E402
import oracle  # noqa: E402

ONLINE = ce.CE_PATH_ROWS_ONLINE
MEAN, SUM, NONE = ce.CE_REDUCE_MEAN, ce.CE_REDUCE_SUM, ce.CE_REDUCE_NONE
BUILDS = 5


@pytest.fixture(scope="module", autouse=True)
def _built():
    ce.build()
    ce.load_library()
    oracle.build()
    yield
    torch.cuda.synchronize()


def _loss_only(z, t, reduction=MEAN, path=ONLINE, split=0):
    B = z.shape[0]
    loss = torch.full((B if reduction == NONE else 1,), float("nan"), device="cuda")
    ce.ce_fwd_bwd_ex(z, t, loss, None, reduction, None, None, path, split)
    torch.cuda.synchronize()
    return loss


def _check_rows(inp, loss_rows, what=""):
    l_ref = oracle.rows(inp.logits, inp.targets, grad=False)
    got = loss_rows.cpu().numpy().astype(np.float64)
    for b in range(inp.workload.B):
        if np.isnan(l_ref[b]):
            assert np.isnan(got[b]), f"{what}: row {b} {got[b]} expected NaN"
            continue
        err = abs(got[b] - l_ref[b])
        assert err <= 1e-5 * abs(l_ref[b]) + 1e-7, \
            f"{what}: row {b} loss {got[b]!r} vs oracle {l_ref[b]!r}"
    return l_ref


def _with_rows(inp, rows_f32):
    """inp with its logits replaced by the fp32 rows (rounded to its dtype)."""
    d = inp.workload.dtype
    if d == "bf16":
        inp.logits = wl.f32_to_bf16_bits(rows_f32)
    elif d == "f16":
        inp.logits = rows_f32.astype(np.float16)
    else:
        inp.logits = np.ascontiguousarray(rows_f32, dtype=np.float32)
    return inp


# (B, C): rows of 1-3 elements, rows shorter than a warp's first step, rows
# that start at every offset mod 16 (odd C), a few steps, many steps
SHAPES = [(8, 1), (40, 3), (300, 1000), (33, 4097), (5, 9001), (7, 20000), (3, 50257),
          (2, 128256), (1, 300001)]


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("reduction", [MEAN, SUM, NONE])
@pytest.mark.parametrize("B,C", SHAPES)
def test_online_path_shapes(B, C, dtype, reduction):
    inp = wl.random_case(B, C, dtype, seed=B * 7 + C + reduction, sigma=3.0)
    z, t = device_inputs(inp)
    loss = _loss_only(z, t, reduction)
    l_ref = oracle.rows_ex(inp.logits, inp.targets, reduction, grad=False)
    if reduction == NONE:
        got = loss.cpu().numpy().astype(np.float64)
        for b in range(B):
            check_loss(float(got[b]), float(l_ref[b]))
    else:
        check_loss(float(loss.item()), oracle.reduce(l_ref, reduction))


@pytest.mark.parametrize("build", range(1, BUILDS + 1))
@pytest.mark.parametrize("B,C,dtype", [(5, 9001, "bf16"), (3, 50257, "f32"), (40, 3, "f16"),
                                       (2, 128256, "bf16"), (1, 300001, "f32")])
def test_every_build(build, B, C, dtype):
    inp = wl.random_case(B, C, dtype, seed=build * 101 + C, sigma=2.0)
    z, t = device_inputs(inp)
    _check_rows(inp, _loss_only(z, t, NONE, ONLINE, build), f"build {build - 1}")


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("C", [1000, 4097, 9001])
def test_target_in_head_vectors_and_tail(C, dtype):
    """Odd C puts the rows at every offset mod 16, so the first elements (head)
    and the last (tail) of a row are read one by one; targets at the row's
    ends, at a vector's first and last elements, and in the middle."""
    B = 48
    inp = wl.random_case(B, C, dtype, seed=C, sigma=2.0)
    picks = [0, 1, 2, 3, 5, 7, 8, 9, 15, 16, 17, C // 2, C - 9, C - 8, C - 2, C - 1]
    inp.targets[:] = np.array([picks[b % len(picks)] for b in range(B)], dtype=np.int32)
    z, t = device_inputs(inp)
    _check_rows(inp, _loss_only(z, t, NONE), f"C={C} {dtype}")


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_rescaled_sums(dtype):
    """Rows whose maximum grows at every step of a warp (ascending), only at
    the start (descending), a dominating target (the loss near 0, its log1p
    form), rows of -inf but for a few elements, and a row where only the
    target is finite (loss 0)."""
    B, C = 8, 20000
    inp = wl.random_case(B, C, dtype, seed=3, sigma=1.0)
    ramp = np.linspace(-8.0, 8.0, C, dtype=np.float32)
    rows = np.empty((B, C), dtype=np.float32)
    rows[0] = ramp
    rows[1] = ramp[::-1]
    rows[2] = np.float32(0.01) * np.arange(C, dtype=np.float32) % np.float32(5.0)
    rows[3] = 0.0
    rows[4] = 1.0
    rows[5] = -np.inf
    rows[5, [0, 777, C - 1]] = [1.0, 3.0, 2.0]
    rows[6] = -np.inf
    rows[7] = np.random.default_rng(5).normal(0, 1, C).astype(np.float32)
    t = np.array([C - 1, 0, 123, 7, 19999, 777, 4321, 50], dtype=np.int32)
    rows[3, t[3]] = 30.0 if dtype != "f16" else 20.0  # the target dominates
    rows[6, t[6]] = 2.5                                # the only finite logit
    rows[7, t[7]] = 12.0
    inp = _with_rows(inp, rows)
    inp.targets[:] = t
    z, tt = device_inputs(inp)
    for build in range(1, BUILDS + 1):
        l_ref = _check_rows(inp, _loss_only(z, tt, NONE, ONLINE, build), f"build {build - 1}")
    assert l_ref[6] == 0.0


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_online_out_of_range_targets(dtype):
    """Reading: an out-of-range target gives that row a NaN loss and one count
    per bad row; other rows are unaffected."""
    B, C = 6, 9000
    inp = wl.random_case(B, C, dtype, seed=11)
    inp.targets[1] = -1
    inp.targets[4] = C
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        ce.ce_get_device_errors(s)  # clear
        z, t = device_inputs(inp)
        rows = torch.full((B,), 0.0, device="cuda")
        ce.ce_fwd_bwd_ex(z, t, rows, None, NONE, None, s, ONLINE, 0)
        mean = torch.full((1,), 0.0, device="cuda")
        ce.ce_fwd_bwd_ex(z, t, mean, None, MEAN, None, s, ONLINE, 0)
        bad, tmo = ce.ce_get_device_errors(s)
    s.synchronize()
    assert (bad, tmo) == (4, 0)
    got = rows.cpu().numpy()
    assert np.isnan(got[1]) and np.isnan(got[4])
    assert np.isnan(mean.item())
    keep = [0, 2, 3, 5]
    l_ref = oracle.rows(inp.logits[keep], inp.targets[keep], grad=False)
    for i, b in enumerate(keep):
        check_loss(float(got[b]), float(l_ref[i]))


@pytest.mark.parametrize("B,C,dtype", [(64, 9001, "bf16"), (64, 50257, "f32"), (16, 128256, "bf16")])
def test_online_bitwise_deterministic(B, C, dtype):
    inp = wl.random_case(B, C, dtype, seed=77)
    z, t = device_inputs(inp)
    ref = _loss_only(z, t, NONE)
    mean = _loss_only(z, t, MEAN)
    for _ in range(5):
        assert torch.equal(_loss_only(z, t, NONE).view(torch.int32), ref.view(torch.int32))
        assert torch.equal(_loss_only(z, t, MEAN).view(torch.int32), mean.view(torch.int32))


def test_online_path_needs_the_loss_alone():
    """A gradient or the softmax forward on the loss-only path: CE_ERR_PATH;
    a build past the last: CE_ERR_PATH."""
    z = torch.zeros(4, 1000, device="cuda")
    t = torch.zeros(4, dtype=torch.int32, device="cuda")
    loss = torch.empty(1, device="cuda")
    with pytest.raises(ce.CEError) as ei:
        ce.ce_fwd_bwd_ex(z, t, loss, torch.empty_like(z), MEAN, None, None, ONLINE, 0)
    assert ei.value.status == 9
    with pytest.raises(ce.CEError) as ei:
        ce.ce_softmax_fwd(z, torch.empty_like(z), None, ONLINE, 0)
    assert ei.value.status == 9
    with pytest.raises(ce.CEError) as ei:
        ce.ce_fwd_bwd_ex(z, t, loss, None, MEAN, None, None, ONLINE, BUILDS + 1)
    assert ei.value.status == 9


@pytest.mark.parametrize("C,dtype", [(32000, "bf16"), (9001, "bf16"), (50257, "f32")])
def test_planner_takes_it_for_the_loss_alone_of_large_batches(C, dtype):
    """CE_PATH_AUTO with no gradient runs the online kernel (the same bits as
    forcing it) once a batch has 8 rows per SM, rows past 8 KB; the full call
    on the same inputs agrees within the loss tolerance."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    B = 8 * sms
    inp = wl.random_case(B, C, dtype, seed=C + 1, sigma=2.0)
    z, t = device_inputs(inp)
    for reduction in (MEAN, NONE):
        auto = _loss_only(z, t, reduction, ce.CE_PATH_AUTO)
        forced = _loss_only(z, t, reduction, ONLINE)
        assert torch.equal(auto.view(torch.int32), forced.view(torch.int32)), reduction
    full = torch.empty(1, device="cuda")
    ce.ce_fwd_bwd_ex(z, t, full, torch.empty_like(z))
    torch.cuda.synchronize()
    check_loss(float(_loss_only(z, t, MEAN, ce.CE_PATH_AUTO).item()), float(full.item()))
    _check_rows(inp, _loss_only(z, t, NONE, ce.CE_PATH_AUTO), f"auto {C} {dtype}")
