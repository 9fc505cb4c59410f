"""GPU parity: the CUDA path through the C-ABI against the fp64 oracle.

Every case is compared element by element: the small ones at once, the
full-size workloads (in the launch configuration the benchmark times) on the
batch loss over every row and on every gradient element, streamed through the
oracle in blocks of rows; the row-sum property is checked on every row, for
16-bit gradients also on the fp32 values before their rounding.
"""

import numpy as np
import pytest

import workloads as wl

from parity import (ROWSUM_ATOL_TIMES_B, check_all_rows, check_full, check_grad, device_inputs,
                    grad_rows_host, run)

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU-only machines
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import softmax_cross_entropy_row_gb300 as ce  # noqa: E402
import oracle  # noqa: E402

AUTO, WARP, SPLIT, STREAM, TWOPASS = (ce.CE_PATH_AUTO, ce.CE_PATH_ROWS_WARP,
                                      ce.CE_PATH_ROW_SPLIT, ce.CE_PATH_STREAM,
                                      ce.CE_PATH_ROW_TWOPASS)
SPLIT_MAX_SLICE_BYTES = 512 * 16 * 16 - 32  # threads x vectors x 16 bytes, less the partial vectors


@pytest.fixture(scope="module", autouse=True)
def _built():
    ce.build()
    ce.load_library()
    oracle.build()
    yield
    torch.cuda.synchronize()


def _case(B, C, dtype, seed, sigma=2.0):
    return wl.random_case(B, C, dtype, seed=seed, sigma=sigma)


# --------------------------------------------------------- small workloads

@pytest.mark.parametrize("name", ["tiny_8x10_f32", "classifier_4096x1000_f32"])
def test_small_workloads_full(name):
    inp = wl.make_inputs(wl.WORKLOADS_BY_NAME[name])
    z, t = device_inputs(inp)
    loss, grad = run(z, t)
    torch.cuda.synchronize()
    check_full(inp, loss, grad, name)


# ------------------------------------------------- edge shapes, every path

WARP_SHAPES = [(1, 1), (3, 2), (8, 3), (5, 5), (7, 7), (64, 10), (33, 31), (9, 33), (300, 1000),
               (17, 1023), (16, 1025), (4, 2047), (5, 2048)]
SPLIT_SHAPES = [(1, 1), (2, 3), (3, 17), (5, 1000), (4, 4099), (3, 8191), (6, 16385), (2, 40000),
                (3, 50257)]
STREAM_SHAPES = [(1, 1), (3, 5), (2, 4095), (2, 4096), (3, 4097), (2, 10000), (2, 50257)]
# rows longer than a warp's registers hold (8 KB .. 48 KB), swept in shared
# memory by the warp kernel: just past 8 KB, ragged, one and several sweeps
# of 8 vectors per lane, the longest row, and many rows per warp (the ring
# wraps)
SWEPT_SHAPES = {"f32": [(1, 2049), (5, 2051), (37, 3001), (6, 4095), (7, 4096), (3, 8191),
                        (4, 12000), (3000, 4500)],
                "bf16": [(1, 4097), (5, 4101), (37, 6001), (6, 8191), (7, 8192), (3, 16383),
                         (4, 24000), (3000, 9001)],
                "f16": [(5, 4101), (9, 16384), (3, 24000)]}
# the two-pass kernel's chunks hold 4096 fp32 / 8192 16-bit elements: rows
# inside one chunk, across a chunk boundary, many chunks, and long rows
TWOPASS_SHAPES = [(1, 1), (3, 2), (5, 5), (7, 31), (4, 1000), (3, 4095), (3, 4096), (2, 4097),
                  (5, 8191), (3, 8193), (6, 16385), (3, 32000), (2, 50257), (2, 128256),
                  (2, 300007)]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("B,C", WARP_SHAPES)
def test_warp_path_shapes(B, C, dtype):
    inp = _case(B, C, dtype, seed=B * 7919 + C)
    z, t = device_inputs(inp)
    loss, grad = run(z, t, WARP)
    torch.cuda.synchronize()
    check_full(inp, loss, grad, f"warp {B}x{C} {dtype}")


@pytest.mark.parametrize("dtype,B,C", [(d, b, c) for d, v in SWEPT_SHAPES.items() for b, c in v])
def test_swept_warp_path_shapes(B, C, dtype):
    inp = _case(B, C, dtype, seed=B * 7919 + C)
    z, t = device_inputs(inp)
    loss, grad = run(z, t, WARP)
    torch.cuda.synchronize()
    check_full(inp, loss, grad, f"swept warp {B}x{C} {dtype}")


def test_swept_warp_path_is_planned_for_medium_rows():
    """Rows past 8 KB for which 8 warps per SM fit (up to ~27 KB) go to the
    warp kernel's swept build; 31 KB rows do not; past 48 KB the forced warp
    path refuses."""
    for C, dt in [(8000, ce.CE_BF16), (4500, ce.CE_F32), (6000, ce.CE_F32), (12000, ce.CE_BF16)]:
        plan = ce.ce_query_plan(16384, C, dt)
        assert plan["path_name"] == "rows_warp", (C, plan)
        assert plan["threads"] in (128, 256, 512), plan
    # 31 KB rows: the split kernel in 128-thread CTAs; 64 KB rows: 512 threads
    plan = ce.ce_query_plan(8192, 16000, ce.CE_BF16)
    assert (plan["path_name"], plan["threads"]) == ("row_split", 128), plan
    plan = ce.ce_query_plan(8192, 32000, ce.CE_BF16)
    assert (plan["path_name"], plan["threads"]) == ("row_split", 512), plan
    z = torch.zeros(2, 12289, device="cuda")  # 49156 bytes: past the swept build
    t = torch.zeros(2, dtype=torch.int32, device="cuda")
    with pytest.raises(ce.CEError) as ei:
        ce.ce_fwd_bwd_path(z, t, torch.empty(1, device="cuda"), torch.empty_like(z), None, WARP, 0)
    assert ei.value.status == 9


@pytest.mark.parametrize("K", [1, 2, 3, 4, 6, 8])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("B,C", SPLIT_SHAPES)
def test_split_path_shapes(B, C, dtype, K):
    inp = _case(B, C, dtype, seed=B * 104729 + C + K, sigma=3.0)
    z, t = device_inputs(inp)
    slice_bytes = -(-(-(-C // K)) // 8) * 8 * inp.workload.elem_bytes
    if slice_bytes > SPLIT_MAX_SLICE_BYTES:
        # a CTA holds at most 128 KB of a row in registers: the forced split is refused
        with pytest.raises(ce.CEError) as ei:
            run(z, t, SPLIT, K)
        assert ei.value.status == 9
        return
    loss, grad = run(z, t, SPLIT, K)
    torch.cuda.synchronize()
    check_full(inp, loss, grad, f"split K={K} {B}x{C} {dtype}")


@pytest.mark.parametrize("K,C", [(1, 30000), (1, 30001), (2, 60000)])
def test_split_path_with_one_slot(K, C):
    """fp32 slices of ~117 KB leave room for one ring slot per CTA: the
    gradient is then stored directly (staging hands a slot back one row late
    and needs a second), every row is computed and no wait gives up."""
    inp = _case(9, C, "f32", seed=C + K)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        ce.ce_get_device_errors(s)  # clear
        z, t = device_inputs(inp)
        loss, grad = run(z, t, SPLIT, K, s)
        assert ce.ce_get_device_errors(s) == (0, 0)
    check_full(inp, loss, grad, f"split K={K} one slot {C}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("B,C", STREAM_SHAPES)
def test_stream_path_shapes(B, C, dtype):
    inp = _case(B, C, dtype, seed=B * 31 + C, sigma=3.0)
    z, t = device_inputs(inp)
    loss, grad = run(z, t, STREAM)
    torch.cuda.synchronize()
    check_full(inp, loss, grad, f"stream {B}x{C} {dtype}")


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("B,C", TWOPASS_SHAPES)
def test_twopass_path_shapes(B, C, dtype):
    inp = _case(B, C, dtype, seed=B * 7 + C + 3, sigma=3.0)
    z, t = device_inputs(inp)
    loss, grad = run(z, t, TWOPASS)
    torch.cuda.synchronize()
    check_full(inp, loss, grad, f"two-pass {B}x{C} {dtype}")


def test_twopass_many_rows_per_cta():
    """More rows than CTAs, so every CTA's ring of chunks wraps many times,
    with ragged rows that start at every 4-byte offset."""
    for B, C, dtype in [(700, 5003, "f32"), (400, 50257, "f32"), (330, 32000, "bf16"),
                        (160, 128256, "bf16"), (2000, 999, "f16")]:
        inp = _case(B, C, dtype, seed=C, sigma=2.0)
        z, t = device_inputs(inp)
        loss, grad = run(z, t, TWOPASS)
        torch.cuda.synchronize()
        check_full(inp, loss, grad, f"two-pass ring wrap {dtype} {B}x{C}")


def test_many_rows_per_cluster():
    """More rows than clusters: the shared-memory rings wrap several times."""
    for B, dtype, C, K in [(1500, "f32", 3000, 1), (1500, "bf16", 9000, 2), (1500, "f32", 20000, 2),
                           (1500, "f32", 50257, 3), (600, "f32", 50257, 4), (100, "f32", 20000, 4),
                           (77, "bf16", 9000, 8), (300, "bf16", 128256, 4)]:
        inp = _case(B, C, dtype, seed=C + K, sigma=2.0)
        z, t = device_inputs(inp)
        loss, grad = run(z, t, SPLIT, K)
        torch.cuda.synchronize()
        check_full(inp, loss, grad, f"ring wrap {dtype} C={C} K={K}")
    inp = _case(20000, 100, "bf16", seed=5)
    z, t = device_inputs(inp)
    loss, grad = run(z, t, WARP)
    torch.cuda.synchronize()
    check_full(inp, loss, grad, "warp ring wrap")


# ------------------------------------------------------------ f16 logits

F16_CASES = [(WARP, 0, 300, 1000), (WARP, 0, 7, 4095), (SPLIT, 1, 5, 20000), (SPLIT, 1, 3, 32000),
             (SPLIT, 2, 4, 50257), (SPLIT, 4, 6, 128256), (SPLIT, 8, 2, 250000),
             (STREAM, 0, 3, 10000), (AUTO, 0, 4, 600000)]


@pytest.mark.parametrize("path,split,B,C", F16_CASES)
def test_f16_logits(path, split, B, C):
    """IEEE binary16 logits on every path: loss to the fp32 bound, gradient
    within 1 f16 ulp of the oracle run on the f16 values."""
    inp = _case(B, C, "f16", seed=B + C, sigma=3.0)
    z, t = device_inputs(inp)
    assert z.dtype == torch.float16
    loss, grad = run(z, t, path, split)
    torch.cuda.synchronize()
    assert grad.dtype == torch.float16
    check_full(inp, loss, grad, f"f16 path {path} K={split} {B}x{C}")


def test_f16_refuses_slices_beyond_64kb():
    """f16 rows are built for slices of at most 8 vectors per thread."""
    inp = _case(2, 40000, "f16", seed=1)
    z, t = device_inputs(inp)
    with pytest.raises(ce.CEError) as ei:
        run(z, t, SPLIT, 1)
    assert ei.value.status == 9


# ------------------------------------------------------ pointer alignment

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("path,split,C", [(WARP, 0, 37), (WARP, 0, 1001), (WARP, 0, 5003),
                                          (SPLIT, 1, 5003),
                                          (SPLIT, 4, 7001), (STREAM, 0, 5003),
                                          (TWOPASS, 0, 3), (TWOPASS, 0, 5003)])
@pytest.mark.parametrize("zoff,goff", [(1, 0), (0, 1), (3, 2), (1, 1)])
def test_unaligned_tensors(dtype, path, split, C, zoff, goff):
    """Logits and grad starting at any element offset (not 16-byte aligned),
    with an unaligned end: the copy cannot cover the first and last bytes."""
    B = 5
    inp = _case(B, C, dtype, seed=C + zoff * 10 + goff, sigma=2.0)
    z0, t = device_inputs(inp)
    n = B * C
    zbuf = torch.empty(n + 16, dtype=z0.dtype, device="cuda")
    zbuf.fill_(float("nan"))
    z = zbuf[zoff:zoff + n].view(B, C)
    z.copy_(z0)
    gbuf = torch.full((n + 16,), 7.0, dtype=z0.dtype, device="cuda")
    g = gbuf[goff:goff + n].view(B, C)
    loss = torch.empty(1, dtype=torch.float32, device="cuda")
    ce.ce_fwd_bwd_path(z, t, loss, g, None, path, split)
    torch.cuda.synchronize()
    check_full(inp, loss, g, f"offsets z+{zoff} g+{goff}")
    # nothing outside the grad tensor was written
    assert torch.all(gbuf[:goff] == 7.0) and torch.all(gbuf[goff + n:] == 7.0)


# ------------------------------------------------------------- data errors

@pytest.mark.parametrize("path,split,C,dtype", [(WARP, 0, 100, "f32"), (WARP, 0, 9000, "bf16"),
                                                (SPLIT, 1, 9000, "bf16"),
                                                (SPLIT, 4, 9000, "f32"), (STREAM, 0, 9000, "f32"),
                                                (TWOPASS, 0, 9000, "f32")])
def test_out_of_range_targets(path, split, C, dtype):
    """Reading: an out-of-range target gives a NaN loss, a softmax/B gradient
    row (no one-hot term) and one count per bad row; other rows unaffected."""
    B = 6
    inp = _case(B, C, dtype, seed=C + path)
    inp.targets[1] = -1
    inp.targets[4] = C
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        ce.ce_get_device_errors(s)  # clear
        z, t = device_inputs(inp)
        loss, grad = run(z, t, path, split, s)
        bad, tmo = ce.ce_get_device_errors(s)
    assert (bad, tmo) == (2, 0)
    assert ce.ce_get_device_errors(s) == (0, 0)
    check_full(inp, loss, grad, "bad targets")


# ------------------------------------------------------ stated properties

@pytest.mark.parametrize("path,split,C,dtype", [(WARP, 0, 1000, "f32"), (WARP, 0, 9001, "bf16"),
                                                (SPLIT, 1, 32000, "bf16"),
                                                (SPLIT, 4, 50257, "f32"), (STREAM, 0, 9000, "bf16"),
                                                (TWOPASS, 0, 50257, "f32"),
                                                (TWOPASS, 0, 128256, "bf16")])
def test_bitwise_deterministic(path, split, C, dtype):
    inp = _case(64, C, dtype, seed=77)
    z, t = device_inputs(inp)
    loss0, grad0 = run(z, t, path, split)
    for _ in range(9):
        loss, grad = run(z, t, path, split)
        assert torch.equal(loss, loss0)
        assert torch.equal(grad.view(torch.int16) if dtype == "bf16" else grad.view(torch.int32),
                           grad0.view(torch.int16) if dtype == "bf16" else grad0.view(torch.int32))


def test_structured_rows_small():
    """The stress recipe (uniform rows, +80 spikes, 30*N(0,1)) and the peaked
    bf16 recipe at sizes the oracle compares element by element."""
    stress = wl.Workload("stress_small", 400, 5003, "f32", seed=4, sigma=30.0,
                         uniform_frac=0.01, spike=80.0)
    peaked = wl.Workload("peaked_small", 256, 12829, "bf16", seed=3, sigma=3.0, peak=8.0)
    for w, paths in [(stress, [(AUTO, 0), (SPLIT, 1), (SPLIT, 2), (SPLIT, 4), (STREAM, 0),
                               (TWOPASS, 0)]),
                     (peaked, [(AUTO, 0), (SPLIT, 1), (SPLIT, 8), (STREAM, 0), (TWOPASS, 0)])]:
        inp = wl.make_inputs(w)
        z, t = device_inputs(inp)
        for path, split in paths:
            loss, grad = run(z, t, path, split)
            torch.cuda.synchronize()
            check_full(inp, loss, grad, f"{w.name} path {path}/{split}")


# ------------------------------------------------------ full-size workloads

EXPECTED_PLAN = {
    "classifier_4096x1000_f32": ("rows_warp", 1),
    "lm_head_8192x32000_bf16": ("row_split", 1),
    "lm_head_4096x128256_bf16_peaked": ("row_twopass", 1),
    "stress_16384x50257_f32": ("row_twopass", 1),
}


def _row_sums_ok(grad, B, dtype):
    worst = 0.0
    for r0 in range(0, grad.shape[0], 512):
        blk = grad[r0:r0 + 512]
        s = blk.double().sum(dim=1).abs()
        if dtype == "f32":
            worst = max(worst, float(s.max()) * B)
        else:
            g = blk.float()
            e = torch.floor(torch.log2(torch.clamp(g.abs(), min=2.0 ** -126)))
            bound = ROWSUM_ATOL_TIMES_B / B + 0.5 * torch.exp2(e - 7).double().sum(dim=1)
            assert torch.all(s <= bound), "bf16 row sums beyond their rounding bound"
    if dtype == "f32":
        assert worst <= ROWSUM_ATOL_TIMES_B, f"row sum {worst:.3g}/B"


@pytest.mark.parametrize("name", ["classifier_4096x1000_f32", "lm_head_8192x32000_bf16",
                                  "lm_head_4096x128256_bf16_peaked", "stress_16384x50257_f32"])
def test_full_size_workload(name):
    w = wl.WORKLOADS_BY_NAME[name]
    plan = ce.ce_query_plan(w.B, w.C, w.dtype_code)
    assert (plan["path_name"], plan["split"]) == EXPECTED_PLAN[name]
    inp = wl.make_inputs(w)
    z, t = device_inputs(inp)
    loss, grad = run(z, t)
    torch.cuda.synchronize()
    check_all_rows(inp, loss, grad, name)
    _row_sums_ok(grad, w.B, w.dtype)
    # uniform rows: softmax is exactly 1/C
    for r in inp.uniform_rows[:4]:
        g = grad_rows_host(grad, [r])[0]
        expect = np.full(w.C, 1.0 / w.C / w.B)
        expect[inp.targets[r]] -= 1.0 / w.B
        check_grad(g[None], expect[None], w.B, w.dtype, "uniform row")
    bad, tmo = ce.ce_get_device_errors()
    assert (bad, tmo) == (0, 0)


@pytest.mark.parametrize("name", ["lm_head_8192x32000_bf16", "lm_head_4096x128256_bf16_peaked"])
def test_bf16_row_sums_before_rounding(name):
    """The row-sum bound 1e-6/B on the fp32 gradient values the kernel rounds
    to bf16 (the test hook records them): a bf16 output can only hold it to
    its rounding.  The recorded values round to exactly the bf16 gradient, and
    recording them leaves the gradient's bits unchanged."""
    w = wl.WORKLOADS_BY_NAME[name]
    inp = wl.make_inputs(w)
    z, t = device_inputs(inp)
    loss0, grad0 = run(z, t)
    loss = torch.empty(1, dtype=torch.float32, device="cuda")
    grad = torch.empty_like(z)
    g32 = torch.empty(z.shape, dtype=torch.float32, device="cuda")
    ce.ce_fwd_bwd_test(z, t, loss, grad, None, AUTO, 0, grad_f32_out=g32)
    torch.cuda.synchronize()
    assert torch.equal(loss, loss0) and torch.equal(grad.view(torch.int16), grad0.view(torch.int16))
    worst = 0.0
    for r0 in range(0, w.B, 512):
        blk = g32[r0:r0 + 512]
        assert torch.equal(blk.to(torch.bfloat16).view(torch.int16),
                           grad[r0:r0 + 512].view(torch.int16)), "recorded values are not the rounded ones"
        worst = max(worst, float(blk.double().sum(dim=1).abs().max()) * w.B)
    assert worst <= ROWSUM_ATOL_TIMES_B, f"{name}: fp32 row sum {worst:.3g}/B before rounding"


def test_stress_workload_other_paths():
    """The streaming path and the cluster split (K = 2) on the full ragged
    stress workload, every element."""
    w = wl.WORKLOADS_BY_NAME["stress_16384x50257_f32"]
    inp = wl.make_inputs(w)
    z, t = device_inputs(inp)
    for path, split in ((STREAM, 0), (SPLIT, 2)):
        loss, grad = run(z, t, path, split)
        torch.cuda.synchronize()
        check_all_rows(inp, loss, grad, f"stress via path {path} K={split}")
        del loss, grad


# --------------------------------------------------------------- runtime

def test_graph_capture_and_replay():
    inp = _case(512, 3000, "bf16", seed=9)
    z, t = device_inputs(inp)
    loss = torch.empty(1, dtype=torch.float32, device="cuda")
    grad = torch.empty_like(z)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        ce.ce_fwd_bwd(z, t, loss, grad, s)  # sizes the stream's workspace
        s.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            ce.ce_fwd_bwd(z, t, loss, grad, s)
    inp2 = _case(512, 3000, "bf16", seed=10)
    z2, t2 = device_inputs(inp2)
    z.copy_(z2)
    t.copy_(t2)
    loss.fill_(float("nan"))
    graph.replay()
    torch.cuda.synchronize()
    check_full(inp2, loss, grad, "graph replay")


def test_graph_survives_workspace_growth():
    """A graph captured before its stream's workspace grows (here: a larger
    batch on the streaming path, which adds per-chunk partials) still replays
    correctly afterwards: the outgrown workspace stays allocated."""
    inp = _case(256, 3000, "f32", seed=21)
    z, t = device_inputs(inp)
    loss = torch.empty(1, dtype=torch.float32, device="cuda")
    grad = torch.empty_like(z)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        ce.ce_fwd_bwd(z, t, loss, grad, s)
        s.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            ce.ce_fwd_bwd(z, t, loss, grad, s)
        big = _case(4000, 5000, "f32", seed=22)
        zb, tb = device_inputs(big)
        lb, gb = run(zb, tb, STREAM, 0, s)
    s.synchronize()
    check_full(big, lb, gb, "the call that grew the workspace")
    inp2 = _case(256, 3000, "f32", seed=23)
    z2, t2 = device_inputs(inp2)
    z.copy_(z2)
    t.copy_(t2)
    loss.fill_(float("nan"))
    with torch.cuda.stream(s):
        graph.replay()
    s.synchronize()
    check_full(inp2, loss, grad, "graph replayed after the growth")
    l_now, g_now = run(z, t, AUTO, 0, s)
    s.synchronize()
    assert torch.equal(l_now, loss) and torch.equal(g_now, grad)


def test_capture_needs_a_sized_workspace():
    z = torch.zeros(4, 8, device="cuda")
    t = torch.zeros(4, dtype=torch.int32, device="cuda")
    loss = torch.empty(1, device="cuda")
    grad = torch.empty_like(z)
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with pytest.raises(ce.CEError) as ei:
            with torch.cuda.graph(graph, stream=s):
                ce.ce_fwd_bwd(z, t, loss, grad, s)
    assert ei.value.status == 8


def test_concurrent_streams():
    cases = [_case(300, 7000, "f32", seed=1), _case(200, 5000, "bf16", seed=2)]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = []
    for inp, s in zip(cases, streams):
        with torch.cuda.stream(s):
            z, t = device_inputs(inp)
            outs.append(run(z, t, AUTO, 0, s))
    torch.cuda.synchronize()
    for inp, (loss, grad) in zip(cases, outs):
        check_full(inp, loss, grad, "concurrent streams")


def test_forced_path_limits():
    z = torch.zeros(2, 100000, device="cuda")
    t = torch.zeros(2, dtype=torch.int32, device="cuda")
    loss = torch.empty(1, device="cuda")
    grad = torch.empty_like(z)
    for path, split in [(WARP, 0), (SPLIT, 5), (SPLIT, 1)]:
        with pytest.raises(ce.CEError) as ei:
            ce.ce_fwd_bwd_path(z, t, loss, grad, None, path, split)
        assert ei.value.status == 9


def test_error_codes_on_device_pointers():
    z = torch.zeros(4, 8, device="cuda")
    t = torch.zeros(4, dtype=torch.int32, device="cuda")
    loss = torch.empty(1, device="cuda")
    grad = torch.empty_like(z)
    raw = ce.ce_fwd_bwd_raw
    assert raw(z.data_ptr(), t.data_ptr(), 4, 8, 0, loss.data_ptr(), grad.data_ptr()) == 0
    assert raw(z.data_ptr(), t.data_ptr(), 4, 8, 0, loss.data_ptr(), z.data_ptr()) == 6
    assert raw(z.data_ptr() + 2, t.data_ptr(), 4, 8, 0, loss.data_ptr(), grad.data_ptr()) == 4
    assert raw(z.data_ptr(), t.data_ptr(), 4, 8, 7, loss.data_ptr(), grad.data_ptr()) == 3
    torch.cuda.synchronize()
