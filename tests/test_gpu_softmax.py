"""GPU parity of the row-wise softmax forward and backward (ce_softmax_fwd,
ce_softmax_bwd) against the fp64 oracle, on every kernel path.

Tolerances, derived from the arithmetic:
  forward, fp32:   |p - p_ref| <= 1e-6 per element and |sum_c p - 1| <= 1e-6
                   per row (the gradient bounds of the loss at B = 1: the
                   forward runs the same row arithmetic without the 1/B);
  forward, 16-bit: |p - p_ref| <= 1 ulp of p_ref in the output type (0 allowed
                   below 2^-126, the kernels flush subnormal fp32 results), and
                   |sum_c p - 1| <= 1e-6 + sum_c ulp(p_c) / 2;
  backward:        the row's dot product is an fp32 sum of at most n = C / 256
                   + 32 rounded terms in sequence, so |dot - dot_ref| <= n 2^-24
                   sum_c |p_c dy_c|; then one subtraction and one product, so
                   |dx - dx_ref| <= |p| (|dot - dot_ref| + 2^-23 |dy - dot|)
                   (+ 2^-126 for flushed products); 16-bit outputs add the
                   rounding to the output type, one ulp at most.
"""

import numpy as np
import pytest

import workloads as wl

from parity import ulp_bf16, ulp_f16

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU-only machines
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import softmax_cross_entropy_row_gb300 as ce  # noqa: E402
import oracle  # noqa: E402

AUTO, WARP, SPLIT, STREAM, TWOPASS = (ce.CE_PATH_AUTO, ce.CE_PATH_ROWS_WARP,
                                      ce.CE_PATH_ROW_SPLIT, ce.CE_PATH_STREAM,
                                      ce.CE_PATH_ROW_TWOPASS)
TORCH_DT = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}

# (path, split, B, C): the warp kernel (ragged and exact rows), the split
# kernel at K = 1 (barrier per row), K = 4 (staged slices) and the pipelined
# K = 2, the streaming path, the two-pass path (short, chunk-sized and long
# rows)
PATHS = [(WARP, 0, 1, 1), (WARP, 0, 7, 7), (WARP, 0, 300, 1000), (WARP, 0, 5, 2047),
         (WARP, 0, 9, 9001),
         (SPLIT, 1, 3, 17), (SPLIT, 1, 5, 20000), (SPLIT, 4, 6, 40000), (SPLIT, 2, 3, 50257),
         (SPLIT, 8, 2, 128256), (STREAM, 0, 1, 1), (STREAM, 0, 3, 10000), (STREAM, 0, 2, 4097),
         (TWOPASS, 0, 1, 1), (TWOPASS, 0, 7, 7), (TWOPASS, 0, 5, 4099), (TWOPASS, 0, 3, 50257),
         (TWOPASS, 0, 2, 300001)]


@pytest.fixture(scope="module", autouse=True)
def _built():
    ce.build()
    ce.load_library()
    oracle.build()
    yield
    torch.cuda.synchronize()


def _to_device(x: np.ndarray, dtype: str):
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def _to_host_typed(t, dtype: str) -> np.ndarray:
    """The tensor's values in the container the oracle reads for `dtype`."""
    if dtype == "bf16":
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def _half_ulp_row_sums(p, dtype: str):
    """sum_c ulp(p_c) / 2 per row in the output type, on the device (exact
    powers of two from the binade of each element)."""
    _, e = torch.frexp(p.double())  # |p| = m 2^e, m in [1/2, 1): binade e - 1
    lo, mant = (-14, 10) if dtype == "f16" else (-126, 7)
    ulp = torch.exp2((torch.clamp(e - 1, min=lo) - mant).double())
    return (0.5 * ulp).sum(dim=1).cpu().numpy()


def _ulp(dtype):
    return ulp_f16 if dtype == "f16" else ulp_bf16


def check_probs(p: np.ndarray, p_ref: np.ndarray, dtype: str, what: str = "") -> None:
    assert p.shape == p_ref.shape
    rs = np.abs(p.sum(axis=1) - 1.0)
    if dtype == "f32":
        err = np.abs(p - p_ref)
        assert float(err.max()) <= 1e-6, f"{what}: max |p - p_ref| = {float(err.max()):.3g}"
        assert float(rs.max()) <= 1e-6, f"{what}: row sum off 1 by {float(rs.max()):.3g}"
        return
    ulp = _ulp(dtype)
    flushed = (p == 0) & (np.abs(p_ref) < 2.0 ** -126)
    bad = (np.abs(p - p_ref) > ulp(p_ref)) & ~flushed
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"{what}: {int(bad.sum())} probabilities beyond 1 ulp, first at {i}: "
                             f"{p[i]!r} vs {p_ref[i]!r}")
    bound = 1e-6 + 0.5 * ulp(p).sum(axis=1)
    assert np.all(rs <= bound), f"{what}: {dtype} row sum beyond its rounding bound"


def check_dx(dx, dx_ref, p, dy, dtype: str, what: str = "") -> None:
    C = p.shape[1]
    n = C / 256 + 32
    dot_abs = np.abs(p * dy).sum(axis=1, keepdims=True)
    dot = (p * dy).sum(axis=1, keepdims=True)
    tol = np.abs(p) * (n * 2.0 ** -24 * dot_abs + 2.0 ** -23 * np.abs(dy - dot)) + 2.0 ** -126
    if dtype != "f32":
        tol = tol + _ulp(dtype)(np.abs(dx_ref) + tol)
    excess = np.abs(dx - dx_ref) - tol
    if (excess > 0).any():
        i = tuple(np.argwhere(excess > 0)[0])
        raise AssertionError(f"{what}: {int((excess > 0).sum())} elements beyond the bound, first "
                             f"at {i}: {dx[i]!r} vs {dx_ref[i]!r} (tol {tol[i]:.3g})")


def _probs(z, **kw):
    p = torch.empty_like(z)
    ce.ce_softmax_fwd(z, p, **kw)
    return p


# ------------------------------------------------------------------ forward

@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("path,split,B,C", PATHS)
def test_forward_on_every_path(path, split, B, C, dtype):
    inp = wl.random_case(B, C, dtype, seed=B * 131 + C + split, sigma=3.0)
    z = _to_device(inp.logits, dtype)
    p = _probs(z, path=path, split=split)
    torch.cuda.synchronize()
    check_probs(p.double().cpu().numpy(), oracle.softmax(inp.logits), dtype,
                f"path {path} K={split} {B}x{C} {dtype}")


def test_forward_special_rows():
    """A constant row gives 1/C; a row with one dominant logit gives a one-hot
    (the others underflow to 0); a uniform shift of the row changes nothing."""
    C = 2000  # within the warp kernel's 8 KB rows
    z = np.zeros((4, C), dtype=np.float32)
    z[1] = 2.5
    z[2, 17] = 200.0
    z[3] = (np.random.default_rng(3).integers(-3000, 3000, C) * 2.0 ** -7).astype(np.float32)
    zs = z.copy()
    zs[3] += np.float32(64.0)  # exact on this grid
    for path, split in [(WARP, 0), (SPLIT, 1), (STREAM, 0)]:
        p = _probs(_to_device(z, "f32"), path=path, split=split).double().cpu().numpy()
        ps = _probs(_to_device(zs, "f32"), path=path, split=split).double().cpu().numpy()
        assert np.allclose(p[0], 1.0 / C, rtol=2e-6, atol=0) and np.allclose(p[1], 1.0 / C, rtol=2e-6)
        assert p[2, 17] == 1.0 and np.count_nonzero(p[2]) == 1
        check_probs(p, oracle.softmax(z), "f32", f"special rows, path {path}")
        check_probs(ps[3:], oracle.softmax(z[3:]), "f32", f"shifted row, path {path}")


@pytest.mark.parametrize("name", ["classifier_4096x1000_f32", "lm_head_8192x32000_bf16",
                                  "lm_head_4096x128256_bf16_peaked"])
def test_forward_full_size(name):
    """The headline shapes through the planner's own choice: sampled rows
    against the oracle element by element, every row's sum."""
    w = wl.WORKLOADS_BY_NAME[name]
    inp = wl.make_inputs(w)
    z = _to_device(inp.logits, w.dtype)
    p = _probs(z)
    torch.cuda.synchronize()
    sums = p.double().sum(dim=1).cpu().numpy()
    ulp_half_sum = 0.0 if w.dtype == "f32" else _half_ulp_row_sums(p, w.dtype)
    assert np.all(np.abs(sums - 1.0) <= 1e-6 + ulp_half_sum), name
    rows = np.unique(np.concatenate([[0, w.B - 1], np.random.default_rng(1).integers(0, w.B, 48)]))
    got = p.index_select(0, torch.as_tensor(rows, device="cuda")).double().cpu().numpy()
    check_probs(got, oracle.softmax(inp.logits, row_ids=rows), w.dtype, name)


# ----------------------------------------------------------------- backward

def _bwd_case(B, C, dtype, seed):
    """Probabilities from the forward of seeded logits and a normal upstream
    gradient, both in `dtype`."""
    inp = wl.random_case(B, C, dtype, seed=seed, sigma=2.0)
    p = _probs(_to_device(inp.logits, dtype))
    g = torch.Generator(device="cpu").manual_seed(seed)
    dy = torch.randn(B, C, generator=g).to(TORCH_DT[dtype]).cuda()
    return p, dy


def _check_bwd(p, dy, dx, dtype, what):
    ph, dyh = _to_host_typed(p, dtype), _to_host_typed(dy, dtype)
    ref = oracle.softmax_bwd(ph, dyh)
    check_dx(dx.double().cpu().numpy(), ref, p.double().cpu().numpy(), dy.double().cpu().numpy(),
             dtype, what)


# rows the register kernels take (16-byte multiples, at most 64 KB: a warp
# per row up to 4 KB, 128 threads per row up to 16 KB -- four rows of a CTA
# at once, groups with unequal row counts -- and 512 beyond) and rows they
# refuse: odd widths and rows beyond 64 KB
BWD_SHAPES = [(1, 4), (3, 8), (64, 1000), (300, 1024), (7, 8192), (2, 16384), (5, 16000),
              (9, 3000), (1030, 2048), (3, 4096),
              (1, 1), (3, 5), (9, 1001), (4, 20000), (2, 50257)]


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("B,C", BWD_SHAPES)
def test_backward_shapes(B, C, dtype):
    p, dy = _bwd_case(B, C, dtype, seed=B * 7 + C)
    dx = torch.empty_like(p)
    ce.ce_softmax_bwd(p, dy, dx)
    torch.cuda.synchronize()
    _check_bwd(p, dy, dx, dtype, f"bwd {B}x{C} {dtype}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_backward_in_place_and_unaligned(dtype):
    """dx written over p or over dy gives the same bits as a separate
    output; tensors at an offset that breaks 16-byte alignment take the
    two-pass kernel and still agree with the oracle."""
    B, C = 6, 4096
    p, dy = _bwd_case(B, C, dtype, seed=99)
    dx = torch.empty_like(p)
    ce.ce_softmax_bwd(p, dy, dx)
    over_p, over_dy = p.clone(), dy.clone()
    ce.ce_softmax_bwd(over_p, dy, over_p)
    ce.ce_softmax_bwd(p, over_dy, over_dy)
    torch.cuda.synchronize()
    assert torch.equal(over_p, dx) and torch.equal(over_dy, dx)
    _check_bwd(p, dy, dx, dtype, f"in place {dtype}")
    # one element in: the rows stay contiguous but lose 16-byte alignment
    flat_p = torch.empty(B * C + 1, dtype=p.dtype, device="cuda")
    flat_dy = torch.empty_like(flat_p)
    flat_dx = torch.empty_like(flat_p)
    pu = flat_p[1:].view(B, C)
    dyu = flat_dy[1:].view(B, C)
    dxu = flat_dx[1:].view(B, C)
    pu.copy_(p)
    dyu.copy_(dy)
    ce.ce_softmax_bwd(pu, dyu, dxu)
    torch.cuda.synchronize()
    _check_bwd(p, dy, dxu, dtype, f"unaligned {dtype}")


@pytest.mark.parametrize("name", ["lm_head_8192x32000_bf16", "classifier_4096x1000_f32"])
def test_backward_full_size(name):
    w = wl.WORKLOADS_BY_NAME[name]
    p, dy = _bwd_case(w.B, w.C, w.dtype, seed=5)
    dx = torch.empty_like(p)
    ce.ce_softmax_bwd(p, dy, dx)
    torch.cuda.synchronize()
    rows = np.unique(np.concatenate([[0, w.B - 1], np.random.default_rng(2).integers(0, w.B, 32)]))
    sel = torch.as_tensor(rows, device="cuda")
    _check_bwd(p.index_select(0, sel), dy.index_select(0, sel), dx.index_select(0, sel), w.dtype,
               name)
