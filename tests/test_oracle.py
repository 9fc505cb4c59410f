"""Pins of the fp64 oracle against facts that do not come from the oracle.

Each test checks the oracle against the mathematics of softmax cross-entropy
(closed forms, invariants, finite differences), an independent multi-precision
restatement, or an independent library (torch CPU fp64).  A plausible slip in
the oracle -- a dropped max shift, a wrong sign, a wrong index, a missing 1/B,
a transposed layout -- fails at least one of them.
"""

import math

import numpy as np
import pytest

import workloads as wl

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _case(z, t):
    z = np.ascontiguousarray(np.asarray(z, dtype=np.float32))
    if z.ndim == 1:
        z = z[None, :]
    t = np.ascontiguousarray(np.asarray(t, dtype=np.int32).reshape(-1))
    return z, t


# ---------------------------------------------------------------- closed forms

@pytest.mark.parametrize("C", [1, 2, 3, 10, 1000, 50257])
@pytest.mark.parametrize("v", [0.0, -7.5, 42.25, 1000.0])
def test_uniform_row_gives_log_c(oracle_mod, C, v):
    """All logits equal: softmax is 1/C, so l = ln C and g = (1/C - [c=t]) / B."""
    B = 4
    z = np.full((B, C), v, dtype=np.float32)
    t = np.arange(B, dtype=np.int32) % C
    L, l, g = oracle_mod.loss_and_grad(z, t)
    assert np.allclose(l, math.log(C), rtol=1e-14, atol=1e-14)
    assert L == pytest.approx(math.log(C), rel=1e-14, abs=1e-14)
    expect = np.full((B, C), 1.0 / C / B)
    expect[np.arange(B), t] -= 1.0 / B
    assert np.allclose(g, expect, rtol=0, atol=1e-16)


@pytest.mark.parametrize("K", [0.5, 3.0, 20.0, 60.0])
def test_dominant_logit(oracle_mod, K):
    """One logit K above C-1 zeros.

    Target on the dominant class: l = log(1 + (C-1) e^-K) (-> 0 as K grows).
    Target on a zero:            l = log(e^K + C - 1).
    """
    C, j = 7, 3
    row = np.zeros(C, dtype=np.float32)
    row[j] = K
    z = np.stack([row, row])
    t = np.array([j, 0], dtype=np.int32)
    l, g = oracle_mod.rows(z, t)
    # log(S) with S near 1 carries an absolute (not relative) error of ~1 ulp of 1
    assert l[0] == pytest.approx(math.log1p((C - 1) * math.exp(-K)), rel=1e-13, abs=1e-15)
    assert l[1] == pytest.approx(K + math.log1p((C - 1) * math.exp(-K)), rel=1e-14)
    p_dom = 1.0 / (1.0 + (C - 1) * math.exp(-K))
    # p - 1 cancels: both sides carry ~1 ulp of 1 (over B = 2) of absolute error
    assert g[0, j] == pytest.approx((p_dom - 1.0) / 2, rel=1e-12, abs=2e-16)
    assert g[1, j] == pytest.approx(p_dom / 2, rel=1e-13)
    assert g[1, 0] == pytest.approx(((1 - p_dom) / (C - 1) - 1.0) / 2, rel=1e-13)


def test_two_classes_is_softplus(oracle_mod):
    """C = 2: l = softplus(z_other - z_target) = log(1 + e^(z_o - z_t))."""
    rng = np.random.default_rng(5)
    z = (rng.standard_normal((64, 2)) * 6).astype(np.float32)
    t = rng.integers(0, 2, 64).astype(np.int32)
    l = oracle_mod.rows(z, t, grad=False)
    zt = z[np.arange(64), t].astype(np.float64)
    zo = z[np.arange(64), 1 - t].astype(np.float64)
    d = zo - zt
    softplus = np.maximum(d, 0) + np.log1p(np.exp(-np.abs(d)))
    assert np.allclose(l, softplus, rtol=1e-14, atol=1e-15)


def test_single_class(oracle_mod):
    """C = 1: the softmax is 1, so l = 0 and g = 0."""
    z = np.array([[3.5], [-2.0], [0.0]], dtype=np.float32)
    t = np.zeros(3, dtype=np.int32)
    L, l, g = oracle_mod.loss_and_grad(z, t)
    assert np.all(l == 0.0) and L == 0.0 and np.all(g == 0.0)


# ------------------------------------------------------------------ invariants

def test_shift_invariance_large_magnitude(oracle_mod):
    """l(z + a) = l(z): exercises the max shift (exp(1000) overflows without it)."""
    rng = np.random.default_rng(7)
    base = rng.integers(-64, 64, size=(5, 300)) / 8.0  # exact in fp32 after +-1024
    t = rng.integers(0, 300, 5).astype(np.int32)
    l0, g0 = oracle_mod.rows(base.astype(np.float32), t)
    for a in (1024.0, -1024.0, 80.0):
        l1, g1 = oracle_mod.rows((base + a).astype(np.float32), t)
        assert np.all(np.isfinite(l1))
        assert np.allclose(l1, l0, rtol=1e-13, atol=1e-12)
        assert np.allclose(g1, g0, rtol=0, atol=1e-16)


def test_permutation_equivariance(oracle_mod):
    rng = np.random.default_rng(11)
    B, C = 6, 37
    z = (rng.standard_normal((B, C)) * 3).astype(np.float32)
    t = rng.integers(0, C, B).astype(np.int32)
    perm = rng.permutation(C)
    inv = np.argsort(perm)
    l0, g0 = oracle_mod.rows(z, t)
    l1, g1 = oracle_mod.rows(np.ascontiguousarray(z[:, perm]), inv[t].astype(np.int32))
    assert np.allclose(l1, l0, rtol=1e-14)
    # the class sum runs in another order, so S differs by a few ulp
    assert np.allclose(g1, g0[:, perm], rtol=1e-14, atol=1e-18)


@pytest.mark.parametrize("shape,sigma", [((16, 10), 1.0), ((9, 1000), 2.0),
                                         ((3, 5000), 30.0), ((5, 3), 0.01)])
def test_row_invariants(oracle_mod, shape, sigma):
    """l >= 0; sum_c g = 0; 0 <= g_c < 1/B off target; -1/B < g_t <= 0;
    and l_b = -log(1 + B g_(b,t_b)) ties the loss to the gradient."""
    B, C = shape
    inp = wl.random_case(B, C, "f32", seed=B * 1000 + C, sigma=sigma)
    L, l, g = oracle_mod.loss_and_grad(inp.logits, inp.targets)
    t = inp.targets
    assert np.all(l >= 0)
    # exact zero up to fp64 rounding of C terms (the required bar is 1e-6 / B)
    assert np.all(np.abs(g.sum(axis=1)) <= 1e-12 / B)
    off = g.copy()
    off[np.arange(B), t] = 0.0
    # the bounds are strict in exact arithmetic; rounding can reach them
    assert np.all(off >= 0) and np.all(off <= 1.0 / B)
    gt = g[np.arange(B), t]
    assert np.all(gt >= -1.0 / B) and np.all(gt <= 0)
    p_t = 1.0 + B * gt
    ok = p_t > 1e-6  # where p_t is not lost to cancellation
    consistent = -np.log(p_t[ok])
    assert np.allclose(consistent, l[ok], rtol=1e-8, atol=1e-10)
    assert L == pytest.approx(math.fsum(l) / B, rel=1e-15)


def test_gradient_matches_finite_differences(oracle_mod):
    """Central differences of L with exact fp32 steps match g to O(h^2)."""
    rng = np.random.default_rng(3)
    B, C = 3, 5
    h = 2.0 ** -10
    z = (rng.integers(-512, 512, size=(B, C)) * h).astype(np.float32)
    t = rng.integers(0, C, B).astype(np.int32)
    L0, _, g = oracle_mod.loss_and_grad(z, t)
    for b in range(B):
        for c in range(C):
            zp = z.copy()
            zm = z.copy()
            zp[b, c] += np.float32(h)
            zm[b, c] -= np.float32(h)
            step = float(zp[b, c]) - float(zm[b, c])
            assert step == 2 * h
            Lp, _, _ = oracle_mod.loss_and_grad(zp, t)
            Lm, _, _ = oracle_mod.loss_and_grad(zm, t)
            assert (Lp - Lm) / step == pytest.approx(g[b, c], abs=2e-7)


# --------------------------------------------- independent restatements / libs

def test_multiprecision_bruteforce(oracle_mod):
    """50-digit restatement without the max shift: l = log(sum e^z) - z_t,
    g = (e^z_c / sum e^z - [c=t]) / B, on tiny inputs in row-major [B, C]."""
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 50
    rng = np.random.default_rng(17)
    for B, C in [(1, 1), (1, 2), (2, 3), (4, 6), (3, 5)]:
        z = (rng.standard_normal((B, C)) * 4).astype(np.float32)
        t = rng.integers(0, C, B).astype(np.int32)
        L, l, g = oracle_mod.loss_and_grad(z, t)
        total = mpmath.mpf(0)
        for b in range(B):
            ex = [mpmath.exp(mpmath.mpf(float(z[b, c]))) for c in range(C)]
            s = mpmath.fsum(ex)
            lb = mpmath.log(s) - mpmath.mpf(float(z[b, t[b]]))
            total += lb
            assert float(lb) == pytest.approx(l[b], rel=1e-14, abs=1e-15)
            for c in range(C):
                gb = (ex[c] / s - (1 if c == t[b] else 0)) / B
                assert float(gb) == pytest.approx(g[b, c], rel=1e-12, abs=1e-16)
        assert float(total / B) == pytest.approx(L, rel=1e-14, abs=1e-15)


def test_against_torch_cross_entropy(oracle_mod):
    """torch CPU fp64 F.cross_entropy(reduction='mean') and its autograd."""
    torch = pytest.importorskip("torch")
    B, C = 64, 333
    inp = wl.random_case(B, C, "f32", seed=99, sigma=5.0)
    L, l, g = oracle_mod.loss_and_grad(inp.logits, inp.targets)
    zt = torch.tensor(inp.logits, dtype=torch.float64, requires_grad=True)
    tt = torch.tensor(inp.targets, dtype=torch.int64)
    loss = torch.nn.functional.cross_entropy(zt, tt, reduction="mean")
    loss.backward()
    assert L == pytest.approx(loss.item(), rel=1e-13)
    per_row = torch.nn.functional.cross_entropy(zt.detach(), tt, reduction="none").numpy()
    assert np.allclose(l, per_row, rtol=1e-13, atol=1e-14)
    # torch evaluates exp(log_softmax) in another order: agreement to ~1e-13 relative
    assert np.allclose(g, zt.grad.numpy(), rtol=1e-12, atol=1e-19)


# --------------------------------------------------------------- dtype, errors

def test_bf16_widening_is_exact(oracle_mod):
    """bf16 bit patterns mean the fp32 values with the low 16 bits zero."""
    bits = np.array([[0x3F80, 0x4000, 0xBF80, 0x3F81, 0x4049, 0x0000, 0xC2A0]],
                    dtype=np.uint16)
    values = np.array([[1.0, 2.0, -1.0, 1.0078125, 3.140625, 0.0, -80.0]],
                      dtype=np.float32)
    t = np.array([4], dtype=np.int32)
    lb, gb = oracle_mod.rows(bits, t)
    lf, gf = oracle_mod.rows(values, t)
    assert lb[0] == lf[0] and np.array_equal(gb, gf)
    same = np.full((1, 77), 0x4049, dtype=np.uint16)
    assert oracle_mod.rows(same, np.array([3], np.int32), grad=False)[0] == pytest.approx(
        math.log(77), rel=1e-14)


@pytest.mark.parametrize("bad", [-1, 10, 2**31 - 1, -(2**31)])
def test_out_of_range_target_is_nan_row(oracle_mod, bad):
    """Reading: a target outside [0, C) makes that row's loss NaN (so L is NaN)
    and its gradient softmax/B with no one-hot term; other rows are unaffected."""
    B, C = 3, 10
    inp = wl.random_case(B, C, "f32", seed=5)
    t = inp.targets.copy()
    t[1] = bad
    L, l, g = oracle_mod.loss_and_grad(inp.logits, t)
    assert math.isnan(L) and math.isnan(l[1])
    assert np.all(np.isfinite(l[[0, 2]]))
    z = inp.logits[1].astype(np.float64)
    p = np.exp(z - z.max())
    p /= p.sum()
    assert np.allclose(g[1], p / B, rtol=1e-14, atol=0)
    l_ok, g_ok = oracle_mod.rows(inp.logits, inp.targets)
    assert np.array_equal(l[[0, 2]], l_ok[[0, 2]]) and np.array_equal(g[[0, 2]], g_ok[[0, 2]])


def test_row_subset_matches_full(oracle_mod):
    inp = wl.random_case(40, 129, "bf16", seed=8, sigma=3.0)
    l, g = oracle_mod.rows(inp.logits, inp.targets)
    ids = np.array([39, 0, 17, 17, 5])
    ls, gs = oracle_mod.rows(inp.logits, inp.targets, row_ids=ids)
    assert np.array_equal(ls, l[ids]) and np.array_equal(gs, g[ids])


def test_fwd_bwd_output_types(oracle_mod):
    """The timed entry point returns the same L and narrows g to the logits' type."""
    for dtype in ("f32", "bf16"):
        inp = wl.random_case(33, 77, dtype, seed=21, sigma=2.0)
        L, l, g = oracle_mod.loss_and_grad(inp.logits, inp.targets)
        out = np.empty_like(inp.logits)
        scratch = np.empty(33, dtype=np.float64)
        L2 = oracle_mod.fwd_bwd(inp.logits, inp.targets, out, scratch)
        assert L2 == L
        if dtype == "f32":
            assert np.array_equal(out, g.astype(np.float32))
        else:
            want = wl.f32_to_bf16_bits(g.astype(np.float32))
            assert np.array_equal(out, want)


def test_rejects_bad_arguments(oracle_mod):
    with pytest.raises(ValueError):
        oracle_mod.rows(np.zeros((2, 3), np.float32), np.zeros(3, np.int32))
    with pytest.raises(ValueError):
        oracle_mod.rows(np.zeros((2, 3), np.float32), np.zeros(2, np.int32), row_ids=[2])
    with pytest.raises(TypeError):
        oracle_mod.rows(np.zeros((2, 3), np.float64), np.zeros(2, np.int32))


# ------------------------------------- reductions and the upstream gradient

def test_reductions_against_torch(oracle_mod):
    """sum and none against torch CPU fp64 F.cross_entropy with autograd, with
    an upstream gradient (a scalar for the sum, one value per row for none)."""
    torch = pytest.importorskip("torch")
    B, C = 48, 257
    inp = wl.random_case(B, C, "f32", seed=5, sigma=4.0)
    zt = torch.tensor(inp.logits, dtype=torch.float64, requires_grad=True)
    tt = torch.tensor(inp.targets, dtype=torch.int64)
    # sum, upstream 0.375
    l_sum, g_sum = oracle_mod.rows_ex(inp.logits, inp.targets, oracle_mod.SUM, upstream=0.375)
    loss = torch.nn.functional.cross_entropy(zt, tt, reduction="sum")
    (0.375 * loss).backward()
    assert oracle_mod.reduce(l_sum, oracle_mod.SUM) == pytest.approx(loss.item(), rel=1e-13)
    assert np.allclose(g_sum, zt.grad.numpy(), rtol=1e-12, atol=1e-18)
    # none, per-row upstream u_b
    u = np.linspace(-2.0, 3.0, B)
    zt.grad = None
    l_none, g_none = oracle_mod.rows_ex(inp.logits, inp.targets, oracle_mod.NONE, upstream=u)
    per_row = torch.nn.functional.cross_entropy(zt, tt, reduction="none")
    (per_row * torch.tensor(u)).sum().backward()
    assert np.allclose(l_none, per_row.detach().numpy(), rtol=1e-13, atol=1e-14)
    assert np.allclose(g_none, zt.grad.numpy(), rtol=1e-12, atol=1e-18)


def test_per_row_gradient_matches_finite_differences(oracle_mod):
    """For none, row b's gradient is d l_b / d z_b: central differences of the
    row loss with exact fp32 steps; other rows' losses do not move."""
    rng = np.random.default_rng(11)
    B, C = 3, 4
    h = 2.0 ** -10
    z = (rng.integers(-512, 512, size=(B, C)) * h).astype(np.float32)
    t = rng.integers(0, C, B).astype(np.int32)
    l0, g = oracle_mod.rows_ex(z, t, oracle_mod.NONE)
    for b in range(B):
        for c in range(C):
            zp, zm = z.copy(), z.copy()
            zp[b, c] += np.float32(h)
            zm[b, c] -= np.float32(h)
            lp = oracle_mod.rows_ex(zp, t, oracle_mod.NONE, grad=False)
            lm = oracle_mod.rows_ex(zm, t, oracle_mod.NONE, grad=False)
            assert (lp[b] - lm[b]) / (2 * h) == pytest.approx(g[b, c], abs=2e-7)
            others = [r for r in range(B) if r != b]
            assert np.array_equal(lp[others], l0[others])


def test_reduction_relations(oracle_mod):
    """The mean is the sum over B, with the gradient over B; the per-row losses
    are the same in every reduction; the upstream gradient scales linearly."""
    inp = wl.random_case(16, 300, "bf16", seed=8, sigma=3.0)
    B = 16
    l_m, g_m = oracle_mod.rows_ex(inp.logits, inp.targets, oracle_mod.MEAN)
    l_s, g_s = oracle_mod.rows_ex(inp.logits, inp.targets, oracle_mod.SUM)
    l_n, g_n = oracle_mod.rows_ex(inp.logits, inp.targets, oracle_mod.NONE)
    assert np.array_equal(l_m, l_s) and np.array_equal(l_m, l_n)
    assert oracle_mod.reduce(l_m, oracle_mod.MEAN) * B == pytest.approx(
        oracle_mod.reduce(l_s, oracle_mod.SUM), rel=1e-14)
    assert np.allclose(g_m * B, g_s, rtol=1e-14, atol=0)
    assert np.array_equal(g_s, g_n)
    _, g_u = oracle_mod.rows_ex(inp.logits, inp.targets, oracle_mod.MEAN, upstream=-2.5)
    assert np.allclose(g_u, -2.5 * g_m, rtol=1e-15, atol=0)
    with pytest.raises(ValueError):
        oracle_mod.rows_ex(inp.logits, inp.targets, 3)
    with pytest.raises(ValueError):
        oracle_mod.rows_ex(inp.logits, inp.targets, oracle_mod.NONE, upstream=1.0)


def test_f16_widening_is_exact(oracle_mod):
    """IEEE binary16 bit patterns mean what numpy's float16 says they mean
    (normal, subnormal, the largest finite value, signed zero)."""
    bits = np.array([[0x3C00, 0x4000, 0xBC00, 0x3555, 0x7BFF, 0x0001, 0x0400, 0x8000]],
                    dtype=np.uint16)
    z16 = bits.view(np.float16)
    t = np.array([0], dtype=np.int32)
    l16, g16 = oracle_mod.rows(z16, t)
    z64 = z16.astype(np.float64)
    assert z64[0, 4] == 65504.0 and z64[0, 5] == 2.0 ** -24 and z64[0, 6] == 2.0 ** -14
    # the same row as fp32 values (exactly representable) gives the same fp64 results
    l32, g32 = oracle_mod.rows(z64.astype(np.float32), t)
    assert np.array_equal(l16, l32) and np.array_equal(g16, g32)


# ------------------------------------------------ row softmax, fwd and bwd

def test_softmax_forward_pins(oracle_mod):
    """Rows sum to 1; a uniform row gives 1/C; shift invariance; the target's
    probability is exp(-l) of the loss oracle; torch CPU fp64 softmax."""
    torch = pytest.importorskip("torch")
    inp = wl.random_case(12, 777, "f32", seed=21, sigma=6.0)
    p = oracle_mod.softmax(inp.logits)
    assert np.allclose(p.sum(axis=1), 1.0, rtol=0, atol=1e-13)
    l = oracle_mod.rows(inp.logits, inp.targets, grad=False)
    assert np.allclose(p[np.arange(12), inp.targets], np.exp(-l), rtol=1e-12, atol=0)
    # shift invariance on a grid where adding 64 is exact in fp32
    zg = (np.random.default_rng(5).integers(-3000, 3000, size=(4, 333)) * 2.0 ** -7).astype(np.float32)
    assert np.allclose(oracle_mod.softmax(zg + np.float32(64.0)), oracle_mod.softmax(zg),
                       rtol=1e-12, atol=0)
    ref = torch.softmax(torch.tensor(inp.logits, dtype=torch.float64), dim=1).numpy()
    assert np.allclose(p, ref, rtol=1e-12, atol=1e-18)
    u = np.full((2, 300), 3.5, dtype=np.float32)
    assert np.allclose(oracle_mod.softmax(u), 1.0 / 300, rtol=1e-15, atol=0)


def test_softmax_backward_is_the_jacobian_product(oracle_mod):
    """dx equals J^T dy with J the softmax Jacobian taken by central finite
    differences of the forward oracle (exact fp32 steps); rows of dx sum to
    0; a row-constant dy gives dx = 0."""
    rng = np.random.default_rng(9)
    B, C = 2, 5
    h = 2.0 ** -12
    z = (rng.integers(-400, 400, size=(B, C)) * 2.0 ** -7).astype(np.float32)
    p = oracle_mod.softmax(z)
    dy = rng.standard_normal((B, C)).astype(np.float32)
    dx = oracle_mod.softmax_bwd(p.astype(np.float32), dy)
    # the oracle takes p in the element type: compare against p widened from fp32
    p32 = p.astype(np.float32).astype(np.float64)
    for b in range(B):
        J = np.empty((C, C))
        for c in range(C):
            zp, zm = z.copy(), z.copy()
            zp[b, c] += np.float32(h)
            zm[b, c] -= np.float32(h)
            J[:, c] = (oracle_mod.softmax(zp)[b] - oracle_mod.softmax(zm)[b]) / (2 * h)
        assert np.allclose(dx[b], J.T @ dy[b].astype(np.float64), rtol=0, atol=5e-6)
    assert np.allclose(dx.sum(axis=1), 0.0, atol=1e-6 * np.abs(p32).sum())
    const = np.full((B, C), 1.25, dtype=np.float32)
    assert np.allclose(oracle_mod.softmax_bwd(p.astype(np.float32), const), 0.0,
                       atol=2e-7)


def test_softmax_backward_against_torch(oracle_mod):
    """torch CPU fp64 autograd of softmax at z = log p (softmax(log p) = p for
    rows summing to 1) with upstream dy."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(13)
    q = rng.random((6, 40))
    p = (q / q.sum(axis=1, keepdims=True))
    dy = rng.standard_normal((6, 40))
    # fp32 inputs to the oracle, the same fp32 values to torch in fp64
    p32, dy32 = p.astype(np.float32), dy.astype(np.float32)
    pt = torch.tensor(p32.astype(np.float64))
    pt = pt / pt.sum(dim=1, keepdim=True)
    z = torch.log(pt).requires_grad_(True)
    torch.softmax(z, dim=1).backward(torch.tensor(dy32.astype(np.float64)))
    dx = oracle_mod.softmax_bwd(p32, dy32)
    assert np.allclose(dx, z.grad.numpy(), rtol=1e-5, atol=1e-7)
