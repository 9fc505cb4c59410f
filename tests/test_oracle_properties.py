"""Property-based pins of the oracle (random small shapes and values): facts
the mathematics fixes for every input, so a dropped term, a wrong sign or a
transposed index anywhere in the oracle fails one of them."""

import numpy as np
import pytest

hyp = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

import oracle  # noqa: E402

SETTINGS = settings(max_examples=60, deadline=None)


@st.composite
def batches(draw, max_b=6, max_c=40):
    """fp32 logits on the 2^-7 grid (so adding an integer stays exact) and
    targets in range."""
    B = draw(st.integers(1, max_b))
    C = draw(st.integers(1, max_c))
    seed = draw(st.integers(0, 2**31 - 1))
    g = np.random.default_rng(seed)
    scale = draw(st.sampled_from([1, 8, 64, 1024]))
    z = (g.integers(-scale * 128, scale * 128, size=(B, C)) * 2.0 ** -7).astype(np.float32)
    t = g.integers(0, C, size=B).astype(np.int32)
    return z, t


@pytest.fixture(scope="module", autouse=True)
def _built():
    oracle.build()


@SETTINGS
@given(batches())
def test_loss_and_gradient_relations(zt):
    z, t = zt
    B, C = z.shape
    l, g = oracle.rows(z, t)
    assert np.all(l >= -1e-12)
    # rows of the gradient sum to 0; entries lie in their ranges
    assert np.allclose(g.sum(axis=1), 0.0, atol=1e-12)
    gt = g[np.arange(B), t]
    assert np.all(gt <= 1e-15) and np.all(gt > -1.0 / B - 1e-15)
    mask = np.ones_like(g, dtype=bool)
    mask[np.arange(B), t] = False
    assert np.all(g[mask] >= 0) and np.all(g[mask] < 1.0 / B + 1e-15)
    # p_t = exp(-l_b) = 1 + B g_t: the loss and the gradient agree (compared
    # as probabilities: 1 + B g_t cancels in fp64 when p_t is tiny)
    assert np.allclose(np.exp(-l), 1.0 + B * gt, rtol=0, atol=1e-13)
    # softmax is the gradient plus the one-hot, times B
    p = oracle.softmax(z)
    onehot = np.zeros_like(p)
    onehot[np.arange(B), t] = 1.0
    assert np.allclose(B * g + onehot, p, rtol=1e-9, atol=1e-13)


@SETTINGS
@given(batches(), st.integers(-64, 64))
def test_shift_and_permutation(zt, shift):
    z, t = zt
    B, C = z.shape
    l, g = oracle.rows(z, t)
    ls, gs = oracle.rows(z + np.float32(shift), t)       # exact on the grid
    assert np.allclose(ls, l, rtol=1e-12, atol=1e-12) and np.allclose(gs, g, atol=1e-15)
    perm = np.random.default_rng(B * 31 + C).permutation(C)
    inv = np.argsort(perm)
    lp, gp = oracle.rows(np.ascontiguousarray(z[:, perm]), inv[t].astype(np.int32))
    assert np.allclose(lp, l, rtol=1e-12, atol=1e-12)
    assert np.allclose(gp, g[:, perm], atol=1e-15)


@SETTINGS
@given(batches(max_b=4, max_c=12))
def test_reductions_and_softmax_backward(zt):
    z, t = zt
    B, C = z.shape
    l = oracle.rows(z, t, grad=False)
    assert np.isclose(oracle.reduce(l, oracle.SUM), l.sum(), rtol=1e-12, atol=1e-12)
    assert np.isclose(oracle.reduce(l, oracle.MEAN), l.sum() / B, rtol=1e-12, atol=1e-12)
    # the gradient of the sum is B times the gradient of the mean
    _, g_mean = oracle.rows_ex(z, t, oracle.MEAN)
    _, g_sum = oracle.rows_ex(z, t, oracle.SUM)
    assert np.allclose(g_sum, B * g_mean, rtol=1e-12, atol=1e-15)
    # softmax backward: rows of dx sum to dot * (1 - sum p), which is 0 up to
    # the fp32 rounding of p; a row-constant dy gives dy * p * (1 - sum p)
    p = oracle.softmax(z)
    p32 = p.astype(np.float32)
    rng = np.random.default_rng(C)
    dy = rng.standard_normal((B, C)).astype(np.float32)
    dx = oracle.softmax_bwd(p32, dy)
    pw = p32.astype(np.float64)
    dot = (pw * dy).sum(axis=1, keepdims=True)
    assert np.allclose(dx.sum(axis=1), (dot * (1.0 - pw.sum(axis=1, keepdims=True)))[:, 0],
                       atol=1e-12)
    # constant dy along a row has no effect
    assert np.allclose(oracle.softmax_bwd(p32, np.full_like(dy, 0.75)),
                       0.75 * pw * (1.0 - pw.sum(axis=1, keepdims=True)), atol=1e-12)
