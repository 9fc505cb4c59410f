"""The stored tiny-workload fixture, and the seeded input generator it came from."""

import json
import math
import os

import numpy as np
import pytest

import workloads as wl

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "tiny_8x10_f32.json")


def _load():
    with open(GOLDEN) as f:
        doc = json.load(f)
    z = np.array([[float.fromhex(v) for v in row] for row in doc["logits_f32_hex"]],
                 dtype=np.float32)
    t = np.array(doc["targets"], dtype=np.int32)
    l = np.array([float.fromhex(v) for v in doc["row_loss"]])
    g = np.array([[float.fromhex(v) for v in row] for row in doc["grad"]])
    return doc, z, t, l, float.fromhex(doc["loss"]), g


def test_fixture_values_are_exact_under_multiprecision():
    """Every stored value agrees with a 50-digit restatement of the definition
    (no max shift, different evaluation order) -- the fixture is pinned by
    something other than the oracle that wrote it."""
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 50
    doc, z, t, l, L, g = _load()
    B, C = z.shape
    total = mpmath.mpf(0)
    for b in range(B):
        ex = [mpmath.exp(mpmath.mpf(float(v))) for v in z[b]]
        s = mpmath.fsum(ex)
        lb = mpmath.log(s) - mpmath.mpf(float(z[b, t[b]]))
        total += lb
        assert float(lb) == pytest.approx(l[b], rel=2e-15)
        for c in range(C):
            gb = (ex[c] / s - (1 if c == t[b] else 0)) / B
            assert float(gb) == pytest.approx(g[b, c], rel=1e-13, abs=1e-18)
    assert float(total / B) == pytest.approx(L, rel=2e-15)


def test_oracle_reproduces_fixture(oracle_mod):
    _, z, t, l, L, g = _load()
    L2, l2, g2 = oracle_mod.loss_and_grad(z, t)
    assert L2 == L and np.array_equal(l2, l) and np.array_equal(g2, g)


def test_generator_reproduces_fixture_inputs():
    """The seeded generator still produces the stored tiny inputs."""
    _, z, t, _, _, _ = _load()
    inp = wl.make_inputs(wl.WORKLOADS_BY_NAME["tiny_8x10_f32"])
    assert np.array_equal(inp.logits, z) and np.array_equal(inp.targets, t)


# ------------------------------------------------------- input generator pins

def test_bf16_rounding_is_nearest_even():
    cases = {
        1.0: 0x3F80,
        1.00390625: 0x3F80,  # halfway between 0x3F80 and 0x3F81: ties to even
        1.01171875: 0x3F82,  # halfway between 0x3F81 and 0x3F82: ties to even
        1.0078125: 0x3F81,
        1.0058594: 0x3F81,   # above the halfway point: rounds up
        -2.0: 0xC000,
        3.14159265: 0x4049,
        0.0: 0x0000,
    }
    x = np.array(list(cases), dtype=np.float32)
    assert wl.f32_to_bf16_bits(x).tolist() == list(cases.values())
    back = wl.bf16_bits_to_f32(np.array(list(cases.values()), dtype=np.uint16))
    assert back[0] == 1.0 and back[5] == -2.0 and back[6] == 3.140625


def test_workload_shapes_and_structure():
    small = [wl.Workload("s", 300, 97, "f32", seed=4, sigma=30.0, uniform_frac=0.01,
                         spike=80.0),
             wl.Workload("p", 64, 50, "bf16", seed=3, sigma=3.0, peak=8.0)]
    a = wl.make_inputs(small[0])
    b = wl.make_inputs(small[0])
    assert np.array_equal(a.logits, b.logits) and np.array_equal(a.targets, b.targets)
    assert a.logits.shape == (300, 97) and a.logits.dtype == np.float32
    assert len(a.uniform_rows) == 3 and len(a.spike_rows) == 3
    assert not set(a.uniform_rows) & set(a.spike_rows)
    for r in a.uniform_rows:
        assert np.all(a.logits[r] == a.logits[r, 0])
    for r, c in zip(a.spike_rows, a.spike_cols):
        assert a.logits[r, c] == 80.0
    assert a.targets.min() >= 0 and a.targets.max() < 97
    p = wl.make_inputs(small[1])
    assert p.logits.dtype == np.uint16
    zt = p.logits_f32()[np.arange(64), p.targets]
    assert np.mean(zt) > 6.0  # the +8 peak sits at the target


def test_full_size_recipes():
    assert [(w.B, w.C, w.dtype) for w in wl.WORKLOADS] == [
        (8, 10, "f32"), (4096, 1000, "f32"), (8192, 32000, "bf16"),
        (4096, 128256, "bf16"), (16384, 50257, "f32")]
    assert wl.WORKLOADS[1].min_bytes == 32_784_388
    assert wl.WORKLOADS[4].min_bytes == 6_587_351_044
    assert math.isclose(wl.WORKLOADS[3].min_bytes, 2_101_362_692)
