"""Seeded synthetic inputs for the softmax cross-entropy row workloads.

This module is shared by the oracle tests, the GPU parity tests and the
benchmark.  It holds no cross-entropy arithmetic: only the random draws, the
round-to-nearest-even narrowing of those draws to bf16, and each workload's
recipe (shape, dtype, value distribution and row structure).

Every array is generated on the host, so the fp64 oracle and the CUDA path
always see byte-identical inputs.  Draws are made in fixed chunks of rows,
each chunk from its own child of a ``numpy.random.SeedSequence``; the result
therefore depends only on the seed, never on how many threads generate it.
"""

from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

# Element-type codes shared with the C-ABI (``ce_dtype``) and the oracle.
DTYPE_F32 = 0
DTYPE_BF16 = 1
DTYPE_F16 = 2
DTYPE_CODES = {"f32": DTYPE_F32, "bf16": DTYPE_BF16, "f16": DTYPE_F16}
ELEM_BYTES = {"f32": 4, "bf16": 2, "f16": 2}

_ROWS_PER_CHUNK = 256


@dataclass(frozen=True)
class Workload:
    """One synthetic logits matrix ``[B, C]`` with int32 class targets.

    sigma        standard deviation of the N(0, sigma^2) logits (drawn in fp32)
    peak         added (in fp32, before any bf16 rounding) at each row's target
    uniform_frac fraction of rows replaced by one constant (the row's first draw)
    spike        value written at one random position of a further disjoint
                 ``uniform_frac`` of rows
    """

    name: str
    B: int
    C: int
    dtype: str
    seed: int
    sigma: float = 1.0
    peak: float = 0.0
    uniform_frac: float = 0.0
    spike: float | None = None
    description: str = field(default="", compare=False)

    @property
    def dtype_code(self) -> int:
        return DTYPE_CODES[self.dtype]

    @property
    def elem_bytes(self) -> int:
        return ELEM_BYTES[self.dtype]

    @property
    def min_bytes(self) -> int:
        """Logits read once + grad written once + int32 targets + fp32 loss."""
        return self.B * self.C * 2 * self.elem_bytes + 4 * self.B + 4


# The five workloads, in order: a tiny correctness case, a classifier head,
# an LM head whose row fits in shared memory, a large-vocabulary LM head that
# needs the split-row path, and a ragged stress case.
WORKLOADS: list[Workload] = [
    Workload("tiny_8x10_f32", 8, 10, "f32", seed=0, sigma=1.0,
             description="B=8, C=10, fp32 logits ~ N(0,1), seed 0"),
    Workload("classifier_4096x1000_f32", 4096, 1000, "f32", seed=1, sigma=2.0,
             description="classifier head, fp32 logits ~ N(0, 2^2)"),
    Workload("lm_head_8192x32000_bf16", 8192, 32000, "bf16", seed=2, sigma=3.0,
             description="LM head, bf16 logits ~ N(0, 3^2)"),
    Workload("lm_head_4096x128256_bf16_peaked", 4096, 128256, "bf16", seed=3,
             sigma=3.0, peak=8.0,
             description="large-vocab LM head, bf16 N(0, 3^2) + 8 at the target"),
    Workload("stress_16384x50257_f32", 16384, 50257, "f32", seed=4, sigma=30.0,
             uniform_frac=0.01, spike=80.0,
             description="ragged stress: 30*N(0,1), 1% uniform rows, 1% rows "
                         "with one logit at +80"),
]

WORKLOADS_BY_NAME = {w.name: w for w in WORKLOADS}


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round finite fp32 values to bf16 (round to nearest, ties to even)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to fp32 (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32)
            << np.uint32(16)).view(np.float32)


def _threads() -> int:
    try:
        n = len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        n = os.cpu_count() or 1
    return max(1, min(16, n))


def _normal_rows(seed: int, B: int, C: int, sigma: float) -> np.ndarray:
    out = np.empty((B, C), dtype=np.float32)
    nchunks = (B + _ROWS_PER_CHUNK - 1) // _ROWS_PER_CHUNK
    children = np.random.SeedSequence([seed, 0x10617]).spawn(max(nchunks, 1))

    def fill(i: int) -> None:
        r0 = i * _ROWS_PER_CHUNK
        r1 = min(B, r0 + _ROWS_PER_CHUNK)
        g = np.random.Generator(np.random.PCG64(children[i]))
        blk = out[r0:r1]
        g.standard_normal(out=blk.reshape(-1), dtype=np.float32)
        if sigma != 1.0:
            np.multiply(blk, np.float32(sigma), out=blk)

    if nchunks <= 1:
        for i in range(nchunks):
            fill(i)
    else:
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(fill, range(nchunks)))
    return out


def make_targets(seed: int, B: int, C: int) -> np.ndarray:
    """Targets uniform in [0, C), int32."""
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 0x7A6])))
    return g.integers(0, C, size=B, dtype=np.int32)


@dataclass
class Inputs:
    """Host arrays of one workload instance.

    ``logits`` is float32 ``[B, C]`` for fp32 workloads and the uint16 bf16 bit
    patterns ``[B, C]`` for bf16 ones.  ``uniform_rows`` / ``spike_rows`` list
    the structured rows (empty unless the recipe has them).
    """

    workload: Workload
    logits: np.ndarray
    targets: np.ndarray
    uniform_rows: np.ndarray
    spike_rows: np.ndarray
    spike_cols: np.ndarray

    def logits_f32(self, rows=None) -> np.ndarray:
        """The logits (or a row subset) as exactly-widened fp32 values."""
        z = self.logits if rows is None else self.logits[rows]
        if self.workload.dtype == "bf16":
            return bf16_bits_to_f32(z)
        if self.workload.dtype == "f16":
            return z.astype(np.float32)
        return z


def make_inputs(w: Workload) -> Inputs:
    """Generate the seeded inputs of workload ``w``."""
    z = _normal_rows(w.seed, w.B, w.C, w.sigma)
    t = make_targets(w.seed, w.B, w.C)
    empty = np.zeros(0, dtype=np.int64)
    uniform_rows, spike_rows, spike_cols = empty, empty, empty
    if w.peak:
        z[np.arange(w.B), t] += np.float32(w.peak)
    if w.uniform_frac:
        n = int(w.B * w.uniform_frac)
        g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([w.seed, 0x5EC])))
        picked = g.choice(w.B, size=2 * n, replace=False).astype(np.int64)
        uniform_rows = np.sort(picked[:n])
        spike_rows = picked[n:]
        for r in uniform_rows:
            z[r, :] = z[r, 0]
        if w.spike is not None:
            spike_cols = g.integers(0, w.C, size=n).astype(np.int64)
            z[spike_rows, spike_cols] = np.float32(w.spike)
        order = np.argsort(spike_rows)
        spike_rows, spike_cols = spike_rows[order], spike_cols[order]
    logits = (f32_to_bf16_bits(z) if w.dtype == "bf16"
              else z.astype(np.float16) if w.dtype == "f16" else z)
    return Inputs(w, logits, t, uniform_rows, spike_rows, spike_cols)


def random_case(B: int, C: int, dtype: str, seed: int, sigma: float = 1.0,
                target_range: tuple[int, int] | None = None) -> Inputs:
    """A small seeded N(0, sigma^2) case for edge-shape tests."""
    w = Workload(f"case_{B}x{C}_{dtype}_{seed}", B, C, dtype, seed=seed, sigma=sigma)
    z = _normal_rows(seed, B, C, sigma)
    if target_range is None:
        t = make_targets(seed, B, C)
    else:
        g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 0xBAD])))
        t = g.integers(target_range[0], target_range[1], size=B, dtype=np.int32)
    logits = (f32_to_bf16_bits(z) if dtype == "bf16"
              else z.astype(np.float16) if dtype == "f16" else z)  # f16: numpy's RNE narrowing
    empty = np.zeros(0, dtype=np.int64)
    return Inputs(w, logits, t, empty, empty, empty)
