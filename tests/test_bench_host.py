"""Host-side arithmetic of bench.py (no GPU): the algorithmic bytes each
measured call must move, and when a recorded DRAM-traffic figure applies."""

import json

import pytest

import bench
import workloads as wl


def test_algorithmic_bytes():
    w = wl.WORKLOADS_BY_NAME["classifier_4096x1000_f32"]
    n = w.B * w.C * 4
    assert w.min_bytes == 2 * n + 4 * w.B + 4             # logits in, gradient out, targets, L
    assert bench.next_row_bytes(w, "plain") == w.min_bytes
    assert bench.next_row_bytes(w, "forward") == n + 4 * w.B + 4
    assert bench.next_row_bytes(w, "sum") == 2 * n + 4 * w.B + 8       # + the scalar upstream
    assert bench.next_row_bytes(w, "none") == 2 * n + 12 * w.B          # + [B] upstream, [B] losses
    assert bench.next_row_bytes(w, "softmax_fwd") == 2 * n
    assert bench.next_row_bytes(w, "softmax_bwd") == 3 * n
    h = wl.WORKLOADS_BY_NAME["lm_head_8192x32000_bf16"]
    assert h.min_bytes == 2 * h.B * h.C * 2 + 4 * h.B + 4


def test_recorded_traffic_applies_only_to_the_captured_kernel_and_launch(tmp_path, monkeypatch):
    plan = {"path": "rows_warp", "split": 1, "ctas": 256, "threads": 512, "smem_bytes": 65536}
    rec = {"w": {"dram_bytes_per_launch": 123, "kernel": "rows_warp",
                 "source_sha": bench.source_hash("rows_warp"), "plan": plan}}
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "source_hash", lambda kernel=None: rec["w"]["source_sha"])
    assert bench.recorded_traffic("w", plan) == 123
    assert bench.recorded_traffic("w", dict(plan, ctas=152)) is None
    assert bench.recorded_traffic("other", plan) is None
    monkeypatch.setattr(bench, "source_hash", lambda kernel=None: "0" * 16)
    assert bench.recorded_traffic("w", plan) is None


def test_device_code_hashes_ignore_the_host_layer():
    """The hashes cover device code only: all of it, or one kernel's file and
    the shared headers (so a change to one kernel leaves the others' records
    valid)."""
    import glob
    import os

    files = glob.glob(os.path.join(bench.ROOT, "softmax_cross_entropy_row_gb300", "csrc", "*"))
    names = {os.path.basename(f) for f in files}
    assert "ce_api.cu" in names and set(bench.HOST_ONLY_SOURCES) <= names
    assert set(bench.KERNEL_SOURCES.values()) | set(bench.SHARED_DEVICE_SOURCES) <= names
    assert len(bench.source_hash()) == 16
    hashes = {k: bench.source_hash(k) for k in bench.KERNEL_SOURCES}
    assert len(set(hashes.values())) == len(hashes)
    # a kernel with an interface header of its own hashes it too (its
    # constants shape the kernel); the others hash their file and the shared
    # headers alone
    assert bench.kernel_source_names("rows_online") == sorted(
        ["ce_rows_online.cu", "ce_rows_online.h"] + list(bench.SHARED_DEVICE_SOURCES))
    assert bench.kernel_source_names("rows_warp") == sorted(
        ["ce_rows_warp.cu"] + list(bench.SHARED_DEVICE_SOURCES))
    assert "ce_api.cu" not in bench.kernel_source_names()


@pytest.mark.parametrize("name", ["classifier_4096x1000_f32", "lm_head_8192x32000_bf16",
                                  "lm_head_4096x128256_bf16_peaked", "stress_16384x50257_f32"])
def test_committed_traffic_matches_the_current_kernels(name):
    """The committed DRAM capture: its reads equal the logits' bytes (the
    logits cross HBM once).  Skipped once the kernels have changed since the
    capture (the bench then reports the traffic as null)."""
    with open(f"{bench.ROOT}/profiles/traffic.json") as f:
        rec = json.load(f)[name]
    if rec["source_sha"] != bench.source_hash(rec["kernel"]):
        pytest.skip("the kernel changed since the capture")
    # DRAM reads match the logits' bytes: the logits cross HBM once; and the
    # traffic per launch is the reads and writes of that launch
    w = wl.WORKLOADS_BY_NAME[name]
    logits = rec["captured_rows"] * w.C * w.elem_bytes
    assert abs(rec["dram_read_bytes_per_launch"] / logits - 1.0) < 0.01
    assert rec["dram_bytes_per_launch"] == (rec["dram_read_bytes_per_launch"]
                                            + rec["dram_write_bytes_per_launch"])
