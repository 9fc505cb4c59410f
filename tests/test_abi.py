"""The C-ABI library builds, loads without a GPU and exports what ce.h declares."""

import ctypes
import os
import re

import pytest

import softmax_cross_entropy_row_gb300 as ce

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ce.h")
TEST_HEADER = os.path.join(ROOT, "include", "ce_testing.h")


def _declared_functions(header=HEADER):
    text = open(header).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ce_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    ce.build()
    return ce.load_library()


def test_header_declares_the_boundary():
    names = _declared_functions()
    assert "ce_fwd_bwd" in names and "ce_status_string" in names
    assert set(names) == set(ce.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions() + _declared_functions(TEST_HEADER):
        assert hasattr(lib, name), f"libce.so does not export {name}"


def _declared_constants(header=HEADER):
    text = re.sub(r"/\*.*?\*/", "", open(header).read(), flags=re.S)
    return {n: int(v) for n, v in re.findall(r"\b(CE_[A-Z0-9_]+)\s*=\s*(-?\d+)", text)}


def test_binding_constants_match_the_header():
    """The binding passes the header's numbers: every dtype, reduction and
    kernel path constant of ce.h has the same value in the Python module, and
    every status has a message of its own."""
    consts = _declared_constants()
    mirrored = [n for n in consts if n.startswith(("CE_PATH_", "CE_REDUCE_"))
                or n in ("CE_F32", "CE_BF16", "CE_F16")]
    assert "CE_PATH_ROWS_ONLINE" in mirrored and len(mirrored) >= 12
    for name in mirrored:
        assert getattr(ce, name) == consts[name], name
    lib = ce.load_library()
    statuses = [v for n, v in consts.items() if n == "CE_OK" or n.startswith("CE_ERR_")]
    messages = {lib.ce_status_string(v).decode() for v in statuses}
    assert len(messages) == len(statuses)


def test_test_header_declares_the_hooks():
    assert set(_declared_functions(TEST_HEADER)) == set(ce.TEST_EXPORTS)


def test_host_side_errors_of_the_test_entry(lib):
    """The test entry point checks its hooks before any CUDA call."""
    f = lib.ce_fwd_bwd_test
    none = ce.TestHooks(-1, 0, None)
    assert f(256, 512, 4, 4, 0, 1024, None, None, 0, 0, ctypes.byref(none)) == 1   # NULL grad
    assert f(256, 512, 4, 4, 7, 1024, 4096, None, 0, 0, None) == 3                 # dtype
    bad = ce.TestHooks(-1, 0, 8194)                                                  # 2 mod 4
    assert f(256, 512, 4, 4, 0, 1024, 4096, None, 0, 0, ctypes.byref(bad)) == 4
    over = ce.TestHooks(-1, 0, 1 << 20)                  # fp32 record over the logits
    assert f(1 << 20, 1 << 24, 4, 4, 0, 1 << 25, 1 << 26, None, 0, 0, ctypes.byref(over)) == 6


def test_status_strings_need_no_gpu(lib):
    for code in range(12):
        s = lib.ce_status_string(code).decode()
        assert s and s != "unknown status"
    assert lib.ce_status_string(99).decode() == "unknown status"
    assert lib.ce_last_cuda_error().decode() == ""


def test_host_side_argument_errors_need_no_gpu(lib):
    """Argument checks run before any CUDA call, so they answer on a CPU machine."""
    f = ce.ce_fwd_bwd_raw
    assert f(0, 0, 4, 4, 0, 0, 0) == 1                      # NULL
    assert f(256, 512, 4, 4, 7, 1024, 4096) == 3            # dtype
    assert f(256, 512, 0, 4, 0, 1024, 4096) == 2            # B = 0
    assert f(256, 512, 4, 0, 0, 1024, 4096) == 2            # C = 0
    assert f(256, 512, 2**31, 4, 0, 1024, 4096) == 2        # B too large
    assert f(258, 512, 4, 4, 0, 1024, 4096) == 4            # fp32 logits at 2 mod 4
    assert f(256, 514, 4, 4, 1, 1024, 4096) == 4            # int32 targets at 2 mod 4
    assert f(1 << 20, 512, 4, 4, 0, 1024, (1 << 20) + 32) == 6  # grad overlaps logits
    assert f(1 << 20, 1 << 24, 4, 4, 0, 1 << 25, (1 << 24) - 32) == 6  # grad covers targets


def test_host_side_errors_of_the_extended_entry_points(lib):
    """Reductions, the upstream gradient and the loss-only forward check their
    arguments before any CUDA call too."""
    ex = lib.ce_fwd_bwd_ex
    fw = lib.ce_forward
    # reduction out of range
    assert ex(256, 512, 4, 4, 0, 3, None, 1024, 4096, None) == 11
    assert fw(256, 512, 4, 4, 0, -1, 1024, None) == 11
    # loss only: the gradient may be NULL, the loss may not
    assert fw(256, 512, 4, 4, 0, 0, None, None) == 1
    assert ex(256, 512, 4, 4, 0, 2, None, None, None, None) == 1
    # misaligned upstream gradient
    assert ex(256, 512, 4, 4, 0, 0, 2050, 1024, 4096, None) == 4
    # per-row losses (4 B bytes) overlapping the logits
    assert ex(1 << 20, 1 << 24, 4, 4, 0, 2, None, (1 << 20) + 16, 1 << 26, None) == 6
    # a per-row upstream gradient overlapping the per-row losses
    assert ex(1 << 20, 1 << 24, 4, 4, 0, 2, 1 << 25, (1 << 25) + 8, 1 << 26, None) == 6
    # the gradient overlapping the scalar upstream gradient
    assert ex(1 << 20, 1 << 24, 4, 4, 0, 0, (1 << 26) + 32, 1 << 25, 1 << 26, None) == 6


def test_host_side_errors_of_the_softmax_entry_points(lib):
    """Row softmax forward and backward: the same checks, before any CUDA call."""
    fw, fp, bw = lib.ce_softmax_fwd, lib.ce_softmax_fwd_path, lib.ce_softmax_bwd
    assert fw(None, 4, 4, 0, 4096, None) == 1                # NULL logits
    assert fw(256, 4, 4, 0, None, None) == 1                 # NULL output
    assert fw(256, 4, 4, 7, 4096, None) == 3                 # dtype
    assert fw(256, 0, 4, 0, 4096, None) == 2                 # B = 0
    assert fp(256, 4, 0, 1, 4096, None, 0, 0) == 2           # C = 0
    assert fw(258, 4, 4, 0, 4096, None) == 4                 # fp32 logits at 2 mod 4
    assert fw(1 << 20, 4, 4, 0, (1 << 20) + 32, None) == 6   # output overlaps logits
    assert bw(None, 512, 4, 4, 0, 4096, None) == 1
    assert bw(256, 512, 4, 4, 7, 4096, None) == 3
    assert bw(256, 512, 4, 4, 1, 4097, None) == 4            # bf16 dx at an odd address
    # dx may be p or dy exactly, but may not overlap them otherwise
    assert bw(1 << 20, 1 << 24, 4, 4, 0, (1 << 20) + 16, None) == 6
    assert bw(1 << 20, 1 << 24, 4, 4, 0, (1 << 24) - 16, None) == 6


def test_host_side_errors_of_the_host_buffer_entry(lib):
    """ce_fwd_bwd_host checks its arguments before any CUDA call as well."""
    h = lib.ce_fwd_bwd_host
    assert h(None, 512, 4, 4, 0, 1024, 4096, None) == 1      # NULL logits
    assert h(256, 512, 4, 4, 0, 1024, None, None) == 1       # NULL gradient
    assert h(256, 512, 4, 4, 0, None, 4096, None) == 1       # NULL loss
    assert h(256, 512, 4, 4, 7, 1024, 4096, None) == 3       # dtype
    assert h(256, 512, 0, 4, 0, 1024, 4096, None) == 2       # B = 0
    assert h(258, 512, 4, 4, 0, 1024, 4096, None) == 4       # fp32 logits at 2 mod 4
    assert h(256, 514, 4, 4, 0, 1024, 4096, None) == 4       # targets at 2 mod 4
    assert h(1 << 20, 512, 4, 4, 0, 1024, (1 << 20) + 32, None) == 6  # gradient over logits
    g = lib.ce_fwd_bwd_host_grad
    assert g(256, 512, 4, 4, 0, 1024, None, None) == 1                 # NULL host gradient
    assert g(256, 512, 4, 4, 1, 1024, 4097, None) == 4                 # bf16 gradient at an odd address
    assert g(1 << 20, 1 << 24, 4, 4, 0, 1 << 25, (1 << 24) - 16, None) == 6  # gradient over targets
    assert g(1 << 20, 1 << 24, 4, 4, 0, (1 << 20) + 4, 1 << 26, None) == 6   # loss inside the logits


def test_no_cpu_fallback_without_library(tmp_path):
    """The binding refuses to run when the CUDA library is absent."""
    import importlib

    mod = importlib.import_module("softmax_cross_entropy_row_gb300")
    with pytest.raises(ImportError):
        mod.load_library(str(tmp_path / "missing_libce.so"))


def test_product_does_not_touch_the_oracle(lib):
    """Neither the library nor the binding loads anything of the oracle."""
    import subprocess
    import sys

    assert not hasattr(lib, "ce_oracle_rows") and not hasattr(lib, "ce_oracle_fwd_bwd")
    code = ("import sys, softmax_cross_entropy_row_gb300 as ce; ce.load_library(); "
            "assert 'oracle' not in sys.modules and 'workloads' not in sys.modules")
    subprocess.run([sys.executable, "-c", code], check=True, cwd=ROOT)


def test_binding_checks_what_the_c_layer_cannot(lib):
    """The wrappers refuse target, loss and upstream-gradient tensors of the
    wrong type or size before calling the library (which sees plain pointers):
    checked here with CPU tensors, which the device entry points refuse too."""
    torch = pytest.importorskip("torch")
    z = torch.zeros(4, 8)
    t = torch.zeros(4, dtype=torch.int32)
    loss = torch.zeros(1)
    g = torch.zeros(4, 8)
    with pytest.raises(ValueError, match="CUDA"):
        ce.ce_fwd_bwd(z, t, loss, g)
    with pytest.raises(ValueError, match="targets"):
        ce.ce_fwd_bwd_host(z, t.long(), loss, g)
    with pytest.raises(ValueError, match="targets"):
        ce.ce_fwd_bwd_host(z, t[:3], loss, g)
    with pytest.raises(ValueError, match="loss_out"):
        ce.ce_fwd_bwd_host(z, t, torch.zeros(1, dtype=torch.float64), g)
    with pytest.raises(ValueError, match="CUDA"):  # the gradient stays on the device
        ce.ce_fwd_bwd_host(z, t, loss, g)
    with pytest.raises(ValueError):  # per-row losses need B elements
        ce._check_io(z, t, loss, ce.CE_REDUCE_NONE, device="cpu")
    with pytest.raises(ValueError, match="grad_scale"):
        ce._check_io(z, t, torch.zeros(4), ce.CE_REDUCE_NONE, torch.zeros(1), device="cpu")
    ce._check_io(z, t, torch.zeros(4), ce.CE_REDUCE_NONE, torch.zeros(4), device="cpu")


def test_the_abi_from_plain_c(lib, tmp_path):
    """A C program that includes include/ce.h and links libce.so (no Python
    in between) gets the documented status codes from every entry point."""
    import shutil
    import subprocess

    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    libdir = os.path.dirname(ce.build())
    exe = tmp_path / "abi_from_c"
    src = os.path.join(ROOT, "tests", "c", "abi_from_c.c")
    subprocess.run(["gcc", "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    src, "-o", str(exe), f"-L{libdir}", "-lce", f"-Wl,-rpath,{libdir}"],
                   check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0, out.stderr
    assert out.stdout.strip() == "ok"

