"""Host-only checks of the C ABI: the library loads, exports every function that
include/*.h declares, and rejects bad arguments before touching the GPU.
No kernel is launched here (these run without a GPU)."""
import ctypes
import glob
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h, encoding="utf-8").read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(",
                             text, flags=re.M):
            if m.group(1) not in ("if", "while", "for", "return", "sizeof"):
                names.add(m.group(1))
    return names


@pytest.fixture(scope="module")
def lr():
    import linear_recurrence_gb300 as m
    m.load_library()
    return m


def test_header_declares_the_boundary():
    names = _declared_functions()
    for f in ("sscan_fwd", "sscan_fwd_ex", "sscan_fwd_fused", "sscan_bwd", "sscan_step", "pscan",
              "sscan_status_string",
              "sscan_get_last_error", "sscan_max_dstate", "sscan_last_launch_count",
              "sscan_last_plan"):
        assert f in names, f


def test_library_exports_every_declared_symbol(lr):
    declared = _declared_functions()
    out = subprocess.run(["nm", "-D", "--defined-only", lr.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    missing = declared - exported
    assert not missing, missing
    assert set(lr.SIGNATURES) == declared
    raw = lr.lib()
    for name in declared:
        assert getattr(raw, name) is not None


def test_status_strings_and_limits(lr):
    assert lr.status_string(0) == "SSCAN_OK"
    assert "INVALID" in lr.status_string(1)
    assert "CUDA" in lr.status_string(2)
    assert "TIMEOUT" in lr.status_string(3)
    assert "UNKNOWN" in lr.status_string(99)
    assert lr.max_dstate() == 64


def test_invalid_calls_return_before_any_cuda_call(lr):
    raw = lr.lib()
    fake = ctypes.c_void_p(0x1000)   # never dereferenced: validation fails first
    # required pointer missing
    assert raw.sscan_fwd(None, fake, fake, fake, fake, None, None, fake, None,
                         1, 1, 1, 1, 0, None) == lr.SSCAN_ERR_INVALID
    assert raw.sscan_fwd(fake, fake, fake, fake, fake, None, None, None, None,
                         1, 1, 1, 1, 0, None) == lr.SSCAN_ERR_INVALID
    # bad dtype, negative size, dstate out of range, unsupported lanes
    assert raw.sscan_fwd(fake, fake, fake, fake, fake, None, None, fake, None,
                         1, 1, 1, 1, 2, None) == lr.SSCAN_ERR_INVALID
    assert raw.sscan_fwd(fake, fake, fake, fake, fake, None, None, fake, None,
                         1, -1, 1, 1, 0, None) == lr.SSCAN_ERR_INVALID
    assert raw.sscan_fwd(fake, fake, fake, fake, fake, None, None, fake, None,
                         1, 1, 1, 0, 0, None) == lr.SSCAN_ERR_INVALID
    assert raw.sscan_fwd(fake, fake, fake, fake, fake, None, None, fake, None,
                         1, 1, 1, 65, 0, None) == lr.SSCAN_ERR_INVALID
    assert raw.sscan_fwd_ex(fake, fake, fake, fake, fake, None, None, fake, None,
                            1, 1, 8, 16, 0, 0, 3, None) == lr.SSCAN_ERR_INVALID
    assert raw.sscan_fwd_ex(fake, fake, fake, fake, fake, None, None, fake, None,
                            1, 1, 8, 16, 0, -1, 0, None) == lr.SSCAN_ERR_INVALID
    # sizes whose element count overflows
    assert raw.sscan_fwd(fake, fake, fake, fake, fake, None, None, fake, None,
                         1 << 40, 1 << 40, 1 << 20, 16, 0, None) == lr.SSCAN_ERR_INVALID
    # unknown option bits, missing pointer with options
    assert raw.sscan_fwd_fused(fake, fake, fake, fake, fake, None, None, None, None, fake, None,
                               1, 1, 8, 16, 0, 4, 0, 0, None) == lr.SSCAN_ERR_INVALID
    assert raw.sscan_fwd_fused(fake, None, fake, fake, fake, None, fake, fake, None, fake, None,
                               1, 1, 8, 16, 0, 3, 0, 0, None) == lr.SSCAN_ERR_INVALID
    assert raw.sscan_step(fake, fake, fake, fake, fake, None, None, fake, 1, 1, 4, 0, None) == \
        lr.SSCAN_ERR_INVALID
    assert raw.sscan_step(fake, fake, fake, fake, fake, None, fake, fake, 1, 1, 65, 0, None) == \
        lr.SSCAN_ERR_INVALID
    assert raw.sscan_step(fake, fake, fake, fake, fake, None, fake, fake, 0, 3, 4, 0, None) == \
        lr.SSCAN_OK
    assert lr.last_plan() == "empty"
    assert raw.sscan_step(fake, fake, fake, fake, fake, None, fake, fake, 1, 1, 0, 0, None) == \
        lr.SSCAN_ERR_INVALID
    assert raw.sscan_bwd(fake, fake, fake, fake, fake, None, None, fake, None, fake, fake, fake, fake,
                         fake, None, None, 1, 1, 8, 65, 0, None) == lr.SSCAN_ERR_INVALID
    assert raw.sscan_bwd(fake, fake, fake, fake, fake, None, None, fake, None, fake, fake, None, fake,
                         fake, None, None, 1, 1, 8, 16, 0, None) == lr.SSCAN_ERR_INVALID
    assert raw.sscan_bwd(fake, fake, fake, fake, fake, None, None, fake, None, fake, fake, fake, fake,
                         fake, None, None, 0, 4, 8, 16, 1, None) == lr.SSCAN_OK
    assert raw.pscan(None, fake, fake, None, 1, 1, None) == lr.SSCAN_ERR_INVALID
    assert raw.pscan(fake, fake, fake, None, -1, 1, None) == lr.SSCAN_ERR_INVALID
    assert lr.last_launch_count() == 0
    assert lr.last_plan() == "rejected"


def test_empty_problems_launch_nothing(lr):
    raw = lr.lib()
    fake = ctypes.c_void_p(0x1000)
    assert raw.sscan_fwd(fake, fake, fake, fake, fake, None, None, fake, None,
                         0, 4, 16, 4, 0, None) == lr.SSCAN_OK
    assert lr.last_launch_count() == 0 and lr.last_plan() == "empty"
    assert raw.pscan(fake, fake, fake, None, 3, 0, None) == lr.SSCAN_OK
    assert lr.last_launch_count() == 0


def test_binding_refuses_cpu_tensors(lr):
    import torch
    u = torch.zeros((1, 2, 4))
    with pytest.raises(ValueError):
        lr.sscan_fwd(u, u, torch.zeros((2, 4)), torch.zeros((1, 4, 4)), torch.zeros((1, 4, 4)))
    with pytest.raises(ValueError):
        lr.pscan(torch.zeros((2, 3)), torch.zeros((2, 3)))


def test_missing_library_fails_loudly(tmp_path):
    import linear_recurrence_gb300 as m
    with pytest.raises((OSError, RuntimeError)):
        m.load_library(str(tmp_path / "no_such_libsscan.so"))


def test_product_path_never_touches_the_oracle():
    pkg = os.path.join(ROOT, "linear_recurrence_gb300")
    for path in glob.glob(os.path.join(pkg, "**", "*.*"), recursive=True):
        if path.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
            text = open(path, encoding="utf-8").read()
            assert "import oracle" not in text and "from oracle" not in text, path
            assert "sscan_oracle" not in text and "_liboracle" not in text, path
    for path in glob.glob(os.path.join(ROOT, "oracle", "*.*")):
        if path.endswith((".py", ".c")):
            text = open(path, encoding="utf-8").read()
            assert "linear_recurrence_gb300" not in text.replace(
                "the product (``linear_recurrence_gb300``)", "").replace(
                "product path (``linear_recurrence_gb300``)", ""), path
