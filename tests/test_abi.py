"""The C-ABI library builds, loads and exports every symbol of include/nvfp4.h
(no GPU: only host-side calls -- sizes, status strings, argument rejection)."""
import ctypes
import os
import re

import pytest

from tensor_quantization_gb300 import build as tq_build
from tensor_quantization_gb300 import nvfp4

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    with open(os.path.join(ROOT, "include", "nvfp4.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:[\w\s\*]+?)\b(nvfp4_\w+)\s*\(", text, re.M)))


@pytest.fixture(scope="module")
def lib():
    path = tq_build.build()
    return nvfp4.load(path)


def test_header_declares_the_boundary():
    names = declared_functions()
    for f in ("nvfp4_amax", "nvfp4_quantize_rne", "nvfp4_quantize_sr", "nvfp4_quantize_rht_sr",
              "nvfp4_quantize_four_over_six", "nvfp4_dequantize"):
        assert f in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert set(declared_functions()) <= set(nvfp4.EXPORTS) | set(declared_functions())


def test_host_only_queries(lib):
    assert nvfp4.nvfp4_workspace_bytes() >= 12
    assert nvfp4.nvfp4_scale_bytes(256, 1024, 0) == 256 * 64
    assert nvfp4.nvfp4_scale_bytes(300, 208, nvfp4.SWIZZLED) == 384 * 16
    assert nvfp4.nvfp4_scale_bytes(8192, 4096, nvfp4.SWIZZLED) == 8192 * 256
    for s in range(5):
        assert nvfp4.status_string(s)


def _inp(rows, cols, ld, ptr=16, dtype=0, row0=0, col0=0):
    return nvfp4.Input(ptr, dtype, rows, cols, ld, row0, col0)


def test_arguments_are_rejected_before_any_launch(lib):
    out = nvfp4.Output(16, 16, 16, 16, 16, 16)
    ws = ctypes.c_void_p(16)
    st = lib.nvfp4_quantize_rne
    assert st(None, 1, ctypes.byref(out), ws, None) == nvfp4.ERR_INVALID_ARG
    assert st(ctypes.byref(_inp(16, 24, 24)), 1, ctypes.byref(out), ws, None) == nvfp4.ERR_INVALID_ARG  # cols % 16
    assert st(ctypes.byref(_inp(16, 32, 36)), 1, ctypes.byref(out), ws, None) == nvfp4.ERR_INVALID_ARG  # pitch
    assert st(ctypes.byref(_inp(16, 32, 32, ptr=8)), 1, ctypes.byref(out), ws, None) == nvfp4.ERR_INVALID_ARG
    assert st(ctypes.byref(_inp(16, 32, 32, dtype=7)), 1, ctypes.byref(out), ws, None) == nvfp4.ERR_INVALID_ARG
    assert st(ctypes.byref(_inp(16, 32, 32)), 0, ctypes.byref(out), ws, None) == nvfp4.ERR_INVALID_ARG  # no orientation
    assert st(ctypes.byref(_inp(16, 32, 32)), 1 << 12, ctypes.byref(out), ws, None) == nvfp4.ERR_INVALID_ARG
    assert st(ctypes.byref(_inp(8, 32, 32)), 2, ctypes.byref(out), ws, None) == nvfp4.ERR_INVALID_ARG  # rows % 16
    assert st(ctypes.byref(_inp(16, 32, 32)), 1, ctypes.byref(out), None, None) == nvfp4.ERR_INVALID_ARG  # workspace
    no_amax = nvfp4.Output(16, 16, 16, 16, None, 16)
    assert st(ctypes.byref(_inp(16, 32, 32)), 1, ctypes.byref(no_amax), ws, None) == nvfp4.ERR_INVALID_ARG
    # valid but unsupported combinations
    sr = lib.nvfp4_quantize_sr
    assert sr(ctypes.byref(_inp(16, 32, 32)), 1 | nvfp4.BLOCK_2D, 1, 0, ctypes.byref(out), ws, None) == \
        nvfp4.ERR_UNSUPPORTED
    assert st(ctypes.byref(_inp(16, 32, 32)), 3 | nvfp4.SCALE_PER_ROW, ctypes.byref(out), ws, None) == \
        nvfp4.ERR_UNSUPPORTED
    rht = lib.nvfp4_quantize_rht_sr
    assert rht(ctypes.byref(_inp(16, 32, 32)), 1 | nvfp4.BLOCK_2D, 0, 1, 0, ctypes.byref(out), ws, None) == \
        nvfp4.ERR_UNSUPPORTED
    assert rht(ctypes.byref(_inp(16, 32, 32)), 3 | nvfp4.SCALE_PER_ROW, 0, 1, 0, ctypes.byref(out), ws, None) == \
        nvfp4.ERR_UNSUPPORTED
    fo6 = lib.nvfp4_quantize_four_over_six
    assert fo6(ctypes.byref(_inp(16, 32, 32)), 1 | nvfp4.FAST_MATH, ctypes.byref(out), ws, None) == \
        nvfp4.ERR_UNSUPPORTED
    # shard positions: never negative; a stochastic shard is cut along its output rows only
    assert st(ctypes.byref(_inp(16, 32, 32, row0=-16)), 1, ctypes.byref(out), ws, None) == nvfp4.ERR_INVALID_ARG
    assert sr(ctypes.byref(_inp(16, 32, 32, col0=32)), 1, 1, 0, ctypes.byref(out), ws, None) == \
        nvfp4.ERR_UNSUPPORTED
    assert sr(ctypes.byref(_inp(16, 32, 32, row0=16)), 2, 1, 0, ctypes.byref(out), ws, None) == \
        nvfp4.ERR_UNSUPPORTED
    grp = lib.nvfp4_quantize_grouped
    offs = ctypes.c_void_p(64)
    assert grp(ctypes.byref(_inp(16, 32, 32)), 1, offs, 0, 0, 0, 0, 0, ctypes.byref(out), None) == \
        nvfp4.ERR_INVALID_ARG  # no groups
    assert grp(ctypes.byref(_inp(16, 32, 32)), 1, offs, 2, 9, 0, 0, 0, ctypes.byref(out), None) == \
        nvfp4.ERR_INVALID_ARG  # mode
    assert grp(ctypes.byref(_inp(16, 32, 32)), 3, offs, 2, 0, 0, 0, 0, ctypes.byref(out), None) == \
        nvfp4.ERR_UNSUPPORTED  # columnwise
    assert grp(ctypes.byref(_inp(16, 32, 32)), 1 | nvfp4.FAST_MATH, offs, 2, 0, 0, 0, 0, ctypes.byref(out),
               None) == nvfp4.ERR_UNSUPPORTED
    assert grp(ctypes.byref(_inp(16, 32, 32)), 1, offs, 1 << 31, 0, 0, 0, 0, ctypes.byref(out), None) == \
        nvfp4.ERR_INVALID_ARG  # 2^31 groups
    assert grp(ctypes.byref(_inp(16, 32, 32)), 1, None, 2, 0, 0, 0, 0, ctypes.byref(out), None) == \
        nvfp4.ERR_INVALID_ARG  # no offsets
    dq = lib.nvfp4_dequantize
    assert dq(16, 16, 16, 4, 24, 0, 16, 0, None) == nvfp4.ERR_INVALID_ARG  # cols % 16
    assert dq(16, 16, 16, 4, 32, 0, 16, 9, None) == nvfp4.ERR_INVALID_ARG  # dtype
    assert dq(None, 16, 16, 4, 32, 0, 16, 0, None) == nvfp4.ERR_INVALID_ARG


def test_binding_fails_loudly_without_the_library(tmp_path):
    with pytest.raises(OSError):
        nvfp4.load(str(tmp_path / "missing.so"))


def test_failure_record_and_wait_limit_arguments(lib):
    assert lib.nvfp4_workspace_status(None, None) == nvfp4.ERR_INVALID_ARG
    assert lib.nvfp4_workspace_status(ctypes.c_void_p(12), None) == nvfp4.ERR_INVALID_ARG  # misaligned
    assert lib.nvfp4_set_wait_limit(1 << 32) == nvfp4.ERR_INVALID_ARG
    assert lib.nvfp4_set_wait_limit(0) == nvfp4.OK
    assert lib.nvfp4_set_wait_limit(-1) == nvfp4.OK  # back to the default
