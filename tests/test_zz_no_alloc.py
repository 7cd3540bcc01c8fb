"""nvfp4_quantize_rht_sr_static: the quantize entry point for callers that
cannot allocate device memory (its amax scratch lives inside the library).

It must give exactly the outputs of nvfp4_quantize_rht_sr with a caller
workspace, and of the CPU oracle, on consecutive calls, through the C ABI:
on the two-kernel path (amax pass, then quantize) and on the one-kernel path
of small rowwise tensors (whose grid barrier uses three scratch words).  This
file is collected last so that a stop at the first failure has already run
every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from tensor_quantization_gb300 import nvfp4
from tensor_quantization_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from tensor_quantization_gb300 import build
    build.build()
    L = nvfp4.load()
    L.nvfp4_quantize_rht_sr_static.argtypes = [ctypes.POINTER(nvfp4.Input), ctypes.c_uint32, ctypes.c_uint16,
                                               ctypes.c_uint64, ctypes.c_uint64, ctypes.POINTER(nvfp4.Output),
                                               ctypes.c_void_p]
    L.nvfp4_quantize_rht_sr_static.restype = ctypes.c_int
    return L


def _outputs(x, flags):
    q = nvfp4.alloc_outputs(x, flags)
    o = nvfp4.make_output(q.codes_row, q.scales_row, q.codes_col, q.scales_col, q.amax, q.global_scale)
    return q, o


def _host(q):
    return {k: getattr(q, k).cpu().numpy() for k in ("codes_row", "scales_row", "codes_col", "scales_col",
                                                      "amax", "global_scale") if getattr(q, k) is not None}


@pytest.mark.parametrize("orient,rows,cols", [("row", 1024, 2048), ("col", 1024, 2048), ("row", 256, 1024)])
def test_static_entry_point_matches_workspace_entry_point(lib, orient, rows, cols):
    w = wl.WORKLOADS["act_rht_sr_8192x4096"].resized(rows, cols)
    x_cpu, mask = wl.make_input(w)
    xb = x_cpu.view(torch.int16).numpy().view(np.uint16)
    want = oracle.quantize(xb, colwise=orient == "col", mode="sr", swizzled=True, rht=True, sign_mask=mask,
                           seed=1, offset=7)
    x = x_cpu.cuda()
    flags = (nvfp4.ROWWISE if orient == "row" else nvfp4.COLWISE) | nvfp4.SWIZZLED
    ref_q, ref_o = _outputs(x, flags)
    ws = torch.zeros(nvfp4.nvfp4_workspace_bytes(), dtype=torch.uint8, device="cuda")
    nvfp4.nvfp4_quantize_rht_sr(x, flags, mask, 1, 7, ref_o, ws)
    torch.cuda.synchronize()
    ref = _host(ref_q)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for _ in range(2):  # two calls in a row: the shared scratch must come back clean
        q, o = _outputs(x, flags)
        st = lib.nvfp4_quantize_rht_sr_static(ctypes.byref(nvfp4.make_input(x)), flags, mask, 1, 7,
                                              ctypes.byref(o), stream)
        assert st == nvfp4.OK, nvfp4.status_string(st)
        torch.cuda.synchronize()
        got = _host(q)
        for k, v in ref.items():
            assert np.array_equal(got[k].view(np.uint8), v.view(np.uint8)), k
        codes, scales = (got["codes_row"], got["scales_row"]) if orient == "row" else \
            (got["codes_col"], got["scales_col"])
        assert np.array_equal(codes, want["codes"])
        assert np.array_equal(scales.ravel(), want["scales"].ravel())
        assert got["global_scale"].view(np.uint32)[0] == want["global_scale"].view(np.uint32)[0]


def test_static_entry_point_rejects_bad_sizes(lib):
    out = nvfp4.Output(16, 16, 16, 16, 16, 16)
    too_big = nvfp4.Input(16, 0, 1 << 31, 16, 16)
    assert lib.nvfp4_quantize_rht_sr_static(ctypes.byref(too_big), nvfp4.ROWWISE, 0, 0, 0, ctypes.byref(out),
                                            None) == nvfp4.ERR_INVALID_ARG
    ragged = nvfp4.Input(16, 0, 16, 24, 24)
    assert lib.nvfp4_quantize_rht_sr_static(ctypes.byref(ragged), nvfp4.ROWWISE, 0, 0, 0, ctypes.byref(out),
                                            None) == nvfp4.ERR_INVALID_ARG
    torch.cuda.synchronize()
