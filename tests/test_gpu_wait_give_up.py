"""A bounded device-side wait that runs out is reported, without a fault or a
hang: the one-kernel path's grid-wide amax barrier (a poll of a global word) is
given a limit of zero polls, so every CTA gives up at once, finishes its work
with the maximum it has seen and counts itself out.  The call's global scale
must come back NaN, the workspace counters zero, the failure record set and
sticky (a later call is poisoned too) until nvfp4_workspace_status reports
NVFP4_ERR_TIMEOUT and clears it; then calls are exact again.  Every copy a CTA
issues is waited for on both passes whatever the barrier returned, so nothing
is in flight when a CTA exits.  TMA waits are not forced to give up."""
import math

import numpy as np
import pytest
import torch

import oracle
from tensor_quantization_gb300 import nvfp4
from tensor_quantization_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from tensor_quantization_gb300 import build
    build.build()
    nvfp4.load()
    yield
    nvfp4.nvfp4_set_wait_limit(-1)


def _call(x, q, ws, rht, mask):
    out = nvfp4.make_output(q.codes_row, q.scales_row, None, None, q.amax, q.global_scale)
    if rht:
        nvfp4.nvfp4_quantize_rht_sr(x, nvfp4.ROWWISE | nvfp4.SWIZZLED, mask, 1, 0, out, ws)
    else:
        nvfp4.nvfp4_quantize_rne(x, nvfp4.ROWWISE, out, ws)
    torch.cuda.synchronize()


def _oracle(x, rht, mask):
    xb = x.cpu().view(torch.int16).numpy().view(np.uint16)
    return oracle.quantize(xb, mode="sr" if rht else "rne", swizzled=rht, rht=rht, sign_mask=mask, seed=1,
                           offset=0)


@pytest.mark.parametrize("rht", [False, True])
def test_grid_barrier_give_up_is_reported_and_recovered(rht):
    w = wl.WORKLOADS["act_rht_sr_8192x4096" if rht else "randn_rne_256x1024"].resized(256, 1024)
    x_cpu, mask = wl.make_input(w)
    x = x_cpu.cuda()  # 2^18 elements: the one-kernel path
    flags = nvfp4.ROWWISE | (nvfp4.SWIZZLED if rht else 0)
    q = nvfp4.alloc_outputs(x, flags)
    ws = torch.zeros(nvfp4.nvfp4_workspace_bytes(), dtype=torch.uint8, device="cuda")
    words = ws.view(torch.int32)
    try:
        nvfp4.nvfp4_set_wait_limit(0)
        _call(x, q, ws, rht, mask)
        assert math.isnan(q.global_scale.item())
        assert words[:3].tolist() == [0, 0, 0]  # the counters came back to zero
        assert words[3].item() != 0  # the failure record
        nvfp4.nvfp4_set_wait_limit(-1)
        _call(x, q, ws, rht, mask)  # a sound call on a workspace with an unread record
        assert math.isnan(q.global_scale.item())
        assert nvfp4.nvfp4_workspace_status(ws) == nvfp4.ERR_TIMEOUT
        assert nvfp4.nvfp4_workspace_status(ws) == nvfp4.OK
        assert words.tolist() == [0] * words.numel()
    finally:
        nvfp4.nvfp4_set_wait_limit(-1)
    _call(x, q, ws, rht, mask)
    o = _oracle(x, rht, mask)
    assert np.array_equal(q.codes_row.cpu().numpy(), o["codes"])
    assert np.array_equal(q.scales_row.cpu().numpy().ravel(), o["scales"].ravel())
    assert q.global_scale.cpu().numpy().view(np.uint32)[0] == o["global_scale"].view(np.uint32)[0]
    assert nvfp4.nvfp4_workspace_status(ws) == nvfp4.OK


def test_the_limit_does_not_touch_the_two_kernel_path():
    w = wl.WORKLOADS["act_rht_sr_8192x4096"].resized(4096, 2048)  # 2^23 elements: amax + quantize kernels
    x_cpu, mask = wl.make_input(w)
    x = x_cpu.cuda()
    q = nvfp4.alloc_outputs(x, nvfp4.ROWWISE | nvfp4.SWIZZLED)
    ws = torch.zeros(nvfp4.nvfp4_workspace_bytes(), dtype=torch.uint8, device="cuda")
    try:
        nvfp4.nvfp4_set_wait_limit(0)
        _call(x, q, ws, True, mask)
    finally:
        nvfp4.nvfp4_set_wait_limit(-1)
    assert nvfp4.nvfp4_workspace_status(ws) == nvfp4.OK
    o = _oracle(x, True, mask)
    assert np.array_equal(q.codes_row.cpu().numpy(), o["codes"])
    assert q.global_scale.cpu().numpy().view(np.uint32)[0] == o["global_scale"].view(np.uint32)[0]
