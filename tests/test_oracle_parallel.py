"""The oracle's parallel orchestration (output row ranges on host threads, the
per-tensor amax as the maximum of slice maxima) gives the single-threaded
oracle's result bit for bit, for every mode, orientation and layout, NaN
included.  It is what the all-cores CPU baseline and the full-size parity
tests run."""
import numpy as np
import pytest
import torch

import oracle


def bits(x: torch.Tensor) -> np.ndarray:
    return x.contiguous().view(torch.int16).numpy().view(np.uint16)


def data(rows, cols, seed, nan=False):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(rows, cols, generator=g) * torch.exp(torch.randn(rows, 1, generator=g))
    x[torch.rand(rows, cols, generator=g) < 0.01] = 0.0
    if nan:
        x[rows - 2, cols // 3] = float("nan")
    return x.to(torch.bfloat16)


CASES = [
    dict(mode="rne"),
    dict(mode="sr", seed=3, offset=5, swizzled=True),
    dict(mode="sr", rht=True, sign_mask=0xA5C3, seed=1, swizzled=True),
    dict(mode="sr", rht=True, sign_mask=0x0F0F, seed=2, colwise=True, swizzled=True),
    dict(mode="rne", block2d=True),
    dict(mode="rne", block2d=True, colwise=True),
    dict(mode="4o6", per_row=True),
    dict(mode="4o6"),
]


@pytest.mark.parametrize("nan", [False, True])
@pytest.mark.parametrize("kw", CASES, ids=lambda kw: "-".join(f"{k}={v}" for k, v in kw.items()))
def test_parallel_oracle_equals_the_single_call(kw, nan):
    x = bits(data(160, 224, 7, nan=nan))
    one = oracle.quantize(x, **kw)
    for threads in (1, 3, 7):
        par = oracle.quantize_parallel(x, threads=threads, **kw)
        for k in ("codes", "scales"):
            assert np.array_equal(par[k], one[k]), (k, threads)
        for k in ("amax", "global_scale"):
            a, b = par[k].view(np.uint32), one[k].view(np.uint32)
            assert np.array_equal(a, b) or (np.isnan(par[k]).all() and np.isnan(one[k]).all()), (k, threads)


@pytest.mark.parametrize("colwise", [False, True])
@pytest.mark.parametrize("rht", [False, True])
def test_parallel_amax_equals_the_single_call(colwise, rht):
    x = bits(data(96, 320, 9))
    want = oracle.amax(x, colwise=colwise, rht=rht, sign_mask=0x1234)[0][0]
    for threads in (1, 2, 5, 64):
        got = oracle.amax_parallel(x, colwise=colwise, rht=rht, sign_mask=0x1234, threads=threads)
        assert np.float32(got).view(np.uint32) == np.float32(want).view(np.uint32)
