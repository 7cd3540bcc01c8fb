"""The RHT amax passes skip the butterfly of a block whose 16 max|v| lies below
a maximum already found (no butterfly output exceeds it: every stage rounds
|a +- b| to at most RN(|a| + |b|)).  The result must still be the oracle's
maximum bit for bit, whatever the data, so these inputs aim at the test's
edges: constant blocks, whose largest output is exactly the bound; a maximum
in the very last rows, found after the shared bound has settled; subnormal
inputs, whose bound is computed on the bit pattern; negative values; NaN and
Inf anywhere.  Each runs through the standalone amax entry point (rowwise and
columnwise) and through quantize calls on the two-kernel path (above 2^22
elements), for one orientation and for both ("在 RTX 5090 (SM120) 上补全 NVFP4
量化相关 kernel", section "随机 Hadamard 变换": the amax is taken over the
transformed values)."""
import numpy as np
import pytest
import torch

import oracle
from tensor_quantization_gb300 import nvfp4

pytestmark = pytest.mark.gpu

R, C = 2048, 4096  # 2^23 elements: amax pass + quantize kernels


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from tensor_quantization_gb300 import build
    build.build()
    nvfp4.load()


def np_bits(x: torch.Tensor) -> np.ndarray:
    x = x.contiguous()
    if x.dtype == torch.bfloat16:
        return x.view(torch.int16).numpy().view(np.uint16)
    return x.numpy()


def same_bits(a, b) -> bool:
    a = np.asarray(a, np.float32).ravel()
    b = np.asarray(b, np.float32).ravel()
    nan = np.isnan(a) & np.isnan(b)
    return a.shape == b.shape and bool(np.all(nan | (a.view(np.uint32) == b.view(np.uint32))))


CASES = ["constant_blocks", "late_max", "one_spike_blocks", "subnormal", "negative", "nan_late", "inf_late",
         "ninf_early"]


def make(case: str, dtype) -> torch.Tensor:
    g = torch.Generator().manual_seed(100 + CASES.index(case))
    if case == "constant_blocks":
        # every 16-block (along rows and along columns) holds one value up to sign
        # patterns that keep it constant in magnitude: the largest butterfly
        # output of such a block is exactly 16 |v|, the skip bound itself
        v = torch.exp(torch.randn(R // 16, C // 16, generator=g) * 2)
        x = v.repeat_interleave(16, 0).repeat_interleave(16, 1)
    elif case == "late_max":
        x = torch.randn(R, C, generator=g)
        x[-1, -16:] *= 1000.0  # in the last tile of rows and of columns
        x[-16:, -1] *= 900.0
    elif case == "one_spike_blocks":
        # one large element per block and tiny others: the bound is 16x the output
        x = torch.randn(R, C, generator=g) * 1e-3
        x[:, ::16] = torch.randn(R, C // 16, generator=g) * 10
    elif case == "subnormal":
        x = torch.randn(R, C, generator=g) * 1e-39
        x[5, 7] = 3e-38
    elif case == "negative":
        x = -torch.rand(R, C, generator=g) * 4
    elif case in ("nan_late", "inf_late", "ninf_early"):
        x = torch.randn(R, C, generator=g)
        if case == "nan_late":
            x[-3, -5] = float("nan")
        elif case == "inf_late":
            x[-1, 100] = float("inf")
        else:
            x[0, 0] = float("-inf")
    else:
        raise ValueError(case)
    return x.to(dtype)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "fp32"])
@pytest.mark.parametrize("case", CASES)
def test_rht_amax_is_exact_with_the_skip(case, dtype):
    x = make(case, dtype)
    xd = x.cuda()
    xb = np_bits(x)
    want = {col: oracle.amax(xb, colwise=col, rht=True) for col in (False, True)}
    ws = torch.zeros(nvfp4.nvfp4_workspace_bytes(), dtype=torch.uint8, device="cuda")
    for col in (False, True):  # standalone entry point
        a = torch.empty(1, device="cuda")
        gs = torch.empty(1, device="cuda")
        nvfp4.nvfp4_amax(xd, nvfp4.COLWISE if col else nvfp4.ROWWISE, True, 0x5A5A,
                         nvfp4.make_output(amax=a, global_scale=gs), ws)
        torch.cuda.synchronize()
        assert same_bits(a.cpu(), want[col][0]), (col, a.item(), want[col][0])
        assert same_bits(gs.cpu(), want[col][1])
    for rowwise, colwise in ((True, False), (False, True), (True, True)):  # consumer calls
        q = nvfp4.quantize(xd, mode="sr", rowwise=rowwise, colwise=colwise, rht=True, sign_mask=0x5A5A, seed=3)
        torch.cuda.synchronize()
        exp = [want[False][0]] * rowwise + [want[True][0]] * colwise
        assert same_bits(q.amax.cpu(), np.concatenate(exp)), (rowwise, colwise, q.amax.cpu(), exp)
    assert int(ws.view(torch.int32).abs().sum()) == 0


def test_both_orientations_codes_from_the_one_read_pass():
    """The two-orientation call on the one-read amax pass gives the oracle's
    codes and scales in both orientations (the maxima differ per orientation)."""
    x = make("late_max", torch.bfloat16)
    mask = 0x3C96
    q = nvfp4.quantize(x.cuda(), mode="sr", rowwise=True, colwise=True, rht=True, swizzled=True, sign_mask=mask,
                       seed=9, offset=4)
    torch.cuda.synchronize()
    xb = np_bits(x)
    for col, codes, scales in ((False, q.codes_row, q.scales_row), (True, q.codes_col, q.scales_col)):
        o = oracle.quantize(xb, colwise=col, mode="sr", swizzled=True, rht=True, sign_mask=mask, seed=9, offset=4)
        assert np.array_equal(codes.cpu().numpy(), o["codes"])
        assert np.array_equal(scales.cpu().numpy().ravel(), o["scales"].ravel())
        assert same_bits(q.global_scale.cpu()[int(col)], o["global_scale"])


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "fp32"])
@pytest.mark.parametrize("case", CASES)
def test_grouped_rht_amax_is_exact_with_the_skip(case, dtype):
    """The grouped amax pass restarts its running maximum for every group
    segment; each group's maximum must still be the oracle's, bit for bit."""
    x = make(case, dtype)
    offs = [0, 700, 701, 701, 1500, 2047, R]
    xb = np_bits(x)
    q = nvfp4.quantize_grouped(x.cuda(), torch.tensor(offs, dtype=torch.int64, device="cuda"), mode="rht_sr",
                               sign_mask=0x5A5A, seed=3)
    torch.cuda.synchronize()
    want = [oracle.amax(xb[o0:o1], rht=True)[0] if o1 > o0 else np.float32([0.0])
            for o0, o1 in zip(offs[:-1], offs[1:])]
    assert same_bits(q.amax.cpu(), np.concatenate([np.asarray(w, np.float32).ravel() for w in want]))
