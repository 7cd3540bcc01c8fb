"""Cross-check of the packed layout against a library routine: cuBLAS's block-
scaled FP4 GEMM (torch._scaled_mm with float4_e2m1fn_x2 operands and
SWIZZLE_32_4_4 float8_e4m3fn block scales) must agree with an fp64 product of
the library's own dequantized operands.  This pins the nibble order, the E2M1
and E4M3 encodings and the swizzled scale layout to how the hardware GEMM
reads them ("nvfp4-sm120" README, sections "Approach" and "Layout": the
quantizer's outputs feed a block-scaled FP4 GEMM directly).  Skipped when the
installed torch or cuBLAS has no NVFP4 GEMM for this GPU.
"""
import numpy as np
import pytest
import torch

from tensor_quantization_gb300 import nvfp4

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    if not hasattr(torch, "float4_e2m1fn_x2"):
        pytest.skip("this torch has no float4_e2m1fn_x2")
    from tensor_quantization_gb300 import build
    build.build()
    nvfp4.load()


def _operand(rows, k, data_seed, **kw):
    g = torch.Generator().manual_seed(data_seed)
    x = (torch.randn(rows, k, generator=g) * torch.exp(torch.randn(rows, 1, generator=g))).to(torch.bfloat16).cuda()
    q = nvfp4.quantize(x, mode=kw.pop("mode", "rne"), swizzled=True, **kw)
    deq = nvfp4.dequantize(q.codes_row, q.scales_row, q.global_scale, rows, k, swizzled=True)
    return q, deq


def _fp4_gemm(qa, qb):
    a = qa.codes_row.view(torch.float4_e2m1fn_x2)
    b = qb.codes_row.view(torch.float4_e2m1fn_x2).t()
    sa = qa.scales_row.view(torch.float8_e4m3fn)
    sb = qb.scales_row.view(torch.float8_e4m3fn)
    try:
        out = torch._scaled_mm(a, b, sa, sb, out_dtype=torch.float32)
    except (RuntimeError, TypeError, NotImplementedError) as e:
        try:
            out = torch._scaled_mm(a, b, sa, sb, out_dtype=torch.bfloat16).float()
        except (RuntimeError, TypeError, NotImplementedError):
            pytest.skip(f"no NVFP4 _scaled_mm here: {str(e).splitlines()[0][:120]}")
    return out * (qa.global_scale * qb.global_scale)


@pytest.mark.parametrize("mode", ["rne", "sr", "rht_sr"])
def test_fp4_gemm_reads_our_layout(mode):
    M, N, K = 256, 384, 1024
    kw = {"rne": dict(mode="rne"), "sr": dict(mode="sr", seed=5),
          "rht_sr": dict(mode="sr", rht=True, sign_mask=0x8421, seed=6)}[mode]
    qa, da = _operand(M, K, 1, **dict(kw))
    qb, db = _operand(N, K, 2, **dict(kw))
    got = _fp4_gemm(qa, qb).double().cpu().numpy()
    want = (da.double() @ db.double().t()).cpu().numpy()
    scale = np.abs(da.double().cpu().numpy()) @ np.abs(db.double().cpu().numpy()).T
    err = np.abs(got - want) / np.maximum(scale, 1e-30)
    assert err.max() < 1e-2, err.max()  # bf16-or-fp32 output rounding and accumulation order only

    # the check has power: the same codes with each 512-byte scale tile reversed
    # (rows and scale columns misplaced inside the tile) are far off
    perm = qa.scales_row.view(-1, 512).flip(1).reshape(-1).contiguous()
    qa_bad = nvfp4.Quantized(qa.codes_row, perm, None, None, qa.amax, qa.global_scale, qa.flags)
    bad = _fp4_gemm(qa_bad, qb).double().cpu().numpy()
    assert (np.abs(bad - want) / np.maximum(scale, 1e-30)).max() > 0.05
