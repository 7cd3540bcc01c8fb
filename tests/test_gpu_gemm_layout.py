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


def _gemm_codes(codes_a, scales_a, gs_a, codes_b, scales_b, gs_b):
    """cuBLAS block-scaled FP4 GEMM of two code arrays (rows x K/2 each): A @ B^T."""
    qa = nvfp4.Quantized(codes_a, scales_a, None, None, None, gs_a, 0)
    qb = nvfp4.Quantized(codes_b, scales_b, None, None, None, gs_b, 0)
    return _fp4_gemm(qa, qb)


def test_wgrad_gemm_of_columnwise_rht_sr_operands():
    """The weight gradient dW = G^T X of a linear layer contracts over the tokens,
    so both operands are quantized columnwise (blocks along the token
    dimension) with the RHT and stochastic rounding ("nvfp4-sm120" README,
    section "Layout": Wgrad takes RHT + SR operands; "在 RTX 5090 (SM120) 上补全
    NVFP4 量化相关 kernel", section "随机 Hadamard 变换").  With the same sign
    mask on both, the transform cancels in the contraction (each block's
    (H16 D / 4)(H16 D / 4)^T = I), so cuBLAS's FP4 GEMM of the columnwise codes
    must give the fp64 product of the operands decoded back to the source basis
    (nvfp4_dequantize_rht), and approximate G^T X itself.  X comes from a
    call that produces both orientations from one amax read (its rowwise codes
    are the forward operand)."""
    T, N, K = 1024, 256, 384
    mask = 0x6A3C
    g = torch.Generator().manual_seed(11)
    G = (torch.randn(T, N, generator=g) * 1e-2).to(torch.bfloat16).cuda()
    X = (torch.randn(T, K, generator=g) * torch.exp(torch.randn(1, K, generator=g))).to(torch.bfloat16).cuda()
    qg = nvfp4.quantize(G, mode="sr", rowwise=False, colwise=True, rht=True, sign_mask=mask, seed=21,
                        swizzled=True)
    qx = nvfp4.quantize(X, mode="sr", rowwise=True, colwise=True, rht=True, sign_mask=mask, seed=22, swizzled=True)
    gs_g, gs_x = qg.global_scale[:1], qx.global_scale[1:2]  # the columnwise scale of X is [1]
    got = _gemm_codes(qg.codes_col, qg.scales_col, gs_g, qx.codes_col, qx.scales_col, gs_x).double().cpu().numpy()
    # both operands decoded to the source basis: [N, T] and [K, T]
    dg = nvfp4.dequantize(qg.codes_col, qg.scales_col, gs_g, N, T, swizzled=True, rht_sign_mask=mask).double()
    dx = nvfp4.dequantize(qx.codes_col, qx.scales_col, gs_x, K, T, swizzled=True, rht_sign_mask=mask).double()
    want = (dg @ dx.t()).cpu().numpy()
    scale = np.abs(dg.cpu().numpy()) @ np.abs(dx.cpu().numpy()).T
    err = np.abs(got - want) / np.maximum(scale, 1e-30)
    assert err.max() < 1e-2, err.max()  # the GEMM's output rounding and accumulation order only
    # and the quantized product estimates the true weight gradient
    exact = (G.double().t() @ X.double()).cpu().numpy()
    gx = np.abs(G.double().cpu().numpy()).T @ np.abs(X.double().cpu().numpy())
    # (the CPU oracle's codes for these inputs give 0.047 and 0.195: each FP4
    # operand carries ~14% relative noise)
    assert (np.abs(got - exact) / np.maximum(gx, 1e-30)).max() < 0.1
    rel = np.linalg.norm(got - exact) / np.linalg.norm(exact)
    assert rel < 0.3, rel  # an unrelated product is off by ~1.4

    # power: without the shared transform (X's columnwise codes made with 8 of
    # the 16 signs flipped) the transform no longer cancels and the product is
    # unrelated to G^T X (1.42 with the oracle's codes)
    qx2 = nvfp4.quantize(X, mode="sr", rowwise=False, colwise=True, rht=True, sign_mask=mask ^ 0x0F0F, seed=22,
                         swizzled=True)
    bad = _gemm_codes(qg.codes_col, qg.scales_col, gs_g, qx2.codes_col, qx2.scales_col,
                      qx2.global_scale[:1]).double().cpu().numpy()
    assert np.linalg.norm(bad - exact) / np.linalg.norm(exact) > 1.0
    # and a scrambled scale tile is far off
    perm = qg.scales_col.view(-1, 512).flip(1).reshape(-1).contiguous()
    bad = _gemm_codes(qg.codes_col, perm, gs_g, qx.codes_col, qx.scales_col, gs_x).double().cpu().numpy()
    assert (np.abs(bad - want) / np.maximum(scale, 1e-30)).max() > 0.05
