"""GPU parity: the sm_103a library (through its C ABI) against the CPU oracle.

Codes, scales (pad bytes included) and the amax / global scale must be
bit-identical.  Small cases span several tiles and ragged tails; the five
workloads also run at full size, in the same call ``bench.py`` times.
"""
import math
import zlib

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


def np_bits(x: torch.Tensor) -> np.ndarray:
    x = x.contiguous()
    if x.dtype == torch.bfloat16:
        return x.view(torch.int16).numpy().view(np.uint16)
    return x.numpy()


def same_float_bits(a, b) -> bool:
    a = np.asarray(a, np.float32).ravel()
    b = np.asarray(b, np.float32).ravel()
    if a.shape != b.shape:
        return False
    both_nan = np.isnan(a) & np.isnan(b)
    return bool(np.all(both_nan | (a.view(np.uint32) == b.view(np.uint32))))


def to_device(x_cpu: torch.Tensor) -> torch.Tensor:
    """Device copy whose row pitch is a multiple of 16 bytes (the ABI's rule)."""
    R, C = x_cpu.shape
    per16 = 16 // x_cpu.element_size()
    ld = (C + per16 - 1) // per16 * per16
    if ld == C or R <= 1:
        return x_cpu.cuda()
    buf = torch.zeros(R, ld, dtype=x_cpu.dtype, device="cuda")
    buf[:, :C] = x_cpu.cuda()
    return buf[:, :C]


def gpu_run(x_cpu: torch.Tensor, x_dev: torch.Tensor | None = None, **kw) -> dict:
    x = to_device(x_cpu) if x_dev is None else x_dev
    q = nvfp4.quantize(x, **kw)
    torch.cuda.synchronize()
    out = {}
    for k in ("codes_row", "scales_row", "codes_col", "scales_col", "amax", "global_scale"):
        t = getattr(q, k)
        out[k] = None if t is None else t.cpu().numpy()
    return out


def oracle_run(x_cpu: torch.Tensor, *, mode="rne", rowwise=True, colwise=False, block2d=False, per_row=False,
               swizzled=False, rht=False, sign_mask=0, seed=0, offset=0, amax=None, row_range=None) -> dict:
    xn = np_bits(x_cpu)
    kw = dict(mode=mode, block2d=block2d, per_row=per_row, swizzled=swizzled, rht=rht, sign_mask=sign_mask,
              seed=seed, offset=offset, row_range=row_range,
              amax_given=None if amax is None else float(np.asarray(amax).ravel()[0]))
    out = {}
    amaxes, scales = [], []
    for orient, on in (("row", rowwise), ("col", colwise)):
        if not on:
            continue
        okw = dict(kw)
        if rht and rowwise and colwise and amax is not None:  # two given amaxes: [0] rows, [1] columns
            okw["amax_given"] = float(np.asarray(amax).ravel()[0 if orient == "row" else 1])
        o = oracle.quantize(xn, colwise=(orient == "col"), **okw)
        out[f"codes_{orient}"] = o["codes"]
        out[f"scales_{orient}"] = o["scales"].ravel()
        amaxes.append(o["amax"])
        scales.append(o["global_scale"])
    if rht and rowwise and colwise:  # one amax per orientation
        out["amax"], out["global_scale"] = np.concatenate(amaxes), np.concatenate(scales)
    else:
        out["amax"], out["global_scale"] = amaxes[-1], scales[-1]
    return out


def oracle_run_all_cores(x_cpu: torch.Tensor, *, mode="rne", rowwise=True, colwise=False, block2d=False,
                         per_row=False, swizzled=False, rht=False, sign_mask=0, seed=0, offset=0, amax=None) -> dict:
    """oracle_run of the whole tensor on every host core (the oracle's row-range
    threads; bit-identical to one thread)."""
    xn = np_bits(x_cpu)
    out, amaxes, scales = {}, [], []
    for i, (orient, on) in enumerate((("row", rowwise), ("col", colwise))):
        if not on:
            continue
        given = None
        if amax is not None:
            a = np.asarray(amax).ravel()
            given = float(a[i if (rht and rowwise and colwise) else 0])
        o = oracle.quantize_parallel(xn, colwise=orient == "col", mode=mode, block2d=block2d, per_row=per_row,
                                     swizzled=swizzled, rht=rht, sign_mask=sign_mask, seed=seed, offset=offset,
                                     amax_given=given)
        out[f"codes_{orient}"] = o["codes"]
        out[f"scales_{orient}"] = o["scales"].ravel()
        amaxes.append(o["amax"])
        scales.append(o["global_scale"])
    if rht and rowwise and colwise:
        out["amax"], out["global_scale"] = np.concatenate(amaxes), np.concatenate(scales)
    else:
        out["amax"], out["global_scale"] = amaxes[-1], scales[-1]
    return out


def assert_parity(g: dict, o: dict, rows_sampled=None):
    for k in ("codes_row", "scales_row", "codes_col", "scales_col"):
        if k not in o:
            continue
        a, b = g[k], o[k]
        if rows_sampled is not None and k.startswith("codes"):
            a, b = a[rows_sampled], b[rows_sampled]
        assert a.shape == b.shape, k
        bad = np.argwhere(a.reshape(b.shape) != b)
        assert bad.size == 0, f"{k}: {len(bad)} mismatches, first at {bad[:5].tolist()}"
    assert same_float_bits(g["amax"], o["amax"]), (g["amax"][:4], o["amax"][:4])
    assert same_float_bits(g["global_scale"], o["global_scale"]), (g["global_scale"][:4], o["global_scale"][:4])


def mixed_input(rows, cols, seed, dtype=torch.bfloat16):
    """Gaussian rows with log-uniform scales, exact zeros, -0 and outliers."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(rows, cols, generator=g) * torch.exp(torch.rand(rows, 1, generator=g) * 6 - 3)
    x[torch.rand(rows, cols, generator=g) < 0.02] = 0.0
    x[torch.rand(rows, cols, generator=g) < 0.01] = -0.0
    x[torch.rand(rows, cols, generator=g) < 0.002] *= 300.0
    return x.to(dtype)


# ------------------------------------------------------ the five workloads
SMALL = {
    "randn_rne_256x1024": (256, 1024),
    "act_rht_sr_8192x4096": (520, 1024),
    "weight_2d_rne_14336x4096": (272, 512),
    "grad_col_rht_sr_16384x8192": (256, 520),
    "rowscaled_4o6_8192x8192": (96, 1024),
    "act_rht_sr_given_8192x4096": (520, 1024),
    "act_rht_sr_rowcol_8192x4096": (528, 1040),
}


def workload_kwargs(w: wl.Workload, mask: int) -> dict:
    return dict(mode=w.mode, rowwise=w.rowwise, colwise=w.colwise, block2d=w.block2d, per_row=w.per_row,
                swizzled=w.swizzled, rht=w.rht, sign_mask=mask, seed=w.philox_seed, offset=w.philox_offset)


def workload_runs(w: wl.Workload, x: torch.Tensor, mask: int) -> tuple[dict, dict]:
    """(GPU call kwargs, oracle kwargs); a given-amax workload passes the
    oracle's amax to both, so the GPU call runs the encode pass alone."""
    kw = workload_kwargs(w, mask)
    if not w.amax_given:
        return kw, kw
    a, _ = oracle.amax(np_bits(x), colwise=w.colwise and not w.rowwise, rht=w.rht, sign_mask=mask)
    return dict(kw, amax=torch.from_numpy(a)), dict(kw, amax=a)


@pytest.mark.parametrize("name", list(SMALL))
def test_workload_small(name):
    w = wl.WORKLOADS[name].resized(*SMALL[name])
    x, mask = wl.make_input(w)
    gkw, okw = workload_runs(w, x, mask)
    assert_parity(gpu_run(x, **gkw), oracle_run(x, **okw))


@pytest.mark.slow
@pytest.mark.parametrize("name", list(wl.WORKLOADS))
def test_workload_full_size(name):
    """Full-size workloads through the call bench.py times, every output byte
    compared with the oracle (run over all host cores)."""
    w = wl.WORKLOADS[name]
    if w.groups:
        pytest.skip("grouped: test_full_size_rht_both_orientations_and_groups covers this input with these group offsets")
    x, mask = wl.make_input(w)
    gkw, kw = workload_runs(w, x, mask)
    g = gpu_run(x, **gkw)
    assert_parity(g, oracle_run_all_cores(x, **kw))
    if w.block2d:
        # 2D: the column codes are the nibble transpose of the row codes
        cr, cc = g["codes_row"], g["codes_col"]
        ur = np.stack([cr & 15, cr >> 4], -1).reshape(cr.shape[0], -1)
        uc = np.stack([cc & 15, cc >> 4], -1).reshape(cc.shape[0], -1)
        assert np.array_equal(ur.T, uc)


# ----------------------------------------------------- the option matrix
MODES = ["rne", "sr", "rht_sr", "4o6"]


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "fp32"])
@pytest.mark.parametrize("swizzled", [False, True], ids=["linear", "swizzled"])
@pytest.mark.parametrize("orient", ["row", "col", "both"])
@pytest.mark.parametrize("mode", MODES)
def test_option_matrix(mode, orient, swizzled, dtype):
    x = mixed_input(160, 208, seed=zlib.crc32(f"{mode}{orient}{swizzled}{dtype}".encode()) & 0xFFFF, dtype=dtype)
    kw = dict(mode="sr" if mode == "rht_sr" else mode, rht=mode == "rht_sr", rowwise=orient in ("row", "both"),
              colwise=orient in ("col", "both"), swizzled=swizzled, sign_mask=0xB4E1, seed=77, offset=5)
    assert_parity(gpu_run(x, **kw), oracle_run(x, **kw))


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "fp32"])
@pytest.mark.parametrize("swizzled", [False, True], ids=["linear", "swizzled"])
@pytest.mark.parametrize("mode", MODES)
def test_per_row(mode, swizzled, dtype):
    x = mixed_input(40, 336, seed=7, dtype=dtype)
    kw = dict(mode="sr" if mode == "rht_sr" else mode, rht=mode == "rht_sr", per_row=True, swizzled=swizzled,
              sign_mask=0x0F0F, seed=3, offset=11)
    assert_parity(gpu_run(x, **kw), oracle_run(x, **kw))


@pytest.mark.parametrize("mode", MODES)
def test_per_row_many_rows_per_cta(mode):
    """Enough rows that every CTA of the staged per-row kernel cycles through
    its row buffers and table slots several times; output rows are compared
    in bands spread over the tensor (the oracle's row range keeps it quick)."""
    rows, cols = 6000, 4096
    x = mixed_input(rows, cols, seed=17)
    x[2999, 77] = float("nan")  # poisons only its own row
    kw = dict(mode="sr" if mode == "rht_sr" else mode, rht=mode == "rht_sr", per_row=True, sign_mask=0x5A3C,
              seed=21, offset=2)
    g = gpu_run(x, **kw)
    for r0, r1 in [(0, 96), (2960, 3040), (rows - 96, rows)]:
        o = oracle_run(x, row_range=(r0, r1), **kw)
        assert np.array_equal(g["codes_row"][r0:r1], o["codes_row"][r0:r1]), (mode, r0)
        assert np.array_equal(g["scales_row"].reshape(rows, -1)[r0:r1], o["scales_row"].reshape(rows, -1)[r0:r1])
        assert same_float_bits(g["amax"][r0:r1], o["amax"][r0:r1])
        assert same_float_bits(g["global_scale"][r0:r1], o["global_scale"][r0:r1])
    assert np.isnan(g["global_scale"][2999]) and not np.isnan(g["global_scale"][2998])


@pytest.mark.parametrize("mode", ["rne", "4o6"])
def test_per_row_long_rows(mode):
    """fp32 rows of 128 KiB exceed the staged kernel's row buffer and take the
    two-read kernel; 64 KiB bf16 rows still fit."""
    for cols, dtype in ((32768, torch.float32), (32768, torch.bfloat16)):
        x = mixed_input(12, cols, seed=18, dtype=dtype)
        kw = dict(mode=mode, per_row=True, swizzled=True)
        assert_parity(gpu_run(x, **kw), oracle_run(x, **kw))


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "fp32"])
@pytest.mark.parametrize("swizzled", [False, True], ids=["linear", "swizzled"])
def test_2d_tiles(swizzled, dtype):
    x = mixed_input(144, 240, seed=9, dtype=dtype)
    for orient in ("row", "col", "both"):
        kw = dict(mode="rne", block2d=True, rowwise=orient != "col", colwise=orient != "row", swizzled=swizzled)
        assert_parity(gpu_run(x, **kw), oracle_run(x, **kw))


# ----------------------------------------------------------- edge cases
def test_single_block_and_tiny_shapes():
    for rows, cols, kw in [(1, 16, dict(mode="rne")), (16, 1, dict(mode="sr", rowwise=False, colwise=True)),
                           (1, 16, dict(mode="sr", rht=True, sign_mask=0xFFFF, seed=2)),
                           (16, 16, dict(mode="rne", block2d=True, colwise=True)),
                           (1, 32, dict(mode="4o6", per_row=True)), (16, 3, dict(mode="rne", rowwise=False,
                                                                                  colwise=True, swizzled=True))]:
        x = mixed_input(rows, cols, seed=rows * 100 + cols)
        assert_parity(gpu_run(x, **kw), oracle_run(x, **kw))


def test_zeros_and_signed_zeros():
    for fill in (0.0, -0.0):
        x = torch.full((32, 64), fill, dtype=torch.bfloat16)
        for kw in (dict(mode="rne"), dict(mode="sr", rht=True, seed=1), dict(mode="4o6", per_row=True)):
            g, o = gpu_run(x, **kw), oracle_run(x, **kw)
            assert_parity(g, o)
            assert np.all(g["codes_row"] == 0) and g["amax"][0] == 0


def test_negative_zero_inside_a_block_keeps_its_sign():
    x = torch.zeros(2, 32)
    x[:, 0] = 3.0
    x[:, 1] = -0.0
    x[:, 2] = -1e-6
    x = x.to(torch.bfloat16)
    for kw in (dict(mode="rne"), dict(mode="sr", seed=4), dict(mode="4o6")):
        g, o = gpu_run(x, **kw), oracle_run(x, **kw)
        assert_parity(g, o)
        assert (g["codes_row"][0, 0] >> 4) == 8  # element 1 = -0 -> code 0x8


@pytest.mark.parametrize("special", ["nan", "inf", "-inf"])
def test_nan_inf_policy(special):
    x = mixed_input(64, 128, seed=12)
    x[17, 45] = float(special)
    for kw in (dict(mode="rne"), dict(mode="sr", rht=True, seed=5), dict(mode="4o6", per_row=True),
               dict(mode="rne", block2d=True, colwise=True), dict(mode="sr", rowwise=False, colwise=True)):
        assert_parity(gpu_run(x, **kw), oracle_run(x, **kw))


@pytest.mark.parametrize("scale", [1e-39, 1e-30, 1e30, 3e38])
def test_extreme_magnitudes_take_the_exact_slow_path(scale):
    x = (mixed_input(48, 96, seed=13, dtype=torch.float32) * scale)
    x = torch.nan_to_num(x, posinf=3.4e38, neginf=-3.4e38)
    for kw in (dict(mode="rne"), dict(mode="sr", seed=9), dict(mode="4o6"), dict(mode="4o6", per_row=True),
               dict(mode="sr", rht=True, seed=1)):
        assert_parity(gpu_run(x, **kw), oracle_run(x, **kw))


def test_subnormal_bf16_inputs():
    bits = torch.randint(1, 0x0080, (32, 64), generator=torch.Generator().manual_seed(3), dtype=torch.int32)
    sign = torch.randint(0, 2, (32, 64), generator=torch.Generator().manual_seed(4), dtype=torch.int32) << 15
    x = (bits | sign).to(torch.int16).view(torch.bfloat16)
    for kw in (dict(mode="rne"), dict(mode="sr", seed=2), dict(mode="4o6"), dict(mode="sr", rht=True, seed=2)):
        assert_parity(gpu_run(x, **kw), oracle_run(x, **kw))


def test_strided_input_rows():
    base = mixed_input(64, 208, seed=14)
    x_dev = base.cuda()[:, 16:192]  # ld = 208 elements, cols = 176
    x_cpu = base[:, 16:192].contiguous()
    for kw in (dict(mode="rne"), dict(mode="sr", rht=True, seed=8), dict(mode="rne", colwise=True),
               dict(mode="4o6", per_row=True), dict(mode="rne", block2d=True, colwise=True)):
        assert_parity(gpu_run(x_cpu, x_dev=x_dev, **kw), oracle_run(x_cpu, **kw))


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "fp32"])
@pytest.mark.parametrize("swizzled", [False, True], ids=["linear", "swizzled"])
def test_rht_both_orientations_from_one_call(swizzled, dtype):
    """RHT + SR into both orientations: each orientation transforms along its own
    blocks and has its own amax ([0] rowwise, [1] columnwise)."""
    x = mixed_input(272, 208, seed=26, dtype=dtype)
    kw = dict(mode="sr", rht=True, rowwise=True, colwise=True, swizzled=swizzled, sign_mask=0x3C5A, seed=13,
              offset=2)
    g, o = gpu_run(x, **kw), oracle_run(x, **kw)
    assert g["amax"].shape == (2,) and g["amax"][0] != g["amax"][1]
    assert_parity(g, o)
    # the same with both amaxes given
    A = torch.from_numpy(o["amax"] * np.float32(1.5)).cuda()
    assert_parity(gpu_run(x, amax=A, **kw), oracle_run(x, amax=A.cpu().numpy(), **kw))


def test_amax_given():
    x = mixed_input(64, 256, seed=15)
    for A in (float(x.float().abs().max()), 7.25, 1e-3):
        for kw in (dict(mode="rne"), dict(mode="sr", seed=1, swizzled=True), dict(mode="4o6", colwise=True)):
            g = gpu_run(x, amax=torch.tensor([A]).cuda(), **kw)
            assert_parity(g, oracle_run(x, amax=A, **kw))


def test_empty_inputs():
    for shape in ((0, 32), (16, 0), (0, 0)):
        x = torch.zeros(*shape, dtype=torch.bfloat16, device="cuda")
        q = nvfp4.quantize(x, mode="rne", rowwise=shape[1] % 16 == 0, colwise=shape[1] % 16 != 0)
        torch.cuda.synchronize()
        assert float(q.amax[0]) == 0.0 and float(q.global_scale[0]) == 0.0


def test_repeated_calls_reuse_the_workspace_and_offsets_change_draws():
    x = mixed_input(128, 256, seed=16)
    kw = dict(mode="sr", rht=True, sign_mask=0x1234, seed=10)
    a = gpu_run(x, offset=0, **kw)
    b = gpu_run(x, offset=0, **kw)
    c = gpu_run(x, offset=1, **kw)
    for k in ("codes_row", "scales_row", "amax"):
        assert np.array_equal(a[k], b[k])
    assert not np.array_equal(a["codes_row"], c["codes_row"])
    assert_parity(c, oracle_run(x, offset=1, **kw))
    ws = nvfp4.Workspace.get(torch.device("cuda"))
    assert int(ws.view(torch.int32)[:2].abs().sum()) == 0  # returned to zero


def test_non_default_stream():
    x = mixed_input(256, 512, seed=17).cuda()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        q = nvfp4.quantize(x, mode="sr", rht=True, sign_mask=5, seed=1, swizzled=True)
    s.synchronize()
    o = oracle_run(x.cpu(), mode="sr", rht=True, sign_mask=5, seed=1, swizzled=True)
    assert np.array_equal(q.codes_row.cpu().numpy(), o["codes_row"])


def test_amax_entry_point():
    x = mixed_input(96, 128, seed=18)
    xd = x.cuda()
    for flags, rht in ((nvfp4.ROWWISE, False), (nvfp4.ROWWISE, True), (nvfp4.COLWISE, True),
                       (nvfp4.ROWWISE | nvfp4.SCALE_PER_ROW, True), (nvfp4.ROWWISE | nvfp4.SCALE_PER_ROW, False)):
        per_row = bool(flags & nvfp4.SCALE_PER_ROW)
        n = 96 if per_row else 1
        a = torch.empty(n, device="cuda")
        gsc = torch.empty(n, device="cuda")
        nvfp4.nvfp4_amax(xd, flags, rht, 0xFFFF, nvfp4.make_output(amax=a, global_scale=gsc),
                         nvfp4.Workspace.get(xd.device))
        torch.cuda.synchronize()
        oa, og = oracle.amax(np_bits(x), colwise=bool(flags & nvfp4.COLWISE), rht=rht, per_row=per_row)
        assert same_float_bits(a.cpu().numpy(), oa) and same_float_bits(gsc.cpu().numpy(), og)


def test_amax_entry_point_dynamic_tiles_and_workspace_reuse():
    """A tensor large enough that the standalone pass hands out most tiles from
    its counter (2048 tiles for at most three CTAs per SM): repeated calls,
    interleaved with quantize calls that share the workspace, give the exact
    amax every time and leave every workspace word zero."""
    x = mixed_input(2048, 8192, seed=41)
    xd = x.cuda()
    ws = nvfp4.Workspace.get(xd.device)
    oa, og = oracle.amax(np_bits(x), rht=True)
    plain = float(x.float().abs().max())
    for it in range(3):
        for rht in (True, False):
            a = torch.empty(1, device="cuda")
            gsc = torch.empty(1, device="cuda")
            nvfp4.nvfp4_amax(xd, nvfp4.ROWWISE, rht, 0xFFFF, nvfp4.make_output(amax=a, global_scale=gsc), ws)
            torch.cuda.synchronize()
            if rht:
                assert same_float_bits(a.cpu().numpy(), oa) and same_float_bits(gsc.cpu().numpy(), og)
            else:
                assert float(a.item()) == plain
            assert int(ws.view(torch.int32).abs().sum()) == 0
        q = nvfp4.quantize(xd, mode="sr", rht=True, sign_mask=0xFFFF, seed=it)
        torch.cuda.synchronize()
        assert same_float_bits(q.amax.cpu().numpy(), oa)
        assert int(ws.view(torch.int32).abs().sum()) == 0


# ------------------------------------------------------------ dequantize
@pytest.mark.parametrize("swizzled", [False, True])
@pytest.mark.parametrize("per_row", [False, True])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16], ids=["fp32", "bf16"])
def test_dequantize(swizzled, per_row, out_dtype):
    x = mixed_input(200, 96, seed=19)
    x[3, 5] = float("nan")
    o = oracle.quantize(np_bits(x), mode="4o6" if per_row else "sr", per_row=per_row, swizzled=swizzled, seed=2)
    ref = oracle.dequantize(o["codes"], o["scales"], o["global_scale"], 200, 96, swizzled=swizzled,
                            per_row=per_row, out_dtype="bf16" if out_dtype == torch.bfloat16 else "fp32")
    got = nvfp4.dequantize(torch.from_numpy(o["codes"]).cuda(), torch.from_numpy(o["scales"].ravel()).cuda(),
                           torch.from_numpy(o["global_scale"]).cuda(), 200, 96, swizzled=swizzled,
                           per_row=per_row, out_dtype=out_dtype)
    torch.cuda.synchronize()
    if out_dtype == torch.bfloat16:
        g = got.cpu().view(torch.int16).numpy().view(np.uint16)
        nan_g = (g & 0x7FFF) > 0x7F80
        nan_r = (ref & 0x7FFF) > 0x7F80
        assert np.array_equal(nan_g, nan_r)
        assert np.array_equal(g[~nan_g], ref[~nan_r])
    else:
        assert same_float_bits(got.cpu().numpy(), ref)


def test_round_trip_through_the_library():
    x = mixed_input(128, 256, seed=20)
    q = nvfp4.quantize(x.cuda(), mode="rne", swizzled=True)
    d = nvfp4.dequantize(q.codes_row, q.scales_row, q.global_scale, 128, 256, swizzled=True)
    torch.cuda.synchronize()
    err = (d.cpu() - x.float()).abs()
    assert math.isfinite(float(err.max()))
    assert float((err <= x.float().abs() * 0.25 + 1e-3 * x.float().abs().max()).float().mean()) > 0.99


# ------------------------------------------------------------- fast math
def _nibbles(codes: np.ndarray) -> np.ndarray:
    c = np.asarray(codes, np.uint8)
    return np.stack([c & 15, c >> 4], -1).reshape(c.shape[0], -1)


FAST_CASES = {
    "row_rne": dict(mode="rne"),
    "row_sr": dict(mode="sr", seed=3, offset=1),
    "row_rht_sr": dict(mode="sr", rht=True, sign_mask=0x9C3A, seed=4, swizzled=True),
    "col_rne": dict(mode="rne", rowwise=False, colwise=True),
    "col_rht_sr": dict(mode="sr", rht=True, sign_mask=0x0FF0, seed=5, rowwise=False, colwise=True),
    "both_sr": dict(mode="sr", colwise=True, seed=6),
    "2d": dict(mode="rne", block2d=True, colwise=True),
    "per_row_rht_sr": dict(mode="sr", rht=True, per_row=True, seed=7),
}


@pytest.mark.parametrize("case", list(FAST_CASES))
def test_fast_math_codes_within_one_step(case):
    """FAST_MATH keeps every scale, and changes at most 0.1% of the codes, each
    to the neighbouring grid value of the same sign."""
    x = mixed_input(512, 1024, seed=zlib.crc32(case.encode()) & 0xFFFF)
    kw = FAST_CASES[case]
    g, o = gpu_run(x, fast_math=True, **kw), oracle_run(x, **kw)
    assert same_float_bits(g["amax"], o["amax"]) and same_float_bits(g["global_scale"], o["global_scale"])
    for orient in ("row", "col"):
        if f"codes_{orient}" not in o:
            continue
        assert np.array_equal(g[f"scales_{orient}"], o[f"scales_{orient}"]), orient
        a, b = _nibbles(g[f"codes_{orient}"]), _nibbles(o[f"codes_{orient}"])
        diff = a != b
        assert diff.mean() <= 1e-3, (orient, diff.mean())
        da, db = a[diff].astype(int), b[diff].astype(int)
        assert np.all((da >> 3) == (db >> 3)) and np.all(np.abs((da & 7) - (db & 7)) == 1), orient


# ------------------------------------------------- shards of one tensor
def test_row_shards_reproduce_the_whole_tensor():
    """Rowwise RHT + SR: shards of whole 128-row bands, each quantized with the
    whole tensor's amax (the maximum of the shards' amax, as an all-reduce
    would give) and its row offset, concatenate to the unsharded output."""
    x = mixed_input(1024, 512, seed=21)
    xd = to_device(x)
    kw = dict(mode="sr", rht=True, sign_mask=0x6B2D, seed=8, offset=3, swizzled=True)
    whole = gpu_run(x, x_dev=xd, **kw)
    bounds = [0, 256, 640, 1024]
    amaxes = []
    for r0, r1 in zip(bounds[:-1], bounds[1:]):
        a = torch.empty(1, device="cuda")
        nvfp4.nvfp4_amax(xd[r0:r1], nvfp4.ROWWISE, True, kw["sign_mask"],
                         nvfp4.make_output(amax=a, global_scale=torch.empty(1, device="cuda")),
                         nvfp4.Workspace.get(xd.device))
        amaxes.append(a)
    A = torch.stack(amaxes).max().reshape(1)
    cs_band = nvfp4.nvfp4_scale_bytes(128, 512, nvfp4.SWIZZLED)
    for r0, r1 in zip(bounds[:-1], bounds[1:]):
        part = gpu_run(x[r0:r1], x_dev=xd[r0:r1], amax=A, row0=r0, **kw)
        assert np.array_equal(part["codes_row"], whole["codes_row"][r0:r1]), r0
        assert np.array_equal(part["scales_row"], whole["scales_row"][r0 // 128 * cs_band:r1 // 128 * cs_band]), r0
        assert same_float_bits(part["global_scale"], whole["global_scale"])


@pytest.mark.parametrize("given", [True, False], ids=["amax_given", "one_kernel"])
@pytest.mark.parametrize("mode", ["sr", "rht_sr"])
@pytest.mark.parametrize("row0", [2 ** 27 + 3, 2 ** 26 - 2], ids=["above_2e32", "across_2e32"])
def test_block_counters_with_a_high_word(row0, mode, given):
    """A row shard far into a tensor: its Philox block counters (row0 * C/16
    onward) have their high word set, or cross 2^32 inside the call, with a
    64-bit seed and offset.  The oracle numbers the same blocks (block_base)."""
    R, C = 256, 1024
    x = mixed_input(R, C, seed=41 + (row0 & 7))
    xb = np_bits(x)
    rht = mode == "rht_sr"
    kw = dict(mode="sr", rht=rht, sign_mask=0x2D4B, seed=0x9E37_79B9_7F4A_7C15, offset=0xD1B5_4A32_D192_ED03,
              swizzled=True)
    A = oracle.amax(xb, rht=rht, sign_mask=kw["sign_mask"])[0]
    want = oracle.quantize(xb, amax_given=float(A[0]) if given else None, block_base=row0 * (C // 16), **kw)
    got = gpu_run(x, amax=torch.from_numpy(A).cuda() if given else None, row0=row0, **kw)
    assert np.array_equal(got["codes_row"], want["codes"])
    assert np.array_equal(got["scales_row"], want["scales"].ravel())
    assert same_float_bits(got["global_scale"], want["global_scale"])


@pytest.mark.parametrize("rht", [False, True])
def test_column_shards_reproduce_the_whole_tensor(rht):
    x = mixed_input(256, 1024, seed=22)
    xd = to_device(x)
    kw = dict(mode="sr", rht=rht, sign_mask=0x1357, seed=9, offset=4, rowwise=False, colwise=True)
    whole = gpu_run(x, x_dev=xd, **kw)
    A = torch.from_numpy(whole["amax"]).cuda()
    for c0, c1 in [(0, 384), (384, 512), (512, 1024)]:
        part = gpu_run(x[:, c0:c1].contiguous(), x_dev=xd[:, c0:c1], amax=A, col0=c0, **kw)
        assert np.array_equal(part["codes_col"], whole["codes_col"][c0:c1]), c0
        assert np.array_equal(part["scales_col"].reshape(c1 - c0, -1), whole["scales_col"].reshape(1024, -1)[c0:c1])


def test_per_row_shards_need_no_exchange():
    x = mixed_input(300, 256, seed=23)
    xd = to_device(x)
    kw = dict(mode="sr", per_row=True, seed=10)
    whole = gpu_run(x, x_dev=xd, **kw)
    for r0, r1 in [(0, 100), (100, 300)]:
        part = gpu_run(x[r0:r1], x_dev=xd[r0:r1], row0=r0, **kw)
        assert np.array_equal(part["codes_row"], whole["codes_row"][r0:r1])
        assert np.array_equal(part["scales_row"].reshape(r1 - r0, -1), whole["scales_row"].reshape(300, -1)[r0:r1])
        assert same_float_bits(part["amax"], whole["amax"][r0:r1])


# ------------------------------------------------- which kernels a call runs
def _kernels_of(fn) -> list[str]:
    """Names of the CUDA kernels launched by fn() (CUPTI through torch.profiler)."""
    from torch.profiler import ProfilerActivity, profile
    torch.cuda.synchronize()
    with profile(activities=[ProfilerActivity.CUDA]) as prof:
        fn()
        torch.cuda.synchronize()
    names = [e.name for e in prof.events() if e.device_type == torch.autograd.DeviceType.CUDA]
    return [n for n in names if "nvfp4" in n or n.startswith(("k_", "void nvfp4", "nvfp4"))]


@pytest.mark.parametrize("case", ["row_rht_sr_bf16", "row_rht_sr_fp32", "row_rne", "row_4o6", "col_rht_sr",
                                  "row_large"])
def test_per_tensor_call_launches(case):
    """A small per-tensor rowwise call is one cooperative kernel (amax pass
    folded in); a large one, or a columnwise one, is the amax kernel and the
    quantize kernel."""
    dtype = torch.float32 if case.endswith("fp32") else torch.bfloat16
    shape = (4096, 2048) if case == "row_large" else (1024, 2048)
    x = to_device(mixed_input(*shape, seed=24, dtype=dtype))
    kw = {"row_rht_sr_bf16": dict(mode="sr", rht=True, sign_mask=3, seed=1, swizzled=True),
          "row_rht_sr_fp32": dict(mode="sr", rht=True, sign_mask=3, seed=1, swizzled=True),
          "row_rne": dict(mode="rne"), "row_4o6": dict(mode="4o6"),
          "col_rht_sr": dict(mode="sr", rht=True, rowwise=False, colwise=True, seed=2),
          "row_large": dict(mode="sr", rht=True, sign_mask=3, seed=1)}[case]
    nvfp4.quantize(x, **kw)  # first call configures the kernels
    names = _kernels_of(lambda: nvfp4.quantize(x, **kw))
    if not names:
        pytest.skip("no kernel activity recorded (CUPTI unavailable)")
    if case == "row_large":
        assert len(names) == 2 and "k_amax" in names[0] and "k_quant_row" in names[1], names
    elif case.startswith("row"):
        assert len(names) == 1 and "k_quant_row_fused" in names[0], names
    else:
        assert len(names) == 2 and "k_amax" in names[0] and "k_quant_col" in names[1], names


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "fp32"])
def test_two_kernel_rowwise_path_ragged(mode, dtype):
    """Per-tensor rowwise tensors above the one-kernel size limit run the amax
    kernel and the TMA quantize kernel: a shape with ragged row and column
    tiles (2100 rows, 129 blocks per row) against the oracle."""
    rows, cols = 2112 if dtype == torch.float32 else 2100, 2064
    x = mixed_input(rows, cols, seed=25, dtype=dtype)
    kw = dict(mode="sr" if mode == "rht_sr" else mode, rht=mode == "rht_sr", swizzled=True, sign_mask=0x2222,
              seed=12, offset=1)
    assert_parity(gpu_run(x, **kw), oracle_run(x, **kw))


@pytest.mark.parametrize("mode", ["rne", "sr", "rht_sr"])
def test_two_kernel_rowwise_path_strided(mode):
    """A strided view (row pitch 2240 elements, 2112 used) above the one-kernel
    limit: the amax pass streams TMA tiles (the load-based pass needs
    contiguous rows), with the skip test when the RHT is on."""
    base = mixed_input(2100, 2240, seed=27)
    x_dev = base.cuda()[:, 64:2176]
    x_cpu = base[:, 64:2176].contiguous()
    kw = dict(mode="sr" if mode == "rht_sr" else mode, rht=mode == "rht_sr", swizzled=True, sign_mask=0x4B1E,
              seed=13, offset=2)
    assert_parity(gpu_run(x_cpu, x_dev=x_dev, **kw), oracle_run(x_cpu, **kw))


# ------------------------------------------------------ grouped scaling
def _oracle_grouped(x, offs, *, mode, swizzled, sign_mask=0, seed=0, offset=0, amax=None):
    """Each row group quantized as a tensor of its own, Philox blocks numbered in
    the whole input (the oracle's row range of the full tensor with the group's
    amax given)."""
    xn = np_bits(x)
    R, C = x.shape
    CS = C // 16
    codes = np.zeros((R, C // 2), np.uint8)
    lin = np.zeros((R, CS), np.uint8)
    amaxes, gscales = [], []
    kw = dict(mode="sr" if mode == "rht_sr" else mode, rht=mode == "rht_sr", sign_mask=sign_mask, seed=seed,
              offset=offset)
    for g in range(len(offs) - 1):
        o0, o1 = int(offs[g]), int(offs[g + 1])
        if o1 == o0:
            A = 0.0 if amax is None else float(amax[g])
            amaxes.append(np.float32(A))
            gscales.append(np.float32(np.float32(A) / np.float32(2688.0)))
            continue
        if amax is None:
            A, _ = oracle.amax(xn[o0:o1], rht=kw["rht"], sign_mask=sign_mask)
            A = float(np.asarray(A).ravel()[0])
        else:
            A = float(amax[g])
        o = oracle.quantize(xn, row_range=(o0, o1), amax_given=A, **kw)
        codes[o0:o1] = o["codes"][o0:o1]
        lin[o0:o1] = o["scales"].reshape(R, CS)[o0:o1]
        amaxes.append(np.asarray(o["amax"]).ravel()[0])
        gscales.append(np.asarray(o["global_scale"]).ravel()[0])
    if swizzled:
        csp = (CS + 3) // 4 * 4
        out = np.zeros(oracle.scale_bytes(R, C, True), np.uint8)
        for r in range(R):
            for j in range(CS):
                out[oracle.swizzle_offset(r, j, csp)] = lin[r, j]
        scales = out
    else:
        scales = lin.ravel()
    return codes, scales, np.array(amaxes, np.float32), np.array(gscales, np.float32)


@pytest.mark.parametrize("mode", ["rne", "sr", "rht_sr", "4o6"])
@pytest.mark.parametrize("swizzled", [False, True], ids=["linear", "swizzled"])
def test_grouped_rows_each_with_its_own_scale(mode, swizzled):
    """Row groups of very different magnitudes (an empty group and a one-row
    group included) against the oracle run per group."""
    x = mixed_input(300, 256, seed=27)
    offs = [0, 40, 40, 41, 170, 300]
    x[41:170] *= 1e-3  # a group of much smaller values: its own scale matters
    kw = dict(mode=mode, swizzled=swizzled, sign_mask=0x6A6A, seed=14, offset=3)
    offs_d = torch.tensor(offs, dtype=torch.int64, device="cuda")
    q = nvfp4.quantize_grouped(to_device(x), offs_d, **kw)
    torch.cuda.synchronize()
    codes, scales, amaxes, gscales = _oracle_grouped(x, offs, **kw)
    assert np.array_equal(q.codes_row.cpu().numpy(), codes)
    assert np.array_equal(q.scales_row.cpu().numpy(), scales)
    assert same_float_bits(q.amax.cpu().numpy(), amaxes)
    assert same_float_bits(q.global_scale.cpu().numpy(), gscales)
    # the same with the amaxes given
    A = torch.from_numpy(amaxes * np.float32(2.0)).cuda()
    q2 = nvfp4.quantize_grouped(to_device(x), offs_d, amax=A, **kw)
    torch.cuda.synchronize()
    codes2, scales2, _, gscales2 = _oracle_grouped(x, offs, amax=amaxes * np.float32(2.0), **kw)
    assert np.array_equal(q2.codes_row.cpu().numpy(), codes2)
    assert np.array_equal(q2.scales_row.cpu().numpy(), scales2)
    assert same_float_bits(q2.global_scale.cpu().numpy(), gscales2)


GROUP_CASES = {
    # rows, cols, dtype, group offsets, mode, strided, amax given, NaN at (row, col)
    "fibonacci_groups": (520, 272, torch.bfloat16, [0, 1, 2, 3, 5, 8, 13, 21, 34, 55, 89, 144, 233, 377, 520],
                         "rht_sr", False, False, None),
    "one_row_groups": (200, 128, torch.bfloat16, list(range(201)), "sr", False, False, None),
    "fp32_strided": (300, 240, torch.float32, [0, 129, 129, 130, 300], "4o6", True, False, None),
    "tile_aligned": (512, 512, torch.bfloat16, [0, 128, 256, 256, 512], "rne", False, False, None),
    "long_rows": (40, 53248, torch.bfloat16, [0, 7, 7, 40], "rht_sr", False, False, None),
    "empty_ends_given_fp32": (260, 96, torch.float32, [0, 0, 0, 130, 130, 260, 260], "sr", False, True, None),
    "nan_in_one_group": (384, 160, torch.bfloat16, [0, 100, 250, 384], "rht_sr", False, False, (120, 37)),
    "fp32_rht": (200, 128, torch.float32, [0, 60, 61, 200], "rht_sr", False, False, None),
    "zero_group": (200, 96, torch.bfloat16, [0, 64, 128, 200], "sr", False, False, None),
    # 64 experts, 10 tokens: most groups empty
    "more_groups_than_rows": (10, 64, torch.bfloat16, [0] * 20 + [3] * 20 + [7] * 10 + [10] * 15, "rht_sr", False,
                              False, None),
}


@pytest.mark.parametrize("case", list(GROUP_CASES))
def test_grouped_tiles(case):
    """Group layouts against the tiles of the grouped kernel: many groups inside
    one tile (their rows look divisors up without a table), a group per row,
    fp32 rows with a pitch, boundaries on tile edges, and rows longer than
    96 KiB; ragged column tiles and pad rows in the swizzled layout."""
    R, C, dtype, offs, mode, strided, given, nan_at = GROUP_CASES[case]
    x = mixed_input(R, C, seed=31 + list(GROUP_CASES).index(case), dtype=dtype)
    x[offs[1]:offs[2]] *= 0.0 if case == "zero_group" else 1e-2  # a group with a scale of its own
    if nan_at:
        x[nan_at] = float("nan")  # poisons its group's amax and scale, no other group
    if strided:
        base = torch.zeros(R, C + 32, dtype=dtype, device="cuda")
        base[:, 16:16 + C] = x.cuda()
        x_dev = base[:, 16:16 + C]
    else:
        x_dev = to_device(x)
    kw = dict(mode=mode, swizzled=True, sign_mask=0x1DB7, seed=15, offset=6)
    offs_d = torch.tensor(offs, dtype=torch.int64, device="cuda")
    A = None
    if given:  # twice each group's own amax (an empty group's stays 0)
        A = _oracle_grouped(x, offs, **kw)[2] * np.float32(2.0)
    q = nvfp4.quantize_grouped(x_dev, offs_d, amax=None if A is None else torch.from_numpy(A).cuda(), **kw)
    torch.cuda.synchronize()
    codes, scales, amaxes, gscales = _oracle_grouped(x, offs, amax=A, **kw)
    if nan_at:
        assert np.isnan(amaxes[1]) and not np.isnan(np.delete(amaxes, 1)).any()
    assert np.array_equal(q.codes_row.cpu().numpy(), codes)
    assert np.array_equal(q.scales_row.cpu().numpy(), scales)
    assert same_float_bits(q.amax.cpu().numpy(), amaxes)
    assert same_float_bits(q.global_scale.cpu().numpy(), gscales)


def test_grouped_empty_input():
    """No rows: every group is empty, its amax and scale 0 (given amaxes kept)."""
    x = torch.empty(0, 64, dtype=torch.bfloat16, device="cuda")
    offs_d = torch.zeros(4, dtype=torch.int64, device="cuda")
    q = nvfp4.quantize_grouped(x, offs_d, mode="rht_sr", sign_mask=0x1234, seed=1)
    torch.cuda.synchronize()
    assert q.amax.cpu().tolist() == [0.0, 0.0, 0.0] and q.global_scale.cpu().tolist() == [0.0, 0.0, 0.0]
    A = torch.tensor([2688.0, 0.0, 5376.0], device="cuda")
    q = nvfp4.quantize_grouped(x, offs_d, mode="sr", amax=A)
    torch.cuda.synchronize()
    assert q.amax.cpu().tolist() == [2688.0, 0.0, 5376.0]
    assert q.global_scale.cpu().tolist() == [1.0, 0.0, 2.0]


def test_grouped_one_group_is_the_per_tensor_result():
    x = mixed_input(256, 512, seed=28)
    offs_d = torch.tensor([0, 256], dtype=torch.int64, device="cuda")
    q = nvfp4.quantize_grouped(to_device(x), offs_d, mode="sr", seed=3, swizzled=True)
    torch.cuda.synchronize()
    o = oracle_run(x, mode="sr", seed=3, swizzled=True)
    assert np.array_equal(q.codes_row.cpu().numpy(), o["codes_row"])
    assert np.array_equal(q.scales_row.cpu().numpy(), o["scales_row"])
    assert same_float_bits(q.amax.cpu().numpy(), o["amax"])


@pytest.mark.parametrize("swizzled", [False, True])
@pytest.mark.parametrize("per_row", [False, True])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16], ids=["fp32", "bf16"])
def test_dequantize_with_inverse_rht(swizzled, per_row, out_dtype):
    x = mixed_input(136, 224, seed=29)
    mask = 0xC3A5
    o = oracle.quantize(np_bits(x), mode="sr", rht=True, sign_mask=mask, per_row=per_row, swizzled=swizzled,
                        seed=7)
    dt = "bf16" if out_dtype == torch.bfloat16 else "fp32"
    ref = oracle.dequantize_rht(o["codes"], o["scales"], o["global_scale"], 136, 224, sign_mask=mask,
                                swizzled=swizzled, per_row=per_row, out_dtype=dt)
    got = nvfp4.dequantize(torch.from_numpy(o["codes"]).cuda(), torch.from_numpy(o["scales"].ravel()).cuda(),
                           torch.from_numpy(o["global_scale"]).cuda(), 136, 224, swizzled=swizzled,
                           per_row=per_row, out_dtype=out_dtype, rht_sign_mask=mask)
    torch.cuda.synchronize()
    if out_dtype == torch.bfloat16:
        assert np.array_equal(got.cpu().view(torch.int16).numpy().view(np.uint16), ref)
    else:
        assert same_float_bits(got.cpu().numpy(), ref)


def test_rht_round_trip_through_the_library():
    """quantize(RHT+SR) then dequantize with the inverse RHT lands near the source."""
    x = mixed_input(256, 512, seed=30, dtype=torch.float32)
    xd = x.cuda()
    q = nvfp4.quantize(xd, mode="sr", rht=True, sign_mask=0x0F0F, seed=8, swizzled=True)
    back = nvfp4.dequantize(q.codes_row, q.scales_row, q.global_scale, 256, 512, swizzled=True,
                            rht_sign_mask=0x0F0F)
    torch.cuda.synchronize()
    err = (back.cpu() - x).reshape(-1, 16).norm(dim=1)
    assert float((err <= 0.5 * x.reshape(-1, 16).norm(dim=1) + 1e-30).float().mean()) > 0.99


@pytest.mark.slow
def test_full_size_rht_both_orientations_and_groups():
    """The headline activation (8192x4096) in both orientations with the RHT
    (linear scales), and as 8 row groups of uneven sizes (an empty and a
    one-row group among them), every output compared with the oracle."""
    w = wl.WORKLOADS["act_rht_sr_8192x4096"]
    x, mask = wl.make_input(w)
    kw = dict(mode="sr", rht=True, rowwise=True, colwise=True, swizzled=False, sign_mask=mask, seed=1)
    assert_parity(gpu_run(x, **kw), oracle_run_all_cores(x, **kw))
    offs = [0, 100, 1124, 1124, 4000, 4001, 6000, 7999, 8192]
    q = nvfp4.quantize_grouped(to_device(x), torch.tensor(offs, dtype=torch.int64, device="cuda"), mode="rht_sr",
                               sign_mask=mask, seed=1, swizzled=True)
    torch.cuda.synchronize()
    xn = np_bits(x)
    codes, scales = np.zeros((8192, 2048), np.uint8), np.zeros(8192 * 256, np.uint8)
    for gi in range(len(offs) - 1):
        o0, o1 = offs[gi], offs[gi + 1]
        A = oracle.amax_parallel(xn[o0:o1], rht=True, sign_mask=mask) if o1 > o0 else 0.0
        if o1 > o0:
            o = oracle.quantize_parallel(xn, mode="sr", rht=True, sign_mask=mask, seed=1, swizzled=True,
                                         row_range=(o0, o1), amax_given=A)
            codes[o0:o1] = o["codes"][o0:o1]
            scales |= o["scales"]  # each group writes its own rows' scale bytes, the rest stay 0
        assert same_float_bits(q.amax[gi:gi + 1].cpu().numpy(), np.float32([A]))
    assert np.array_equal(q.codes_row.cpu().numpy(), codes)
    assert np.array_equal(q.scales_row.cpu().numpy(), scales)


def test_calls_on_two_streams_at_once():
    """Two per-tensor quantizations in flight on two streams (each stream has its
    own workspace in the binding) give the same results as one after the other."""
    xa, xb = mixed_input(4096, 2048, seed=31), mixed_input(4096, 2048, seed=32)
    da, db = to_device(xa), to_device(xb)
    kw = dict(mode="sr", rht=True, sign_mask=0x1111, seed=9, swizzled=True)
    ra, rb = gpu_run(xa, x_dev=da, **kw), gpu_run(xb, x_dev=db, **kw)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    for _ in range(3):
        with torch.cuda.stream(s1):
            qa = nvfp4.quantize(da, stream=s1, **kw)
        with torch.cuda.stream(s2):
            qb = nvfp4.quantize(db, stream=s2, **kw)
        torch.cuda.synchronize()
        assert np.array_equal(qa.codes_row.cpu().numpy(), ra["codes_row"])
        assert np.array_equal(qb.codes_row.cpu().numpy(), rb["codes_row"])
        assert same_float_bits(qa.amax.cpu().numpy(), ra["amax"]) and same_float_bits(qb.amax.cpu().numpy(), rb["amax"])
