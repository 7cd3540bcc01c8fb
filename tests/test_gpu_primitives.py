"""The library's device primitives on the GPU, one at a time.

The hardware casts (cvt.rn.satfinite.e2m1x2 / e4m3x2 and their decodes) are
checked against the oracle's converters over dense sweeps of every binade they
can see, which also fixes operand order, nibble order, NaN, -0 and
saturation.  The per-block exact division is checked against CUDA's own IEEE
division on random and near-midpoint quotients.  The four-over-six
candidate error (every product and sum individually rounded, pinned tree
order) is checked against the oracle's on a million blocks.
"""
import ctypes
import os
import subprocess

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


@pytest.fixture(scope="module")
def probes(tmp_path_factory):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from tensor_quantization_gb300 import build
    so = str(tmp_path_factory.mktemp("probes") / "libprobes.so")
    subprocess.run([build.nvcc(), *build.ARCH, "-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-shared",
                    "-I", build.CSRC, os.path.join(HERE, "gpu_probes.cu"), "-o", so], check=True)
    torch.zeros(1, device="cuda")  # create the context first
    lib = ctypes.CDLL(so)
    vp, i64, u64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64, ctypes.c_int
    lib.probe_e2m1.argtypes = [vp, i64, vp]
    lib.probe_e2m1_order.argtypes = [vp]
    lib.probe_sr.argtypes = [vp, vp, i64, vp]
    lib.probe_sr_f16.argtypes = [vp, vp, i64, vp]
    lib.probe_e2m1_f16.argtypes = [vp]
    lib.probe_e4m3.argtypes = [vp, i64, vp]
    lib.probe_e4m3_value.argtypes = [vp]
    lib.probe_e2m1_value.argtypes = [vp]
    lib.probe_div.argtypes = [u64, i64, i32, vp, vp]
    lib.probe_cand_err.argtypes = [vp, vp, vp, i64, vp]
    lib.probe_cand_err_neg.argtypes = [vp, vp, vp, i64, vp]
    return lib


def ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def dense_floats(exp_lo, exp_hi, mant_bits, seed):
    """Every sign, every binade 2^exp_lo..2^exp_hi, the top mant_bits of the
    significand enumerated, the remaining bits random."""
    rng = np.random.default_rng(seed)
    e = np.arange(exp_lo + 127, exp_hi + 128, dtype=np.uint32)
    top = np.arange(1 << mant_bits, dtype=np.uint32) << (23 - mant_bits)
    grid = (e[:, None] << 23 | top[None, :]).ravel()
    low = rng.integers(0, 1 << (23 - mant_bits), grid.size, dtype=np.uint32)
    bits = np.concatenate([grid, grid | low, grid | ((1 << (23 - mant_bits)) - 1)])
    bits = np.concatenate([bits, bits | 0x80000000])
    return bits.view(np.float32)


SPECIALS = np.array([0.0, -0.0, np.inf, -np.inf, np.nan, -np.nan, 1e-45, -1e-45, 3.4e38, -3.4e38,
                     0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0, 7.0, 448.0, 464.0, 480.0, 1e9],
                    np.float32)


def run_cast(fn, vals):
    q = torch.from_numpy(vals).cuda()
    out = torch.empty(vals.size, dtype=torch.uint8, device="cuda")
    assert fn(ptr(q), vals.size, ptr(out)) == 0
    return out.cpu().numpy()


def test_e2m1_cast_matches_oracle(probes):
    vals = np.concatenate([dense_floats(-24, 4, 12, 1), SPECIALS,
                           np.random.default_rng(2).integers(0, 2 ** 32, 1 << 20, dtype=np.uint32).view(np.float32)])
    got = run_cast(probes.probe_e2m1, vals)
    ref = oracle.e2m1_rne_array(vals)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(float(vals[i]), int(got[i]), int(ref[i])) for i in bad[:8]]


def test_e2m1_pack_order(probes):
    out = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert probes.probe_e2m1_order(ptr(out)) == 0
    w = int(out.item()) & 0xFFFFFFFF
    assert [(w >> (4 * k)) & 15 for k in range(8)] == [1, 2, 3, 4, 5, 6, 7, 9]


def test_sr_round_matches_oracle(probes):
    rng = np.random.default_rng(3)
    q = np.concatenate([dense_floats(-12, 3, 10, 4), SPECIALS[np.isfinite(SPECIALS)]])
    q = q[np.abs(q) < 8.0]
    q = np.repeat(q, 3)
    r = rng.integers(0, 256, q.size, dtype=np.uint8)
    qt, rt = torch.from_numpy(q).cuda(), torch.from_numpy(r).cuda()
    out = torch.empty(q.size, dtype=torch.uint8, device="cuda")
    assert probes.probe_sr(ptr(qt), ptr(rt), q.size, ptr(out)) == 0
    got = out.cpu().numpy()
    ref = oracle.e2m1_sr_array(q, r)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(float(q[i]), int(r[i]), int(got[i]), int(ref[i])) for i in bad[:8]]


def test_sr_f16_pair_matches_oracle(probes):
    # the fast path's stochastic rounding: quotients at 2^-14 scale, truncated
    # to f16 pairs, dithered per 16-bit lane, cast from f16x2
    rng = np.random.default_rng(13)
    q = np.concatenate([dense_floats(-30, 3, 10, 14), SPECIALS[np.isfinite(SPECIALS)]])
    q = q[np.abs(q) < 16.0]
    q = np.repeat(q, 4)
    r = rng.integers(0, 256, q.size, dtype=np.uint8)
    qt, rt = torch.from_numpy(q).cuda(), torch.from_numpy(r).cuda()
    out = torch.empty(q.size, dtype=torch.uint8, device="cuda")
    assert probes.probe_sr_f16(ptr(qt), ptr(rt), q.size, ptr(out)) == 0
    got = out.cpu().numpy()
    ref = oracle.e2m1_sr_array(q, r)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(float(q[i]), int(r[i]), int(got[i]), int(ref[i])) for i in bad[:8]]


def test_e2m1_f16_cast_matches_oracle(probes):
    # every f16 pattern (the fast path never feeds it NaN), in both halves of the pair
    out = torch.empty(65536, dtype=torch.uint8, device="cuda")
    assert probes.probe_e2m1_f16(ptr(out)) == 0
    got = out.cpu().numpy()
    with np.errstate(invalid="ignore"):  # NaN patterns widen to NaN
        vals = np.arange(65536, dtype=np.uint16).view(np.float16).astype(np.float32)
    keep = ~np.isnan(vals)
    ref = oracle.e2m1_rne_array(vals)
    bad = np.nonzero((got != ref) & keep)[0]
    assert bad.size == 0, [(float(vals[i]), int(got[i]), int(ref[i])) for i in bad[:8]]


def test_e4m3_cast_matches_oracle(probes):
    vals = np.concatenate([dense_floats(-12, 10, 12, 5), SPECIALS,
                           np.random.default_rng(6).integers(0, 2 ** 32, 1 << 20, dtype=np.uint32).view(np.float32)])
    got = run_cast(probes.probe_e4m3, vals)
    ref = oracle.e4m3_rn_array(vals)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(float(vals[i]), int(got[i]), int(ref[i])) for i in bad[:8]]


def test_decodes_match_oracle(probes):
    out = torch.empty(256, device="cuda")
    assert probes.probe_e4m3_value(ptr(out)) == 0
    got = out.cpu().numpy()
    for b in range(256):
        ref = oracle.e4m3_value(b)
        assert (np.isnan(got[b]) and np.isnan(ref)) or np.float32(ref).view(np.uint32) == got[b].view(np.uint32)
    out = torch.empty(512, device="cuda")
    assert probes.probe_e2m1_value(ptr(out)) == 0
    got = out.cpu().numpy()
    for b in range(256):
        assert got[2 * b] == oracle.e2m1_value(b & 15) and got[2 * b + 1] == oracle.e2m1_value(b >> 4)
        assert np.signbit(got[2 * b]) == bool(b & 8)


@pytest.mark.parametrize("kind", [0, 1, 2, 3, 4])
def test_exact_division(probes, kind):
    bad = torch.zeros(1, dtype=torch.int64, device="cuda")
    first = torch.zeros(12, device="cuda")
    n = 1 << 26
    for seed in range(8):
        assert probes.probe_div(seed + 100 * kind, n, kind, ptr(bad), ptr(first)) == 0
    assert int(bad.item()) == 0, first.cpu().numpy().reshape(-1, 3)[:4]


@pytest.mark.parametrize("form", ["codes", "negated_values"])
def test_four_over_six_candidate_error_matches_oracle(probes, form):
    """Bit-exact squared errors, so that no multiply is fused into the add or
    subtract that follows it (that would change which candidate wins a
    near-tie).  Half of the blocks carry the RNE codes of y/d (errors of a real
    candidate), half random codes (every code value against every divisor).
    Both forms: from the packed codes, and from the negated f16x2 values the
    fast encoder takes straight from its casts."""
    n = 1 << 20
    rng = np.random.default_rng(31)
    y = (rng.standard_normal((n, 16)) * np.exp2(rng.integers(-30, 30, (n, 1)))).astype(np.float32)
    S = rng.integers(1, 127, n).astype(np.uint32)
    S[rng.random(n) < 0.01] = 0
    g = np.exp2(rng.uniform(-40, 20, n)).astype(np.float32) * np.float32(1.0 + rng.random(n).astype(np.float32))
    sf = np.array([oracle.e4m3_value(int(b)) for b in range(256)], np.float32)[S]
    d = np.where(S == 0, np.float32(0), sf * g).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.where(d[:, None] == 0, np.float32(0), y / d[:, None]).astype(np.float32)
    codes = oracle.e2m1_rne_array(q).reshape(n, 16).astype(np.int32)
    rand = rng.random(n) < 0.5
    codes[rand] = rng.integers(0, 16, (int(rand.sum()), 16))
    want = oracle.candidate_error_array(y, codes, S, g)
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    yt, ct, dt = (torch.from_numpy(np.ascontiguousarray(a)).cuda() for a in (y, packed, d))
    out = torch.empty(n, dtype=torch.float32, device="cuda")
    fn = probes.probe_cand_err if form == "codes" else probes.probe_cand_err_neg
    assert fn(ptr(yt), ptr(ct), ptr(dt), n, ptr(out)) == 0
    got = out.cpu().numpy()
    same = (got.view(np.uint32) == want.view(np.uint32)) | (np.isnan(got) & np.isnan(want))
    bad = np.flatnonzero(~same)
    assert bad.size == 0, f"{bad.size} blocks differ, first {bad[:4].tolist()}: {got[bad[:4]]} vs {want[bad[:4]]}"
