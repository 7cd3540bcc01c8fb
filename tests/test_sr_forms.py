"""The two bit-level forms of stochastic rounding that the kernels use,
re-enacted in numpy on the CPU and compared with the oracle's SR rule.

The kernels never compute (|q| - a)/(b - a) + (r + 0.5)/256 >= 1 directly.
The slow path scales q by 2^-126 (toward zero) so that the E2M1 grid sits at
the fp32 patterns with 22 low zero bits, adds the dither (r + 0.5) * 2^14 to
the bits and clears them; the fast path scales q by 2^-14, truncates to fp16
(grid above bit 9), adds 2r + 1 to the 16-bit pattern and clears the low 9
bits, then casts the grid value times 2^14 with round-to-nearest.  These tests
check, without a GPU, that both encodings make exactly the oracle's decision
on dense sweeps of every binade (the GPU tests then check that the hardware
instructions behave as re-enacted here).
"""
import numpy as np

import oracle


def dense_q(seed):
    """|q| < 16 over every binade from 2^-30, the top 10 significand bits
    enumerated, the rest random; plus grid points, midpoints and both signs."""
    rng = np.random.default_rng(seed)
    e = np.arange(-30 + 127, 3 + 128, dtype=np.uint32)
    top = np.arange(1 << 10, dtype=np.uint32) << 13
    grid = (e[:, None] << 23 | top[None, :]).ravel()
    low = rng.integers(0, 1 << 13, grid.size, dtype=np.uint32)
    bits = np.concatenate([grid, grid | low, grid | 0x1FFF])
    q = bits.view(np.float32)
    special = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, 8.0, 12.0, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0,
                        7.0, 6.5, 15.5], np.float32)
    q = np.concatenate([q, special])
    return np.concatenate([q, -q])


def trunc_to_f16_bits(x):
    """fp16 pattern of |x| rounded toward zero (|x| < 2^15), sign apart."""
    a = np.abs(x.astype(np.float64))
    h = np.zeros(a.shape, np.uint32)
    sub = a < 2.0 ** -14
    h[sub] = np.floor(a[sub] * 2.0 ** 24).astype(np.uint32)
    nz = ~sub
    ex = np.floor(np.log2(a[nz])).astype(np.int64)
    # guard log2 rounding at binade edges
    ex = np.where(2.0 ** ex > a[nz], ex - 1, ex)
    ex = np.where(2.0 ** (ex + 1) <= a[nz], ex + 1, ex)
    mant = np.floor((a[nz] / 2.0 ** ex - 1.0) * 1024.0).astype(np.int64)
    h[nz] = (((ex + 15) << 10) | mant).astype(np.uint32)
    return h


def f16_bits_value(h):
    return h.astype(np.uint16).view(np.float16).astype(np.float64)


def fast_path_codes(q, r):
    """sr_pair_f16 on one lane: truncate q * 2^-14 to fp16, add 2r + 1 to the
    magnitude bits, clear the low 9, scale back, cast with RNE (saturating)."""
    qs = q.astype(np.float64) * 2.0 ** -14  # exact
    h = trunc_to_f16_bits(qs)
    h = (h + 2 * r.astype(np.uint32) + 1) & 0xFE00
    v = f16_bits_value(h) * 2.0 ** 14
    v = np.where(np.signbit(q), -v, v).astype(np.float32)
    return oracle.e2m1_rne_array(v)


def slow_path_codes(q, r):
    """sr_round2 on one element: q * 2^-126 toward zero, add (r + 0.5) * 2^14
    to the fp32 magnitude bits, clear the low 22, scale back, cast with RNE."""
    a = np.abs(q.astype(np.float64)) * 2.0 ** -126
    # fp32 toward zero: the subnormal step is 2^-149, the normal step
    # 2^(e - 23); |q| < 16 keeps every value below 2^-122
    bits = np.zeros(q.shape, np.uint64)
    sub = a < 2.0 ** -126
    bits[sub] = np.floor(a[sub] * 2.0 ** 149).astype(np.uint64)
    nz = ~sub
    ex = np.floor(np.log2(a[nz])).astype(np.int64)
    ex = np.where(2.0 ** ex > a[nz], ex - 1, ex)
    ex = np.where(2.0 ** (ex + 1) <= a[nz], ex + 1, ex)
    mant = np.floor((a[nz] / 2.0 ** ex - 1.0) * 2.0 ** 23).astype(np.int64)
    bits[nz] = (((ex + 127) << 23) | mant).astype(np.uint64)
    bits = (bits + (r.astype(np.uint64) << 14) + 0x2000) & 0x7FC00000
    v = bits.astype(np.uint32).view(np.float32).astype(np.float64) * 2.0 ** 126
    v = np.where(np.signbit(q), -v, v).astype(np.float32)
    return oracle.e2m1_rne_array(v)


def test_fast_path_form_matches_oracle_sr():
    q = dense_q(1)
    for r in (np.zeros(q.size, np.uint8), np.full(q.size, 255, np.uint8),
              np.random.default_rng(2).integers(0, 256, q.size, dtype=np.uint8)):
        got = fast_path_codes(q, r)
        ref = oracle.e2m1_sr_array(q, r)
        bad = np.flatnonzero(got != ref)
        assert bad.size == 0, [(float(q[i]), int(r[i]), int(got[i]), int(ref[i])) for i in bad[:6]]


def test_slow_path_form_matches_oracle_sr():
    q = dense_q(3)
    q = q[np.abs(q) < 8.0]
    for r in (np.zeros(q.size, np.uint8), np.full(q.size, 255, np.uint8),
              np.random.default_rng(4).integers(0, 256, q.size, dtype=np.uint8)):
        got = slow_path_codes(q, r)
        ref = oracle.e2m1_sr_array(q, r)
        bad = np.flatnonzero(got != ref)
        assert bad.size == 0, [(float(q[i]), int(r[i]), int(got[i]), int(ref[i])) for i in bad[:6]]


def test_forms_are_sensitive_to_the_half_step():
    """Dropping the +1 (the 0.5 of the dither) must break the fast form on
    thresholds that the sweep reaches, so the test above can fail."""
    q = dense_q(5)
    r = np.random.default_rng(6).integers(0, 256, q.size, dtype=np.uint8)
    qs = q.astype(np.float64) * 2.0 ** -14
    h = (trunc_to_f16_bits(qs) + 2 * r.astype(np.uint32)) & 0xFE00  # no + 1
    v = np.where(np.signbit(q), -1, 1) * f16_bits_value(h) * 2.0 ** 14
    wrong = oracle.e2m1_rne_array(v.astype(np.float32))
    assert np.any(wrong != oracle.e2m1_sr_array(q, r))
