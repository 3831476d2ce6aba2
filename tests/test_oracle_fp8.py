"""Pins for the oracle's e4m3 format, rounding, quantiser and Hadamard rotation.

Each check ties the oracle to something outside it: values printed in the
pages (tests/golden/e4m3_page_values.txt), PyTorch's float8_e4m3fn cast,
SciPy's Sylvester Hadamard matrix, or a closed form. The mutation tests at the
end plant plausible mistakes in copies of the oracle and show that a pin
catches each of them.
"""
import math
import os

import numpy as np
import pytest
import scipy.linalg
import torch

from oracle import fp8

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e4m3_page_values.txt")


def _golden_rows():
    rows = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            val, code, *_ = line.split()
            rows.append((float(val), int(code, 16)))
    return rows


@pytest.mark.parametrize("value,code", _golden_rows())
def test_page_printed_codes(value, code):
    got = int(fp8.e4m3_rne(np.array([value]))[0])
    assert got == code, f"{value} -> {got:#x}, pages say {code:#x}"
    if code & 0x7F:
        assert fp8.e4m3_decode(np.array([code], np.uint8))[0] == value


def test_underflow_threshold_and_min_normal():
    # ZYFA post, "Precision and Underflow": below 2^-10 -> 0; 2^-10 itself is a
    # tie between 0 and 2^-9 and goes to the even code 0; just above -> 2^-9.
    t = 2.0 ** -10
    assert fp8.e4m3_rne(np.array([t]))[0] == 0x00
    assert fp8.e4m3_rne(np.array([np.nextafter(t, 1.0)]))[0] == 0x01
    assert fp8.e4m3_decode(np.array([0x01], np.uint8))[0] == 2.0 ** -9
    assert fp8.e4m3_decode(np.array([0x08], np.uint8))[0] == 2.0 ** -6
    # subnormals lose precision: spacing 2^-9 below 2^-6
    assert fp8.e4m3_decode(np.array([0x07], np.uint8))[0] == 7 * 2.0 ** -9


def test_code_steps_by_8_per_binade():
    # ZYFA post, "Lean P": the code grows by 8 each time the value doubles.
    for e in range(-6, 8):
        a = int(fp8.e4m3_rne(np.array([2.0 ** e]))[0])
        b = int(fp8.e4m3_rne(np.array([2.0 ** (e + 1)]))[0])
        assert b - a == 8


def test_decode_matches_torch_float8():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = fp8.e4m3_decode(codes.numpy())
    np.testing.assert_array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    np.testing.assert_array_equal(got[ok], ref[ok])


def _torch_e4m3(x32: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x32, dtype=np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_rne_matches_torch_on_every_bf16_pattern():
    bits = np.arange(65536, dtype=np.uint32) << 16
    x = bits.view(np.float32)
    keep = np.isfinite(x) & (np.abs(x) <= 448.0)
    x = x[keep]
    np.testing.assert_array_equal(fp8.e4m3_rne(x), _torch_e4m3(x))


def test_rne_matches_torch_on_random_fp32():
    rng = np.random.default_rng(7)
    mag = 2.0 ** rng.uniform(-14, math.log2(448.0), size=400_000)
    x = (mag * rng.choice([-1.0, 1.0], size=mag.size)).astype(np.float32)
    # exact midpoints between codes exercise ties-to-even
    mids = ((fp8.E4M3_VALUES[:-1] + fp8.E4M3_VALUES[1:]) / 2).astype(np.float32)
    x = np.concatenate([x, mids, -mids])
    np.testing.assert_array_equal(fp8.e4m3_rne(x), _torch_e4m3(x))


def test_saturation_and_signed_zero():
    got = fp8.e4m3_rne(np.array([449.0, 1e6, -1e6, -0.0, -1e-6, 0.0]))
    assert list(got) == [0x7E, 0x7E, 0xFE, 0x80, 0x80, 0x00]


def _bf16_block(rng, S, H, D, scale=1.0):
    x = torch.from_numpy(rng.standard_normal((1, S, H, D)).astype(np.float32) * scale)
    return x.to(torch.bfloat16).to(torch.float32).numpy()


def test_quantiser_scale_is_amax_over_448():
    rng = np.random.default_rng(1)
    x = _bf16_block(rng, 256, 2, 128)
    codes, scales = fp8.quantize_fp8(x)
    for h in range(2):
        for j in range(2):
            blk = x[0, j * 128:(j + 1) * 128, h, :]
            amax = np.float32(np.abs(blk).max())
            assert scales[0, h, j] == np.float32(amax / np.float32(448.0))
            # the element that attains amax maps to the largest code
            r, c = np.unravel_index(np.argmax(np.abs(blk)), blk.shape)
            assert codes[0, j * 128 + r, h, c] & 0x7F == 0x7E


def test_quantiser_zero_block_guard():
    # "FP8 GEMM on CDNA4" section 2.2: all-zero block -> scale 1, codes 0.
    x = np.zeros((1, 128, 1, 128), np.float32)
    codes, scales = fp8.quantize_fp8(x)
    assert scales[0, 0, 0] == 1.0
    assert not codes.any()


def test_quantiser_error_bound_and_ragged_tail():
    rng = np.random.default_rng(2)
    x = _bf16_block(rng, 300, 3, 192, scale=3.0)
    codes, scales = fp8.quantize_fp8(x)
    assert scales.shape == (1, 3, 3)
    deq = fp8.dequantize_fp8(codes, scales)
    # RNE to 3 mantissa bits: error <= 2^-4 relative for normals, and
    # <= 2^-10 * scale absolute in the subnormal range.
    tok_blk = np.arange(300) // 128
    sc = scales[0][:, tok_blk].T[None, :, :, None]
    bound = np.maximum(np.abs(x) * 2.0 ** -4, sc * 2.0 ** -10) * (1 + 1e-6)
    assert np.all(np.abs(deq - x) <= bound)
    # the tail block is quantised from its own 44 rows only
    tail = x[0, 256:, 1, :]
    assert scales[0, 1, 2] == np.float32(np.float32(np.abs(tail).max()) / np.float32(448))


def test_fwht_matches_scipy_hadamard():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((64, 128)).astype(np.float32)
    H = scipy.linalg.hadamard(128).astype(np.float64)
    ref = x.astype(np.float64) @ H.T / math.sqrt(128.0)
    got = fp8.fwht128_fp32(x).astype(np.float64)
    # 7 rounded stages plus the scale: a few float32 ulps of sum |x| / sqrt(128)
    bound = 10 * 2.0 ** -24 * np.abs(x).sum(axis=1, keepdims=True) / math.sqrt(128.0)
    assert np.all(np.abs(got - ref) <= bound)


def test_sylvester_orthogonality_and_involution():
    H = scipy.linalg.hadamard(128).astype(np.float64)
    np.testing.assert_array_equal(H @ H.T, 128 * np.eye(128))
    rng = np.random.default_rng(4)
    x = rng.standard_normal((16, 128)).astype(np.float32)
    back = fp8.fwht128_fp32(fp8.fwht128_fp32(x))
    np.testing.assert_allclose(back, x, rtol=0, atol=1e-5)


def test_rotation_leaves_qk_unchanged():
    # ZYFA post, "FP8 Error in Full-Model Inference": the rotation of Q and K
    # leaves QK^T unchanged.
    rng = np.random.default_rng(5)
    q = rng.standard_normal((32, 128)).astype(np.float32)
    k = rng.standard_normal((32, 128)).astype(np.float32)
    qr = fp8.fwht128_fp32(q).astype(np.float64)
    kr = fp8.fwht128_fp32(k).astype(np.float64)
    np.testing.assert_allclose(qr @ kr.T, q.astype(np.float64) @ k.astype(np.float64).T,
                               rtol=0, atol=2e-4)


def test_rotation_spreads_outlier_channel():
    x = np.zeros((1, 128), np.float32)
    x[0, 17] = 100.0
    y = fp8.fwht128_fp32(x)
    np.testing.assert_allclose(np.abs(y), 100.0 / math.sqrt(128.0), rtol=1e-6)


def test_quantiser_hadamard_flag_rotates_before_amax():
    rng = np.random.default_rng(6)
    x = _bf16_block(rng, 128, 1, 128)
    c1, s1 = fp8.quantize_fp8(x, hadamard=True)
    c2, s2 = fp8.quantize_fp8(fp8.fwht128_fp32(x), hadamard=False)
    np.testing.assert_array_equal(c1, c2)
    np.testing.assert_array_equal(s1, s2)


# ---------------------------------------------------------------- mutations --
# Each planted mistake lives in a local copy of an oracle step and must be
# caught by one of the pins above (re-run here on the mutant).

def _rne_ties_odd(q):
    q = np.asarray(q, np.float64)
    a = np.abs(q)
    idx = np.searchsorted(fp8.E4M3_VALUES, a, side="left")
    hi = np.clip(idx, 0, 126)
    lo = np.clip(idx - 1, 0, 126)
    d_hi = np.abs(fp8.E4M3_VALUES[hi] - a)
    d_lo = np.abs(a - fp8.E4M3_VALUES[lo])
    pick_lo = (d_lo < d_hi) | ((d_lo == d_hi) & (lo % 2 == 1))   # wrong tie rule
    mag = np.where(a > 448, 126, np.where(pick_lo, lo, hi))
    return (mag | np.where(np.signbit(q), 0x80, 0)).astype(np.uint8)


def test_mutant_tie_rule_is_caught():
    mids = ((fp8.E4M3_VALUES[:-1] + fp8.E4M3_VALUES[1:]) / 2).astype(np.float32)
    assert not np.array_equal(_rne_ties_odd(mids), _torch_e4m3(mids))


def test_mutant_bias8_format_is_caught():
    # a bias-8 ("fnuz") table would put 1.0 at code 0x40, not 0x38
    def mag(code):
        e, m = (code >> 3) & 0xF, code & 7
        return m * 2.0 ** -10 if e == 0 else (1 + m / 8) * 2.0 ** (e - 8)
    table = np.array([mag(c) for c in range(127)])
    assert int(np.argmin(np.abs(table - 1.0))) != _golden_rows()[0][1]


def test_mutant_unnormalised_fwht_is_caught():
    rng = np.random.default_rng(8)
    x = rng.standard_normal((4, 128)).astype(np.float32)
    bad = fp8.fwht128_fp32(x) * np.float32(math.sqrt(128.0))    # dropped 1/sqrt(128)
    H = scipy.linalg.hadamard(128) / math.sqrt(128.0)
    assert np.max(np.abs(bad - x @ H.T)) > 1.0


def test_mutant_wrong_max_is_caught():
    # A scale of amax/480 saturates the largest element at 448, so its
    # dequantised value misses the RNE error bound of the error-bound pin.
    rng = np.random.default_rng(9)
    x = _bf16_block(rng, 128, 1, 128)
    amax = np.float32(np.abs(x).max())
    bad_scale = np.float32(amax / np.float32(480.0))              # wrong format max
    q = (x / bad_scale).astype(np.float32)
    deq = fp8.e4m3_decode(fp8.e4m3_rne(q)) * np.float64(bad_scale)
    bound = np.maximum(np.abs(x) * 2.0 ** -4, bad_scale * 2.0 ** -10) * (1 + 1e-6)
    assert np.any(np.abs(deq - x) > bound)


# ------------------------------------------------- division, pinned exactly --
# Reading: the quantiser divides, code = RNE_e4m3(fl32(y / s)) with an IEEE
# float32 division ("FP8 GEMM on CDNA4", 2.2: scale = amax / max, values
# divided by the scale). The cases below (bf16 y, bf16 amax) are ones where
# multiplying by the rounded reciprocal, fl32(y * fl32(1 / s)), gives another
# code: y / s lands exactly on an e4m3 rounding midpoint, which the division
# keeps (and the tie goes to the even code) while the reciprocal moves it to
# one side. Expected codes come from exact rational arithmetic only.
from fractions import Fraction

DIVISION_CASES = [(1.2734375, 1.9431114196777344e-05), (2.84375, 8.058547973632812e-05),
                  (3.0625, 0.00016689300537109375)]


def _rn_f32(x: Fraction) -> Fraction:
    """x > 0 rounded to the nearest float32 (ties to an even significand), exactly."""
    e = x.numerator.bit_length() - x.denominator.bit_length()
    if Fraction(2) ** e > x:
        e -= 1
    ulp = Fraction(2) ** (max(e, -126) - 23)
    n, r = divmod(x, ulp)
    n = int(n)
    if r > ulp / 2 or (r == ulp / 2 and n % 2 == 1):
        n += 1
    return n * ulp


def _e4m3_exact(x: Fraction) -> int:
    """Code of the e4m3 value nearest to x >= 0 (ties to the even code), by
    search over the 127 non-negative finite codes, saturating at 448."""
    best, best_d = 0, None
    for c in range(0x7F):
        e, m = c >> 3, c & 7
        v = Fraction(m, 8) * Fraction(2) ** -6 if e == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)
        d = abs(v - x)
        if best_d is None or d < best_d or (d == best_d and c % 2 == 0):
            best, best_d = c, d
    return best


@pytest.mark.parametrize("amax,y", DIVISION_CASES)
def test_quantiser_divides_in_float32(amax, y):
    s_exact = _rn_f32(Fraction(amax) / 448)
    want = _e4m3_exact(_rn_f32(Fraction(y) / s_exact))
    via_reciprocal = _e4m3_exact(_rn_f32(Fraction(y) * _rn_f32(1 / s_exact)))
    assert want != via_reciprocal                       # the case tells the two readings apart
    x = np.zeros((1, 128, 1, 128), np.float32)
    x[0, 0, 0, 0] = amax                                # fixes the block's scale
    x[0, 1, 0, 0] = y
    x[0, 2, 0, 0] = -y
    codes, scales = fp8.quantize_fp8(x)
    assert Fraction(float(scales[0, 0, 0])) == s_exact
    assert int(codes[0, 1, 0, 0]) == want
    assert int(codes[0, 2, 0, 0]) == 0x80 | want        # sign bit over the same magnitude
