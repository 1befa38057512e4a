"""Pins for the oracle's number formats (CPU only).

Each check ties the oracle to something other than itself: the FP8
definition's special values (golden file), brute-force nearest-value search,
torch's and numpy's own casts, and closed-form bounds of the quantizers.
"""
import os

import numpy as np
import pytest
import torch

from oracle import formats as F

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def all_bf16_finite() -> np.ndarray:
    bits = np.arange(1 << 16, dtype=np.uint32) << 16
    x = bits.view(np.float32)
    return x[np.isfinite(x)]


def test_fp8_golden_points():
    rows = [l.split() for l in open(os.path.join(GOLDEN, "fp8_format_points.txt"))
            if l.strip() and not l.startswith("#")]
    assert len(rows) >= 16
    for fmt, code, val in rows:
        m = F.FP8[fmt]
        got = m.decode(np.array([int(code, 16)]))[0]
        want = float(val)
        if np.isnan(want):
            assert np.isnan(got), (fmt, code)
        else:
            assert got == want, (fmt, code, got, want)
            if np.isfinite(want):
                enc = m.encode(np.array([want], np.float32), saturate=True)[0]
                assert enc == int(code, 16), (fmt, code, hex(enc))


@pytest.mark.parametrize("fmt", ["fp8_e4m3", "fp8_e5m2"])
def test_fp8_every_finite_code_round_trips(fmt):
    m = F.FP8[fmt]
    codes = np.arange(256)
    vals = m.decode(codes)
    fin = np.isfinite(vals)
    back = m.encode(vals[fin].astype(np.float32), saturate=True)
    assert np.array_equal(back, codes[fin].astype(np.uint8))


def _bruteforce_fp8(v: np.ndarray, m) -> np.ndarray:
    """Nearest finite code by exhaustive search; ties to the even code; clamp to
    max magnitude (satfinite); sign kept."""
    codes = np.arange(128)
    vals = m.decode(codes)
    ok = np.isfinite(vals)
    codes, vals = codes[ok], vals[ok]
    order = np.argsort(vals)
    codes, vals = codes[order], vals[order]
    a = np.abs(v.astype(np.float64))
    a = np.minimum(a, m.max_finite)
    hi = np.clip(np.searchsorted(vals, a, side="left"), 0, len(vals) - 1)
    lo = np.clip(hi - 1, 0, len(vals) - 1)
    dlo, dhi = a - vals[lo], vals[hi] - a
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (codes[hi] % 2 == 0))
    out = np.where(pick_hi, codes[hi], codes[lo]).astype(np.int64)
    out |= np.signbit(v).astype(np.int64) << 7
    return out.astype(np.uint8)


@pytest.mark.parametrize("fmt", ["fp8_e4m3", "fp8_e5m2"])
@pytest.mark.parametrize("scale", [1.0, 0.0371, 3.0e-3])
def test_fp8_encode_equals_bruteforce_on_all_bf16(fmt, scale):
    x = all_bf16_finite()
    inv = F.inverse_scale(np.float32(scale))
    with np.errstate(over="ignore"):
        v = x * inv
    v = v[np.isfinite(v)]
    m = F.FP8[fmt]
    assert np.array_equal(m.encode(v, saturate=True), _bruteforce_fp8(v, m))


@pytest.mark.parametrize("fmt,tdtype", [("fp8_e4m3", torch.float8_e4m3fn),
                                        ("fp8_e5m2", torch.float8_e5m2)])
def test_fp8_in_range_equals_torch_cast(fmt, tdtype):
    """Scale 1.0 is a plain cast (PR #4893 item 2): inside the finite range the
    code equals torch's own round-to-nearest cast."""
    m = F.FP8[fmt]
    x = all_bf16_finite()
    x = x[np.abs(x) <= m.max_finite]
    ours = F.quant_fp8(x, F.inverse_scale(1.0), fmt)
    ref = torch.from_numpy(x).to(tdtype).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_fp8_saturates():
    for fmt, mx in (("fp8_e4m3", 448.0), ("fp8_e5m2", 57344.0)):
        m = F.FP8[fmt]
        v = np.array([mx * 1.2, -mx * 1.2, np.inf, -np.inf, 1e30], np.float32)
        dec = m.decode(m.encode(v, saturate=True))
        assert np.array_equal(dec, [mx, -mx, mx, -mx, mx])


def test_f16_rounding_equals_numpy_cast():
    x = all_bf16_finite()
    rng = np.random.default_rng(0)
    y = (rng.standard_normal(200000) * np.exp(rng.uniform(-20, 12, 200000))).astype(np.float32)
    for v in (x, y):
        with np.errstate(over="ignore"):
            ref = v.astype(np.float16).astype(np.float32)
        assert np.array_equal(F.to_f16(v), ref, equal_nan=True)


def test_calibrate_is_correctly_rounded_division():
    rng = np.random.default_rng(1)
    for _ in range(200):
        x = (rng.standard_normal(1000) * rng.uniform(0.01, 50)).astype(np.float32)
        amax = np.float64(np.abs(x).max())
        assert F.calibrate(x, "absmax/127") == np.float32(amax / 127.0)
        assert F.calibrate(x, "absmax/448") == np.float32(amax / 448.0)
    assert F.calibrate(np.zeros(4, np.float32), "absmax/127") == 1.0
    assert F.calibrate(x, "1.0") == 1.0


def test_int8_error_bound_and_extremes():
    """|dequant(quant(x)) - x| <= scale/2 whenever |x| <= 127*scale; the tensor's
    absmax maps to +-127; beyond the range codes saturate at -128 / 127."""
    rng = np.random.default_rng(2)
    x = (rng.standard_normal(200000) * 3).astype(np.float32)
    x[7] = -np.abs(x).max() * 1.01
    scale = F.calibrate(x, "absmax/127")
    inv = F.inverse_scale(scale)
    c = F.quant_int8(x, inv)
    xh = F.dequant_sym(c, "int8", scale)
    # half a step plus the float32 rounding of x*inv (a few ulps of 127)
    assert np.all(np.abs(xh - x) <= scale * (0.5 + 2e-5))
    assert c.view(np.int8)[7] == -127
    assert c.view(np.int8).max() <= 127 and c.view(np.int8).min() >= -127
    big = np.array([130, -130, 1000, -1000, 127.49, -128.4], np.float32) * scale
    cb = F.quant_int8(big, inv).view(np.int8)
    assert list(cb) == [127, -128, 127, -128, 127, -128]


def test_int8_rounds_half_to_even():
    c = F.quant_int8(np.array([2.5, 3.5, -2.5, -3.5, 0.5, -0.5], np.float32), np.float32(1))
    assert list(c.view(np.int8)) == [2, 4, -2, -4, 0, 0]


@pytest.mark.parametrize("fmt", ["int4_asym", "uint8_asym"])
def test_asym_codes_range_and_min_max_reconstruction(fmt):
    levels = F.ASYM_LEVELS[fmt]
    rng = np.random.default_rng(3)
    rows = (rng.standard_normal((4000, 128)) * rng.uniform(0.1, 20, (4000, 1))).astype(np.float32)
    rows[:, 5] *= 8  # outlier channel
    c, s, z = F.quant_asym(rows, fmt)
    assert c.min() >= 0 and c.max() <= levels
    i_min = rows.argmin(axis=1)
    i_max = rows.argmax(axis=1)
    r = np.arange(rows.shape[0])
    mn, mx = rows[r, i_min].astype(np.float64), rows[r, i_max].astype(np.float64)
    # the zero point is the row minimum rounded to fp16
    assert np.all(np.abs(z - mn) <= np.abs(mn) * 2.0 ** -11 + 2.0 ** -25)
    assert np.all(c[r, i_min] == 0)
    assert np.all(c[r, i_max] == levels)
    xh = F.dequant_asym(c, s, z)
    assert np.all(xh[r, i_min] == z)
    # every element within half a step (plus fp16 rounding of s and z)
    tol = s.astype(np.float64) * 0.5 + levels * s * 2.0 ** -11 + np.abs(mn) * 2.0 ** -11 + 1e-6
    assert np.all(np.abs(xh - rows) <= tol[:, None])


def test_asym_constant_row_gets_unit_scale():
    rows = np.full((3, 64), 0.75, np.float32)
    c, s, z = F.quant_asym(rows, "int4_asym")
    assert np.all(s == 1.0) and np.all(z == 0.75) and np.all(c == 0)


def test_int4_nibble_order():
    c = np.array([[1, 2, 3, 4, 15, 0]], np.uint8)
    p = F.pack_int4(c)
    assert list(p[0]) == [0x21, 0x43, 0x0F]
    assert np.array_equal(F.unpack_int4(p), c)


def test_capacity_ratios_reproduce_pr4893_blocks_and_kvarn_range():
    """Bytes per token per kv-head: 16-bit KV 2*D; 8-bit KV D; int4 asymmetric
    D/2 codes + 2 fp16 meta.  8-bit doubles the block count of the PR table
    exactly; int4 asymmetric lands inside KVarN's 3-5x capacity claim."""
    d = 128
    b16 = 2 * d
    b8 = F.bytes_per_row("int8", d)
    b4 = F.bytes_per_row("int4_asym", d) + 2 * 2
    rows = [l.split() for l in open(os.path.join(GOLDEN, "pr4893_gpu_blocks.txt"))
            if l.strip() and not l.startswith("#")]
    for _, blocks16, _, blocks8 in rows:
        assert int(blocks16) * b16 // b8 == int(blocks8)
    line = [l for l in open(os.path.join(GOLDEN, "kvarn_capacity.txt"))
            if l.strip() and not l.startswith("#")][0]
    lo, hi = [float(v) for v in line.split()]
    assert lo <= b16 / b4 <= hi
