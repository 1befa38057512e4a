"""Pins for the oracle's rotation and variance normalisation (CPU only)."""
import math

import numpy as np
import pytest
import scipy.linalg

from oracle import hadamard as H
from oracle import kvarn as K
from oracle import formats as F

DIMS = [2, 4, 8, 16, 32, 64, 128, 256]


def test_h2_is_the_textbook_matrix():
    assert np.array_equal(H.sylvester(2), [[1, 1], [1, -1]])


@pytest.mark.parametrize("d", DIMS)
def test_sylvester_closed_form_library_and_orthogonality(d):
    h = H.sylvester(d)
    i, j = np.meshgrid(np.arange(d), np.arange(d), indexing="ij")
    pop = np.vectorize(lambda v: bin(int(v)).count("1"))(i & j)
    assert np.array_equal(h, (-1.0) ** pop)
    assert np.array_equal(h, scipy.linalg.hadamard(d))
    assert np.array_equal(h @ h.T, d * np.eye(d))


@pytest.mark.parametrize("d", DIMS)
def test_butterfly_equals_matrix_exactly_on_integers(d):
    rng = np.random.default_rng(d)
    x = rng.integers(-1000, 1000, size=(50, d)).astype(np.float64)
    assert np.array_equal(H.fwht_stages(x), x @ H.sylvester(d).T)


@pytest.mark.parametrize("d", [64, 128, 256])
def test_float32_rotation_close_to_exact_and_orthonormal(d):
    rng = np.random.default_rng(7)
    x = rng.standard_normal((300, d)).astype(np.float32)
    signs = np.where(rng.integers(0, 2, d) == 0, 1, -1).astype(np.int8)
    y = H.rotate_f32(x, signs)
    exact = ((x.astype(np.float64) * signs) @ H.sylvester(d).T) / math.sqrt(d)
    # log2(D) rounded add stages + one multiply: relative to the row norm
    norm = np.linalg.norm(x, axis=1, keepdims=True)
    assert np.all(np.abs(y - exact) <= (math.log2(d) + 2) * 2.0 ** -23 * norm)
    assert np.allclose(np.linalg.norm(y, axis=1), norm[:, 0], rtol=1e-5)
    back = H.unrotate_f32(y, signs)
    assert np.all(np.abs(back - x) <= 2 * (math.log2(d) + 2) * 2.0 ** -23 * norm)
    assert np.allclose(H.unrotate_f64(exact, signs), x, atol=1e-12)


def test_rotation_scale_values():
    assert H.rotation_scale(64) == 0.125 and H.rotation_scale(256) == 0.0625
    assert H.rotation_scale(128) == np.float32(1 / math.sqrt(128))


def test_hadamard_rows_bf16_output_is_rounded_f32_result():
    rng = np.random.default_rng(9)
    x = rng.standard_normal((20, 128)).astype(np.float32)
    x = (x.view(np.uint32) & 0xFFFF0000).view(np.float32)  # bf16 values
    y32 = H.hadamard_rows(x, None, False, "f32")
    y16 = H.hadamard_rows(x, None, False, "bf16")
    assert np.all((y16.view(np.uint32) & 0xFFFF) == 0)
    assert np.all(np.abs(y16 - y32) <= np.abs(y32) * 2.0 ** -8)


def _bf16(bits):
    return (np.asarray(bits, np.uint32) << 16).view(np.float32)


@pytest.mark.parametrize("sign", [1.0, -1.0])
def test_hadamard_rows_bf16_rounds_ties_to_even(sign):
    """D = 64, so cR = 1/8 exactly and a row a*e0 + b*e1 rotates to (a + b)/8
    and (a - b)/8 (alternating positions) with no rounding before the bf16
    store; b = 2^-8 puts these on or off bf16 ties:
      a = 1:          a + b = 1 + 2^-8, halfway between 1 (even) and 1 + 2^-7:
                      ties-to-even gives 1, ties-away or rounding up 1 + 2^-7;
                      a - b = 1 - 2^-8 is a bf16 value (no rounding).
      a = 1 + 2^-7:   a + b = 1 + 3*2^-8, halfway between 1 + 2^-7 (odd) and
                      1 + 2^-6 (even): ties-to-even rounds up, ties-to-odd or
                      truncation stay at 1 + 2^-7;
                      a - b = 1 + 2^-8, a tie again: ties-to-even gives 1."""
    d = 64
    cases = ((1.0, 1.0, 1.0 + 2.0 ** -7, 1.0 - 2.0 ** -8),
             (1.0 + 2.0 ** -7, 1.0 + 2.0 ** -6, 1.0 + 2.0 ** -7, 1.0))
    b = 2.0 ** -8
    for a, plus_even, plus_wrong, minus_even in cases:
        x = np.zeros((1, d), np.float32)
        x[0, 0], x[0, 1] = sign * a, sign * b
        y32 = H.hadamard_rows(x, None, False, "f32")
        y16 = H.hadamard_rows(x, None, False, "bf16")
        assert np.all(y32[0, 0::2] == np.float32(sign * (a + b) / 8))  # exact in float32
        assert np.all(y32[0, 1::2] == np.float32(sign * (a - b) / 8))
        assert np.all(y16[0, 0::2] == np.float32(sign * plus_even / 8))
        assert np.all(y16[0, 0::2] != np.float32(sign * plus_wrong / 8))
        assert np.all(y16[0, 1::2] == np.float32(sign * minus_even / 8))


def test_hadamard_rows_bf16_rounding_matches_torch():
    """Random rows, and rows whose float32 result sits exactly on bf16 ties:
    the bf16 store equals torch's float32 -> bfloat16 conversion (round to
    nearest, ties to even)."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(21)
    x = _bf16(rng.integers(0x3000, 0x4300, size=(64, 64)) | (rng.integers(0, 2, (64, 64)) << 15))
    x[:32] = 0
    # rows a e0 + b e1 with (a + b) on a tie: a any bf16, b = half an ulp of a
    a = _bf16(rng.integers(0x3E00, 0x4100, size=32) | (rng.integers(0, 2, 32) << 15))
    ulp_half = (a.view(np.uint32) & 0x7F800000).view(np.float32) * np.float32(2.0 ** -8)
    x[:32, 0], x[:32, 1] = a, ulp_half * np.sign(a)
    for inverse in (False, True):
        y32 = H.hadamard_rows(x, None, inverse, "f32")
        y16 = H.hadamard_rows(x, None, inverse, "bf16")
        ref = torch.from_numpy(y32).to(torch.bfloat16).to(torch.float32).numpy()
        assert np.array_equal(y16.view(np.uint32), ref.view(np.uint32))
    ties = (H.hadamard_rows(x[:32], None, False, "f32").view(np.uint32) & 0xFFFF) == 0x8000
    assert ties.sum() >= 32 * 16  # the tie rows really do land on ties


def test_tree_sum_order_is_pinned():
    """Group sums go left to right; groups combine largest offset first."""
    d = 128
    row = np.zeros(d, np.float32)
    row[0:3] = [2.0 ** 24, 1.0, 1.0]  # left to right: 2^24+1 -> 2^24, +1 -> 2^24
    assert K.tree_sum(row[None])[0] == 2.0 ** 24
    row = np.zeros(d, np.float32)
    row[0], row[8], row[24] = 2.0 ** 24, 1.0, 1.0  # group sums s0=2^24, s1=1, s3=1
    # offsets 8,4,2 first give s1+s3 = 2, then s0 + 2 is exact; offset 1 first
    # would lose both ones to round-half-even
    assert K.tree_sum(row[None])[0] == 2.0 ** 24 + 2


def test_tree_sum_matches_exact_sum():
    rng = np.random.default_rng(11)
    x = rng.integers(-2 ** 10, 2 ** 10, size=(100, 128)).astype(np.float32)
    assert np.array_equal(K.tree_sum(x), x.sum(axis=1))  # exact for small integers
    y = rng.standard_normal((100, 128)).astype(np.float32)
    ref = np.array([math.fsum(r) for r in y.astype(np.float64)])
    assert np.all(np.abs(K.tree_sum(y) - ref) <= 128 * 2.0 ** -23 * np.abs(y).sum(axis=1))


def test_sigma16_is_fp16_of_population_std():
    rng = np.random.default_rng(12)
    x = (rng.standard_normal((2000, 128)) * rng.uniform(0.01, 30, (2000, 1))).astype(np.float32)
    s16 = K.row_sigma16(x)
    ref = x.astype(np.float64).std(axis=1)
    assert np.all(np.abs(s16 - ref) <= ref * (2.0 ** -11 + 1e-5))
    assert np.all(F.to_f16(s16) == s16)
    assert np.all(K.row_sigma16(np.full((2, 128), 3.0, np.float32)) == 1.0)


def test_normalised_rotated_rows_have_unit_variance_and_round_trip():
    rng = np.random.default_rng(13)
    x = (rng.standard_normal((500, 128)) * rng.uniform(0.1, 10, (500, 1))).astype(np.float32)
    x[:, 3] += 5.0
    signs = np.where(rng.integers(0, 2, 128) == 0, 1, -1).astype(np.int8)
    y, s16 = K.normalise_rotate(x, signs)
    # the rotation preserves the norm, so mean square of y = (var + mean^2)/sigma^2
    ms = (x.astype(np.float64) ** 2).mean(axis=1) / s16.astype(np.float64) ** 2
    assert np.allclose((y.astype(np.float64) ** 2).mean(axis=1), ms, rtol=1e-4)
    back = H.unrotate_f64(y, signs) * s16[:, None]
    assert np.allclose(back, x, rtol=1e-4, atol=1e-4 * np.abs(x).max())


def test_kvarn_quant_error_bound():
    rng = np.random.default_rng(14)
    x = (rng.standard_normal((500, 128)) * rng.uniform(0.1, 10, (500, 1))).astype(np.float32)
    signs = np.where(rng.integers(0, 2, 128) == 0, 1, -1).astype(np.int8)
    for fmt in ("int4_asym", "uint8_asym"):
        c, s, z, sig = K.kvarn_quant(x, fmt, signs)
        y_hat = F.dequant_asym(c, s, z)
        x_hat = H.unrotate_f64(y_hat * sig[:, None], signs)
        # error in the rotated domain is <= s/2 per element; rotation is orthonormal
        bound = np.sqrt(128) * (s * 0.5 * 1.01 + np.abs(z) * 2 ** -11) * sig
        assert np.all(np.linalg.norm(x_hat - x, axis=1) <= bound)
