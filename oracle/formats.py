"""Oracle: cache number formats (test infrastructure only).

Plain, slow, obviously-correct restatement of every code format the cache
stores.  Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline leg
may import this package; the library never does.

Formats and the passages they follow:

* INT8, symmetric, one fp32 scale per tensor (per layer):
  "vllm-int8-kv-cache-for-ampere-sm86" project summary -- an INT8 KV cache
  with calibrated per-layer scaling values.
* FP8 E4M3 (the same summary emulates E4M3 for a part of the cache;
  `fp8` = `fp8_e4m3` in vLLM PR #4893 'Load FP8 kv-cache scaling factors
  from checkpoints', item 1) and FP8 E5M2 (same item), each with a
  kv_scale; uncalibrated means scale 1.0 (PR #4893 item 2; the modelium guide
  'vLLM FP8 KV-кеш', section 'Что проверить перед сменой dtype?').
  Bit layouts follow the OCP 8-bit floating point definition: E4M3FN (bias 7,
  no infinities, max 448) and E5M2 (bias 15, IEEE-like, max 57344).
* Asymmetric INT4 (and UINT8) with a scale and a zero point per token and
  kv-head: vLLM issue #4025 'Support for 4-bit KV Cache in paged-attention op',
  section 'methods', items 1-3; the 'asymmetric quantization' of the KVarN
  article (section 'Contexte Technique').

The code-producing arithmetic is the fixed float32 formula of the library's
contract: x * inv_scale in IEEE float32, round half to even, saturate.
numpy's float32 ufuncs are IEEE round-to-nearest and never fuse a multiply
with an add, so every step below is one correctly rounded operation.
"""
from __future__ import annotations

import numpy as np

F32 = np.float32


# ---------------------------------------------------------------------------
# Generic IEEE-style binary formats (used for fp8 e4m3 / e5m2 and fp16)
# ---------------------------------------------------------------------------
class MiniFloat:
    """A binary floating point format: sign, `ebits` exponent bits, `mbits`
    mantissa bits, exponent bias, largest finite value."""

    def __init__(self, name, ebits, mbits, bias, max_finite, has_inf):
        self.name, self.ebits, self.mbits, self.bias = name, ebits, mbits, bias
        self.max_finite = float(max_finite)
        self.has_inf = has_inf
        self.emin = 1 - bias  # exponent of the smallest normal number
        self.nbits = 1 + ebits + mbits

    def decode(self, codes) -> np.ndarray:
        """Value of every code, float64 (NaN for NaN codes)."""
        c = np.asarray(codes).astype(np.int64)
        sign = (c >> (self.ebits + self.mbits)) & 1
        e = (c >> self.mbits) & ((1 << self.ebits) - 1)
        m = c & ((1 << self.mbits) - 1)
        emax_field = (1 << self.ebits) - 1
        sub = np.ldexp(m.astype(np.float64), self.emin - self.mbits)
        nor = np.ldexp((m + (1 << self.mbits)).astype(np.float64), e - self.bias - self.mbits)
        v = np.where(e == 0, sub, nor)
        if self.has_inf:  # IEEE-like: top exponent is inf / NaN
            v = np.where((e == emax_field) & (m == 0), np.inf, v)
            v = np.where((e == emax_field) & (m != 0), np.nan, v)
        else:  # E4M3FN: only S.1111.111 is NaN
            v = np.where((e == emax_field) & (m == (1 << self.mbits) - 1), np.nan, v)
        return np.where(sign == 1, -v, v)

    def nan_code(self) -> int:
        return (1 << (self.nbits - 1)) - 1  # 0x7F for fp8, 0x7FFF for f16

    def inf_code(self) -> int:
        return ((1 << self.ebits) - 1) << self.mbits

    def encode(self, x, saturate: bool) -> np.ndarray:
        """Round float32 values to this format, to nearest with ties to even.

        `saturate`: finite overflow (and +-inf) clamps to +-max_finite (the
        'satfinite' rule); otherwise it becomes +-inf.  NaN -> the positive
        all-ones NaN code.  The sign of zero (and of values rounding to zero)
        is kept.
        """
        x = np.asarray(x, dtype=np.float32)
        a = np.abs(x.astype(np.float64))
        neg = np.signbit(x)
        nan = np.isnan(x)
        inf = np.isinf(x)
        a_f = np.where(nan | inf, 0.0, a)
        _, e2 = np.frexp(a_f)  # a = f * 2**e2, f in [0.5, 1)
        exp = np.maximum(e2 - 1, self.emin)
        quantum = np.ldexp(1.0, exp - self.mbits)
        r = np.rint(a_f / quantum) * quantum  # exact division; rint = half-even
        over = r > self.max_finite
        # encode r (finite, <= max)
        r_c = np.where(over, 0.0, r)
        _, e2r = np.frexp(r_c)
        er = e2r - 1
        is_sub = r_c < np.ldexp(1.0, self.emin)
        mant_sub = (r_c / np.ldexp(1.0, self.emin - self.mbits)).astype(np.int64)
        mant_nor = (r_c / np.ldexp(1.0, er - self.mbits)).astype(np.int64) - (1 << self.mbits)
        efield = np.where(is_sub, 0, er + self.bias).astype(np.int64)
        mant = np.where(is_sub, mant_sub, mant_nor)
        code = (efield << self.mbits) | mant
        max_code = int(self.encode_scalar_max())
        if saturate:
            code = np.where(over | inf, max_code, code)
        else:
            code = np.where(over | inf, self.inf_code(), code)
        code = code | (neg.astype(np.int64) << (self.nbits - 1))
        code = np.where(nan, self.nan_code(), code)
        dtype = np.uint8 if self.nbits == 8 else np.uint16
        return code.astype(dtype)

    def encode_scalar_max(self) -> int:
        """Code of +max_finite."""
        e = int(np.floor(np.log2(self.max_finite)))
        m = int(self.max_finite / 2.0 ** (e - self.mbits)) - (1 << self.mbits)
        return ((e + self.bias) << self.mbits) | m


E4M3 = MiniFloat("fp8_e4m3", ebits=4, mbits=3, bias=7, max_finite=448.0, has_inf=False)
E5M2 = MiniFloat("fp8_e5m2", ebits=5, mbits=2, bias=15, max_finite=57344.0, has_inf=True)
F16 = MiniFloat("fp16", ebits=5, mbits=10, bias=15, max_finite=65504.0, has_inf=True)
FP8 = {"fp8_e4m3": E4M3, "fp8_e5m2": E5M2}


def to_f16(x) -> np.ndarray:
    """float32 -> nearest fp16 value (ties to even, overflow to inf), as float32."""
    bits = F16.encode(np.asarray(x, np.float32), saturate=False)
    return F16.decode(bits).astype(np.float32)


def f16_bits(x) -> np.ndarray:
    """fp16 bit patterns of float32 values that are exact fp16 numbers."""
    return F16.encode(np.asarray(x, np.float32), saturate=False)


# ---------------------------------------------------------------------------
# Per-tensor calibration (one scale per layer's K or V)
# ---------------------------------------------------------------------------
QMAX = {"int8": 127.0, "fp8_e4m3": 448.0}


def calibrate(x: np.ndarray, rule: str) -> np.float32:
    """Per-tensor scale: absmax/127 (int8), absmax/448 (E4M3) or 1.0.

    Follows the per-layer scaling values of the INT8 KV summary and the
    kv_scale of PR #4893 (scale 1.0 when uncalibrated).  absmax is exact;
    the division is one IEEE float32 division.  An all-zero tensor gets 1.0.
    """
    if rule == "1.0":
        return F32(1.0)
    qmax = {"absmax/127": 127.0, "absmax/448": 448.0}[rule]
    amax = F32(np.max(np.abs(np.asarray(x, np.float32)))) if np.size(x) else F32(0)
    if amax == 0:
        return F32(1.0)
    return F32(amax) / F32(qmax)


def calibrate_heads(x_thd: np.ndarray, rule: str) -> np.ndarray:
    """One scale per kv-head of x [T, Hkv, D]: calibrate() over each head's
    values (the per-attention-head scales that PR #4893's thread leaves as a
    later step)."""
    x_thd = np.asarray(x_thd, np.float32)
    return np.array([calibrate(x_thd[:, h, :], rule) for h in range(x_thd.shape[1])], np.float32)


def inverse_scale(scale) -> np.float32:
    """inv = 1/scale, one IEEE float32 division, computed once per call."""
    return F32(1.0) / F32(scale)


# ---------------------------------------------------------------------------
# Symmetric per-tensor formats
# ---------------------------------------------------------------------------
def quant_int8(x, inv) -> np.ndarray:
    """code = clamp(rne(x * inv), -128, 127), stored as two's complement bytes."""
    v = np.asarray(x, np.float32) * F32(inv)
    c = np.clip(np.rint(v), -128, 127).astype(np.int8)
    return c.view(np.uint8)


def quant_fp8(x, inv, fmt: str) -> np.ndarray:
    """code = fp8_rn_satfinite(x * inv) for fmt in {fp8_e4m3, fp8_e5m2}."""
    v = np.asarray(x, np.float32) * F32(inv)
    return FP8[fmt].encode(v, saturate=True)


def dequant_sym(codes, fmt: str, scale) -> np.ndarray:
    """x_hat = value(code) * scale, float64."""
    codes = np.asarray(codes, np.uint8)
    if fmt == "int8":
        v = codes.view(np.int8).astype(np.float64)
    else:
        v = FP8[fmt].decode(codes)
    return v * float(scale)


# ---------------------------------------------------------------------------
# Asymmetric per-(token, kv-head) formats: int4 (packed) and uint8
# ---------------------------------------------------------------------------
ASYM_LEVELS = {"int4_asym": 15, "uint8_asym": 255}


def asym_params(rows: np.ndarray, levels: int):
    """Scale and zero point of each row (last axis), as fp16 values in float32.

    s16 = fp16(fp32(mx - mn) / levels), replaced by 1 when it rounds to 0;
    z16 = fp16(mn): the zero point is a float offset, so code 0 reconstructs
    the row minimum up to fp16 rounding (issue #4025, 'methods' item 1).
    """
    rows = np.asarray(rows, np.float32)
    mn = rows.min(axis=-1)
    mx = rows.max(axis=-1)
    s = to_f16((mx - mn) / F32(levels))
    s = np.where(s == 0, F32(1.0), s).astype(np.float32)
    z = to_f16(mn)
    return s, z


def quant_asym(rows: np.ndarray, fmt: str):
    """Codes (unpacked, uint8 in [0, levels]), s16 and z16 for each row.

    code = clamp(rne((x - z16) * (1/s16)), 0, levels) in float32.
    """
    levels = ASYM_LEVELS[fmt]
    rows = np.asarray(rows, np.float32)
    s, z = asym_params(rows, levels)
    inv = (F32(1.0) / s).astype(np.float32)
    v = (rows - z[..., None]) * inv[..., None]
    c = np.clip(np.rint(v), 0, levels).astype(np.uint8)
    return c, s, z


def pack_int4(codes: np.ndarray) -> np.ndarray:
    """Two 4-bit codes per byte: element 2i in the low nibble, 2i+1 in the high."""
    c = np.asarray(codes, np.uint8)
    return (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8)


def unpack_int4(packed: np.ndarray) -> np.ndarray:
    p = np.asarray(packed, np.uint8)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out


def dequant_asym(codes_unpacked, s, z) -> np.ndarray:
    """x_hat = code * s16 + z16, float64."""
    c = np.asarray(codes_unpacked).astype(np.float64)
    return c * np.asarray(s, np.float64)[..., None] + np.asarray(z, np.float64)[..., None]


# ---------------------------------------------------------------------------
# The unquantized 16-bit cache (PR #4893 item 1: --kv-cache-dtype auto keeps
# the model's 16-bit KV; here bfloat16, the write path's input type)
# ---------------------------------------------------------------------------
def quant_bf16(x) -> np.ndarray:
    """Stored bytes of bf16-valued float32 inputs: the value's own 16 bits,
    little-endian, two bytes per element (no scale, no rounding: the inputs
    are bf16 already)."""
    x = np.ascontiguousarray(x, np.float32)
    bits = (x.view(np.uint32) >> 16).astype("<u2")
    if np.any((x.view(np.uint32) & 0xFFFF) != 0):
        raise ValueError("bf16 cache input must be bf16 values")
    return bits.view(np.uint8).reshape(x.shape[:-1] + (2 * x.shape[-1],))


def dequant_bf16(codes) -> np.ndarray:
    """Values of stored bf16 rows (bytes [..., 2D]) as float64 [..., D]."""
    c = np.ascontiguousarray(codes, np.uint8)
    bits = c.view("<u2").astype(np.uint32) << 16
    return bits.view(np.float32).astype(np.float64)


def bytes_per_row(fmt: str, head_dim: int) -> int:
    """Stored code bytes per (token, kv-head)."""
    return head_dim // 2 if fmt == "int4_asym" else head_dim * (2 if fmt == "bf16" else 1)
