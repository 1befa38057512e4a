"""Oracle: quantize-and-scatter into the paged cache (test infrastructure only).

vLLM issue #4025 ('Support for 4-bit KV Cache in paged-attention op',
section 'methods', items 1-2) asks for an op that computes the quantization
parameters and a `write_to_paged_cache` that stores the quantized KV in the
paged cache; the INT8 summary ('vllm-int8-kv-cache-for-ampere-sm86') and
vLLM PR #4893 (item 1) do the same with per-tensor scales.

Layouts (all caller-owned, row-major):
  codes  [num_blocks, block_size, num_kv_heads, D'] bytes, D' = D (8-bit)
         or D/2 (int4, two codes per byte);
  meta   [num_blocks, num_kv_heads, F, block_size] fp16 bit patterns, for the
         asymmetric formats only; fields F = (scale, zero point) or, with the
         KVarN rotation, (scale, zero point, sigma).
Token t goes to slot = slot_mapping[t] (block = slot // bs, offset = slot %
bs); a negative slot skips the token.  Slots that are not written keep their
previous bytes.
"""
from __future__ import annotations

import numpy as np

from . import formats as F
from .kvarn import kvarn_quant

SYMMETRIC = ("int8", "fp8_e4m3", "fp8_e5m2")
ASYMMETRIC = ("int4_asym", "uint8_asym")


def meta_fields(fmt: str, kvarn: bool) -> int:
    if fmt in ASYMMETRIC:
        return 3 if kvarn else 2
    return 0


def encode_rows(rows: np.ndarray, fmt: str, scale, kvarn: bool, signs):
    """Quantize rows [N, D] -> (codes [N, D'] uint8, meta [N, F] fp16 bits)."""
    rows = np.asarray(rows, np.float32)
    n = rows.shape[0]
    if fmt == "bf16":  # the 16-bit cache stores the values themselves
        if kvarn:
            raise ValueError("the rotation is only defined with asymmetric formats")
        return F.quant_bf16(rows), np.zeros((n, 0), np.uint16)
    if fmt in SYMMETRIC:
        if kvarn:
            raise ValueError("the rotation is only defined with asymmetric formats")
        inv = F.inverse_scale(scale)
        codes = F.quant_int8(rows, inv) if fmt == "int8" else F.quant_fp8(rows, inv, fmt)
        return codes, np.zeros((n, 0), np.uint16)
    if fmt not in ASYMMETRIC:
        raise ValueError(fmt)
    if kvarn:
        c, s, z, sig = kvarn_quant(rows, fmt, signs)
        meta = np.stack([F.f16_bits(s), F.f16_bits(z), F.f16_bits(sig)], axis=-1)
    else:
        c, s, z = F.quant_asym(rows, fmt)
        meta = np.stack([F.f16_bits(s), F.f16_bits(z)], axis=-1)
    if fmt == "int4_asym":
        c = F.pack_int4(c)
    return c, meta


def decode_rows(codes: np.ndarray, meta: np.ndarray, fmt: str, scale, kvarn: bool,
                signs, head_dim: int) -> np.ndarray:
    """Dequantize stored rows back to float64 [N, D] (un-rotating for KVarN)."""
    if fmt == "bf16":
        return F.dequant_bf16(codes)
    if fmt in SYMMETRIC:
        return F.dequant_sym(codes, fmt, scale)
    c = F.unpack_int4(codes) if fmt == "int4_asym" else np.asarray(codes, np.uint8)
    s = F.F16.decode(meta[..., 0])
    z = F.F16.decode(meta[..., 1])
    y = F.dequant_asym(c, s, z)
    if kvarn:
        from .hadamard import unrotate_f64
        sig = F.F16.decode(meta[..., 2])
        y = unrotate_f64(y * sig[..., None], signs)
    return y


def alloc_cache(num_blocks, block_size, num_kv_heads, head_dim, fmt, kvarn, fill=0xAA):
    """Fresh cache arrays filled with a poison byte (codes) / bit pattern (meta)."""
    dp = F.bytes_per_row(fmt, head_dim)
    codes = np.full((num_blocks, block_size, num_kv_heads, dp), fill, np.uint8)
    nf = meta_fields(fmt, kvarn)
    meta = np.full((num_blocks, num_kv_heads, nf, block_size), fill * 0x101, np.uint16)
    return codes, meta


def write_cache(codes, meta, rows_thd: np.ndarray, slot_mapping, block_size, fmt, scale,
                kvarn=False, signs=None):
    """Quantize x [T, Hkv, D] and scatter into (codes, meta) in place.

    `scale` is one value for the tensor, or (symmetric formats) an array of
    one value per kv-head, head h's rows quantized with scale[h]."""
    rows_thd = np.asarray(rows_thd, np.float32)
    t, hkv, d = rows_thd.shape
    slots = np.asarray(slot_mapping, np.int64)
    keep = slots >= 0
    if np.ndim(scale) == 1:
        parts = [encode_rows(rows_thd[:, h, :], fmt, scale[h], kvarn, signs) for h in range(hkv)]
        c = np.stack([p[0] for p in parts], axis=1)[keep]
        m = np.stack([p[1] for p in parts], axis=1)[keep]
    else:
        c, m = encode_rows(rows_thd.reshape(t * hkv, d), fmt, scale, kvarn, signs)
        c = c.reshape(t, hkv, -1)[keep]
        m = m.reshape(t, hkv, -1)[keep]
    blk = slots[keep] // block_size
    off = slots[keep] % block_size
    codes[blk, off] = c
    if meta.shape[2]:
        for f in range(meta.shape[2]):
            meta[blk[:, None], np.arange(hkv)[None, :], f, off[:, None]] = m[..., f]
    return codes, meta


def gather_sequence(codes, meta, block_table_row, ctx, block_size, kv_head):
    """Stored codes [ctx, D'] and meta [ctx, F] of one sequence and kv-head."""
    t = np.arange(int(ctx))
    blk = np.asarray(block_table_row)[t // block_size].astype(np.int64)
    off = t % block_size
    c = codes[blk, off, kv_head]
    m = meta[blk, kv_head, :, off] if meta.shape[2] else np.zeros((int(ctx), 0), np.uint16)
    return c, m
