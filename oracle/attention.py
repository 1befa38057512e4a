"""Oracle: single-token paged decode attention in float64 (test infrastructure only).

vLLM issue #4025 ('Support for 4-bit KV Cache in paged-attention op',
section 'methods', item 3): the paged-attention op takes the quantization
parameters, reads the quantized cache, converts it back to floating point and
then computes attention as usual.  PR #4893's side note (decode of an FP8
cache goes through the paged-attention kernel) is the same operation for
the fp8 formats.  This oracle is that definition, written out:

    for every sequence s and query head h (kv-head h // G, G = Hq / Hkv):
        k_t, v_t = dequantized cache rows of the sequence's tokens t < ctx
        s_t      = sm_scale * <q, k_t>
        out      = sum_t softmax(s)_t v_t        (ctx = 0 -> out = 0)

all in float64, dequantizing token by token from the block table.
"""
from __future__ import annotations

import numpy as np

from .cache import decode_rows, gather_sequence


def softmax_average(q: np.ndarray, k: np.ndarray, v: np.ndarray, sm_scale: float) -> np.ndarray:
    """Plain float64 attention of queries q [G, D] over keys/values [n, D]."""
    if k.shape[0] == 0:
        return np.zeros((q.shape[0], v.shape[1]))
    s = float(sm_scale) * (q.astype(np.float64) @ k.T)
    s = s - s.max(axis=1, keepdims=True)
    p = np.exp(s)
    p /= p.sum(axis=1, keepdims=True)
    return p @ v


def dequant_sequence(codes, meta, block_table_row, ctx, block_size, kv_head, fmt, scale,
                     kvarn, signs, head_dim):
    c, m = gather_sequence(codes, meta, block_table_row, ctx, block_size, kv_head)
    return decode_rows(c, m, fmt, scale, kvarn, signs, head_dim)


def paged_decode(query, k_codes, k_meta, v_codes, v_meta, block_table, context_lens,
                 block_size, k_fmt, v_fmt, k_scale, v_scale, sm_scale, kvarn=False,
                 signs=None, pairs=None) -> np.ndarray:
    """out [S, Hq, D] float64.  `pairs`: optional list of (seq, kv_head) to
    compute (others stay 0), for sampled checks at large sizes."""
    query = np.asarray(query, np.float64)
    s_count, hq, d = query.shape
    hkv = k_codes.shape[2]
    g = hq // hkv
    out = np.zeros((s_count, hq, d))
    if pairs is None:
        pairs = [(s, h) for s in range(s_count) for h in range(hkv)]
    # a scale may be one per kv-head (symmetric formats)
    head = lambda sc, h: sc[h] if np.ndim(sc) == 1 else sc
    for s, h in pairs:
        ctx = int(context_lens[s])
        k = dequant_sequence(k_codes, k_meta, block_table[s], ctx, block_size, h, k_fmt,
                             head(k_scale, h), kvarn, signs, d)
        v = dequant_sequence(v_codes, v_meta, block_table[s], ctx, block_size, h, v_fmt,
                             head(v_scale, h), kvarn, signs, d)
        out[s, h * g:(h + 1) * g] = softmax_average(query[s, h * g:(h + 1) * g], k, v, sm_scale)
    return out


def paged_decode_classes(query, classes, seq_class, block_table, context_lens, k_fmt, v_fmt,
                         k_scale, v_scale, sm_scale, kvarn=False, signs=None) -> np.ndarray:
    """paged_decode over a cache of several page classes (the KVarN article's
    variable page sizes, section 'Perspective'): classes[c] = (k codes, k meta,
    v codes, v meta, block size) of pool c; sequence s reads pool
    seq_class[s] through its row of the block table.  Each sequence's attention
    is the plain definition over its own tokens, whatever its page size."""
    query = np.asarray(query, np.float64)
    s_count, hq, d = query.shape
    out = np.zeros((s_count, hq, d))
    for c, (kc, km, vc, vm, bs) in enumerate(classes):
        pairs = [(s, h) for s in range(s_count) if int(seq_class[s]) == c
                 for h in range(kc.shape[2])]
        if pairs:
            out += paged_decode(query, kc, km, vc, vm, block_table, context_lens, bs, k_fmt,
                                v_fmt, k_scale, v_scale, sm_scale, kvarn, signs, pairs=pairs)
    return out


def default_sm_scale(head_dim: int) -> np.float32:
    """float32(1/sqrt(D)), the usual attention scale."""
    return np.float32(1.0 / np.sqrt(np.float64(head_dim)))
