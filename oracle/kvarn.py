"""Oracle: KVarN pre-quantization (test infrastructure only).

KVarN ('KVarN : le backend natif pour la quantification du cache KV',
section 'Contexte Technique') quantizes the KV cache after a Hadamard
rotation and a variance normalisation, with asymmetric quantization and no
calibration (same article, same section and the one after it).  The article
fixes neither the statistic nor the order; the reading implemented here is:

1. per (token, kv-head) row of D values, sigma = population standard
   deviation in float32, summed by a fixed tree (below); sigma16 = fp16(sigma),
   1 if it rounds to 0;
2. y = x * (1 / sigma16);
3. y = cR * H_D (d . y)  (see oracle.hadamard);
4. asymmetric quantization of y per row (oracle.formats.quant_asym).

Fixed summation tree for a row of D values (float32, one rounding per add):
the row is cut into D/8 groups of 8 consecutive values; each group is summed
left to right; then for o = D/16, D/32, ..., 1 every group sum s_j becomes
s_j + s_(j xor o).  All group sums end equal; that value is the total.
mean = total * (1/D) (exact: D is a power of two); the squared deviations
(x - mean) * (x - mean) are summed by the same tree; var = that * (1/D);
sigma = correctly rounded float32 square root.
"""
from __future__ import annotations

import numpy as np

from .formats import to_f16, quant_asym
from .hadamard import rotate_f32

F32 = np.float32


def tree_sum(rows: np.ndarray) -> np.ndarray:
    """Fixed-order float32 sum of the last axis (length D, a multiple of 8)."""
    rows = np.asarray(rows, np.float32)
    d = rows.shape[-1]
    g = rows.reshape(rows.shape[:-1] + (d // 8, 8))
    s = g[..., 0].copy()
    for k in range(1, 8):
        s = s + g[..., k]
    ngroups = d // 8
    o = ngroups // 2
    idx = np.arange(ngroups)
    while o >= 1:
        s = s + s[..., idx ^ o]
        o //= 2
    return s[..., 0]


def row_sigma16(rows: np.ndarray) -> np.ndarray:
    """fp16 standard deviation of each row (as float32), 1 where it is 0."""
    rows = np.asarray(rows, np.float32)
    d = rows.shape[-1]
    inv_d = F32(1.0 / d)
    mean = tree_sum(rows) * inv_d
    dev = rows - mean[..., None]
    var = tree_sum(dev * dev) * inv_d
    sigma = np.sqrt(var).astype(np.float32)
    s16 = to_f16(sigma)
    return np.where(s16 == 0, F32(1.0), s16).astype(np.float32)


def normalise_rotate(rows: np.ndarray, signs):
    """Steps 1-3: returns (rotated rows in float32, sigma16)."""
    rows = np.asarray(rows, np.float32)
    s16 = row_sigma16(rows)
    inv = (F32(1.0) / s16).astype(np.float32)
    y = rows * inv[..., None]
    return rotate_f32(y, signs), s16


def kvarn_quant(rows: np.ndarray, fmt: str, signs):
    """Steps 1-4: (unpacked codes, s16, z16, sigma16) for each row."""
    y, s16 = normalise_rotate(rows, signs)
    c, s, z = quant_asym(y, fmt)
    return c, s, z, s16
