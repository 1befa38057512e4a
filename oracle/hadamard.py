"""Oracle: Walsh-Hadamard rotation (test infrastructure only).

The KVarN article ('KVarN : le backend natif pour la quantification du cache
KV', section 'Contexte Technique') combines a Hadamard rotation with variance
normalisation and asymmetric quantization.  The rotation used here is the
orthonormal natural-order (Sylvester) Walsh-Hadamard matrix with a +-1
diagonal applied first:

    forward:  y = cR * H_D (d . x)          cR = float32(1/sqrt(D))
    inverse:  x = d . (cR * H_D y)

Two independent statements of H_D live here: the explicit Sylvester matrix
(Kronecker powers of [[1, 1], [1, -1]]) for dequantization in float64, and
the fixed-order float32 butterfly whose rounding the cache codes depend on:
stages h = 1, 2, 4, ..., D/2 in increasing order, each pair (i, i + h) with
i & h == 0 becoming (a + b, a - b), one IEEE add each.
"""
from __future__ import annotations

import numpy as np


def sylvester(d: int) -> np.ndarray:
    """H_d by the Sylvester recursion H_2n = [[H_n, H_n], [H_n, -H_n]] (float64)."""
    if d < 1 or d & (d - 1):
        raise ValueError("D must be a power of two")
    h = np.ones((1, 1))
    base = np.array([[1.0, 1.0], [1.0, -1.0]])
    while h.shape[0] < d:
        h = np.kron(base, h)
    return h


def rotation_scale(d: int) -> np.float32:
    """cR = float32(1 / sqrt(D)) (1/8 exactly for D = 64)."""
    return np.float32(1.0 / np.sqrt(np.float64(d)))


def fwht_stages(x: np.ndarray) -> np.ndarray:
    """Unnormalised transform H_D x along the last axis, in x's dtype, by the
    fixed stage order h = 1, 2, ..., D/2 (one rounded add per output)."""
    y = np.array(x, copy=True)
    d = y.shape[-1]
    h = 1
    lead = y.shape[:-1]
    while h < d:
        v = y.reshape(lead + (d // (2 * h), 2, h))
        a = v[..., 0, :]
        b = v[..., 1, :]
        y = np.stack([a + b, a - b], axis=-2).reshape(lead + (d,))
        h *= 2
    return y


def rotate_f32(x: np.ndarray, signs) -> np.ndarray:
    """Forward rotation in float32: cR * FWHT(d . x)."""
    x = np.asarray(x, np.float32)
    d = x.shape[-1]
    if signs is not None:
        x = x * np.asarray(signs, np.float32)
    return fwht_stages(x) * rotation_scale(d)


def unrotate_f32(y: np.ndarray, signs) -> np.ndarray:
    """Inverse rotation in float32: d . (cR * FWHT(y))."""
    y = np.asarray(y, np.float32)
    d = y.shape[-1]
    x = fwht_stages(y) * rotation_scale(d)
    if signs is not None:
        x = x * np.asarray(signs, np.float32)
    return x


def unrotate_f64(y: np.ndarray, signs) -> np.ndarray:
    """Exact inverse of the orthonormal rotation in float64 with the explicit
    matrix: x = d . (H y) / sqrt(D)."""
    y = np.asarray(y, np.float64)
    d = y.shape[-1]
    x = (y @ sylvester(d).T) / np.sqrt(d)
    if signs is not None:
        x = x * np.asarray(signs, np.float64)
    return x


def hadamard_rows(x: np.ndarray, signs, inverse: bool, dtype: str) -> np.ndarray:
    """What the standalone in-place transform leaves in a [rows, D] buffer.

    dtype "f32": float32 in and out.  dtype "bf16": float32 values that are
    exact bf16 in, computed in float32, rounded to bf16 (nearest, ties to
    even) on the way out; returned as float32.
    """
    f = unrotate_f32 if inverse else rotate_f32
    y = f(np.asarray(x, np.float32), signs)
    if dtype == "bf16":
        u = y.view(np.uint32).astype(np.uint64)
        y = (((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint32) << 16).view(np.float32)
    return y
