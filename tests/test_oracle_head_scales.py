"""Pins for per-kv-head scales of the symmetric formats in the oracle (CPU only).

A per-head scale replaces the per-tensor scale of the INT8 summary / PR #4893
with one value per kv-head.  Pinned against the per-tensor definitions it
generalises and against identities of the attention it feeds."""
import numpy as np
import pytest

from oracle import attention as A
from oracle import cache as C
from oracle import formats as F
from quantized_paged_kv_kvq_gb300 import workloads as W


def _wl(name="llama8b_int8"):
    return W.workload(name, num_seqs=3, ctx_lo=5, ctx_hi=60)


def _write(wl, fmt, x, scale):
    codes, meta = C.alloc_cache(wl.num_blocks, wl.block_size, wl.num_kv_heads, wl.head_dim,
                                fmt, False)
    C.write_cache(codes, meta, x, wl.slot_mapping, wl.block_size, fmt, scale)
    return codes, meta


def test_calibrate_heads_matches_each_head_and_the_tensor():
    wl = _wl()
    for rule in ("absmax/127", "absmax/448"):
        per = F.calibrate_heads(wl.key, rule)
        assert per.shape == (wl.num_kv_heads,) and per.dtype == np.float32
        for h in range(wl.num_kv_heads):
            assert per[h] == F.calibrate(wl.key[:, h, :], rule)
        # the tensor's absmax is the largest head absmax; the division is monotone
        assert per.max() == F.calibrate(wl.key, rule)


@pytest.mark.parametrize("fmt", ["int8", "fp8_e4m3", "fp8_e5m2"])
def test_equal_head_scales_reduce_to_the_tensor_scale(fmt):
    wl = _wl()
    sc = np.float32(0.037)
    a, _ = _write(wl, fmt, wl.key, sc)
    b, _ = _write(wl, fmt, wl.key, np.full(wl.num_kv_heads, sc, np.float32))
    assert np.array_equal(a, b)


def test_a_head_scale_changes_only_that_heads_codes():
    wl = _wl()
    scales = F.calibrate_heads(wl.key, "absmax/127")
    a, _ = _write(wl, "int8", wl.key, scales)
    s2 = scales.copy()
    s2[3] *= np.float32(2)
    b, _ = _write(wl, "int8", wl.key, s2)
    diff = np.any(a != b, axis=(0, 1, 3))
    assert diff[3] and not diff[np.arange(wl.num_kv_heads) != 3].any()


def test_int8_error_bound_per_head():
    wl = _wl()
    scales = F.calibrate_heads(wl.key, "absmax/127")
    codes, meta = _write(wl, "int8", wl.key, scales)
    for s in range(wl.num_seqs):
        for h in range(wl.num_kv_heads):
            c, m = C.gather_sequence(codes, meta, wl.block_table[s], wl.context_lens[s],
                                     wl.block_size, h)
            xr = C.decode_rows(c, m, "int8", scales[h], False, None, wl.head_dim)
            start = int(np.sum(wl.context_lens[:s]))
            x = wl.key[start:start + int(wl.context_lens[s]), h, :].astype(np.float64)
            assert np.max(np.abs(xr - x)) <= scales[h] / 2 * (1 + 1e-6)


def test_attention_with_head_scales_obeys_the_scale_identities():
    """Scaling head h's K scale by c is scaling its logits by c (sm_scale * c);
    scaling its V scale by c scales its output by c; equal scales equal the
    tensor scale."""
    wl = _wl()
    ks = F.calibrate_heads(wl.key, "absmax/127")
    vs = F.calibrate_heads(wl.value, "absmax/127")
    kc, km = _write(wl, "int8", wl.key, ks)
    vc, vm = _write(wl, "int8", wl.value, vs)
    sm = A.default_sm_scale(wl.head_dim)
    run = lambda k_s, v_s, smx: A.paged_decode(wl.query, kc, km, vc, vm, wl.block_table,
                                               wl.context_lens, wl.block_size, "int8", "int8",
                                               k_s, v_s, smx)
    base = run(ks, vs, sm)
    g = wl.num_q_heads // wl.num_kv_heads
    h = 5
    ks2 = ks.astype(np.float64).copy()
    ks2[h] *= 3.0
    heads = slice(h * g, (h + 1) * g)
    np.testing.assert_allclose(run(ks2, vs, sm)[:, heads], run(ks, vs, 3.0 * np.float64(sm))[:, heads],
                               rtol=1e-12, atol=1e-12)
    vs2 = vs.astype(np.float64).copy()
    vs2[h] *= 0.5
    np.testing.assert_allclose(run(ks, vs2, sm)[:, heads], 0.5 * base[:, heads], rtol=1e-12,
                               atol=1e-15)
    other = np.ones(wl.num_q_heads, bool)
    other[heads] = False
    np.testing.assert_array_equal(run(ks2, vs2, sm)[:, other], base[:, other])
    # all heads at one value == that value as the tensor scale
    one = np.float32(0.04)
    np.testing.assert_array_equal(run(np.full(wl.num_kv_heads, one), np.full(wl.num_kv_heads, one), sm),
                                  run(one, one, sm))
