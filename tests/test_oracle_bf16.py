"""Pins for the oracle's unquantized 16-bit cache (PR #4893 item 1: with
--kv-cache-dtype auto the KV cache keeps the model's 16-bit values).

The stored bytes of a bf16 cache are the values' own bits, so the format is
pinned by an exact round trip over every bf16 value, by its byte order, and by
attention over a paged bf16 cache reducing to plain dense attention on the
inputs (no quantization anywhere)."""
import numpy as np
import pytest

from oracle import attention as OA
from oracle import cache as OC
from oracle import formats as OF
from quantized_paged_kv_kvq_gb300 import workloads as W


def _all_finite_bf16():
    bits = np.arange(1 << 16, dtype=np.uint32) << 16
    x = bits.view(np.float32)
    return x[np.isfinite(x)]


def test_round_trip_of_every_bf16_value_is_exact():
    x = _all_finite_bf16()
    x = x[: x.size // 64 * 64].reshape(-1, 64)
    codes = OF.quant_bf16(x)
    assert codes.shape == (x.shape[0], 128) and codes.dtype == np.uint8
    back = OF.dequant_bf16(codes)
    assert np.array_equal(back.astype(np.float32).view(np.uint32), x.view(np.uint32))


def test_byte_order_is_little_endian_bf16():
    x = np.array([[1.0, -2.0, 0.0, -0.0, 0.5, 3.0, 65280.0, 2.0 ** -133]], np.float32)
    c = OF.quant_bf16(x)
    # 1.0 = 0x3F80, -2.0 = 0xC000, +0, -0 = 0x8000, 0.5 = 0x3F00, 3.0 = 0x4040,
    # 65280 = 0x477F, 2^-133 = 0x0001 (the smallest subnormal)
    assert list(c[0]) == [0x80, 0x3F, 0x00, 0xC0, 0x00, 0x00, 0x00, 0x80, 0x00, 0x3F, 0x40,
                          0x40, 0x7F, 0x47, 0x01, 0x00]


def test_non_bf16_input_is_rejected():
    with pytest.raises(ValueError):
        OF.quant_bf16(np.array([[1.0 + 2.0 ** -12] * 8], np.float32))


def test_paged_bf16_cache_gives_dense_attention_on_the_inputs():
    """Write a seeded workload into a paged bf16 cache (shuffled blocks), decode
    with the paged oracle, and compare with softmax attention computed straight
    from the generator's K / V arrays."""
    wl = W.workload("llama8b_int8", num_seqs=3, ctx_lo=1, ctx_hi=90, num_q_heads=8,
                    num_kv_heads=2)
    kc, km = OC.alloc_cache(wl.num_blocks, wl.block_size, wl.num_kv_heads, wl.head_dim, "bf16",
                            False)
    vc, vm = OC.alloc_cache(wl.num_blocks, wl.block_size, wl.num_kv_heads, wl.head_dim, "bf16",
                            False)
    OC.write_cache(kc, km, wl.key, wl.slot_mapping, wl.block_size, "bf16", 1.0)
    OC.write_cache(vc, vm, wl.value, wl.slot_mapping, wl.block_size, "bf16", 1.0)
    sm = OA.default_sm_scale(wl.head_dim)
    out = OA.paged_decode(wl.query, kc, km, vc, vm, wl.block_table, wl.context_lens,
                          wl.block_size, "bf16", "bf16", 1.0, 1.0, sm)
    starts = np.concatenate([[0], np.cumsum(wl.context_lens)])
    g = wl.num_q_heads // wl.num_kv_heads
    for s in range(wl.num_seqs):
        k = wl.key[starts[s]:starts[s + 1]].astype(np.float64)
        v = wl.value[starts[s]:starts[s + 1]].astype(np.float64)
        for h in range(wl.num_q_heads):
            q = wl.query[s, h].astype(np.float64)
            logits = float(sm) * (k[:, h // g] @ q)
            p = np.exp(logits - logits.max())
            ref = (p / p.sum()) @ v[:, h // g]
            assert np.allclose(out[s, h], ref, rtol=0, atol=1e-12)
