"""Host-side pins of the decode-step append (CPU only).

kvq_decode_append stores the step's row of sequence s at position
context_lens[s] - 1, i.e. at slot block_table[s][(n-1) // bs] * bs + (n-1) % bs.
These tests pin that addressing against the workload's own slot mapping and
check, on the oracle, that writing all rows but each sequence's last and then
the last rows at those slots builds the same cache as writing every row."""
import numpy as np
import pytest

from oracle import cache as OC
from oracle import formats as OF
from quantized_paged_kv_kvq_gb300 import workloads as W

from kvq_testing import new_token_rows


def _slot_of_last(wl):
    n = wl.context_lens.astype(np.int64)
    out = np.full(wl.num_seqs, -1, np.int64)
    for s in range(wl.num_seqs):
        if n[s] > 0:
            p = n[s] - 1
            out[s] = int(wl.block_table[s, p // wl.block_size]) * wl.block_size + p % wl.block_size
    return out


@pytest.mark.parametrize("name,kw", [("tiny_int8", {}),
                                     ("llama8b_int8", dict(num_seqs=9, ctx_lo=0, ctx_hi=90)),
                                     ("kvarn_131k", dict(num_seqs=5, ctx_lo=1, ctx_hi=200))])
def test_last_position_slot_is_the_slot_mapping_entry(name, kw):
    wl = W.workload(name, **kw)
    rows, has = new_token_rows(wl)
    slots = _slot_of_last(wl)
    assert np.array_equal(slots[has], wl.slot_mapping[rows[has]])
    assert np.all(slots[~has] == -1)


@pytest.mark.parametrize("name", ["llama8b_int8", "llama70b_int4", "kvarn_131k"])
def test_write_all_but_last_then_last_equals_write_all(name):
    lens = np.array([5, 0, 16, 33, 1, 17], np.int32)
    wl = W.workload(name, num_seqs=len(lens), context_lens=lens)
    rows, has = new_token_rows(wl)
    scale = OF.calibrate(wl.key, wl.k_scale_rule) if wl.k_scale_rule else np.float32(1.0)

    def cache():
        return OC.alloc_cache(wl.num_blocks, wl.block_size, wl.num_kv_heads, wl.head_dim,
                              wl.k_fmt, wl.kvarn, 0xAA)

    full_c, full_m = cache()
    OC.write_cache(full_c, full_m, wl.key, wl.slot_mapping, wl.block_size, wl.k_fmt, scale,
                   wl.kvarn, wl.signs)
    two_c, two_m = cache()
    first = wl.slot_mapping.copy()
    first[rows[has]] = -1
    OC.write_cache(two_c, two_m, wl.key, first, wl.block_size, wl.k_fmt, scale, wl.kvarn,
                   wl.signs)
    assert not np.array_equal(two_c, full_c)  # the last rows are still missing
    OC.write_cache(two_c, two_m, wl.key[rows[has]], _slot_of_last(wl)[has], wl.block_size,
                   wl.k_fmt, scale, wl.kvarn, wl.signs)
    assert np.array_equal(two_c, full_c)
    assert np.array_equal(two_m, full_m)
