"""Fused new-token append + decode (kvq_decode_append) on the GPU against the oracle.

A decode step brings one new key / value row per sequence, stored into the
paged cache and attended to in the same step (issue #4025 'Support for 4-bit KV
Cache in paged-attention op', section 'methods', items 2-3, for the decoding
phase).  Here the new row of each sequence is the last position of its
context: the cache write leaves it out and the append call stores it.  After
the call the whole cache must equal, byte for byte, the oracle's cache of all
tokens, and the output must match the oracle's attention over that cache."""
import numpy as np
import pytest
import torch

from oracle import attention as OA
from quantized_paged_kv_kvq_gb300 import kvq
from quantized_paged_kv_kvq_gb300 import workloads as W

from kvq_testing import (GpuRun, OracleRun, append_step, assert_attention_close,
                         new_token_rows, out_numpy, random_workspace)

pytestmark = pytest.mark.gpu

SMALL = {
    "tiny_int8": dict(),
    "llama8b_int8": dict(num_seqs=6, ctx_lo=1, ctx_hi=700),
    "llama8b_e4m3k_int8v": dict(num_seqs=6, ctx_lo=1, ctx_hi=700),
    "llama8b_e5m2": dict(num_seqs=6, ctx_lo=1, ctx_hi=700),
    "llama70b_int4": dict(num_seqs=4, ctx_lo=1, ctx_hi=900),
    "kvarn_131k": dict(num_seqs=3, ctx_lo=1, ctx_hi=900),
    "llama8b_bf16": dict(num_seqs=6, ctx_lo=1, ctx_hi=700),
}


def assert_cache_equals_oracle(g, o, what):
    kc, km, vc, vm = g.cache_numpy()
    assert np.array_equal(kc, o.kc), f"{what}: K codes"
    assert np.array_equal(vc, o.vc), f"{what}: V codes"
    if o.km.shape[2]:
        assert np.array_equal(km, o.km), f"{what}: K meta"
        assert np.array_equal(vm, o.vm), f"{what}: V meta"


@pytest.mark.parametrize("name", list(SMALL))
def test_append_matches_oracle(name):
    wl = W.workload(name, **SMALL[name])
    g, out = append_step(wl)
    o = OracleRun(wl)
    assert_cache_equals_oracle(g, o, name)
    assert_attention_close(out_numpy(out), o.decode(), name)
    assert kvq.kvq_get_device_error() == 0


@pytest.mark.parametrize("name", ["llama8b_int8", "llama70b_int4", "kvarn_131k"])
@pytest.mark.parametrize("ctas", [1, 3, 64, 0])
def test_append_split_variants(name, ctas):
    """The range that holds a sequence's last tile stores its new row, whether
    the sequence is whole in one range or split over several."""
    wl = W.workload(name, **dict(SMALL[name], ctx_lo=200, ctx_hi=2500))
    g, out = append_step(wl, num_ctas=ctas)
    o = OracleRun(wl)
    assert_cache_equals_oracle(g, o, f"{name} ctas={ctas}")
    assert_attention_close(out_numpy(out), o.decode(), f"{name} ctas={ctas}")


@pytest.mark.parametrize("name", ["llama8b_int8", "kvarn_131k"])
@pytest.mark.parametrize("ctas", [1, 2, 5])
def test_append_many_sequences_per_range(name, ctas):
    """More than 32 sequences end in one range (the walk takes them 32 at a
    time), with empty sequences, one-token sequences and full last tiles."""
    rng = np.random.default_rng(7)
    lens = rng.integers(1, 60, size=75).astype(np.int32)
    lens[[3, 40, 41, 74]] = 0
    lens[[5, 33]] = 1
    lens[[10, 50]] = [16, 48]
    wl = W.workload(name, num_seqs=len(lens), context_lens=lens)
    g, out = append_step(wl, num_ctas=ctas)
    o = OracleRun(wl)
    assert_cache_equals_oracle(g, o, f"{name} ctas={ctas}")
    got = out_numpy(out)
    assert np.all(got[lens == 0] == 0)
    assert_attention_close(got, o.decode(), f"{name} ctas={ctas}")
    assert kvq.kvq_get_device_error() == 0


@pytest.mark.parametrize("name", ["llama8b_int8", "llama70b_int4", "kvarn_131k"])
@pytest.mark.parametrize("ctas", [3, 0])
def test_append_equals_write_then_decode(name, ctas):
    """The fused call gives the codes and the output (bit for bit, same ranges)
    of a cache write of the new rows followed by kvq_paged_decode."""
    wl = W.workload(name, **dict(SMALL[name], ctx_lo=100, ctx_hi=1500))
    g, out = append_step(wl, num_ctas=ctas)
    h = GpuRun(wl)
    h.write()
    ref = h.decode(num_ctas=ctas)
    for a, b in zip(g.cache_numpy(), h.cache_numpy()):
        if a is not None:
            assert np.array_equal(a, b)
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))


@pytest.mark.parametrize("bs", [8, 32, 64, 128])
def test_append_block_sizes(bs):
    wl = W.workload("llama8b_int8", num_seqs=5, ctx_lo=1, ctx_hi=600, block_size=bs)
    g, out = append_step(wl, num_ctas=0)
    o = OracleRun(wl)
    assert_cache_equals_oracle(g, o, f"block_size={bs}")
    assert_attention_close(out_numpy(out), o.decode(), f"block_size={bs}")


@pytest.mark.parametrize("name", ["llama8b_int8", "llama8b_e4m3k_int8v"])
def test_append_per_head_scales(name):
    wl = W.workload(name, **SMALL[name])
    g, out = append_step(wl, head_scales=True)
    o = OracleRun(wl, head_scales=True)
    assert_cache_equals_oracle(g, o, name)
    assert_attention_close(out_numpy(out), o.decode(), name)


def test_append_bad_block_id_writes_nothing():
    """A block id outside the cache sets the block-range error bit and the
    append stores nothing (the rest of the cache is untouched)."""
    wl = W.workload("llama8b_int8", num_seqs=3, ctx_lo=20, ctx_hi=80)
    g = GpuRun(wl)
    g.write()
    before = [x.copy() for x in g.cache_numpy() if x is not None]
    bt = g.block_table.clone()
    s = 1
    n = int(wl.context_lens[s])
    bt[s, (n - 1) // wl.block_size] = wl.num_blocks + 5  # only the new token's block
    rows, _ = new_token_rows(wl)
    r = torch.from_numpy(rows).to(g.key.device)
    out = torch.empty_like(g.query)
    kvq.kvq_get_device_error()  # clear
    kvq.kvq_decode_append(g.cache, g.key[r].contiguous() * 3, g.value[r].contiguous() * 3,
                          g.query, out, bt, g.context_lens, wl.max_context_len,
                          float(OA.default_sm_scale(wl.head_dim)), random_workspace(g, 1), 1)
    bits = kvq.kvq_get_device_error()
    assert bits & 2
    after = [x for x in g.cache_numpy() if x is not None]
    # sequences 0 and 2 took their (tripled) new rows; sequence 1 wrote nothing
    changed = [np.any(a != b, axis=tuple(range(1, a.ndim))) for a, b in zip(after, before)]
    bad_blocks = {int(wl.block_table[s, (n - 1) // wl.block_size])}
    for s2 in (0, 2):
        n2 = int(wl.context_lens[s2])
        blk = int(wl.block_table[s2, (n2 - 1) // wl.block_size])
        assert changed[0][blk]
    assert not any(c[b] for c in changed for b in bad_blocks)
