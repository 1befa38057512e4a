"""Paged-decode parity on the GPU against the float64 oracle."""
import numpy as np
import pytest
import torch

from quantized_paged_kv_kvq_gb300 import kvq
from quantized_paged_kv_kvq_gb300 import workloads as W

from kvq_testing import GpuRun, OracleRun, assert_attention_close, out_numpy

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


@pytest.mark.parametrize("name", list(SMALL))
def test_decode_matches_oracle(name):
    wl = W.workload(name, **SMALL[name])
    g = GpuRun(wl)
    g.write()
    got = out_numpy(g.decode())
    ref = OracleRun(wl).decode()
    assert_attention_close(got, ref, name)
    assert kvq.kvq_get_device_error() == 0


@pytest.mark.parametrize("name", ["llama8b_int8", "llama70b_int4", "kvarn_131k",
                                  "llama8b_e4m3k_int8v", "llama8b_bf16"])
@pytest.mark.parametrize("ctas", [1, 3, 7, 64, 0])
def test_split_invariance(name, ctas):
    """1, 3, 7, 64 stream-K ranges (and the automatic count) agree with the
    oracle: sequences are whole, or split between several CTAs."""
    wl = W.workload(name, **dict(SMALL[name], ctx_lo=200, ctx_hi=2500))
    g = GpuRun(wl)
    g.write()
    got = out_numpy(g.decode(num_ctas=ctas))
    ref = OracleRun(wl).decode()
    assert_attention_close(got, ref, f"{name} ctas={ctas}")


@pytest.mark.parametrize("name", ["llama8b_int8", "kvarn_131k"])
@pytest.mark.parametrize("ctas", [33, 200])
def test_long_sequence_merges_in_two_levels(name, ctas):
    """One long sequence next to short ones, split over more than 32 ranges:
    the split results are merged team by team, then across teams."""
    lens = np.array([4000, 37, 1, 300], np.int32)
    wl = W.workload(name, num_seqs=len(lens), context_lens=lens)
    g = GpuRun(wl)
    g.write()
    got = out_numpy(g.decode(num_ctas=ctas))
    assert_attention_close(got, OracleRun(wl).decode(), f"{name} ctas={ctas}")
    assert kvq.kvq_get_device_error() == 0


@pytest.mark.parametrize("name", ["llama8b_int8", "llama70b_int4", "kvarn_131k", "tiny_int8",
                                  "llama8b_e5m2", "llama8b_bf16"])
def test_context_length_edge_cases(name):
    bs = W.WORKLOADS[name]["block_size"]
    lens = np.array([0, 1, bs - 1, bs, bs + 1, 15, 16, 17, 63, 64, 65, 0, 2 * bs + 3], np.int32)
    wl = W.workload(name, num_seqs=len(lens), context_lens=lens)
    g = GpuRun(wl)
    g.write()
    ref = OracleRun(wl).decode()
    for ctas in (0, 1, 5):
        got = out_numpy(g.decode(num_ctas=ctas))
        assert_attention_close(got, ref, f"{name} ctas={ctas}")
        assert np.all(got[lens == 0] == 0)


def test_block_permutation_gives_identical_output():
    wl = W.workload("llama8b_int8", num_seqs=4, ctx_lo=100, ctx_hi=600)
    g = GpuRun(wl)
    g.write()
    out1 = g.decode(num_ctas=5).clone()
    perm = torch.from_numpy(np.random.default_rng(2).permutation(wl.num_blocks)).cuda()
    kc2 = torch.empty_like(g.cache.k_cache)
    vc2 = torch.empty_like(g.cache.v_cache)
    kc2[perm] = g.cache.k_cache
    vc2[perm] = g.cache.v_cache
    g.cache.k_cache, g.cache.v_cache = kc2, vc2
    bt = g.block_table.long()
    g.block_table = torch.where(bt >= 0, perm[bt.clamp(min=0)], bt).int().contiguous()
    out2 = g.decode(num_ctas=5)
    assert torch.equal(out1, out2)


@pytest.mark.parametrize("name", ["llama8b_int8", "kvarn_131k", "llama70b_int4", "llama8b_bf16"])
def test_block_sizes_agree(name):
    """Pages of 8, 16, 32, 64 and 128 tokens: codes bit-exact with the oracle's
    cache of the same page size, outputs within tolerance and alike."""
    lens = np.array([33, 100, 257, 5, 300], np.int32)
    outs = []
    for bs in (8, 16, 32, 64, 128):
        wl = W.workload(name, num_seqs=len(lens), context_lens=lens, block_size=bs)
        g = GpuRun(wl)
        g.write()
        o = OracleRun(wl)
        kc, km, vc, vm = g.cache_numpy()
        assert np.array_equal(kc, o.kc) and np.array_equal(vc, o.vc), f"bs={bs}: codes differ"
        if km is not None:
            assert np.array_equal(km, o.km) and np.array_equal(vm, o.vm), f"bs={bs}: meta differs"
        for ctas in (0, 7):
            outs.append(out_numpy(g.decode(num_ctas=ctas)))
            assert_attention_close(outs[-1], o.decode(), f"{name} bs={bs} ctas={ctas}")
    for other in outs[1:]:
        assert_attention_close(outs[0], other, f"{name}: page sizes")
    assert kvq.kvq_get_device_error() == 0


SMALL_PAGE_SHAPES = {
    "int8_d64_2heads": ("tiny_int8", {}),
    "int4_d64_2heads": ("llama70b_int4", dict(num_q_heads=8, num_kv_heads=2, head_dim=64)),
    "kvarn_d128_2heads": ("kvarn_131k", dict(num_q_heads=8, num_kv_heads=2)),
    "kvarn_d64_2heads": ("kvarn_131k", dict(num_q_heads=8, num_kv_heads=2, head_dim=64)),
    "fp8_d128_4heads": ("llama8b_e4m3k_int8v", dict(num_q_heads=16, num_kv_heads=4)),
    "bf16_d128_2heads": ("llama8b_bf16", dict(num_q_heads=8, num_kv_heads=2)),
    "bf16_d64_2heads": ("llama8b_bf16", dict(num_q_heads=8, num_kv_heads=2, head_dim=64)),
}


@pytest.mark.parametrize("shape", list(SMALL_PAGE_SHAPES))
@pytest.mark.parametrize("bs", [8, 16])
def test_small_pages_few_heads(shape, bs):
    """8-token pages (a tile spans two pages; the second may be absent) and
    16-token pages with fewer than 8 kv-heads per CTA, around page edges."""
    name, kw = SMALL_PAGE_SHAPES[shape]
    lens = np.array([1, 7, 8, 9, 15, 16, 17, 24, 25, 0, 100, 333], np.int32)
    wl = W.workload(name, **dict(kw, num_seqs=len(lens), context_lens=lens, block_size=bs))
    g = GpuRun(wl)
    g.write()
    o = OracleRun(wl)
    kc, km, vc, vm = g.cache_numpy()
    assert np.array_equal(kc, o.kc) and np.array_equal(vc, o.vc), f"{shape} bs={bs}: codes"
    if km is not None:
        assert np.array_equal(km, o.km) and np.array_equal(vm, o.vm), f"{shape} bs={bs}: meta"
    ref = o.decode()
    for ctas in (1, 5, 0):
        got = out_numpy(g.decode(num_ctas=ctas))
        assert np.all(got[lens == 0] == 0)
        assert_attention_close(got, ref, f"{shape} bs={bs} ctas={ctas}")
    assert kvq.kvq_get_device_error() == 0


def test_bad_block_id_is_flagged_not_faulted():
    wl = W.workload("tiny_int8")
    g = GpuRun(wl)
    g.write()
    bt = g.block_table.clone()
    bt[0, 0] = wl.num_blocks + 100  # outside the cache
    g.block_table = bt
    g.decode()
    assert kvq.kvq_get_device_error() & kvq.DEVERR_BLOCK_RANGE
    assert kvq.kvq_get_device_error() == 0


def test_decode_is_deterministic():
    wl = W.workload("llama70b_int4", num_seqs=3, ctx_lo=500, ctx_hi=1500)
    g = GpuRun(wl)
    g.write()
    a = g.decode().clone()
    b = g.decode()
    assert torch.equal(a, b)


@pytest.mark.parametrize("name", ["llama8b_int8", "llama8b_e4m3k_int8v", "llama8b_e5m2",
                                  "llama70b_int4", "kvarn_131k", "llama8b_bf16"])
def test_decode_full_size_sampled(name):
    """The full-size workload, written and decoded in the launch configuration
    the benchmark times; a sample of (sequence, kv-head) pairs is computed by
    the oracle from its own cache of those sequences."""
    wl = W.workload(name)
    g = GpuRun(wl)
    g.write()
    got = out_numpy(g.decode())
    rng = np.random.default_rng(7)
    seqs = sorted(rng.choice(wl.num_seqs, size=min(2, wl.num_seqs), replace=False).tolist())
    heads = sorted(rng.choice(wl.num_kv_heads, size=2, replace=False).tolist())
    pairs = [(s, h) for s in seqs for h in heads]
    ref = OracleRun(wl, seqs=seqs).decode(pairs=pairs)
    gq = wl.gqa
    rows = [(s, h * gq + j) for s, h in pairs for j in range(gq)]
    sel_got = np.stack([got[s, q] for s, q in rows])
    sel_ref = np.stack([ref[s, q] for s, q in rows])
    assert_attention_close(sel_got, sel_ref, name)
    assert np.all(np.isfinite(got))
    assert kvq.kvq_get_device_error() == 0


@pytest.mark.parametrize("name", ["llama8b_int8", "llama8b_e4m3k_int8v"])
@pytest.mark.parametrize("ctas", [1, 7, 0])
def test_per_head_scales_decode(name, ctas):
    """Decode with per-kv-head scales matches the oracle with the same scales
    (and differs from the per-tensor result, so the scales are used)."""
    wl = W.workload(name, num_seqs=4, ctx_lo=50, ctx_hi=700)
    g = GpuRun(wl, head_scales=True)
    g.write()
    got = out_numpy(g.decode(num_ctas=ctas))
    assert_attention_close(got, OracleRun(wl, head_scales=True).decode(), f"{name} ctas={ctas}")
    assert kvq.kvq_get_device_error() == 0


@pytest.mark.parametrize("name", ["llama8b_int8", "kvarn_131k", "llama8b_bf16"])
def test_query_out_of_range_is_flagged(name):
    """A query value beyond what the decode's query conversion holds (fp16's
    65504 for the quantized formats; an infinity for the 16-bit cache) sets
    KVQ_DEVERR_QUERY_RANGE; a query in range sets nothing."""
    wl = W.workload(name, num_seqs=3, ctx_lo=50, ctx_hi=300)
    g = GpuRun(wl)
    g.write()
    g.decode(num_ctas=2)
    assert kvq.kvq_get_device_error() == 0
    big = 1.0e6 if name != "llama8b_bf16" else float("inf")
    g.query[1, 0, 5] = big
    g.decode(num_ctas=2)
    assert kvq.kvq_get_device_error() & kvq.DEVERR_QUERY_RANGE
