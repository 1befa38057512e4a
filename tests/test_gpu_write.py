"""Cache-write parity on the GPU: codes and metadata bit-exact vs the oracle."""
import numpy as np
import pytest
import torch

from oracle import cache as OC
from oracle import formats as OF
from quantized_paged_kv_kvq_gb300 import kvq
from quantized_paged_kv_kvq_gb300 import workloads as W

from kvq_testing import GpuRun, OracleRun, bf16, blocks_of

pytestmark = pytest.mark.gpu

SMALL = {
    "tiny_int8": dict(),
    "llama8b_int8": dict(num_seqs=5, ctx_lo=1, ctx_hi=300),
    "llama8b_e4m3k_int8v": dict(num_seqs=5, ctx_lo=1, ctx_hi=300),
    "llama8b_e5m2": dict(num_seqs=5, ctx_lo=1, ctx_hi=300),
    "llama70b_int4": dict(num_seqs=4, ctx_lo=1, ctx_hi=300),
    "kvarn_131k": dict(num_seqs=3, ctx_lo=1, ctx_hi=300),
    "llama8b_bf16": dict(num_seqs=5, ctx_lo=1, ctx_hi=300),
}


@pytest.mark.parametrize("name", list(SMALL))
def test_write_bitexact_small(name):
    wl = W.workload(name, **SMALL[name])
    g = GpuRun(wl)
    o = OracleRun(wl)
    assert np.float32(g.k_scale) == o.k_scale and np.float32(g.v_scale) == o.v_scale
    g.write()
    kc, km, vc, vm = g.cache_numpy()
    assert np.array_equal(kc, o.kc), "K codes"
    assert np.array_equal(vc, o.vc), "V codes"
    if o.km.shape[2]:
        assert np.array_equal(km, o.km), "K meta"
        assert np.array_equal(vm, o.vm), "V meta"
    assert kvq.kvq_get_device_error() == 0


# More kv-heads than one warp pass holds: a token's rows take several passes,
# which the write spreads over different warps (head_dim 128: 8 rows a pass, so
# 24 rows are three passes; head_dim 64: 16 rows a pass, so the first pass
# holds K and V rows and the second is partly empty).
MANY_HEADS = {
    "kvarn_d128_12heads": ("kvarn_131k", dict(num_q_heads=12, num_kv_heads=12)),
    "kvarn_d64_12heads": ("kvarn_131k", dict(num_q_heads=12, num_kv_heads=12, head_dim=64)),
    "int4_d128_12heads": ("llama70b_int4", dict(num_q_heads=12, num_kv_heads=12)),
}


@pytest.mark.parametrize("shape", list(MANY_HEADS))
def test_write_bitexact_many_heads(shape):
    name, kw = MANY_HEADS[shape]
    wl = W.workload(name, **dict(kw, num_seqs=3, ctx_lo=1, ctx_hi=300))
    g = GpuRun(wl)
    o = OracleRun(wl)
    g.write()
    kc, km, vc, vm = g.cache_numpy()
    assert np.array_equal(kc, o.kc) and np.array_equal(vc, o.vc), f"{shape}: codes"
    assert np.array_equal(km, o.km) and np.array_equal(vm, o.vm), f"{shape}: meta"
    assert kvq.kvq_get_device_error() == 0


def _all_bf16_finite():
    bits = np.arange(1 << 16, dtype=np.uint32) << 16
    x = bits.view(np.float32)
    return np.where(np.isfinite(x), x, 0).astype(np.float32)


@pytest.mark.parametrize("fmt", ["fp8_e4m3", "fp8_e5m2", "int8"])
@pytest.mark.parametrize("scale", [1.0, 0.0371, 3.0e-3])
def test_write_every_bf16_value(fmt, scale):
    """All 65536 bf16 bit patterns (non-finite ones replaced by 0) through the
    cache write, against the oracle's formula."""
    x = _all_bf16_finite().reshape(512, 1, 128)
    t = x.shape[0]
    nb = t // 16
    slots = np.arange(t, dtype=np.int64)
    cache = kvq.alloc_kv_cache(fmt, fmt, nb, 16, 1, 128, scale, scale, fill=0)
    xd = bf16(x)
    with np.errstate(over="ignore"):
        kvq.kvq_write_cache(cache, xd, xd, torch.from_numpy(slots).cuda())
        kc = cache.k_cache.cpu().numpy().reshape(t, 128)
        inv = OF.inverse_scale(np.float32(scale))
        ref = (OF.quant_int8(x.reshape(t, 128), inv) if fmt == "int8"
               else OF.quant_fp8(x.reshape(t, 128), inv, fmt))
    bad = np.nonzero(kc != ref)
    assert bad[0].size == 0, (
        f"{bad[0].size} mismatches, first input {x.reshape(t, 128)[bad][:4]}, "
        f"gpu {kc[bad][:4]}, oracle {ref[bad][:4]}")


def test_write_asym_all_bf16_rows():
    """Asymmetric codes on rows cut from every bf16 value of moderate size."""
    x = _all_bf16_finite()
    x = x[(np.abs(x) < 1e4) & (np.abs(x) > 1e-30)][:32768 * 2]
    x = x[: (x.size // 128) * 128].reshape(-1, 1, 128)
    rng = np.random.default_rng(0)
    x = x[:, :, rng.permutation(128)]
    t = x.shape[0] - x.shape[0] % 16
    x = np.ascontiguousarray(x[:t])
    slots = np.arange(t, dtype=np.int64)
    for fmt in ("int4_asym", "uint8_asym"):
        cache = kvq.alloc_kv_cache(fmt, fmt, t // 16, 16, 1, 128, fill=0)
        xd = bf16(x)
        kvq.kvq_write_cache(cache, xd, xd, torch.from_numpy(slots).cuda())
        kc, km = OC.alloc_cache(t // 16, 16, 1, 128, fmt, False, 0)
        OC.write_cache(kc, km, x, slots, 16, fmt, 1.0)
        assert np.array_equal(cache.k_cache.cpu().numpy(), kc)
        assert np.array_equal(cache.k_meta.view(torch.int16).cpu().numpy().view(np.uint16), km)


def test_calibrate_matches_oracle():
    rng = np.random.default_rng(3)
    for n in (1, 7, 8, 1000, 123457):
        x = W.round_to_bf16((rng.standard_normal(n) * rng.uniform(0.01, 100)).astype(np.float32))
        out = torch.empty(1, dtype=torch.float32, device="cuda")
        for rule, qmax in (("absmax/127", 127.0), ("absmax/448", 448.0)):
            kvq.kvq_calibrate_scale(bf16(x), qmax, out)
            assert np.float32(out.item()) == OF.calibrate(x, rule)
    kvq.kvq_calibrate_scale(bf16(np.zeros(64, np.float32)), 127.0, out)
    assert out.item() == 1.0


def test_negative_slots_skip_and_bad_slots_flag():
    wl = W.workload("tiny_int8")
    g = GpuRun(wl, fill=0x5C)
    slots = wl.slot_mapping.copy()
    slots[::3] = -1
    slots[1] = wl.num_blocks * wl.block_size + 5  # past the cache: skipped, flagged
    kvq.kvq_write_cache(g.cache, g.key, g.value, torch.from_numpy(slots).cuda())
    assert kvq.kvq_get_device_error() & kvq.DEVERR_SLOT_RANGE
    assert kvq.kvq_get_device_error() == 0  # read clears
    kc = g.cache.k_cache.cpu().numpy()
    skipped = wl.slot_mapping[::3]
    assert np.all(kc[skipped // 16, skipped % 16] == 0x5C)
    assert np.all(kc[wl.slot_mapping[1] // 16, wl.slot_mapping[1] % 16] == 0x5C)
    o = OracleRun(wl, fill=0x5C)
    ok = slots >= 0
    ok[1] = False
    kc_o, _ = OC.alloc_cache(wl.num_blocks, 16, wl.num_kv_heads, wl.head_dim, "int8", False, 0x5C)
    OC.write_cache(kc_o, np.zeros((wl.num_blocks, wl.num_kv_heads, 0, 16), np.uint16),
                   wl.key[ok], wl.slot_mapping[ok], 16, "int8", o.k_scale)
    assert np.array_equal(kc, kc_o)


def test_strided_key_value_views():
    """key/value as views of a fused [T, 2*Hkv*D] buffer (token stride 2*Hkv*D)."""
    wl = W.workload("llama8b_int8", num_seqs=3, ctx_lo=10, ctx_hi=80)
    g = GpuRun(wl)
    t, h, d = wl.key.shape
    fused = torch.cat([g.key.reshape(t, h * d), g.value.reshape(t, h * d)], dim=1)
    kview = fused[:, : h * d].view(t, h, d)
    vview = fused[:, h * d:].view(t, h, d)
    assert kview.stride(0) == 2 * h * d
    kvq.kvq_write_cache(g.cache, kview, vview, g.slots)
    o = OracleRun(wl)
    kc, _, vc, _ = g.cache_numpy()
    assert np.array_equal(kc, o.kc) and np.array_equal(vc, o.vc)


@pytest.mark.parametrize("name", ["llama8b_int8", "kvarn_131k"])
def test_write_full_size_sampled(name):
    """Full-size workload written in one launch; a sample of sequences checked
    bit-exact against the oracle (which writes only those sequences)."""
    wl = W.workload(name)
    g = GpuRun(wl)
    g.write()
    torch.cuda.synchronize()
    rng = np.random.default_rng(1)
    seqs = sorted(rng.choice(wl.num_seqs, size=min(3, wl.num_seqs), replace=False).tolist())
    o = OracleRun(wl, seqs=seqs)
    blks = torch.from_numpy(blocks_of(wl, seqs).astype(np.int64)).cuda()
    kc = g.cache.k_cache[blks].cpu().numpy()
    vc = g.cache.v_cache[blks].cpu().numpy()
    bl = blocks_of(wl, seqs)
    assert np.array_equal(kc, o.kc[bl]) and np.array_equal(vc, o.vc[bl])
    if g.cache.k_meta is not None:
        km = g.cache.k_meta[blks].view(torch.int16).cpu().numpy().view(np.uint16)
        vm = g.cache.v_meta[blks].view(torch.int16).cpu().numpy().view(np.uint16)
        assert np.array_equal(km, o.km[bl]) and np.array_equal(vm, o.vm[bl])
    assert kvq.kvq_get_device_error() == 0


@pytest.mark.parametrize("name", ["llama8b_int8", "llama8b_e4m3k_int8v", "tiny_int8"])
def test_per_head_scales_calibration_and_codes_bit_exact(name):
    """Per-kv-head scales: the GPU calibration equals the oracle's per head, and
    the codes written with them equal the oracle's."""
    wl = W.workload(name, num_seqs=3, ctx_lo=20, ctx_hi=300)
    g = GpuRun(wl, head_scales=True)
    o = OracleRun(wl, head_scales=True)
    for attr, ref in (("k_head_scales", o.k_scale), ("v_head_scales", o.v_scale)):
        got = getattr(g.cache, attr)
        assert got is not None and np.array_equal(got.cpu().numpy(), np.asarray(ref, np.float32))
    g.write()
    kc, _, vc, _ = g.cache_numpy()
    assert np.array_equal(kc, o.kc) and np.array_equal(vc, o.vc)
    assert kvq.kvq_get_device_error() == 0


@pytest.mark.parametrize("name", ["kvarn_131k", "llama8b_int8"])
def test_prefill_chunk_write_bit_exact(name):
    """A prefill chunk (new tokens over sequence 0's first pages, as the long-context
    shape's chunked prefill writes them) lands bit-exact over an existing cache."""
    wl = W.workload(name, num_seqs=2, ctx_lo=3000, ctx_hi=3000)
    pc = W.prefill_chunk(wl, 2048, seed=5)
    g = GpuRun(wl)
    o = OracleRun(wl)
    g.write()
    kvq.kvq_write_cache(g.cache, bf16(pc["key"]), bf16(pc["value"]),
                        torch.from_numpy(pc["slot_mapping"]).cuda())
    for codes, meta, x, fmt, sc in ((o.kc, o.km, pc["key"], wl.k_fmt, o.k_scale),
                                    (o.vc, o.vm, pc["value"], wl.v_fmt, o.v_scale)):
        OC.write_cache(codes, meta, x, pc["slot_mapping"], wl.block_size, fmt, sc, wl.kvarn,
                       wl.signs)
    kc, km, vc, vm = g.cache_numpy()
    assert np.array_equal(kc, o.kc) and np.array_equal(vc, o.vc)
    if o.km.shape[2]:
        assert np.array_equal(km, o.km) and np.array_equal(vm, o.vm)
    assert kvq.kvq_get_device_error() == 0
