"""A cache whose sequences use pages of different sizes (the KVarN article's
variable page sizes, section 'Perspective'): two pools, of 16- and 64-token
pages, each sequence in one of them.  Each pool is written with kvq_write_cache
(codes bit-exact against the oracle's pool), and kvq_decode_mixed decodes over
both (within the tolerance of the oracle, and bit-identical to the decode of
the same tokens in one pool of 16-token pages: a 16-token tile is the same
whatever page holds it) or runs the fused decode step with each sequence's new
token stored into its own pool."""
import numpy as np
import pytest
import torch

from oracle import attention as OA
from oracle import cache as OC
from quantized_paged_kv_kvq_gb300 import kvq
from quantized_paged_kv_kvq_gb300 import workloads as W

from kvq_testing import (GpuRun, OracleRun, assert_attention_close, bf16, gpu_scale,
                         oracle_scale, out_numpy, random_workspace)

pytestmark = pytest.mark.gpu

SHAPES = {
    "llama8b_int8": dict(num_seqs=7, ctx_lo=1, ctx_hi=700),
    "llama70b_int4": dict(num_seqs=5, ctx_lo=1, ctx_hi=900),
    "kvarn_131k": dict(num_seqs=4, ctx_lo=1, ctx_hi=900),
    "llama8b_bf16": dict(num_seqs=6, ctx_lo=1, ctx_hi=600),
}


class Mixed:
    """The GPU pools of a mixed-page layout, written from the workload's tokens
    (all of them, or all but each sequence's last)."""

    def __init__(self, wl, mp, drop_last=False):
        self.wl, self.mp = wl, mp
        self.key, self.value, self.query = bf16(wl.key), bf16(wl.value), bf16(wl.query)
        self.signs = None if wl.signs is None else torch.from_numpy(wl.signs).cuda()
        ks, vs = gpu_scale(self.key, wl.k_scale_rule), gpu_scale(self.value, wl.v_scale_rule)
        last = set((np.cumsum(wl.context_lens.astype(np.int64)) - 1).tolist())
        self.classes = []
        for c, bs in enumerate(mp["block_sizes"]):
            cache = kvq.alloc_kv_cache(wl.k_fmt, wl.v_fmt, mp["num_blocks"][c], bs,
                                       wl.num_kv_heads, wl.head_dim, ks, vs, wl.kvarn,
                                       self.signs, fill=0xAA)
            tok, slots = mp["tokens"][c], mp["slots"][c].copy()
            if drop_last:
                slots[np.isin(tok, list(last))] = -1
            if tok.size:
                t = torch.from_numpy(tok).cuda()
                kvq.kvq_write_cache(cache, self.key[t], self.value[t],
                                    torch.from_numpy(slots).cuda())
            self.classes.append(cache)
        self.seq_class = torch.from_numpy(mp["seq_class"]).cuda()
        self.table = torch.from_numpy(mp["block_table"]).cuda()
        self.lens = torch.from_numpy(wl.context_lens).cuda()

    def decode(self, num_ctas, new_rows=None):
        wl = self.wl
        n = kvq.kvq_decode_workspace_size(self.classes[0], wl.num_seqs, wl.num_q_heads,
                                          wl.max_context_len, num_ctas)
        ws = torch.empty(max(n, 16) // 4 + 4, dtype=torch.float32, device="cuda")
        ws.view(torch.int32).random_()
        out = torch.full_like(self.query, float("nan"))
        nk, nv = (None, None) if new_rows is None else new_rows
        kvq.kvq_decode_mixed(self.classes, self.seq_class, self.query, out, self.table,
                             self.lens, wl.max_context_len,
                             float(OA.default_sm_scale(wl.head_dim)), ws, num_ctas,
                             new_key=nk, new_value=nv)
        return out


def oracle_pools(wl, mp):
    ks, vs = oracle_scale(wl.key, wl.k_scale_rule), oracle_scale(wl.value, wl.v_scale_rule)
    pools = []
    for c, bs in enumerate(mp["block_sizes"]):
        kc, km = OC.alloc_cache(mp["num_blocks"][c], bs, wl.num_kv_heads, wl.head_dim, wl.k_fmt,
                                wl.kvarn)
        vc, vm = OC.alloc_cache(mp["num_blocks"][c], bs, wl.num_kv_heads, wl.head_dim, wl.v_fmt,
                                wl.kvarn)
        t = mp["tokens"][c]
        OC.write_cache(kc, km, wl.key[t], mp["slots"][c], bs, wl.k_fmt, ks, wl.kvarn, wl.signs)
        OC.write_cache(vc, vm, wl.value[t], mp["slots"][c], bs, wl.v_fmt, vs, wl.kvarn, wl.signs)
        pools.append((kc, km, vc, vm, bs))
    ref = OA.paged_decode_classes(wl.query, pools, mp["seq_class"], mp["block_table"],
                                  wl.context_lens, wl.k_fmt, wl.v_fmt, ks, vs,
                                  OA.default_sm_scale(wl.head_dim), wl.kvarn, wl.signs)
    return pools, ref


def assert_pools_equal(m, pools, what):
    for c, (kc, km, vc, vm, _) in enumerate(pools):
        g = m.classes[c]
        assert np.array_equal(g.k_cache.cpu().numpy(), kc), f"{what}: class {c} K codes"
        assert np.array_equal(g.v_cache.cpu().numpy(), vc), f"{what}: class {c} V codes"
        if g.k_meta is not None:
            gm = lambda t: t.view(torch.int16).cpu().numpy().view(np.uint16)
            assert np.array_equal(gm(g.k_meta), km), f"{what}: class {c} K meta"
            assert np.array_equal(gm(g.v_meta), vm), f"{what}: class {c} V meta"


@pytest.mark.parametrize("name", list(SHAPES))
def test_mixed_pages_write_and_decode(name):
    wl = W.workload(name, **SHAPES[name])
    mp = W.mixed_pages(wl, (16, 64))
    m = Mixed(wl, mp)
    pools, ref = oracle_pools(wl, mp)
    assert_pools_equal(m, pools, name)
    uniform = GpuRun(wl)
    uniform.write()
    for ctas in (0, 1, 7, 33):
        got = m.decode(ctas)
        assert_attention_close(out_numpy(got), ref, f"{name} ctas={ctas}")
        assert torch.equal(got.view(torch.int16), uniform.decode(num_ctas=ctas).view(torch.int16))
    assert kvq.kvq_get_device_error() == 0


@pytest.mark.parametrize("name", list(SHAPES))
def test_mixed_pages_fused_append(name):
    """Every token but each sequence's last written per pool; the decode step
    stores the last ones into their own pools and attends over all."""
    wl = W.workload(name, **SHAPES[name])
    mp = W.mixed_pages(wl, (16, 64))
    m = Mixed(wl, mp, drop_last=True)
    rows = np.where(wl.context_lens > 0, np.cumsum(wl.context_lens.astype(np.int64)) - 1, 0)
    r = torch.from_numpy(rows).cuda()
    got = m.decode(5, new_rows=(m.key[r].contiguous(), m.value[r].contiguous()))
    pools, ref = oracle_pools(wl, mp)
    assert_pools_equal(m, pools, f"{name} append")
    assert_attention_close(out_numpy(got), ref, f"{name} append")
    assert kvq.kvq_get_device_error() == 0


def test_bad_page_class_is_flagged_not_faulted():
    wl = W.workload("llama8b_int8", **SHAPES["llama8b_int8"])
    mp = W.mixed_pages(wl, (16, 64))
    m = Mixed(wl, mp)
    m.seq_class[0] = 9
    m.decode(3)
    assert kvq.kvq_get_device_error() & kvq.DEVERR_CLASS_RANGE
    assert kvq.kvq_get_device_error() == 0
