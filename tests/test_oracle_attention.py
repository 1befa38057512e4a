"""Pins for the oracle's cache scatter and float64 paged attention (CPU only)."""
import numpy as np
import pytest
import scipy.special

from oracle import attention as A
from oracle import cache as C
from oracle import formats as F
from quantized_paged_kv_kvq_gb300 import workloads as W


def _write_all(wl, scale_k=None, scale_v=None):
    kc, km = C.alloc_cache(wl.num_blocks, wl.block_size, wl.num_kv_heads, wl.head_dim,
                           wl.k_fmt, wl.kvarn)
    vc, vm = C.alloc_cache(wl.num_blocks, wl.block_size, wl.num_kv_heads, wl.head_dim,
                           wl.v_fmt, wl.kvarn)
    ks = scale_k if scale_k is not None else (
        F.calibrate(wl.key, wl.k_scale_rule) if wl.k_scale_rule else np.float32(1))
    vs = scale_v if scale_v is not None else (
        F.calibrate(wl.value, wl.v_scale_rule) if wl.v_scale_rule else np.float32(1))
    C.write_cache(kc, km, wl.key, wl.slot_mapping, wl.block_size, wl.k_fmt, ks, wl.kvarn, wl.signs)
    C.write_cache(vc, vm, wl.value, wl.slot_mapping, wl.block_size, wl.v_fmt, vs, wl.kvarn,
                  wl.signs)
    return kc, km, vc, vm, ks, vs


def _decode(wl, kc, km, vc, vm, ks, vs, table=None):
    return A.paged_decode(wl.query, kc, km, vc, vm, wl.block_table if table is None else table,
                          wl.context_lens, wl.block_size, wl.k_fmt, wl.v_fmt, ks, vs,
                          A.default_sm_scale(wl.head_dim), wl.kvarn, wl.signs)


def small(name, **kw):
    base = dict(num_seqs=3, ctx_lo=1, ctx_hi=70)
    if name == "kvarn_131k":
        base.update(ctx_lo=1, ctx_hi=90)
    base.update(kw)
    return W.workload(name, **base)


NAMES = ["tiny_int8", "llama8b_int8", "llama8b_e4m3k_int8v", "llama8b_e5m2",
         "llama70b_int4", "kvarn_131k"]


@pytest.mark.parametrize("name", NAMES)
def test_paged_equals_dense_bruteforce(name):
    """Dequantize each sequence into a dense array by walking tokens one by one,
    then run textbook attention with scipy's softmax."""
    wl = small(name)
    kc, km, vc, vm, ks, vs = _write_all(wl)
    out = _decode(wl, kc, km, vc, vm, ks, vs)
    g = wl.gqa
    sm = float(A.default_sm_scale(wl.head_dim))
    for s in range(wl.num_seqs):
        ctx = int(wl.context_lens[s])
        for h in range(wl.num_kv_heads):
            krows, vrows = [], []
            for t in range(ctx):
                slot = int(wl.block_table[s, t // wl.block_size]) * wl.block_size + t % wl.block_size
                b, o = divmod(slot, wl.block_size)
                krows.append(C.decode_rows(kc[b, o, h][None], km[b, h, :, o][None], wl.k_fmt, ks,
                                           wl.kvarn, wl.signs, wl.head_dim)[0])
                vrows.append(C.decode_rows(vc[b, o, h][None], vm[b, h, :, o][None], wl.v_fmt, vs,
                                           wl.kvarn, wl.signs, wl.head_dim)[0])
            k, v = np.array(krows), np.array(vrows)
            for j in range(g):
                q = wl.query[s, h * g + j].astype(np.float64)
                p = scipy.special.softmax(sm * (k @ q))
                np.testing.assert_allclose(out[s, h * g + j], p @ v, rtol=1e-12, atol=1e-12)


def test_written_rows_dequantize_close_to_inputs():
    for name in NAMES:
        wl = small(name)
        kc, km, vc, vm, ks, vs = _write_all(wl)
        for s in range(wl.num_seqs):
            ctx = int(wl.context_lens[s])
            start = int(wl.context_lens[:s].sum())
            k = A.dequant_sequence(kc, km, wl.block_table[s], ctx, wl.block_size, 0, wl.k_fmt, ks,
                                   wl.kvarn, wl.signs, wl.head_dim)
            ref = wl.key[start:start + ctx, 0].astype(np.float64)
            rel = np.linalg.norm(k - ref) / max(np.linalg.norm(ref), 1e-30)
            # int4 with outlier channels is coarse; e5m2 keeps 2 mantissa bits
            bound = {"int4_asym": 0.3, "fp8_e5m2": 0.1}.get(wl.k_fmt, 0.07)
            assert rel < bound, (name, rel)


def test_unwritten_slots_keep_poison():
    wl = small("llama70b_int4")
    kc, km, vc, vm, _, _ = _write_all(wl)
    used = np.zeros((wl.num_blocks, wl.block_size), bool)
    used[wl.slot_mapping // wl.block_size, wl.slot_mapping % wl.block_size] = True
    assert np.all(kc[~used] == 0xAA)
    assert np.all(km.transpose(0, 3, 1, 2)[~used] == 0xAAAA)
    assert not np.any(np.all(kc[used] == 0xAA, axis=(-1, -2)))


def test_negative_slots_are_skipped():
    wl = small("tiny_int8")
    slots = wl.slot_mapping.copy()
    slots[::2] = -1
    kc, km = C.alloc_cache(wl.num_blocks, wl.block_size, wl.num_kv_heads, wl.head_dim, "int8", False)
    C.write_cache(kc, km, wl.key, slots, wl.block_size, "int8", np.float32(0.05))
    skipped = wl.slot_mapping[::2]
    assert np.all(kc[skipped // wl.block_size, skipped % wl.block_size] == 0xAA)


def test_single_token_context_returns_its_value():
    wl = small("llama8b_int8", context_lens=np.array([1, 1, 1]))
    kc, km, vc, vm, ks, vs = _write_all(wl)
    out = _decode(wl, kc, km, vc, vm, ks, vs)
    for s in range(3):
        for h in range(wl.num_kv_heads):
            v0 = A.dequant_sequence(vc, vm, wl.block_table[s], 1, wl.block_size, h, "int8", vs,
                                    False, None, wl.head_dim)[0]
            for j in range(wl.gqa):
                assert np.array_equal(out[s, h * wl.gqa + j], v0)


def test_equal_keys_average_values_and_dominant_key_wins():
    wl = small("llama8b_int8", context_lens=np.array([40, 33, 17]))
    wl.key[:] = wl.key[0]  # all keys identical
    kc, km, vc, vm, ks, vs = _write_all(wl)
    out = _decode(wl, kc, km, vc, vm, ks, vs)
    for s in range(3):
        ctx = int(wl.context_lens[s])
        v = A.dequant_sequence(vc, vm, wl.block_table[s], ctx, wl.block_size, 2, "int8", vs,
                               False, None, wl.head_dim)
        np.testing.assert_allclose(out[s, 2 * wl.gqa], v.mean(axis=0), rtol=1e-12, atol=1e-12)
    # a key aligned with the query and 1000x larger takes all the weight
    wl = small("llama8b_int8", context_lens=np.array([40, 33, 17]))
    start = int(wl.context_lens[:1].sum())
    wl.key[start + 5, 0] = W.round_to_bf16(wl.query[1, 0] * 1000.0)
    kc, km, vc, vm, ks, vs = _write_all(wl)
    out = _decode(wl, kc, km, vc, vm, ks, vs)
    v = A.dequant_sequence(vc, vm, wl.block_table[1], 33, wl.block_size, 0, "int8", vs, False,
                           None, wl.head_dim)
    np.testing.assert_allclose(out[1, 0], v[5], atol=1e-9)


def test_block_table_permutation_invariance():
    wl = small("llama8b_e4m3k_int8v")
    kc, km, vc, vm, ks, vs = _write_all(wl)
    out = _decode(wl, kc, km, vc, vm, ks, vs)
    rng = np.random.default_rng(5)
    perm = rng.permutation(wl.num_blocks)  # block b moves to perm[b]
    kc2, vc2 = np.empty_like(kc), np.empty_like(vc)
    kc2[perm], vc2[perm] = kc, vc
    km2, vm2 = np.empty_like(km), np.empty_like(vm)
    km2[perm], vm2[perm] = km, vm
    table = np.where(wl.block_table >= 0, perm[np.maximum(wl.block_table, 0)], -1)
    out2 = _decode(wl, kc2, km2, vc2, vm2, ks, vs, table=table)
    assert np.array_equal(out, out2)


def test_empty_context_gives_zero():
    wl = small("tiny_int8", context_lens=np.array([0, 5, 0]))
    kc, km, vc, vm, ks, vs = _write_all(wl)
    out = _decode(wl, kc, km, vc, vm, ks, vs)
    assert np.all(out[0] == 0) and np.all(out[2] == 0) and np.any(out[1] != 0)


def test_mixed_page_classes_give_the_single_class_result():
    from oracle import attention as OA
    """Attention does not depend on page sizes: the same tokens written into two
    pools of 16- and 64-token pages (each sequence in one pool) decode to
    exactly the result of one pool of 16-token pages, and the layout puts every
    token at its own slot of its own class."""
    from oracle import cache as OC
    from oracle import formats as OF
    from quantized_paged_kv_kvq_gb300 import workloads as W
    for name in ("llama8b_int8", "llama70b_int4", "kvarn_131k"):
        wl = W.workload(name, num_seqs=5, ctx_lo=1, ctx_hi=150, num_q_heads=8, num_kv_heads=2)
        mp = W.mixed_pages(wl, (16, 64))
        assert set(np.unique(mp["seq_class"])) <= {0, 1}
        for c, bs in enumerate(mp["block_sizes"]):  # slots are distinct and inside the pool
            assert np.unique(mp["slots"][c]).size == mp["slots"][c].size
            assert mp["slots"][c].size == 0 or mp["slots"][c].max() < mp["num_blocks"][c] * bs
        ks = OF.calibrate(wl.key, wl.k_scale_rule) if wl.k_scale_rule else np.float32(1)
        vs = OF.calibrate(wl.value, wl.v_scale_rule) if wl.v_scale_rule else np.float32(1)
        classes = []
        for c, bs in enumerate(mp["block_sizes"]):
            kc, km = OC.alloc_cache(mp["num_blocks"][c], bs, 2, wl.head_dim, wl.k_fmt, wl.kvarn)
            vc, vm = OC.alloc_cache(mp["num_blocks"][c], bs, 2, wl.head_dim, wl.v_fmt, wl.kvarn)
            t = mp["tokens"][c]
            OC.write_cache(kc, km, wl.key[t], mp["slots"][c], bs, wl.k_fmt, ks, wl.kvarn, wl.signs)
            OC.write_cache(vc, vm, wl.value[t], mp["slots"][c], bs, wl.v_fmt, vs, wl.kvarn,
                           wl.signs)
            classes.append((kc, km, vc, vm, bs))
        sm = OA.default_sm_scale(wl.head_dim)
        got = OA.paged_decode_classes(wl.query, classes, mp["seq_class"], mp["block_table"],
                                      wl.context_lens, wl.k_fmt, wl.v_fmt, ks, vs, sm, wl.kvarn,
                                      wl.signs)
        kc, km = OC.alloc_cache(wl.num_blocks, wl.block_size, 2, wl.head_dim, wl.k_fmt, wl.kvarn)
        vc, vm = OC.alloc_cache(wl.num_blocks, wl.block_size, 2, wl.head_dim, wl.v_fmt, wl.kvarn)
        OC.write_cache(kc, km, wl.key, wl.slot_mapping, wl.block_size, wl.k_fmt, ks, wl.kvarn,
                       wl.signs)
        OC.write_cache(vc, vm, wl.value, wl.slot_mapping, wl.block_size, wl.v_fmt, vs, wl.kvarn,
                       wl.signs)
        ref = OA.paged_decode(wl.query, kc, km, vc, vm, wl.block_table, wl.context_lens,
                              wl.block_size, wl.k_fmt, wl.v_fmt, ks, vs, sm, wl.kvarn, wl.signs)
        assert np.array_equal(got, ref), name
