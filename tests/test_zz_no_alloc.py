"""kvq_paged_decode_static: the decode entry point for callers that cannot
allocate device memory (its split-K scratch is a fixed array inside the
library).  Kept in its own file, collected last, so that a stop-at-first-
failure run has already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

from quantized_paged_kv_kvq_gb300 import kvq
from quantized_paged_kv_kvq_gb300 import workloads as W

from kvq_testing import GpuRun, OracleRun, assert_attention_close, out_numpy

pytestmark = pytest.mark.gpu


def _static_decode(g, ctas):
    wl = g.wl
    out = torch.full_like(g.query, float("nan"))  # a stale or skipped output cannot pass
    sm = float(np.float32(1.0 / np.sqrt(wl.head_dim)))
    kvq.kvq_paged_decode_static(g.cache, g.query, out, g.block_table, g.context_lens,
                                wl.max_context_len, sm, ctas)
    torch.cuda.synchronize()
    return out


def test_static_scratch_decode_matches_workspace_decode_twice():
    cap = kvq.kvq_paged_decode_static_capacity()
    runs = [(W.workload("llama8b_int8", num_seqs=6, ctx_lo=300, ctx_hi=2000), 16),
            (W.workload("llama70b_int4", num_seqs=3, ctx_lo=100, ctx_hi=900), 7)]
    for wl, ctas in runs:  # two calls in a row, different shapes
        g = GpuRun(wl)
        g.write()
        need = kvq.kvq_decode_workspace_size(g.cache, wl.num_seqs, wl.num_q_heads,
                                             wl.max_context_len, ctas)
        assert 0 < need <= cap  # the call really goes through the scratch
        ref = out_numpy(g.decode(num_ctas=ctas))
        got = out_numpy(_static_decode(g, ctas))
        assert np.all(np.isfinite(got))
        assert_attention_close(got, ref, f"static vs workspace, {wl.name}")
    assert kvq.kvq_get_device_error() == 0


@pytest.mark.parametrize("ctas", [64, 0])
def test_static_scratch_long_sequence_against_oracle(ctas):
    """One long KVarN sequence over 64 ranges (more than 32: merged in two
    levels, whose team tags and claims sit deeper in the scratch) and over the
    automatic grid (a size that depends on the SM count), after the calls
    above have left their own contents in the scratch."""
    lens = np.array([8192], np.int32)
    wl = W.workload("kvarn_131k", num_seqs=1, context_lens=lens)
    g = GpuRun(wl)
    g.write()
    need = kvq.kvq_decode_workspace_size(g.cache, wl.num_seqs, wl.num_q_heads,
                                         wl.max_context_len, ctas)
    assert 0 < need <= kvq.kvq_paged_decode_static_capacity()
    got = out_numpy(_static_decode(g, ctas))
    assert np.all(np.isfinite(got))
    assert_attention_close(got, OracleRun(wl).decode(), f"static, kvarn 8192 tokens, ctas={ctas}")
    assert kvq.kvq_get_device_error() == 0


def test_static_scratch_rejects_sizes_beyond_capacity():
    lib = kvq.load_library()
    d = kvq._CacheDesc(1, 1, 8, 128, 16, 4096, 0, 0.1, 0.1, None, None, None)
    fake = 0x10000  # never dereferenced: the size check comes first
    # 4096 CTAs x 2 slots x 64 heads x 130 floats: far beyond 16 MiB
    st = lib.kvq_paged_decode_static(ctypes.byref(d), fake, fake, fake, fake, 2000, 64, fake,
                                     512, fake, 8192, 0.088, 4096, None)
    assert st == 3  # KVQ_ERR_WORKSPACE
