"""The decode calls recorded into a CUDA graph, as a serving loop records its
decode step, and replayed with new inputs.

A replay re-runs the recorded launch with the same arguments, so the
completion tags and merge claims it finds in the workspace are those of the
replay before it; a capturing call clears them first (a memset node).  Each
replay here is compared bit for bit with a direct call on the same inputs and
grid, over a grid whose ranges split sequences (merges in every replay)."""
import numpy as np
import pytest
import torch

from oracle import attention as OA
from quantized_paged_kv_kvq_gb300 import kvq
from quantized_paged_kv_kvq_gb300 import workloads as W

from kvq_testing import GpuRun, new_token_rows

pytestmark = pytest.mark.gpu

CTAS = 7


def workspace(g, ctas):
    wl = g.wl
    n = kvq.kvq_decode_workspace_size(g.cache, wl.num_seqs, wl.num_q_heads, wl.max_context_len,
                                      ctas)
    ws = torch.empty(max(n, 16) // 4 + 4, dtype=torch.float32, device="cuda")
    ws.view(torch.int32).random_()
    return ws


@pytest.mark.parametrize("name", ["llama8b_int8", "kvarn_131k"])
def test_decode_replayed_from_a_graph_matches_direct_calls(name):
    shape = dict(num_seqs=6, ctx_lo=300, ctx_hi=1500) if name != "kvarn_131k" else \
        dict(num_seqs=2, ctx_lo=3000, ctx_hi=3000)
    wl = W.workload(name, **shape)
    g = GpuRun(wl)
    g.write()
    sm = float(OA.default_sm_scale(wl.head_dim))
    q = g.query.clone()
    out = torch.empty_like(q)
    ws = workspace(g, CTAS)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):  # first use outside the capture
        kvq.kvq_paged_decode(g.cache, q, out, g.block_table, g.context_lens, wl.max_context_len,
                             sm, ws, CTAS)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        kvq.kvq_paged_decode(g.cache, q, out, g.block_table, g.context_lens, wl.max_context_len,
                             sm, ws, CTAS)
    gen = torch.Generator(device="cuda").manual_seed(11)
    for _ in range(4):
        q.copy_(torch.randn(q.shape, device="cuda", generator=gen).to(torch.bfloat16))
        graph.replay()
        torch.cuda.synchronize()
        ref = torch.empty_like(q)
        kvq.kvq_paged_decode(g.cache, q, ref, g.block_table, g.context_lens, wl.max_context_len,
                             sm, workspace(g, CTAS), CTAS)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    assert kvq.kvq_get_device_error() == 0


def test_append_step_replayed_from_a_graph():
    """The fused decode step in a graph: every replay stores the step's rows
    (the same slots, new values) and attends; equal to direct calls."""
    wl = W.workload("llama8b_int8", num_seqs=6, ctx_lo=300, ctx_hi=1500)
    g = GpuRun(wl)
    g.write()
    sm = float(OA.default_sm_scale(wl.head_dim))
    rows, _ = new_token_rows(wl)
    r = torch.from_numpy(rows).cuda()
    nk, nv = g.key[r].contiguous(), g.value[r].contiguous()
    q = g.query.clone()
    out = torch.empty_like(q)
    ws = workspace(g, CTAS)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        kvq.kvq_decode_append(g.cache, nk, nv, q, out, g.block_table, g.context_lens,
                              wl.max_context_len, sm, ws, CTAS)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        kvq.kvq_decode_append(g.cache, nk, nv, q, out, g.block_table, g.context_lens,
                              wl.max_context_len, sm, ws, CTAS)
    gen = torch.Generator(device="cuda").manual_seed(12)
    for _ in range(3):
        for t in (q, nk, nv):
            t.copy_(torch.randn(t.shape, device="cuda", generator=gen).to(torch.bfloat16))
        graph.replay()
        torch.cuda.synchronize()
        got_cache = (g.cache.k_cache.clone(), g.cache.v_cache.clone())
        ref = torch.empty_like(q)
        kvq.kvq_decode_append(g.cache, nk, nv, q, ref, g.block_table, g.context_lens,
                              wl.max_context_len, sm, workspace(g, CTAS), CTAS)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
        assert torch.equal(got_cache[0], g.cache.k_cache) and torch.equal(got_cache[1], g.cache.v_cache)
    assert kvq.kvq_get_device_error() == 0
