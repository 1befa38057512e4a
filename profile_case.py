"""Run one seeded workload's cache write and decode a few times on the GPU.

A small, fixed case for a profiler to capture (the bench's full-size workloads are
too large for a multi-pass capture):

  python profile_case.py kvarn_131k num_seqs=1 ctx_lo=32768 ctx_hi=32768

Arguments after the workload name override its generator settings (integers).
Everything goes through the library's public calls; nothing is checked here.
"""
from __future__ import annotations

import os
import sys

import numpy as np
import torch

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
from quantized_paged_kv_kvq_gb300 import build as kbuild  # noqa: E402
from quantized_paged_kv_kvq_gb300 import kvq  # noqa: E402
from quantized_paged_kv_kvq_gb300 import workloads as W  # noqa: E402


def run(name: str, repeats: int = 3, **overrides) -> None:
    kbuild.build()
    wl = W.workload(name, **overrides)
    dev = torch.device("cuda", 0)
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev).to(torch.bfloat16)
    key, value, query = bf(wl.key), bf(wl.value), bf(wl.query)
    slots = torch.from_numpy(wl.slot_mapping).to(dev)
    table = torch.from_numpy(wl.block_table).to(dev)
    lens = torch.from_numpy(wl.context_lens).to(dev)
    signs = None if wl.signs is None else torch.from_numpy(wl.signs).to(dev)
    qmax = {"absmax/127": 127.0, "absmax/448": 448.0}

    def scale(x, rule):
        if rule not in qmax:
            return 1.0
        o = torch.empty(1, dtype=torch.float32, device=dev)
        kvq.kvq_calibrate_scale(x.reshape(-1), qmax[rule], o)
        return float(o.item())

    cache = kvq.alloc_kv_cache(wl.k_fmt, wl.v_fmt, wl.num_blocks, wl.block_size,
                               wl.num_kv_heads, wl.head_dim, scale(key, wl.k_scale_rule),
                               scale(value, wl.v_scale_rule), wl.kvarn, signs, device=dev)
    out = torch.empty_like(query)
    sm = float(np.float32(1.0 / np.sqrt(wl.head_dim)))
    nbytes = kvq.kvq_decode_workspace_size(cache, wl.num_seqs, wl.num_q_heads,
                                           wl.max_context_len, 0)
    ws = torch.empty(max(nbytes, 16) // 4 + 4, dtype=torch.float32, device=dev)
    print(f"{name}: {wl.num_seqs} sequences, {wl.num_tokens} tokens")
    for _ in range(repeats):
        kvq.kvq_write_cache(cache, key, value, slots)
        kvq.kvq_paged_decode(cache, query, out, table, lens, wl.max_context_len, sm, ws, 0)
        torch.cuda.synchronize()
    print("device error bits:", kvq.kvq_get_device_error())


def main(argv=None) -> None:
    argv = sys.argv[1:] if argv is None else argv
    kw = {}
    for a in argv[1:]:
        k, v = a.split("=", 1)
        kw[k] = int(v)
    run(argv[0], **kw)


if __name__ == "__main__":
    main()
