"""Shared helpers for the parity tests: run a workload through the CUDA
library and, independently, through the CPU oracle on the same inputs."""
from __future__ import annotations

import numpy as np
import torch

from oracle import attention as OA
from oracle import cache as OC
from oracle import formats as OF
from quantized_paged_kv_kvq_gb300 import kvq
from quantized_paged_kv_kvq_gb300 import workloads as W

# attention tolerance of the float64 oracle comparison (max-abs, mean-abs)
TOL_MAX = 2e-2
TOL_MEAN = 2e-3
QMAX = {"absmax/127": 127.0, "absmax/448": 448.0}


def bf16(x: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(device).to(torch.bfloat16)


def gpu_scale(x_dev: torch.Tensor, rule) -> float:
    """Per-tensor scale computed by the library's calibration kernel."""
    if rule is None or rule == "1.0":
        return 1.0
    out = torch.empty(1, dtype=torch.float32, device=x_dev.device)
    kvq.kvq_calibrate_scale(x_dev.reshape(-1), QMAX[rule], out)
    return float(out.item())


def oracle_scale(x: np.ndarray, rule) -> np.float32:
    if rule is None:
        return np.float32(1.0)
    return OF.calibrate(x, rule)


class GpuRun:
    """Device tensors of a workload plus the library's cache after the write."""

    def __init__(self, wl: W.Workload, fill: int = 0xAA, device="cuda", head_scales=False):
        self.wl = wl
        self.key = bf16(wl.key, device)
        self.value = bf16(wl.value, device)
        self.query = bf16(wl.query, device)
        self.slots = torch.from_numpy(wl.slot_mapping).to(device)
        self.block_table = torch.from_numpy(wl.block_table).to(device)
        self.context_lens = torch.from_numpy(wl.context_lens).to(device)
        self.signs = None if wl.signs is None else torch.from_numpy(
            np.ascontiguousarray(wl.signs)).to(device)
        self.k_scale = gpu_scale(self.key, wl.k_scale_rule)
        self.v_scale = gpu_scale(self.value, wl.v_scale_rule)
        self.cache = kvq.alloc_kv_cache(wl.k_fmt, wl.v_fmt, wl.num_blocks, wl.block_size,
                                        wl.num_kv_heads, wl.head_dim, self.k_scale, self.v_scale,
                                        wl.kvarn, self.signs, device=device, fill=fill)
        if head_scales:  # per-kv-head scales, calibrated on the GPU
            qmax = {"absmax/127": 127.0, "absmax/448": 448.0}
            for x, rule, attr in ((self.key, wl.k_scale_rule, "k_head_scales"),
                                  (self.value, wl.v_scale_rule, "v_head_scales")):
                if rule in qmax:
                    hs = torch.empty(wl.num_kv_heads, dtype=torch.float32, device=device)
                    kvq.kvq_calibrate_head_scales(x, qmax[rule], hs)
                    setattr(self.cache, attr, hs)

    def write(self):
        kvq.kvq_write_cache(self.cache, self.key, self.value, self.slots)

    def decode(self, num_ctas: int = 0, sm_scale=None, out=None) -> torch.Tensor:
        wl = self.wl
        sm = float(OA.default_sm_scale(wl.head_dim)) if sm_scale is None else sm_scale
        nbytes = kvq.kvq_decode_workspace_size(self.cache, wl.num_seqs, wl.num_q_heads,
                                               wl.max_context_len, num_ctas)
        # arbitrary bytes: the counters inside must not depend on the contents
        ws = torch.empty(max(nbytes, 16) // 4 + 4, dtype=torch.float32, device=self.query.device)
        ws.view(torch.int32).random_()
        if out is None:
            out = torch.empty_like(self.query)
        kvq.kvq_paged_decode(self.cache, self.query, out, self.block_table, self.context_lens,
                             wl.max_context_len, sm, ws, num_ctas)
        return out

    def cache_numpy(self):
        c = self.cache
        km = None if c.k_meta is None else c.k_meta.view(torch.int16).cpu().numpy().view(np.uint16)
        vm = None if c.v_meta is None else c.v_meta.view(torch.int16).cpu().numpy().view(np.uint16)
        return c.k_cache.cpu().numpy(), km, c.v_cache.cpu().numpy(), vm


class OracleRun:
    """The oracle's own cache for (a subset of the tokens of) a workload."""

    def __init__(self, wl: W.Workload, seqs=None, fill: int = 0xAA, head_scales=False):
        self.wl = wl
        self.k_scale = oracle_scale(wl.key, wl.k_scale_rule)
        self.v_scale = oracle_scale(wl.value, wl.v_scale_rule)
        if head_scales:  # per-kv-head scales where the format is calibrated
            if wl.k_scale_rule not in (None, "1.0"):
                self.k_scale = OF.calibrate_heads(wl.key, wl.k_scale_rule)
            if wl.v_scale_rule not in (None, "1.0"):
                self.v_scale = OF.calibrate_heads(wl.value, wl.v_scale_rule)
        kc, km = OC.alloc_cache(wl.num_blocks, wl.block_size, wl.num_kv_heads, wl.head_dim,
                                wl.k_fmt, wl.kvarn, fill)
        vc, vm = OC.alloc_cache(wl.num_blocks, wl.block_size, wl.num_kv_heads, wl.head_dim,
                                wl.v_fmt, wl.kvarn, fill)
        if seqs is None:
            sel = slice(None)
            key, value, slots = wl.key, wl.value, wl.slot_mapping
        else:
            starts = np.concatenate([[0], np.cumsum(wl.context_lens)])
            idx = np.concatenate([np.arange(starts[s], starts[s + 1]) for s in seqs])
            key, value, slots = wl.key[idx], wl.value[idx], wl.slot_mapping[idx]
        OC.write_cache(kc, km, key, slots, wl.block_size, wl.k_fmt, self.k_scale, wl.kvarn,
                       wl.signs)
        OC.write_cache(vc, vm, value, slots, wl.block_size, wl.v_fmt, self.v_scale, wl.kvarn,
                       wl.signs)
        self.kc, self.km, self.vc, self.vm = kc, km, vc, vm

    def decode(self, pairs=None, sm_scale=None) -> np.ndarray:
        wl = self.wl
        sm = OA.default_sm_scale(wl.head_dim) if sm_scale is None else sm_scale
        return OA.paged_decode(wl.query, self.kc, self.km, self.vc, self.vm, wl.block_table,
                               wl.context_lens, wl.block_size, wl.k_fmt, wl.v_fmt, self.k_scale,
                               self.v_scale, sm, wl.kvarn, wl.signs, pairs=pairs)


def random_workspace(g, num_ctas):
    wl = g.wl
    n = kvq.kvq_decode_workspace_size(g.cache, wl.num_seqs, wl.num_q_heads, wl.max_context_len,
                                      num_ctas)
    ws = torch.empty(max(n, 16) // 4 + 4, dtype=torch.float32, device=g.key.device)
    ws.view(torch.int32).random_()  # contents on entry must not matter
    return ws


def new_token_rows(wl):
    """Token index of each sequence's last position (0 where the sequence is empty)."""
    lens = wl.context_lens.astype(np.int64)
    last = np.cumsum(lens) - 1
    has = lens > 0
    return np.where(has, last, 0), has


def append_step(wl, num_ctas=0, head_scales=False):
    """Cache write of every token but each sequence's last, then one
    kvq_decode_append call with the last tokens; returns (GpuRun, out)."""
    g = GpuRun(wl, head_scales=head_scales)
    rows, has = new_token_rows(wl)
    slots = wl.slot_mapping.copy()
    slots[rows[has]] = -1
    dev = g.key.device
    kvq.kvq_write_cache(g.cache, g.key, g.value, torch.from_numpy(slots).to(dev))
    r = torch.from_numpy(rows).to(dev)
    new_k, new_v = g.key[r].contiguous(), g.value[r].contiguous()
    out = torch.empty_like(g.query)
    kvq.kvq_decode_append(g.cache, new_k, new_v, g.query, out, g.block_table, g.context_lens,
                          wl.max_context_len, float(OA.default_sm_scale(wl.head_dim)),
                          random_workspace(g, num_ctas), num_ctas)
    return g, out


def blocks_of(wl: W.Workload, seqs) -> np.ndarray:
    out = []
    for s in seqs:
        n = (int(wl.context_lens[s]) + wl.block_size - 1) // wl.block_size
        out.append(wl.block_table[s, :n])
    return np.concatenate(out) if out else np.zeros(0, np.int32)


def assert_attention_close(got: np.ndarray, ref: np.ndarray, what: str = ""):
    err = np.abs(got.astype(np.float64) - ref)
    mx, mean = float(err.max()) if err.size else 0.0, float(err.mean()) if err.size else 0.0
    assert mx <= TOL_MAX and mean <= TOL_MEAN, f"{what}: max-abs {mx:.3e}, mean-abs {mean:.3e}"
    return mx, mean


def out_numpy(out: torch.Tensor) -> np.ndarray:
    return out.float().cpu().numpy().astype(np.float64)
