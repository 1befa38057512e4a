#!/usr/bin/env python3
"""Benchmark of the quantized paged KV cache hot path on GB300.

One step = the whole path on one batch of synthetic input: quantize-and-
scatter every context token into the paged cache (kvq_write_cache, one
launch), then single-token paged decode over it (kvq_paged_decode, one
stream-K launch that also merges sequences split between CTAs).  Inputs are
resident in HBM before the timed region; L2 is flushed (a 2x-L2 memset, then a
2x-L2 read) before each of the two kernels, outside the CUDA-event pairs.
One JSON line on stdout (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the CPU oracle, as the reference arm

Multi-GPU (torchrun, one rank per GPU): every rank runs its own seeded
replica of the workload (independent sequences; no data-path collective),
barrier + max-over-ranks timing; value = bytes of all ranks / max time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

DEFAULT_WORKLOAD = "llama8b_int8"
METRIC = "quantized paged decode: effective KV GB/s vs HBM peak; decode & cache-write tok/s"
FALLBACK_HBM_GBS = 6800.0
# the kernel's own code (the instance units only list template arguments)
DECODE_SOURCES = ["decode.cuh", "decode_launch.cuh", "kvq_device.cuh", "quant_row.cuh"]
WRITE_SOURCES = ["write.cu", "kvq_device.cuh", "quant_row.cuh"]
WRITE_ASYM_SOURCES = ["write_asym.cu", "kvq_device.cuh", "quant_row.cuh"]


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["kvq", "reference"], default="kvq")
    p.add_argument("--workload", default=DEFAULT_WORKLOAD,
                   help="the headline workload (timed for exactly --steps steps)")
    p.add_argument("--workloads", default="all",
                   help="other workloads measured in the same run: all, none, or a comma list")
    p.add_argument("--ctas", type=int, default=0, help="decode CTAs per kv-head group (0 = auto)")
    p.add_argument("--e2e-steps", type=int, default=20)
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--chunk-tokens", type=int, default=16384,
                   help="prefill-chunk write timed where sequence 0 is at least this long (0: off)")
    p.add_argument("--no-append", action="store_true",
                   help="skip the fused append-and-decode step timing")
    p.add_argument("--cpu-seconds", type=float, default=12.0,
                   help="target CPU time of the oracle baseline sample")
    return p.parse_args(argv)


# ---------------------------------------------------------------------------
# algorithmic bytes (what the kernels must move at minimum)
# ---------------------------------------------------------------------------
def kv_bytes_per_token(wl) -> int:
    from quantized_paged_kv_kvq_gb300.kvq import meta_fields, row_bytes
    d = wl.head_dim
    per_head = (row_bytes(wl.k_fmt, d) + row_bytes(wl.v_fmt, d)
                + 2 * meta_fields(wl.k_fmt, wl.kvarn) + 2 * meta_fields(wl.v_fmt, wl.kvarn))
    return wl.num_kv_heads * per_head


def kv_cache_bytes(case) -> int:
    """Bytes of the cached codes and metadata a decode reads."""
    return int(case.wl.context_lens.astype("int64").sum()) * kv_bytes_per_token(case.wl)


def decode_bytes(wl) -> int:
    """Codes + metadata of every context token (once, whatever the GQA ratio),
    the query, the output, the used block-table entries and the lengths."""
    ctx = int(wl.context_lens.astype("int64").sum())
    blocks = int(((wl.context_lens.astype("int64") + wl.block_size - 1) // wl.block_size).sum())
    q = wl.num_seqs * wl.num_q_heads * wl.head_dim * 2
    return ctx * kv_bytes_per_token(wl) + 2 * q + 4 * blocks + 4 * wl.num_seqs


def write_bytes(wl) -> int:
    """bf16 K and V read + codes/metadata written + the slot id, per token."""
    t = wl.num_tokens
    return t * (2 * wl.num_kv_heads * wl.head_dim * 2 + kv_bytes_per_token(wl) + 8)


def source_hash(names) -> str:
    h = hashlib.sha256()
    for name in names:
        with open(os.path.join(ROOT, "quantized_paged_kv_kvq_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def decode_source_hash() -> str:
    return source_hash(DECODE_SOURCES)


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


KERNEL_SOURCES = {"decode_partition": DECODE_SOURCES, "write_cache": WRITE_SOURCES,
                  "write_asym": WRITE_ASYM_SOURCES}


def profiled_traffic(workload: str, kernel: str = "decode_partition"):
    """DRAM bytes per launch of a kernel on a workload, from the machine-readable
    record of its ncu capture (profiles/<kernel>_<workload>.json), if that
    capture was taken on the kernel's current sources; else None."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.json")
    if not os.path.exists(path):
        return None
    try:
        with open(path) as f:
            rec = json.load(f)
        if rec.get("source_sha256_16") != source_hash(KERNEL_SOURCES[kernel]):
            return None
        return float(rec["dram_bytes_per_launch"])
    except (OSError, ValueError, KeyError, TypeError):
        return None


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [l.strip().split(",") for l in self.file if l.count(",") >= 8]
        self.file.close()
        os.unlink(self.file.name)
        if not rows:
            return None
        sm = sorted(float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit())
        smax = max((float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()),
                   default=None)
        reasons = sorted({name for r in rows for name, v in zip(self.REASONS, r[5:9])
                          if "Active" in v and "Not" not in v})
        return {"sm_mhz": sm[len(sm) // 2] if sm else None, "sm_max_mhz": smax,
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------------------
# CPU oracle timing (cpu_baseline leg and the reference arm)
# ---------------------------------------------------------------------------
def oracle_sample(workload: str, seed_offset: int, budget_s: float, token_cap=None):
    """Run the oracle, sequence by sequence, until `budget_s` of CPU time; returns
    (kv bytes decoded, decode seconds, tokens written, write seconds, seqs used)."""
    import numpy as np
    from oracle import attention as OA
    from oracle import cache as OC
    from oracle import formats as OF
    from quantized_paged_kv_kvq_gb300 import workloads as W
    wl = W.workload(workload, seed=W.SEEDS[workload] + seed_offset)
    ks = OF.calibrate(wl.key, wl.k_scale_rule) if wl.k_scale_rule else np.float32(1)
    vs = OF.calibrate(wl.value, wl.v_scale_rule) if wl.v_scale_rule else np.float32(1)
    starts = np.concatenate([[0], np.cumsum(wl.context_lens.astype(np.int64))])
    per_tok = kv_bytes_per_token(wl)
    kv, tdec, ntok, twr, used = 0, 0.0, 0, 0.0, 0
    sm = OA.default_sm_scale(wl.head_dim)
    for s in range(wl.num_seqs):
        sl = slice(starts[s], starts[s + 1])
        if token_cap is not None:
            sl = slice(starts[s], min(starts[s + 1], starts[s] + token_cap))
        kc, km = OC.alloc_cache(wl.num_blocks, wl.block_size, wl.num_kv_heads, wl.head_dim,
                                wl.k_fmt, wl.kvarn)
        vc, vm = OC.alloc_cache(wl.num_blocks, wl.block_size, wl.num_kv_heads, wl.head_dim,
                                wl.v_fmt, wl.kvarn)
        t0 = time.process_time()
        OC.write_cache(kc, km, wl.key[sl], wl.slot_mapping[sl], wl.block_size, wl.k_fmt, ks,
                       wl.kvarn, wl.signs)
        OC.write_cache(vc, vm, wl.value[sl], wl.slot_mapping[sl], wl.block_size, wl.v_fmt, vs,
                       wl.kvarn, wl.signs)
        t1 = time.process_time()
        ctx = np.array(wl.context_lens)
        ctx[s] = sl.stop - sl.start
        OA.paged_decode(wl.query, kc, km, vc, vm, wl.block_table, ctx, wl.block_size, wl.k_fmt,
                        wl.v_fmt, ks, vs, sm, wl.kvarn, wl.signs,
                        pairs=[(s, h) for h in range(wl.num_kv_heads)])
        t2 = time.process_time()
        n = sl.stop - sl.start
        kv += n * per_tok
        ntok += n
        twr += t1 - t0
        tdec += t2 - t1
        used += 1
        if twr + tdec >= budget_s:
            break
    return int(kv), float(tdec), int(ntok), float(twr), int(used)


def cpu_baseline_subprocess(workload: str, budget_s: float):
    """Time the oracle single-threaded in a fresh process (BLAS pinned to 1 thread)."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    code = ("import json,bench;r=bench.oracle_sample(%r,0,%r);print(json.dumps(r))"
            % (workload, budget_s))
    out = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True,
                         text=True, timeout=600)
    if out.returncode != 0:
        return None
    kv, tdec, ntok, twr, used = json.loads(out.stdout.strip().splitlines()[-1])
    return {"value": round(kv / tdec / 1e9, 6) if tdec > 0 else None, "unit": "GB/s",
            "cores": 1, "kind": "oracle",
            "sample": f"{used} sequence(s) of {workload} (all {ntok} of their tokens): "
                      f"float32 quantize-and-scatter then float64 decode, single thread",
            "write_tok_s": round(ntok / twr, 3) if twr > 0 else None,
            "decode_seconds": round(tdec, 3), "write_seconds": round(twr, 3)}


def cpu_model() -> str:
    import platform
    part = None
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key = line.split(":", 1)[0].strip().lower()
                if key in ("model name", "cpu model", "hardware"):
                    return line.split(":", 1)[1].strip()
                if key == "cpu part" and part is None:  # Arm: implementer-specific part id
                    part = line.split(":", 1)[1].strip()
    except OSError:
        pass
    name = platform.processor() or platform.machine()
    return f"{name} (CPU part {part})" if part else name


def cpu_baseline_all_cores(workload: str, budget_s: float, procs: int):
    """The same oracle sample in `procs` concurrent single-threaded processes (one per
    host core, each on its own seeded copy of the workload); the rate is the sum of
    the processes' rates, each measured in its own CPU time."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    children = []
    for i in range(procs):
        code = ("import json,bench;r=bench.oracle_sample(%r,%d,%r);print(json.dumps(r))"
                % (workload, 1 + i, budget_s))
        children.append(subprocess.Popen([sys.executable, "-c", code], cwd=ROOT, env=env,
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True))
    rate, done = 0.0, 0
    for c in children:
        try:
            out, _ = c.communicate(timeout=600)
        except subprocess.TimeoutExpired:
            c.kill()
            continue
        if c.returncode != 0 or not out.strip():
            continue
        kv, tdec, _, _, _ = json.loads(out.strip().splitlines()[-1])
        if tdec > 0:
            rate += kv / tdec
            done += 1
    if done == 0:
        return None
    return {"value": round(rate / 1e9, 6), "unit": "GB/s", "cores": done,
            "sample": f"{done} concurrent single-thread processes, each as the one-core sample",
            "cpu_model": cpu_model()}


def run_reference(args, rank: int):
    if rank != 0:
        return
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ.setdefault(v, "1")
    from quantized_paged_kv_kvq_gb300 import workloads as W
    wl_meta = W.WORKLOADS[args.workload]
    kv_total, t_total, tok_total, tw_total = 0, 0.0, 0, 0.0
    # each step: one sequence (round robin), capped at 256 tokens, write + decode
    cap = 256
    for step in range(args.warmup + args.steps):
        kv, tdec, ntok, twr, _ = oracle_sample_one(args.workload, step, cap)
        if step >= args.warmup:
            kv_total += kv
            t_total += tdec
            tok_total += ntok
            tw_total += twr
    value = kv_total / t_total / 1e9 if t_total > 0 else None
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * (t_total + tw_total) / max(args.steps, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "impl": "reference",
        "config": {"workload": args.workload, "num_seqs": wl_meta["num_seqs"],
                   "num_q_heads": wl_meta["num_q_heads"], "num_kv_heads": wl_meta["num_kv_heads"],
                   "head_dim": wl_meta["head_dim"], "block_size": wl_meta["block_size"],
                   "step_sample": f"one sequence per step (round robin), first {cap} tokens"},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"{args.steps} steps x one sequence's first {cap} tokens: "
                                   "float32 quantize-and-scatter + float64 decode, one thread"},
        "cache_write_tok_s": tok_total / tw_total if tw_total > 0 else None,
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


_REF_CACHE = {}


def oracle_sample_one(workload: str, step: int, cap: int):
    """One reference step: oracle write + decode of one sequence (first `cap` tokens)."""
    import numpy as np
    from oracle import attention as OA
    from oracle import cache as OC
    from oracle import formats as OF
    from quantized_paged_kv_kvq_gb300 import workloads as W
    if workload not in _REF_CACHE:
        wl = W.workload(workload, **({"num_seqs": min(W.WORKLOADS[workload]["num_seqs"], 16)}))
        ks = OF.calibrate(wl.key, wl.k_scale_rule) if wl.k_scale_rule else np.float32(1)
        vs = OF.calibrate(wl.value, wl.v_scale_rule) if wl.v_scale_rule else np.float32(1)
        kc, km = OC.alloc_cache(wl.num_blocks, wl.block_size, wl.num_kv_heads, wl.head_dim,
                                wl.k_fmt, wl.kvarn)
        vc, vm = OC.alloc_cache(wl.num_blocks, wl.block_size, wl.num_kv_heads, wl.head_dim,
                                wl.v_fmt, wl.kvarn)
        starts = np.concatenate([[0], np.cumsum(wl.context_lens.astype(np.int64))])
        _REF_CACHE[workload] = (wl, ks, vs, kc, km, vc, vm, starts)
    wl, ks, vs, kc, km, vc, vm, starts = _REF_CACHE[workload]
    s = step % wl.num_seqs
    n = int(min(wl.context_lens[s], cap))
    sl = slice(starts[s], starts[s] + n)
    t0 = time.process_time()
    OC.write_cache(kc, km, wl.key[sl], wl.slot_mapping[sl], wl.block_size, wl.k_fmt, ks,
                   wl.kvarn, wl.signs)
    OC.write_cache(vc, vm, wl.value[sl], wl.slot_mapping[sl], wl.block_size, wl.v_fmt, vs,
                   wl.kvarn, wl.signs)
    t1 = time.process_time()
    ctx = np.array(wl.context_lens)
    ctx[s] = n
    OA.paged_decode(wl.query, kc, km, vc, vm, wl.block_table, ctx, wl.block_size, wl.k_fmt,
                    wl.v_fmt, ks, vs, OA.default_sm_scale(wl.head_dim), wl.kvarn, wl.signs,
                    pairs=[(s, h) for h in range(wl.num_kv_heads)])
    t2 = time.process_time()
    return n * kv_bytes_per_token(wl), t2 - t1, n, t1 - t0, 1


# ---------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------
def aggregate(per_rank_times, per_rank_units):
    """Whole-job throughput: units of all ranks / the slowest rank's time."""
    t = max(per_rank_times)
    return (sum(per_rank_units) / t) if t > 0 else float("nan")


def max_over_ranks(values, device=None):
    """Element-wise maximum of a list of floats over all ranks (identity at N=1)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor(values, dtype=torch.float64, device=device)
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def write_kernel_name(wl) -> str:
    return "write_asym" if wl.k_fmt.endswith("_asym") else "write_cache"


class Case:
    """One workload resident on the device: inputs, calibrated cache, output,
    decode workspace and an L2 flush; every call goes through the public API."""

    def __init__(self, name, dev, seed, ctas, l2_bytes):
        import numpy as np
        import torch
        from quantized_paged_kv_kvq_gb300 import kvq
        from quantized_paged_kv_kvq_gb300 import workloads as W
        self.kvq, self.dev, self.ctas, self.l2_bytes = kvq, dev, ctas, l2_bytes
        self.wl = wl = W.workload(name, seed=seed, with_data=False)
        data = W.device_data(wl, dev, seed)
        self.key, self.value, self.query = data["key"], data["value"], data["query"]
        self.slots = torch.from_numpy(wl.slot_mapping).to(dev)
        self.block_table = torch.from_numpy(wl.block_table).to(dev)
        self.ctx_lens = torch.from_numpy(wl.context_lens).to(dev)
        self.signs = None if wl.signs is None else torch.from_numpy(wl.signs).to(dev)
        qmax = {"absmax/127": 127.0, "absmax/448": 448.0}

        def scale(x, rule):  # offline per-tensor calibration (untimed), on the GPU
            if rule not in qmax:
                return 1.0
            o = torch.empty(1, dtype=torch.float32, device=dev)
            kvq.kvq_calibrate_scale(x.reshape(-1), qmax[rule], o)
            return float(o.item())

        self.cache = kvq.alloc_kv_cache(wl.k_fmt, wl.v_fmt, wl.num_blocks, wl.block_size,
                                        wl.num_kv_heads, wl.head_dim,
                                        scale(self.key, wl.k_scale_rule),
                                        scale(self.value, wl.v_scale_rule), wl.kvarn,
                                        self.signs, device=dev)
        self.out = torch.empty_like(self.query)
        self.sm_scale = float(np.float32(1.0 / np.sqrt(wl.head_dim)))
        self.ws_bytes = kvq.kvq_decode_workspace_size(self.cache, wl.num_seqs, wl.num_q_heads,
                                                      wl.max_context_len, ctas)
        self.ws = torch.empty(max(self.ws_bytes, 16) // 4 + 4, dtype=torch.float32, device=dev)
        # L2 flush: write one buffer of 2x L2, then read another of 2x L2, so a
        # timed kernel starts with an L2 that holds none of its data and no dirty
        # lines (whose write-back would otherwise land inside the timed kernel)
        n = max(2 * l2_bytes, 256 << 20)
        self.flush_w = torch.empty(n, dtype=torch.uint8, device=dev)
        self.flush_r = torch.ones(n // 4, dtype=torch.int32, device=dev)
        # each sequence's last token, for the decode step that brings its own token
        last = np.cumsum(wl.context_lens.astype(np.int64)) - 1
        self.has_new = wl.context_lens > 0
        rows = torch.from_numpy(np.where(self.has_new, last, 0)).to(dev)
        self.new_k = self.key[rows].contiguous()
        self.new_v = self.value[rows].contiguous()
        self.last_slots = torch.from_numpy(
            np.where(self.has_new, wl.slot_mapping[np.where(self.has_new, last, 0)], -1)).to(dev)

    def flush_l2(self):
        self.flush_w.zero_()
        self.flush_r.sum()

    def write(self):
        self.kvq.kvq_write_cache(self.cache, self.key, self.value, self.slots)

    def decode(self):
        wl = self.wl
        self.kvq.kvq_paged_decode(self.cache, self.query, self.out, self.block_table,
                                  self.ctx_lens, wl.max_context_len, self.sm_scale, self.ws,
                                  self.ctas)

    def append_decode(self, new_k=None, new_v=None, query=None, ctx_lens=None):
        wl = self.wl
        self.kvq.kvq_decode_append(self.cache, self.new_k if new_k is None else new_k,
                                   self.new_v if new_v is None else new_v,
                                   self.query if query is None else query, self.out,
                                   self.block_table,
                                   self.ctx_lens if ctx_lens is None else ctx_lens,
                                   wl.max_context_len, self.sm_scale, self.ws, self.ctas)


def _events(n):
    import torch
    return [torch.cuda.Event(enable_timing=True) for _ in range(n)]


def time_steps(case, warmup, steps):
    """`steps` steps of the whole path (flush, write, flush, decode); returns the
    per-step write and decode times (ms) from CUDA events on the current stream."""
    import numpy as np
    import torch

    def step(ev):
        case.flush_l2()
        ev[0].record()
        case.write()
        ev[1].record()
        case.flush_l2()
        ev[2].record()
        case.decode()
        ev[3].record()

    for _ in range(warmup):
        step(_events(4))
    torch.cuda.synchronize()
    evs = [_events(4) for _ in range(steps)]
    for ev in evs:
        step(ev)
    torch.cuda.synchronize()
    w = np.array([e[0].elapsed_time(e[1]) for e in evs])
    d = np.array([e[2].elapsed_time(e[3]) for e in evs])
    return w, d


def time_write_back_to_back(case, launches):
    """Cache writes one after another with no flush between them, between one
    pair of events: a launch's dirty lines are written back during the next
    ones, so the time per launch includes its DRAM writes (all but the last
    launch's, 1/launches of them)."""
    import torch
    case.flush_l2()
    e0, e1 = _events(2)
    e0.record()
    for _ in range(launches):
        case.write()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) * 1e3 / launches


def time_decode_back_to_back(case, launches):
    """Decodes one after another with no flush between them, between one pair
    of events (the launch overhead of all but the first is hidden behind the
    previous kernel, as in a serving loop).  Where the cache is larger than L2,
    each launch still reads it from DRAM (the loads carry an evict-first
    policy); a smaller cache stays in L2 and the number is not an HBM one."""
    import torch
    case.flush_l2()
    e0, e1 = _events(2)
    e0.record()
    for _ in range(launches):
        case.decode()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) * 1e3 / launches


def time_decode_graph(case, n, reps=3):
    """Decode time per launch when the steps are replayed from a CUDA graph, as
    a serving loop launches its decode: one graph of n x (L2 flush, decode) and
    one of the n flushes alone, each replayed between a pair of events; the
    difference over n.  The flush before every launch stays, so each decode
    still reads the cache from DRAM."""
    import torch
    s = torch.cuda.Stream(device=case.dev)

    def capture(fn):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            fn()  # warm-up outside the capture (first-use allocations)
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=s):
            fn()
        return g

    def both():
        for _ in range(n):
            case.flush_l2()
            case.decode()

    def flushes():
        for _ in range(n):
            case.flush_l2()

    def replay_us(g):
        ts = []
        for _ in range(reps):
            e0, e1 = _events(2)
            torch.cuda.synchronize()
            e0.record()
            g.replay()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1) * 1e3)
        return sorted(ts)[len(ts) // 2]

    ga, gb = capture(both), capture(flushes)
    us = (replay_us(ga) - replay_us(gb)) / n
    del ga, gb
    return us


def time_each(case, fn, n, warmup=3):
    """Median (us) of `fn` over n launches, L2 flushed before each."""
    import numpy as np
    import torch

    def one(ev):
        case.flush_l2()
        ev[0].record()
        fn()
        ev[1].record()

    for _ in range(warmup):
        one(_events(2))
    evs = [_events(2) for _ in range(n)]
    for ev in evs:
        one(ev)
    torch.cuda.synchronize()
    return float(np.median([e[0].elapsed_time(e[1]) for e in evs])) * 1e3


def time_append(case, n):
    """One decode step that brings one new token per sequence: the fused
    append-and-decode launch, and a cache write of those tokens followed by
    the decode (both with a flushed L2)."""
    kvq, wl = case.kvq, case.wl
    fused = time_each(case, case.append_decode, n)
    unfused = time_each(case, lambda: (kvq.kvq_write_cache(case.cache, case.new_k, case.new_v,
                                                           case.last_slots), case.decode()), n)
    return {"fused_append_decode_us": fused, "write_then_decode_us": unfused, "steps": n,
            "stat": "median, L2 flushed before each step", "tokens_per_step": int(case.has_new.sum())}


def time_chunk(case, tokens, n, seed, hbm):
    """The write of a `tokens`-token prefill chunk into sequence 0's pages (the
    long-context shape's prefill step), L2 flushed before each."""
    import torch
    from quantized_paged_kv_kvq_gb300 import workloads as W
    wl = case.wl
    if tokens <= 0 or int(wl.context_lens[0]) < tokens:
        return None
    rows = torch.arange(tokens, device=case.dev)  # sequence 0's first tokens
    ck, cv = case.key[rows].contiguous(), case.value[rows].contiguous()
    cs = torch.from_numpy(W.slots_for_context(wl.context_lens[:1] * 0 + tokens,
                                              wl.block_table[:1], wl.block_size)).to(case.dev)
    us = time_each(case, lambda: case.kvq.kvq_write_cache(case.cache, ck, cv, cs), n)
    cbytes = tokens * (2 * wl.num_kv_heads * wl.head_dim * 2 + kv_bytes_per_token(wl) + 8)
    return {"tokens": tokens, "us": us, "tok_s": tokens / us * 1e6, "gbs": cbytes / us / 1e3,
            "frac_of_hbm": cbytes / us / 1e3 / hbm, "bytes": cbytes, "steps": n,
            "stat": "median, L2 flushed before each write"}


def e2e_decode_step(case, n, dbytes, world):
    """A decode step through the public API with host buffers: every step copies
    its inputs from pinned host memory (the query, each sequence's new key and
    value row and the context lengths, packed in one buffer: one copy), runs
    kvq_decode_append (store the new rows, attend over the cache resident in
    HBM) and copies the output back."""
    import torch
    srcs = (case.query, case.new_k, case.new_v, case.ctx_lens)
    sizes = [x.numel() * x.element_size() for x in srcs]
    offs, o = [], 0
    for sz in sizes:  # 16-byte aligned pieces of one packed buffer
        offs.append(o)
        o += (sz + 15) // 16 * 16
    h_buf = torch.empty(o, dtype=torch.uint8).pin_memory()
    d_buf = torch.empty(o, dtype=torch.uint8, device=case.dev)

    def views(buf):
        return [buf[a:a + sz].view(x.dtype).view(x.shape) for a, sz, x in zip(offs, sizes, srcs)]

    for h, x in zip(views(h_buf), srcs):
        h.copy_(x.cpu())
    d_q, d_k, d_v, d_ctx = views(d_buf)
    h_out = torch.empty(case.out.shape, dtype=case.out.dtype).pin_memory()

    def step():
        d_buf.copy_(h_buf, non_blocking=True)
        case.append_decode(new_k=d_k, new_v=d_v, query=d_q, ctx_lens=d_ctx)
        h_out.copy_(case.out, non_blocking=True)

    for _ in range(3):
        step()
    torch.cuda.synchronize()
    e0, e1 = _events(2)
    w0 = time.perf_counter()
    e0.record()
    for _ in range(n):
        step()
    e1.record()
    torch.cuda.synchronize()
    wall = time.perf_counter() - w0
    t = max_over_ranks([e0.elapsed_time(e1) / 1e3], case.dev)[0]
    return {"value": world * dbytes * n / t / 1e9, "unit": "GB/s", "h2d_bytes_per_step": o,
            "d2h_bytes_per_step": h_out.numel() * h_out.element_size(), "steps": n,
            "ms_per_step": 1e3 * t / n, "wall_ms_per_step": 1e3 * wall / n,
            "call": "kvq_decode_append", "tokens_per_step": int(case.has_new.sum())}


def e2e_full_context(case, n, dbytes, world):
    """Write-everything-then-decode through the public API with host buffers:
    every step copies all bf16 keys and values of the context (and the query,
    slots, block table, lengths) from pinned host memory, writes the whole
    cache, decodes and copies the output back -- a prefill-sized step, bound
    by the host-to-device copy."""
    import torch
    srcs = (case.key, case.value, case.query, case.slots, case.block_table, case.ctx_lens)
    h_in = [x.cpu().pin_memory() for x in srcs]
    d_in = [torch.empty_like(x) for x in srcs]
    h_out = torch.empty(case.out.shape, dtype=case.out.dtype).pin_memory()
    kvq, wl = case.kvq, case.wl

    def step():
        for h, d in zip(h_in, d_in):
            d.copy_(h, non_blocking=True)
        kvq.kvq_write_cache(case.cache, d_in[0], d_in[1], d_in[3])
        kvq.kvq_paged_decode(case.cache, d_in[2], case.out, d_in[4], d_in[5], wl.max_context_len,
                             case.sm_scale, case.ws, case.ctas)
        h_out.copy_(case.out, non_blocking=True)

    for _ in range(3):
        step()
    torch.cuda.synchronize()
    e0, e1 = _events(2)
    e0.record()
    for _ in range(n):
        step()
    e1.record()
    torch.cuda.synchronize()
    t = max_over_ranks([e0.elapsed_time(e1) / 1e3], case.dev)[0]
    h2d = sum(x.numel() * x.element_size() for x in h_in)
    return {"value": world * dbytes * n / t / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": h_out.numel() * h_out.element_size(), "steps": n,
            "ms_per_step": 1e3 * t / n}


def roofline(kernel, workload, nbytes, seconds_per_launch, hbm, peak_note):
    achieved = nbytes / seconds_per_launch / 1e9
    return {"bound": "hbm", "kernel": kernel + "_kernel", "achieved": achieved, "peak": hbm,
            "peak_source": peak_note, "unit": "GB/s", "frac": achieved / hbm,
            "traffic": profiled_traffic(workload, kernel), "algorithmic_bytes": nbytes}


def measure_case(args, case, rank, world, hbm, peak_note, steps, headline=False):
    """Time one workload: the whole-path steps (with clocks sampled meanwhile),
    back-to-back writes, the decode step with its own token and, where the
    first sequence is long enough, the prefill-chunk write."""
    import numpy as np
    import torch
    import torch.distributed as dist
    wl, dev = case.wl, case.dev
    for _ in range(args.warmup):  # untimed warm-up steps
        time_steps(case, 0, 1)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    sampler = ClockSampler(dev.index or 0)
    sampler.start()
    time.sleep(0.3)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    w0 = time.perf_counter()
    w_ms, d_ms = time_steps(case, 0, steps)
    if world > 1:
        dist.barrier()
    wall = time.perf_counter() - w0
    clocks = sampler.stop()
    t_write, t_dec = float(w_ms.sum()) / 1e3, float(d_ms.sum()) / 1e3
    t_write, t_dec, wall = max_over_ranks([t_write, t_dec, wall], dev)
    dbytes, wbytes = decode_bytes(wl), write_bytes(wl)
    pct = lambda x: {f"p{q}": round(float(np.percentile(x, q)) * 1e3, 3) for q in (10, 50, 90)}
    b2b = max_over_ranks([time_write_back_to_back(case, max(8, min(steps, 50)))], dev)[0]
    d2b = max_over_ranks([time_decode_back_to_back(case, max(8, min(steps, 200)))], dev)[0]
    dgr = max_over_ranks([time_decode_graph(case, max(4, min(steps, 50)))], dev)[0]
    n_side = max(3, min(steps, 200))
    app = None if args.no_append else time_append(case, n_side)
    chunk = time_chunk(case, args.chunk_tokens, n_side, W_SEED(wl.name) + 7 + 100 * rank, hbm)
    r = {
        "steps": steps,
        "decode_us": 1e6 * t_dec / steps, "decode_us_pct": pct(d_ms),
        "decode_gbs": world * dbytes * steps / t_dec / 1e9,
        "decode_frac_of_hbm": dbytes * steps / t_dec / 1e9 / hbm,
        "decode_tok_s": world * wl.num_seqs * steps / t_dec,
        "decode_bytes": dbytes, "decode_split": case.ws_bytes > 0,
        "cache_write_us": 1e6 * t_write / steps, "cache_write_us_pct": pct(w_ms),
        "cache_write_gbs": world * wbytes * steps / t_write / 1e9,
        "cache_write_frac_of_hbm": wbytes * steps / t_write / 1e9 / hbm,
        "cache_write_tok_s": world * wl.num_tokens * steps / t_write,
        "write_bytes": wbytes,
        "cache_write_back_to_back_us": b2b,
        "cache_write_back_to_back_frac_of_hbm": wbytes / (b2b * 1e-6) / 1e9 / hbm,
        "decode_back_to_back_us": d2b,
        "decode_back_to_back_frac_of_hbm": dbytes / (d2b * 1e-6) / 1e9 / hbm,
        "decode_back_to_back_cache_exceeds_l2": kv_cache_bytes(case) > case.l2_bytes,
        "decode_graph_us": dgr,
        "decode_graph_frac_of_hbm": dbytes / (dgr * 1e-6) / 1e9 / hbm,
        "roofline_decode": roofline("decode_partition", wl.name, dbytes, t_dec / steps, hbm,
                                    peak_note),
        "roofline_write": roofline(write_kernel_name(wl), wl.name, wbytes, t_write / steps, hbm,
                                   peak_note),
        "decode_step_append": app,
        "prefill_chunk_write": chunk,
        "clocks": clocks,
        "wall_s_timed_region": wall,
        "shape": {"num_seqs": wl.num_seqs, "num_q_heads": wl.num_q_heads,
                  "num_kv_heads": wl.num_kv_heads, "head_dim": wl.head_dim,
                  "block_size": wl.block_size, "k_fmt": wl.k_fmt, "v_fmt": wl.v_fmt,
                  "kvarn": wl.kvarn, "context_tokens": int(wl.context_lens.sum())},
    }
    return r, t_write, t_dec


def W_SEED(name):
    from quantized_paged_kv_kvq_gb300 import workloads as W
    return W.SEEDS[name]


def quantized_vs_bf16(per):
    """Decode and write time of each 8-bit cache of the Llama-3-8B shape against
    the unquantized 16-bit cache on the same shape and inputs (the comparison
    the pages' FP8 / INT8 numbers are about), where both were measured."""
    ref = per.get("llama8b_bf16")
    if not ref:
        return None
    out = {"reference": "llama8b_bf16", "decode_us": ref["decode_us"],
           "cache_write_us": ref["cache_write_us"]}
    for name in ("llama8b_int8",):
        if name in per:
            out[name] = {"decode_us": per[name]["decode_us"],
                         "decode_speedup": ref["decode_us"] / per[name]["decode_us"],
                         "kv_bytes_ratio": per[name]["decode_bytes"] / ref["decode_bytes"]}
    return out


def run_kvq(args, rank: int, world: int, local_rank: int):
    import torch
    import torch.distributed as dist

    from quantized_paged_kv_kvq_gb300 import build as kbuild
    kbuild.build()
    from quantized_paged_kv_kvq_gb300 import workloads as W

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    hbm, peak_src = measured_peaks()
    peak_note = f"{peak_src} hbm_gbs (burst copy)"
    K = args.steps

    # ---- the headline workload: exactly K timed steps, then the side legs
    case = Case(args.workload, dev, W.SEEDS[args.workload] + 100 * rank, args.ctas, l2)
    head, t_write, t_dec = measure_case(args, case, rank, world, hbm, peak_note, K, headline=True)
    wl = case.wl
    dbytes = decode_bytes(wl)
    e2e = e2e_full = None
    if not args.no_e2e:
        n_e2e = max(1, min(args.e2e_steps, K))
        e2e = e2e_decode_step(case, max(n_e2e, 20), dbytes, world)
        e2e_full = e2e_full_context(case, n_e2e, dbytes, world)
    ws_desc = case.ws_bytes
    del case
    torch.cuda.empty_cache()

    # ---- every other configuration, each with its own clocks
    names = [] if args.workloads == "none" else (
        list(W.WORKLOADS) if args.workloads == "all" else args.workloads.split(","))
    per = {args.workload: head}
    n_cfg = min(max(K, 50), 500)
    for name in names:
        if name in per:
            continue
        c = Case(name, dev, W.SEEDS[name] + 100 * rank, args.ctas, l2)
        per[name], _, _ = measure_case(args, c, rank, world, hbm, peak_note, n_cfg)
        del c
        torch.cuda.empty_cache()

    if world > 1:
        dist.barrier()
    if rank != 0:
        dist.destroy_process_group()
        return
    cpu = None if args.no_cpu_baseline or world > 1 else cpu_baseline_subprocess(
        args.workload, args.cpu_seconds)
    if cpu is not None:  # context: the oracle over every host core at once
        cpu["cpu_model"] = cpu_model()
        cpu["all_cores"] = cpu_baseline_all_cores(args.workload, args.cpu_seconds / 2,
                                                  min(os.cpu_count() or 1, 16))
    rl_d, rl_w = head["roofline_decode"], head["roofline_write"]
    line = {
        "metric": METRIC, "value": head["decode_gbs"], "unit": "GB/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": 1e3 * (t_write + t_dec) / K,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u8",
        "data": "synthetic",
        "config": {"workload": args.workload, "num_seqs": wl.num_seqs,
                   "num_q_heads": wl.num_q_heads, "num_kv_heads": wl.num_kv_heads,
                   "head_dim": wl.head_dim, "block_size": wl.block_size,
                   "k_fmt": wl.k_fmt, "v_fmt": wl.v_fmt, "kvarn": wl.kvarn,
                   "context_tokens": int(wl.context_lens.sum()),
                   "decode_ctas": args.ctas or "auto",
                   "l2": "flushed before the write and before the decode (2xL2 memset, "
                         "then a 2xL2 read), outside the timed events",
                   "inputs": "drawn on the device (torch generator) by the workload recipe"},
        "decode_tok_s": head["decode_tok_s"], "decode_us": head["decode_us"],
        "decode_us_pct": head["decode_us_pct"], "decode_split": ws_desc > 0,
        "cache_write_tok_s": head["cache_write_tok_s"],
        "cache_write_gbs": head["cache_write_gbs"], "cache_write_us": head["cache_write_us"],
        "cache_write_us_pct": head["cache_write_us_pct"],
        "cache_write_frac_of_hbm": head["cache_write_frac_of_hbm"],
        "cache_write_back_to_back_us": head["cache_write_back_to_back_us"],
        "cache_write_back_to_back_frac_of_hbm": head["cache_write_back_to_back_frac_of_hbm"],
        "decode_back_to_back_us": head["decode_back_to_back_us"],
        "decode_back_to_back_frac_of_hbm": head["decode_back_to_back_frac_of_hbm"],
        "decode_graph_us": head["decode_graph_us"],
        "decode_graph_frac_of_hbm": head["decode_graph_frac_of_hbm"],
        "decode_bytes": head["decode_bytes"], "write_bytes": head["write_bytes"],
        "wall_s_timed_region": head["wall_s_timed_region"],
        # the dominant kernel of the step (largest share of its time) first
        "roofline": rl_w if t_write >= t_dec else rl_d,
        "roofline_decode": rl_d,
        "roofline_write": rl_w,
        "decode_frac_of_hbm": head["decode_frac_of_hbm"],
        "e2e": e2e,
        "e2e_full_context": e2e_full,
        "decode_step_append": head["decode_step_append"],
        # the long-context configuration's prefill chunk (where the run measured it)
        "prefill_chunk_write": (per.get("kvarn_131k") or {}).get("prefill_chunk_write"),
        "gpu_launches": 2 * K,  # one write and one decode launch per timed step
        "clocks": head["clocks"],
        "cpu_baseline": cpu,
        "workloads": {k: {kk: vv for kk, vv in v.items()} for k, v in per.items()},
        "quantized_vs_bf16": quantized_vs_bf16(per),
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main(argv=None):
    args = parse_args(argv)
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank)
        return
    run_kvq(args, rank, world, local_rank)


if __name__ == "__main__":
    main()
