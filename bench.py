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
DECODE_SOURCES = ["decode.cuh", "decode_launch.cuh", "kvq_device.cuh", "quant_row.cuh",
                  "decode_d128_sym.cu", "decode_d128_asym.cu", "decode_d64_sym.cu",
                  "decode_d64_asym.cu"]
WRITE_SOURCES = ["write.cu", "kvq_device.cuh", "quant_row.cuh"]
WRITE_ASYM_SOURCES = ["write_asym.cu", "kvq_device.cuh", "quant_row.cuh"]


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["kvq", "reference"], default="kvq")
    p.add_argument("--workload", default=DEFAULT_WORKLOAD)
    p.add_argument("--ctas", type=int, default=0, help="decode CTAs per kv-head group (0 = auto)")
    p.add_argument("--e2e-steps", type=int, default=20)
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--chunk-tokens", type=int, default=16384,
                   help="prefill-chunk write timed when sequence 0 is at least this long (0: off)")
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


def profiled_traffic(workload: str, kernel: str = "decode_partition"):
    """DRAM bytes per launch of a kernel from its committed ncu summary
    (profiles/<kernel>_<workload>.md), if that was taken on the current
    sources of the kernel; else None."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    if not os.path.exists(path):
        return None
    vals = {}
    with open(path) as f:
        for line in f:
            if ":" in line and line.strip().startswith("- "):
                k, v = line.strip()[2:].split(":", 1)
                vals[k.strip()] = v.strip().strip("`")
    if kernel == "decode_partition":
        ok = vals.get("decode_source_sha256_16") == decode_source_hash()
    elif kernel == "write_asym":
        ok = vals.get("write_source_sha256_16") == source_hash(WRITE_ASYM_SOURCES)
    else:
        ok = vals.get("write_source_sha256_16") == source_hash(WRITE_SOURCES)
    if not ok:
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
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


def run_kvq(args, rank: int, world: int, local_rank: int):
    import numpy as np
    import torch
    import torch.distributed as dist

    from quantized_paged_kv_kvq_gb300 import build as kbuild
    kbuild.build()
    from quantized_paged_kv_kvq_gb300 import kvq
    from quantized_paged_kv_kvq_gb300 import workloads as W

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    wl = W.workload(args.workload, seed=W.SEEDS[args.workload] + 100 * rank)
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev).to(torch.bfloat16)
    key, value, query = bf(wl.key), bf(wl.value), bf(wl.query)
    slots = torch.from_numpy(wl.slot_mapping).to(dev)
    block_table = torch.from_numpy(wl.block_table).to(dev)
    ctx_lens = torch.from_numpy(wl.context_lens).to(dev)
    signs = None if wl.signs is None else torch.from_numpy(wl.signs).to(dev)
    qmax = {"absmax/127": 127.0, "absmax/448": 448.0}

    def scale(x, rule):  # offline per-tensor calibration (untimed), on the GPU
        if rule is None or rule == "1.0":
            return 1.0
        o = torch.empty(1, dtype=torch.float32, device=dev)
        kvq.kvq_calibrate_scale(x.reshape(-1), qmax[rule], o)
        return float(o.item())

    cache = kvq.alloc_kv_cache(wl.k_fmt, wl.v_fmt, wl.num_blocks, wl.block_size,
                               wl.num_kv_heads, wl.head_dim, scale(key, wl.k_scale_rule),
                               scale(value, wl.v_scale_rule), wl.kvarn, signs, device=dev)
    out = torch.empty_like(query)
    sm_scale = float(np.float32(1.0 / np.sqrt(wl.head_dim)))
    P = args.ctas
    ws_bytes = kvq.kvq_decode_workspace_size(cache, wl.num_seqs, wl.num_q_heads,
                                             wl.max_context_len, P)
    ws = torch.empty(max(ws_bytes, 16) // 4 + 4, dtype=torch.float32, device=dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    # L2 flush: write one buffer of 2x L2, then read another of 2x L2, so the
    # timed kernels start with an L2 that holds none of their data and no dirty
    # lines (whose write-back would otherwise land inside the next timed kernel)
    flush_w = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device=dev)
    flush_r = torch.ones(max(2 * l2, 256 << 20) // 4, dtype=torch.int32, device=dev)

    def flush_l2():
        flush_w.zero_()
        flush_r.sum()
    dargs = (cache, query, out, block_table, ctx_lens, wl.max_context_len, sm_scale, ws, P)

    def step(ev):
        flush_l2()
        ev[0].record()
        kvq.kvq_write_cache(cache, key, value, slots)
        ev[1].record()
        flush_l2()
        ev[2].record()
        kvq.kvq_paged_decode(*dargs)
        ev[3].record()

    mk = lambda: [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    for _ in range(args.warmup):
        step(mk())
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    events = [mk() for _ in range(args.steps)]
    sampler = ClockSampler(local_rank)
    sampler.start()
    time.sleep(0.3)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    w0 = time.perf_counter()
    for ev in events:
        step(ev)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    wall = time.perf_counter() - w0
    clocks = sampler.stop()
    w_ms = np.array([e[0].elapsed_time(e[1]) for e in events])
    d_ms = np.array([e[2].elapsed_time(e[3]) for e in events])
    t_write, t_dec = float(w_ms.sum()) / 1e3, float(d_ms.sum()) / 1e3
    pct = lambda x: {f"p{q}": round(float(np.percentile(x, q)) * 1e3, 3) for q in (10, 50, 90)}
    t_write, t_dec, wall = max_over_ranks([t_write, t_dec, wall], dev)
    dbytes, wbytes = decode_bytes(wl), write_bytes(wl)
    K = args.steps
    gbs = aggregate([t_dec], [world * dbytes * K]) / 1e9
    hbm, peak_src = measured_peaks()
    achieved = dbytes / (t_dec / K) / 1e9
    achieved_w = wbytes / (t_write / K) / 1e9
    peak_note = f"{peak_src} hbm_gbs (burst copy)"
    rl_decode = {"bound": "hbm", "kernel": "decode_partition_kernel", "achieved": achieved,
                 "peak": hbm, "peak_source": peak_note, "unit": "GB/s", "frac": achieved / hbm,
                 "traffic": profiled_traffic(args.workload, "decode_partition"),
                 "algorithmic_bytes": dbytes}
    wkern = "write_asym" if wl.k_fmt.endswith("_asym") else "write_cache"
    rl_write = {"bound": "hbm", "kernel": wkern + "_kernel", "achieved": achieved_w,
                "peak": hbm, "peak_source": peak_note, "unit": "GB/s", "frac": achieved_w / hbm,
                "traffic": profiled_traffic(args.workload, wkern),
                "algorithmic_bytes": wbytes}

    # one decode step that brings its own token (one per sequence): the fused
    # append-and-decode launch against a cache write of those tokens followed by
    # the decode (both with a flushed L2; outside the timed region above)
    step_lat = None
    if not args.no_append:
        last = np.cumsum(wl.context_lens.astype(np.int64)) - 1
        has = wl.context_lens > 0
        rows = torch.from_numpy(np.where(has, last, 0)).to(dev)
        new_k, new_v = key[rows].contiguous(), value[rows].contiguous()
        last_slots = torch.from_numpy(np.where(has, wl.slot_mapping[np.where(has, last, 0)],
                                               -1)).to(dev)
        n_app = max(3, min(K, 200))

        def fused(ev):
            flush_l2()
            ev[0].record()
            kvq.kvq_decode_append(cache, new_k, new_v, query, out, block_table, ctx_lens,
                                  wl.max_context_len, sm_scale, ws, P)
            ev[1].record()

        def unfused(ev):
            flush_l2()
            ev[0].record()
            kvq.kvq_write_cache(cache, new_k, new_v, last_slots)
            kvq.kvq_paged_decode(*dargs)
            ev[1].record()

        res = {}
        for name, fn in (("fused", fused), ("unfused", unfused)):
            for _ in range(3):
                fn(mk())
            evs = [mk() for _ in range(n_app)]
            for ev in evs:
                fn(ev)
            torch.cuda.synchronize()
            ms = np.array([e[0].elapsed_time(e[1]) for e in evs])
            res[name] = max_over_ranks([float(np.median(ms)) * 1e3], dev)[0]
        step_lat = {"fused_append_decode_us": res["fused"],
                    "write_then_decode_us": res["unfused"], "steps": n_app,
                    "stat": "median, L2 flushed before each step", "tokens_per_step": int(has.sum())}

    # a prefill chunk: the write of `chunk_tokens` new tokens into sequence 0's
    # pages (the long-context shape's prefill step), L2 flushed before each
    chunk = None
    C = args.chunk_tokens
    if C > 0 and int(wl.context_lens[0]) >= C:
        pc = W.prefill_chunk(wl, C, seed=W.SEEDS[args.workload] + 7 + 100 * rank)
        ck, cv = bf(pc["key"]), bf(pc["value"])
        cs = torch.from_numpy(pc["slot_mapping"]).to(dev)
        n_ch = max(3, min(K, 200))

        def chunk_write(ev):
            flush_l2()
            ev[0].record()
            kvq.kvq_write_cache(cache, ck, cv, cs)
            ev[1].record()

        for _ in range(3):
            chunk_write(mk())
        evs = [mk() for _ in range(n_ch)]
        for ev in evs:
            chunk_write(ev)
        torch.cuda.synchronize()
        us = max_over_ranks([float(np.median([e[0].elapsed_time(e[1]) for e in evs])) * 1e3],
                            dev)[0]
        cbytes = C * (2 * wl.num_kv_heads * wl.head_dim * 2 + kv_bytes_per_token(wl) + 8)
        chunk = {"tokens": C, "us": us, "tok_s": C / us * 1e6, "gbs": cbytes / us / 1e3,
                 "frac_of_hbm": cbytes / us / 1e3 / hbm, "steps": n_ch,
                 "stat": "median, L2 flushed before each write"}

    # end to end through the public API: pinned host inputs in, result out
    e2e = None
    if not args.no_e2e:
        pin = lambda t: t.cpu().pin_memory()
        h_in = [pin(x) for x in (key, value, query, slots, block_table, ctx_lens)]
        d_in = [torch.empty_like(x) for x in (key, value, query, slots, block_table, ctx_lens)]
        h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        n_e2e = max(1, min(args.e2e_steps, K))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

        def e2e_step():
            for h, d in zip(h_in, d_in):
                d.copy_(h, non_blocking=True)
            kvq.kvq_write_cache(cache, d_in[0], d_in[1], d_in[3])
            kvq.kvq_paged_decode(cache, d_in[2], out, d_in[4], d_in[5], wl.max_context_len,
                                 sm_scale, ws, P)
            h_out.copy_(out, non_blocking=True)

        for _ in range(3):
            e2e_step()
        torch.cuda.synchronize()
        e0.record()
        for _ in range(n_e2e):
            e2e_step()
        e1.record()
        torch.cuda.synchronize()
        t_e2e = max_over_ranks([e0.elapsed_time(e1) / 1e3], dev)[0]
        h2d = sum(x.numel() * x.element_size() for x in h_in)
        e2e = {"value": world * dbytes * n_e2e / t_e2e / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": h_out.numel() * 2,
               "steps": n_e2e, "ms_per_step": 1e3 * t_e2e / n_e2e}

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
    launches = 2 * K  # one write and one decode launch per step
    line = {
        "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": 1e3 * (t_write + t_dec) / K,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u8",
        "data": "synthetic",
        "config": {"workload": args.workload, "num_seqs": wl.num_seqs,
                   "num_q_heads": wl.num_q_heads, "num_kv_heads": wl.num_kv_heads,
                   "head_dim": wl.head_dim, "block_size": wl.block_size,
                   "k_fmt": wl.k_fmt, "v_fmt": wl.v_fmt, "kvarn": wl.kvarn,
                   "context_tokens": int(wl.context_lens.sum()),
                   "decode_ctas": P or "auto", "l2": "flushed before the write and before the decode (2xL2 memset, "
                   "then a 2xL2 read), outside the timed events"},
        "decode_tok_s": world * wl.num_seqs * K / t_dec,
        "decode_us": 1e6 * t_dec / K, "decode_us_pct": pct(d_ms),
        "decode_split": ws_bytes > 0,
        "cache_write_tok_s": world * wl.num_tokens * K / t_write,
        "cache_write_gbs": world * wbytes * K / t_write / 1e9,
        "cache_write_us": 1e6 * t_write / K, "cache_write_us_pct": pct(w_ms),
        "cache_write_frac_of_hbm": (wbytes * K / t_write / 1e9) / hbm,
        "decode_bytes": dbytes, "write_bytes": wbytes,
        "wall_s_timed_region": wall,
        # the dominant kernel of the step (largest share of its time) first
        "roofline": rl_write if t_write >= t_dec else rl_decode,
        "roofline_decode": rl_decode,
        "roofline_write": rl_write,
        "decode_frac_of_hbm": gbs / world / hbm,
        "e2e": e2e,
        "decode_step_append": step_lat,
        "prefill_chunk_write": chunk,
        "gpu_launches": launches,
        "clocks": clocks,
        "cpu_baseline": cpu,
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
