"""Host-side logic of bench.py, on CPU: the whole-job aggregation over ranks
(two gloo ranks), the algorithmic byte counts, and the reference arm (the
oracle) printing its JSON line."""
import io
import json
import os
import socket
import sys
from contextlib import redirect_stdout

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    # rank r "took" 1 + r seconds for 10 units of work
    t = bench.max_over_ranks([1.0 + rank, 0.5 * (rank + 1)])
    out[rank] = (t, bench.aggregate(t[:1] * world, [10.0] * world))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_and_aggregate_with_two_gloo_ranks():
    world = 2
    out = mp.Manager().dict()
    mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
    for r in range(world):
        t, value = out[r]
        assert t == [2.0, 1.0]  # element-wise maximum over the ranks
        assert value == pytest.approx(20.0 / 2.0)  # all units / the slowest time


def test_aggregate_single_rank_and_degenerate():
    assert bench.aggregate([2.0], [8.0]) == 4.0
    assert bench.aggregate([0.5, 2.0], [3.0, 5.0]) == 4.0
    assert bench.max_over_ranks([3.0, 1.5]) == [3.0, 1.5]


def test_algorithmic_bytes_match_the_layout():
    from quantized_paged_kv_kvq_gb300 import workloads as W
    wl = W.workload("llama8b_int8", num_seqs=3, ctx_lo=20, ctx_hi=40)
    # int8 K and V, 8 kv-heads x 128 dims, no metadata: 2048 bytes per token
    assert bench.kv_bytes_per_token(wl) == 2048
    ctx = int(wl.context_lens.sum())
    blocks = int(((wl.context_lens + 15) // 16).sum())
    q = 3 * 32 * 128 * 2
    assert bench.decode_bytes(wl) == ctx * 2048 + 2 * q + 4 * blocks + 4 * 3
    assert bench.write_bytes(wl) == wl.num_tokens * (2 * 8 * 128 * 2 + 2048 + 8)
    kv = W.workload("kvarn_131k", num_seqs=1, ctx_lo=40, ctx_hi=41)
    # int4 K (64 B) + uint8 V (128 B) + 3 fp16 metadata fields each, per kv-head
    assert bench.kv_bytes_per_token(kv) == 8 * (64 + 128 + 6 + 6)


def test_reference_arm_prints_its_line():
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.main(["--impl", "reference", "--steps", "2", "--warmup", "0",
                    "--workload", "tiny_int8"])
    line = json.loads(buf.getvalue().strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] == 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0
    assert line["config"]["workload"] == "tiny_int8"


def test_oracle_baseline_over_several_cores():
    """The all-cores oracle baseline runs concurrent single-thread processes and
    sums their rates; each process's rate is positive, so the sum exceeds none."""
    r = bench.cpu_baseline_all_cores("tiny_int8", 0.2, 2)
    assert r is not None and r["cores"] == 2 and r["value"] > 0
    one = bench.cpu_baseline_subprocess("tiny_int8", 0.2)
    assert one is not None and one["cores"] == 1 and one["value"] > 0
    assert isinstance(bench.cpu_model(), str) and bench.cpu_model()


def test_profiled_traffic_reads_json_sidecars(tmp_path, monkeypatch):
    """A sidecar counts only while its source hash is that of the kernel's
    current sources; a missing or malformed one gives None."""
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", tmp_path)
    assert bench.profiled_traffic("w", "decode_partition") is None
    monkeypatch.setattr(bench, "ROOT", ROOT)
    good = bench.source_hash(bench.DECODE_SOURCES)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "source_hash", lambda names: good)
    rec = {"kernel": "decode_partition", "workload": "w", "source_sha256_16": good,
           "dram_bytes_per_launch": 12345}
    (tmp_path / "profiles" / "decode_partition_w.json").write_text(json.dumps(rec))
    assert bench.profiled_traffic("w", "decode_partition") == 12345.0
    rec["source_sha256_16"] = "0" * 16
    (tmp_path / "profiles" / "decode_partition_w.json").write_text(json.dumps(rec))
    assert bench.profiled_traffic("w", "decode_partition") is None
    (tmp_path / "profiles" / "decode_partition_w.json").write_text("{not json")
    assert bench.profiled_traffic("w", "decode_partition") is None


def test_committed_sidecars_name_their_kernel_and_workload():
    import glob
    from quantized_paged_kv_kvq_gb300 import workloads as W
    for path in glob.glob(os.path.join(ROOT, "profiles", "*.json")):
        rec = json.load(open(path))
        assert rec["kernel"] in bench.KERNEL_SOURCES and rec["workload"] in W.WORKLOADS
        assert os.path.basename(path) == f"{rec['kernel']}_{rec['workload']}.json"
        assert int(rec["dram_bytes_per_launch"]) > 0


def test_layout_only_workload_has_the_same_layout():
    """The bench draws its tensors on the device but takes the paged layout
    (lengths, block table, slots) from the same seeded generator."""
    from quantized_paged_kv_kvq_gb300 import workloads as W
    for name, kw in (("llama8b_int8", dict(num_seqs=5, ctx_lo=10, ctx_hi=300)),
                     ("kvarn_131k", dict(num_seqs=2, ctx_lo=33, ctx_hi=70))):
        a = W.workload(name, **kw)
        b = W.workload(name, with_data=False, **kw)
        assert b.key is None and b.value is None and b.query is None
        for f in ("context_lens", "block_table", "slot_mapping"):
            assert np.array_equal(getattr(a, f), getattr(b, f))
        assert a.num_blocks == b.num_blocks and a.extra == b.extra
        if a.kvarn:
            assert b.signs is not None and set(np.unique(b.signs)) <= {-1, 1}
