"""Batches with more sequences than a decode CTA has threads, and at that
boundary.

A CTA finds its stream-K range with a block scan of the sequences' tile counts:
in one pass (a sequence per thread, with each sequence boundary weighted on the
partition's line) when the batch has at most as many sequences as threads, else
in chunks (no boundary weight).  Both partitions are checked against the oracle
over several grids, with empty sequences among the others, for 8 kv-heads per
CTA (256 threads) and for 2 (64 threads), the append path included."""
import numpy as np
import pytest

from quantized_paged_kv_kvq_gb300 import kvq
from quantized_paged_kv_kvq_gb300 import workloads as W

from kvq_testing import GpuRun, OracleRun, append_step, assert_attention_close, out_numpy

pytestmark = pytest.mark.gpu


def lens_mix(n, seed, hi):
    rng = np.random.default_rng(seed)
    lens = rng.integers(1, hi, size=n).astype(np.int32)
    lens[rng.random(n) < 0.1] = 0  # some empty sequences among the others
    return lens


@pytest.mark.parametrize("name,n", [("llama8b_int8", 256), ("llama8b_int8", 257),
                                    ("llama8b_int8", 300), ("tiny_int8", 64),
                                    ("tiny_int8", 65), ("tiny_int8", 150)])
def test_one_pass_and_chunked_range_scans(name, n):
    lens = lens_mix(n, 100 + n, 120)
    wl = W.workload(name, num_seqs=n, context_lens=lens)
    g = GpuRun(wl)
    g.write()
    ref = OracleRun(wl).decode()
    outs = {}
    for ctas in (0, 3, 64, 500):
        got = out_numpy(g.decode(num_ctas=ctas))
        assert_attention_close(got, ref, f"{name} n={n} ctas={ctas}")
        assert np.all(got[lens == 0] == 0)
        outs[ctas] = got
    assert np.array_equal(out_numpy(g.decode(num_ctas=64)), outs[64])  # deterministic
    assert kvq.kvq_get_device_error() == 0


@pytest.mark.parametrize("n", [256, 300])
def test_append_with_many_sequences(n):
    lens = lens_mix(n, 7 + n, 100)
    wl = W.workload("llama8b_int8", num_seqs=n, context_lens=lens)
    for ctas in (0, 5):
        g, out = append_step(wl, num_ctas=ctas)
        assert_attention_close(out_numpy(out), OracleRun(wl).decode(), f"append n={n} ctas={ctas}")
        assert kvq.kvq_get_device_error() == 0
