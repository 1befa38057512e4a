"""The decode kernel's bounded pipeline waits, made to run out on purpose.

Every mbarrier wait of the decode kernel polls a bounded number of times; the
first wait that runs out raises KVQ_DEVERR_TIMEOUT, and its CTA stops loading,
publishes nothing and returns once no copy it issued is in flight.  The test
hook kvq_debug_arm_wait_timeout makes one CTA's producer never issue the loads
of one tile (nothing is in flight for it, and nothing faults): the waits for
that tile run out, the launch ends by itself within the short poll limit, the
error word says so, and the next launch (the hook disarms itself) gives the
same output as before on the same context."""
import time

import numpy as np
import pytest

from quantized_paged_kv_kvq_gb300 import kvq
from quantized_paged_kv_kvq_gb300 import workloads as W

from kvq_testing import GpuRun, append_step, out_numpy

pytestmark = pytest.mark.gpu

POLLS = 1 << 14

CASES = {
    # name: (workload, overrides, CTAs, tile withheld in CTA 0's range)
    "int8_first_tile": ("llama8b_int8", dict(num_seqs=4, ctx_lo=300, ctx_hi=600), 4, 0),
    "int8_after_refills": ("llama8b_int8", dict(num_seqs=4, ctx_lo=300, ctx_hi=600), 4, 10),
    "int8_8_token_pages": ("llama8b_int8", dict(num_seqs=4, ctx_lo=300, ctx_hi=600,
                                               block_size=8), 4, 5),
    "int8_short_ranges": ("llama8b_int8", dict(num_seqs=4, ctx_lo=300, ctx_hi=600), 16, 1),
    "kvarn": ("kvarn_131k", dict(num_seqs=2, ctx_lo=500, ctx_hi=900), 5, 3),
    "int4": ("llama70b_int4", dict(num_seqs=3, ctx_lo=400, ctx_hi=900), 6, 2),
}


@pytest.mark.parametrize("case", list(CASES))
def test_a_wait_that_runs_out_ends_the_launch(case):
    name, kw, ctas, tile = CASES[case]
    wl = W.workload(name, **kw)
    g = GpuRun(wl)
    g.write()
    tiles = int(((wl.context_lens + 15) // 16).sum())
    assert tile < tiles // ctas  # the tile lies inside CTA 0's range
    ref = out_numpy(g.decode(num_ctas=ctas))
    assert kvq.kvq_get_device_error() == 0
    kvq.kvq_debug_arm_wait_timeout(POLLS, 0, tile)
    t0 = time.perf_counter()
    g.decode(num_ctas=ctas)
    bits = kvq.kvq_get_device_error()  # synchronizes with the launch
    elapsed = time.perf_counter() - t0
    assert bits & kvq.DEVERR_TIMEOUT, f"no timeout reported (bits {bits})"
    assert elapsed < 5.0, f"the launch took {elapsed:.2f} s to give up"
    # the hook disarmed itself and the context is still usable
    again = out_numpy(g.decode(num_ctas=ctas))
    assert kvq.kvq_get_device_error() == 0
    assert np.array_equal(again, ref)


def test_a_wait_that_runs_out_in_the_fused_append():
    wl = W.workload("llama8b_int8", num_seqs=4, ctx_lo=300, ctx_hi=600)
    kvq.kvq_debug_arm_wait_timeout(POLLS, 0, 4)
    append_step(wl, num_ctas=4)
    assert kvq.kvq_get_device_error() & kvq.DEVERR_TIMEOUT
    _, out = append_step(wl, num_ctas=4)
    assert kvq.kvq_get_device_error() == 0
    assert np.all(np.isfinite(out_numpy(out)))
