"""Standalone rotation on the GPU: bit-exact vs the oracle's float32 butterfly."""
import numpy as np
import pytest
import torch

from oracle import hadamard as OH
from quantized_paged_kv_kvq_gb300 import kvq
from quantized_paged_kv_kvq_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("inverse", [False, True])
@pytest.mark.parametrize("with_signs", [False, True])
def test_hadamard_bitexact(d, dtype, inverse, with_signs):
    rng = np.random.default_rng(d + 7 * inverse)
    rows = 1000 + 3  # ragged tail of a warp's row group
    x = (rng.standard_normal((rows, d)) * rng.uniform(0.01, 100, (rows, 1))).astype(np.float32)
    if dtype == "bf16":
        x = W.round_to_bf16(x)
    signs = np.where(rng.integers(0, 2, d) == 0, 1, -1).astype(np.int8) if with_signs else None
    xt = torch.from_numpy(x).cuda()
    if dtype == "bf16":
        xt = xt.to(torch.bfloat16)
    st = None if signs is None else torch.from_numpy(signs).cuda()
    kvq.kvq_hadamard(xt, st, inverse)
    got = xt.float().cpu().numpy()
    ref = OH.hadamard_rows(x, signs, inverse, dtype)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


def test_hadamard_round_trip_and_orthonormality():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((4096, 128)).astype(np.float32)
    signs = torch.from_numpy(np.where(rng.integers(0, 2, 128) == 0, 1, -1).astype(np.int8)).cuda()
    xt = torch.from_numpy(x).cuda()
    kvq.kvq_hadamard(xt, signs, False)
    y = xt.cpu().numpy()
    assert np.allclose(np.linalg.norm(y, axis=1), np.linalg.norm(x, axis=1), rtol=1e-5)
    kvq.kvq_hadamard(xt, signs, True)
    assert np.allclose(xt.cpu().numpy(), x, atol=1e-5)


def test_hadamard_empty_is_noop():
    x = torch.empty((0, 128), dtype=torch.float32, device="cuda")
    kvq.kvq_hadamard(x)
