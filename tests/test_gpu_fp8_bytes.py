"""Every byte value through the decode's V conversion, exactly.

With a context of one token, softmax gives that token weight 1, so the output
is its dequantized value row: the code's value times the V scale, rounded to
bf16.  Rows holding all 256 byte values of the FP8 formats (E4M3, E5M2) and of
int8, with a power-of-two scale, make every product exact and every value
representable in bf16 (3 or 2 mantissa bits), so the output must equal the
oracle's table of the format bit for bit, NaN and infinity codes included
(OCP FP8 formats; int8 as two's complement); negative zero may come out as
+0, since the output is a sum that starts at +0."""
import numpy as np
import pytest
import torch

from oracle import formats as OF
from quantized_paged_kv_kvq_gb300 import kvq

pytestmark = pytest.mark.gpu

D, HKV, BS = 128, 2, 16


def byte_rows():
    """[seq, head, D] byte values: each of the 256 values in every sequence,
    in a different order per sequence (the lane mapping sees each byte at
    several dims)."""
    base = np.arange(256, dtype=np.uint8).reshape(HKV, D)
    rows = [base, base[:, ::-1], np.roll(base.reshape(-1), 77).reshape(HKV, D),
            np.random.default_rng(5).permutation(256).astype(np.uint8).reshape(HKV, D)]
    return np.stack(rows)


def bf16_bits_of(x64: np.ndarray) -> np.ndarray:
    """bf16 bit patterns of values that bf16 holds exactly (NaN: any NaN)."""
    f32 = x64.astype(np.float32)
    bits = f32.view(np.uint32)
    assert np.all(np.isnan(f32) | ((bits & 0xFFFF) == 0)), "value not exact in bf16"
    return (bits >> 16).astype(np.uint16)


@pytest.mark.parametrize("fmt", ["fp8_e4m3", "fp8_e5m2", "int8"])
@pytest.mark.parametrize("ctas", [1, 0])
def test_every_v_byte_decodes_exactly(fmt, ctas):
    rows = byte_rows()
    S = rows.shape[0]
    v_scale = 2.0 ** -4 if fmt != "fp8_e5m2" else 1.0
    cache = kvq.alloc_kv_cache(fmt, fmt, S, BS, HKV, D, 2.0 ** -3, v_scale, fill=0)
    for s in range(S):  # sequence s: one token, in block s
        cache.v_cache[s, 0] = torch.from_numpy(rows[s]).cuda()
    query = torch.randn(S, HKV, D, device="cuda").to(torch.bfloat16)
    out = torch.full_like(query, float("nan"))
    table = torch.arange(S, dtype=torch.int32, device="cuda").reshape(S, 1)
    lens = torch.ones(S, dtype=torch.int32, device="cuda")
    n = kvq.kvq_decode_workspace_size(cache, S, HKV, 1, ctas)
    ws = torch.empty(max(n, 16) // 4 + 4, dtype=torch.float32, device="cuda")
    kvq.kvq_paged_decode(cache, query, out, table, lens, 1, 0.0883883, ws, ctas)
    assert kvq.kvq_get_device_error() == 0
    got = out.view(torch.int16).cpu().numpy().view(np.uint16)
    want = OF.dequant_sym(rows.reshape(-1), fmt, v_scale).reshape(rows.shape)
    nan = np.isnan(want)
    got_f = out.float().cpu().numpy()
    assert np.array_equal(np.isnan(got_f), nan), f"{fmt}: NaN codes differ"
    zero = lambda b: np.where(b == 0x8000, 0, b)  # -0 and +0 (a sum that starts at +0)
    exp = zero(bf16_bits_of(want))
    bad = (zero(got) != exp) & ~nan
    assert not bad.any(), (f"{fmt}: bytes {np.unique(rows[bad]).tolist()[:16]} decode to "
                           f"{got[bad][:8].tolist()}, expected {exp[bad][:8].tolist()}")
    if fmt == "fp8_e5m2":  # the infinities are in the table
        assert np.isinf(got_f).sum() == 2 * S
