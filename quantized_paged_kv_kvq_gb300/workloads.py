"""Seeded synthetic workloads for the quantized paged KV cache.

This module only draws random inputs (queries, keys, values, context lengths,
block tables, slot mappings, the rotation sign vector).  It holds none of the
method's arithmetic: no scale, no quantization, no attention.  Both the CUDA
path and the CPU oracle are fed from here, so they see identical inputs.

The shapes stand in for the serving workloads the source pages measure on
(Llama-3-8B on one L4 in vLLM PR #4893 'Load FP8 kv-cache scaling factors from
checkpoints', benchmark table; Llama 3 70B in vLLM issue #4025 'Support for
4-bit KV Cache in paged-attention op', thread): only the attention head shapes
are taken, no model weights and no dataset content.

Every floating point tensor is returned as float32 whose values are exactly
representable in bfloat16 (the cache-write input dtype), rounded to nearest
with ties to even from a float32 normal draw.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import numpy as np

# Cache formats understood by the library (names mirror include/kvq.h).
FORMATS = ("bf16", "int8", "fp8_e4m3", "fp8_e5m2", "int4_asym", "uint8_asym")


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round a float32 array to the nearest bfloat16 value (ties to even).

    Plain input preparation: the generator draws float32 normals and hands out
    bfloat16-valued tensors.  Returns float32 holding exact bf16 values.
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return (rounded.astype(np.uint32) << 16).view(np.float32)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Upper 16 bits of float32 values that are exact bfloat16 numbers."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    return (x.view(np.uint32) >> 16).astype(np.uint16)


@dataclass
class Workload:
    name: str
    seed: int
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    k_fmt: str
    v_fmt: str
    kvarn: bool
    # per-tensor scale rule for symmetric formats: "absmax/127", "absmax/448" or "1.0"
    k_scale_rule: Optional[str]
    v_scale_rule: Optional[str]
    context_lens: np.ndarray  # int32 [S]
    block_table: np.ndarray  # int32 [S, max_blocks]; -1 past the last used block
    num_blocks: int
    slot_mapping: np.ndarray  # int64 [T]; token order = sequences concatenated
    key: np.ndarray  # float32 (bf16-exact) [T, Hkv, D]
    value: np.ndarray  # float32 (bf16-exact) [T, Hkv, D]
    query: np.ndarray  # float32 (bf16-exact) [S, Hq, D]
    signs: Optional[np.ndarray] = None  # int8 [D] of +-1 (rotation diagonal)
    extra: dict = field(default_factory=dict)

    @property
    def num_tokens(self) -> int:
        return int(self.slot_mapping.shape[0])

    @property
    def gqa(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens.max()) if self.context_lens.size else 0

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_table.shape[1])


def _paged_layout(rng, context_lens, block_size, spare_blocks):
    """Random block permutation: each sequence gets ceil(ctx/bs) blocks."""
    need = [(int(c) + block_size - 1) // block_size for c in context_lens]
    total = int(sum(need))
    num_blocks = total + spare_blocks
    perm = rng.permutation(num_blocks).astype(np.int32)
    max_blocks = max(max(need) if need else 1, 1)
    table = np.full((len(need), max_blocks), -1, dtype=np.int32)
    pos = 0
    for s, n in enumerate(need):
        table[s, :n] = perm[pos:pos + n]
        pos += n
    return table, num_blocks


def slots_for_context(context_lens, block_table, block_size) -> np.ndarray:
    """Slot of every context token, sequences concatenated (slot = block*bs + offset)."""
    out = []
    for s, ctx in enumerate(context_lens):
        t = np.arange(int(ctx), dtype=np.int64)
        out.append(block_table[s, t // block_size].astype(np.int64) * block_size + t % block_size)
    return np.concatenate(out) if out else np.zeros(0, np.int64)


def _normal(rng, shape):
    return rng.standard_normal(size=shape, dtype=np.float32)


def _with_outliers(rng, x, channels_per_head, factor):
    """Multiply `channels_per_head` seeded channels of every kv-head by `factor`."""
    t, hkv, d = x.shape
    for h in range(hkv):
        ch = rng.choice(d, size=channels_per_head, replace=False)
        x[:, h, ch] *= np.float32(factor)
    return x


def _per_token_magnitude(rng, x, sigma):
    """Scale every (token, head) row by exp(N(0, sigma)) so row norms differ."""
    t, hkv, _ = x.shape
    m = np.exp(rng.normal(0.0, sigma, size=(t, hkv, 1))).astype(np.float32)
    return x * m


def make_workload(
    name: str,
    seed: int,
    num_seqs: int,
    num_q_heads: int,
    num_kv_heads: int,
    head_dim: int,
    block_size: int,
    ctx_lo: int,
    ctx_hi: int,
    k_fmt: str,
    v_fmt: str,
    k_scale_rule: Optional[str],
    v_scale_rule: Optional[str],
    kvarn: bool = False,
    k_outliers: tuple = (0, 1.0),
    token_magnitude_sigma: float = 0.0,
    spare_blocks: int = 4,
    context_lens: Optional[np.ndarray] = None,
    with_data: bool = True,
) -> Workload:
    # two independent streams: the paged layout (lengths, block permutation) and
    # the tensor data, so that changing the block size keeps the same K/V/q
    rng = np.random.Generator(np.random.PCG64(seed))
    if context_lens is None:
        context_lens = rng.integers(ctx_lo, ctx_hi + 1, size=num_seqs).astype(np.int32)
    else:
        context_lens = np.asarray(context_lens, dtype=np.int32)
    table, nb = _paged_layout(rng, context_lens, block_size, spare_blocks)
    slots = slots_for_context(context_lens, table, block_size)
    t = int(slots.shape[0])
    recipe = dict(k_outliers=tuple(k_outliers), token_magnitude_sigma=token_magnitude_sigma)
    if not with_data:  # the paged layout only; tensors come from device_data()
        signs = None
        if kvarn:
            srng = np.random.Generator(np.random.PCG64([seed, 2]))
            signs = np.where(srng.integers(0, 2, size=head_dim) == 0, 1, -1).astype(np.int8)
        return Workload(
            name=name, seed=seed, num_seqs=num_seqs, num_q_heads=num_q_heads,
            num_kv_heads=num_kv_heads, head_dim=head_dim, block_size=block_size,
            k_fmt=k_fmt, v_fmt=v_fmt, kvarn=kvarn, k_scale_rule=k_scale_rule,
            v_scale_rule=v_scale_rule, context_lens=context_lens, block_table=table,
            num_blocks=nb, slot_mapping=slots, key=None, value=None, query=None, signs=signs,
            extra=recipe)
    rng = np.random.Generator(np.random.PCG64([seed, 1]))
    key = _normal(rng, (t, num_kv_heads, head_dim))
    if k_outliers[0]:
        key = _with_outliers(rng, key, k_outliers[0], k_outliers[1])
    value = _normal(rng, (t, num_kv_heads, head_dim))
    if token_magnitude_sigma:  # keys only: values keep unit scale
        key = _per_token_magnitude(rng, key, token_magnitude_sigma)
    query = _normal(rng, (num_seqs, num_q_heads, head_dim))
    signs = None
    if kvarn:
        # d_i = +1 where bit i of a seeded 64-bit draw stream is 0, else -1
        words = rng.integers(0, 2**63, size=(head_dim + 63) // 64, dtype=np.int64).astype(np.uint64)
        bits = np.array([(int(words[i // 64]) >> (i % 64)) & 1 for i in range(head_dim)])
        signs = np.where(bits == 0, 1, -1).astype(np.int8)
    return Workload(
        name=name, seed=seed, num_seqs=num_seqs, num_q_heads=num_q_heads,
        num_kv_heads=num_kv_heads, head_dim=head_dim, block_size=block_size,
        k_fmt=k_fmt, v_fmt=v_fmt, kvarn=kvarn, k_scale_rule=k_scale_rule,
        v_scale_rule=v_scale_rule, context_lens=context_lens, block_table=table,
        num_blocks=nb, slot_mapping=slots, key=round_to_bf16(key),
        value=round_to_bf16(value), query=round_to_bf16(query), signs=signs, extra=recipe,
    )


# The five workloads (and the e5m2 variant of the third), by what they are.
WORKLOADS = {
    # tiny int8 paged decode, one layer
    "tiny_int8": dict(num_seqs=4, num_q_heads=8, num_kv_heads=2, head_dim=64, block_size=16,
                      ctx_lo=17, ctx_hi=200, k_fmt="int8", v_fmt="int8",
                      k_scale_rule="absmax/127", v_scale_rule="absmax/127"),
    # Llama-3-8B-shaped int8 decode layer
    "llama8b_int8": dict(num_seqs=64, num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=16,
                         ctx_lo=256, ctx_hi=4096, k_fmt="int8", v_fmt="int8",
                         k_scale_rule="absmax/127", v_scale_rule="absmax/127",
                         k_outliers=(4, 10.0)),
    # same shape, K as E4M3 bytes with a per-tensor scale, V int8; batch 128
    "llama8b_e4m3k_int8v": dict(num_seqs=128, num_q_heads=32, num_kv_heads=8, head_dim=128,
                                block_size=16, ctx_lo=512, ctx_hi=8192, k_fmt="fp8_e4m3",
                                v_fmt="int8", k_scale_rule="absmax/448",
                                v_scale_rule="absmax/127", k_outliers=(4, 10.0)),
    # same, K and V fp8 e5m2 at scale 1.0 (uncalibrated)
    "llama8b_e5m2": dict(num_seqs=128, num_q_heads=32, num_kv_heads=8, head_dim=128,
                         block_size=16, ctx_lo=512, ctx_hi=8192, k_fmt="fp8_e5m2",
                         v_fmt="fp8_e5m2", k_scale_rule="1.0", v_scale_rule="1.0",
                         k_outliers=(4, 10.0)),
    # the same Llama-3-8B shape and inputs with the unquantized 16-bit cache
    # (the --kv-cache-dtype auto baseline every quantized format is compared with)
    "llama8b_bf16": dict(num_seqs=64, num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=16,
                         ctx_lo=256, ctx_hi=4096, k_fmt="bf16", v_fmt="bf16",
                         k_scale_rule=None, v_scale_rule=None, k_outliers=(4, 10.0)),
    # Llama-3-70B-shaped INT4 asymmetric decode layer (GQA 8)
    "llama70b_int4": dict(num_seqs=32, num_q_heads=64, num_kv_heads=8, head_dim=128,
                          block_size=16, ctx_lo=8192, ctx_hi=32768, k_fmt="int4_asym",
                          v_fmt="int4_asym", k_scale_rule=None, v_scale_rule=None,
                          k_outliers=(8, 8.0)),
    # KVarN-style long context: 4 x 131072 tokens, block size 32
    "kvarn_131k": dict(num_seqs=4, num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=32,
                       ctx_lo=131072, ctx_hi=131072, k_fmt="int4_asym", v_fmt="uint8_asym",
                       k_scale_rule=None, v_scale_rule=None, kvarn=True,
                       k_outliers=(4, 10.0), token_magnitude_sigma=0.5),
}

SEEDS = {"tiny_int8": 1001, "llama8b_int8": 1002, "llama8b_bf16": 1002, "llama8b_e4m3k_int8v": 1003,
         "llama8b_e5m2": 1013, "llama70b_int4": 1004, "kvarn_131k": 1005}


def workload(name: str, **overrides) -> Workload:
    """Build a named workload; `overrides` may shrink it (e.g. num_seqs, ctx_hi)."""
    kw = dict(WORKLOADS[name])
    kw.update(overrides)
    seed = kw.pop("seed", SEEDS[name])
    return make_workload(name=name, seed=seed, **kw)


def device_data(wl: Workload, device, seed: Optional[int] = None) -> dict:
    """The tensors of a layout-only workload (with_data=False), drawn on the
    device with torch's generator by the same recipe as make_workload: normal
    q, K, V; the seeded outlier channels of K; KVarN's per-row magnitudes of
    K; every value rounded to bfloat16 (nearest, ties to even).  The values
    differ from the numpy stream (another generator) but follow the same
    distributions; used where only sizes and statistics matter (timing).
    Returns bf16 tensors key, value [T, Hkv, D] and query [S, Hq, D]."""
    import torch
    seed = wl.seed if seed is None else seed
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    t, hkv, d = wl.num_tokens, wl.num_kv_heads, wl.head_dim
    rng = np.random.Generator(np.random.PCG64([seed, 3]))

    def normal(shape):
        return torch.randn(shape, generator=g, device=device, dtype=torch.float32)

    key = normal((t, hkv, d))
    n_out, factor = wl.extra.get("k_outliers", (0, 1.0))
    if n_out:
        for h in range(hkv):
            ch = torch.from_numpy(rng.choice(d, size=n_out, replace=False)).to(device)
            key[:, h, ch] *= float(factor)
    sigma = wl.extra.get("token_magnitude_sigma", 0.0)
    if sigma:
        key *= torch.exp(torch.randn((t, hkv, 1), generator=g, device=device) * sigma)
    value = normal((t, hkv, d))
    query = normal((wl.num_seqs, wl.num_q_heads, d))
    return dict(key=key.to(torch.bfloat16), value=value.to(torch.bfloat16),
                query=query.to(torch.bfloat16))


def mixed_pages(wl: Workload, block_sizes=(16, 64), seed: Optional[int] = None,
                spare_blocks: int = 4) -> dict:
    """Lay wl's sequences out over page classes of different sizes (one pool per
    class): sequence s takes a seeded class; its pages are a random permutation
    within that class's pool.  Returns seq_class (uint8 [S]), block_table
    (int32 [S, max_context_len / smallest page size], ids in the sequence's
    pool, -1 past its pages),
    num_blocks per class, and per class the token indices (into wl's token
    order, sequences concatenated) and their slots in that pool."""
    rng = np.random.Generator(np.random.PCG64([wl.seed if seed is None else seed, 4]))
    S = wl.num_seqs
    seq_class = rng.integers(0, len(block_sizes), size=S).astype(np.uint8)
    need = [(int(c) + block_sizes[k] - 1) // block_sizes[k]
            for c, k in zip(wl.context_lens, seq_class)]
    # the table is as wide as max_context_len at the smallest page size
    width = max(-(-int(wl.max_context_len) // min(block_sizes)), 1)
    table = np.full((S, width), -1, np.int32)
    num_blocks = []
    for k, bs in enumerate(block_sizes):
        members = [s for s in range(S) if seq_class[s] == k]
        total = sum(need[s] for s in members) + spare_blocks
        perm = rng.permutation(total).astype(np.int32)
        pos = 0
        for s in members:
            table[s, :need[s]] = perm[pos:pos + need[s]]
            pos += need[s]
        num_blocks.append(total)
    starts = np.concatenate([[0], np.cumsum(wl.context_lens.astype(np.int64))])
    tokens, slots = [], []
    for k, bs in enumerate(block_sizes):
        idx, sl = [], []
        for s in range(S):
            if seq_class[s] != k:
                continue
            t = np.arange(int(wl.context_lens[s]), dtype=np.int64)
            idx.append(starts[s] + t)
            sl.append(table[s, t // bs].astype(np.int64) * bs + t % bs)
        tokens.append(np.concatenate(idx) if idx else np.zeros(0, np.int64))
        slots.append(np.concatenate(sl) if sl else np.zeros(0, np.int64))
    return dict(seq_class=seq_class, block_table=table, num_blocks=num_blocks,
                block_sizes=tuple(block_sizes), tokens=tokens, slots=slots)


def prefill_chunk(wl: Workload, num_tokens: int, seed: int) -> dict:
    """A prefill chunk of `num_tokens` new tokens for sequence 0 of `wl`,
    written at positions [0, num_tokens) of that sequence's blocks."""
    rng = np.random.Generator(np.random.PCG64(seed))
    d, hkv = wl.head_dim, wl.num_kv_heads
    key = _normal(rng, (num_tokens, hkv, d))
    value = _normal(rng, (num_tokens, hkv, d))
    t = np.arange(num_tokens, dtype=np.int64)
    if num_tokens > int(wl.context_lens[0]):
        raise ValueError("chunk longer than sequence 0")
    slots = wl.block_table[0, t // wl.block_size].astype(np.int64) * wl.block_size + t % wl.block_size
    return dict(key=round_to_bf16(key), value=round_to_bf16(value), slot_mapping=slots)
