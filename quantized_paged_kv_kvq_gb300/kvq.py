"""Python binding of libkvq.so (argument marshalling only).

Every function here has the name of the C entry point it calls and does
nothing but turn torch tensors into pointers and sizes; all work runs in the
library's CUDA kernels on the current torch stream.  The library must have
been built (quantized_paged_kv_kvq_gb300.build); importing this module
without it raises, and there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkvq.so")

FMT = {"int8": 1, "fp8_e4m3": 2, "fp8_e5m2": 3, "int4_asym": 4, "uint8_asym": 5, "bf16": 6}
FLAG_VARNORM_ROTATE = 1
STATUS = {0: "KVQ_OK", 1: "KVQ_ERR_INVALID_ARGUMENT", 2: "KVQ_ERR_UNSUPPORTED",
          3: "KVQ_ERR_WORKSPACE", 4: "KVQ_ERR_CUDA"}
DEVERR_SLOT_RANGE = 1
DEVERR_BLOCK_RANGE = 2
DEVERR_CONTEXT_RANGE = 4
DEVERR_COMBINE = 8
DEVERR_TIMEOUT = 16
DEVERR_CLASS_RANGE = 32
DEVERR_QUERY_RANGE = 64


class KvqError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {STATUS.get(status, status)}")
        self.status = status


class _CacheDesc(ctypes.Structure):
    _fields_ = [("k_fmt", ctypes.c_int32), ("v_fmt", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("block_size", ctypes.c_int32), ("num_blocks", ctypes.c_int32),
                ("flags", ctypes.c_uint32), ("k_scale", ctypes.c_float),
                ("v_scale", ctypes.c_float), ("k_meta", ctypes.c_void_p),
                ("v_meta", ctypes.c_void_p), ("signs", ctypes.c_void_p),
                ("k_head_scales", ctypes.c_void_p), ("v_head_scales", ctypes.c_void_p)]


_P = ctypes.c_void_p
_I32, _I64, _F32, _SZ = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
_DESC = ctypes.POINTER(_CacheDesc)

# name -> (restype, argtypes)
SIGNATURES = {
    "kvq_write_cache": (_I32, [_DESC, _P, _P, _P, _P, _I64, _I64, _P, _I64, _P]),
    "kvq_decode_workspace_size": (_I32, [_DESC, _I32, _I32, _I32, ctypes.POINTER(_SZ)]),
    "kvq_decode_workspace_size_ex": (_I32, [_DESC, _I32, _I32, _I32, _I32, ctypes.POINTER(_SZ)]),
    "kvq_paged_decode": (_I32, [_DESC, _P, _P, _P, _P, _I32, _I32, _P, _I32, _P, _I32, _F32, _P,
                                _SZ, _P]),
    "kvq_paged_decode_ex": (_I32, [_DESC, _P, _P, _P, _P, _I32, _I32, _P, _I32, _P, _I32, _F32,
                                   _I32, _P, _SZ, _P]),
    "kvq_decode_append": (_I32, [_DESC, _P, _P, _P, _P, _I64, _I64, _P, _P, _I32, _I32, _P, _I32,
                                 _P, _I32, _F32, _I32, _P, _SZ, _P]),
    "kvq_paged_decode_static": (_I32, [_DESC, _P, _P, _P, _P, _I32, _I32, _P, _I32, _P, _I32,
                                       _F32, _I32, _P]),
    "kvq_decode_mixed": (_I32, [_DESC, _I32, ctypes.POINTER(_P), ctypes.POINTER(_P), _P, _P, _P,
                                _I64, _I64, _P, _P, _I32, _I32, _P, _I32, _P, _I32, _F32, _I32,
                                _P, _SZ, _P]),
    "kvq_paged_decode_static_capacity": (_SZ, []),
    "kvq_hadamard": (_I32, [_P, _I32, _I64, _I32, _P, _I32, _P]),
    "kvq_calibrate_scale": (_I32, [_P, _I64, _F32, _P, _P]),
    "kvq_calibrate_head_scales": (_I32, [_P, _I64, _I32, _I32, _I64, _F32, _P, _P]),
    "kvq_debug_arm_wait_timeout": (_I32, [_I32, _I32, _I32]),
    "kvq_get_device_error": (_I32, [_P, ctypes.POINTER(ctypes.c_uint32)]),
    "kvq_status_string": (ctypes.c_char_p, [_I32]),
    "kvq_version": (ctypes.c_char_p, []),
}

_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libkvq.so (once) and declare its entry points; raises if absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with "
                          "`python -m quantized_paged_kv_kvq_gb300.build`")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _check(status: int, what: str):
    if status != 0:
        raise KvqError(status, what)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


@dataclass
class KVCache:
    """One layer's paged cache: caller-owned device tensors + description.

    k_cache / v_cache: uint8 [num_blocks, block_size, num_kv_heads, row_bytes]
    k_meta / v_meta:   fp16 [num_blocks, num_kv_heads, F, block_size] (asymmetric formats)
    signs:             int8 [head_dim] of +-1 (KVarN rotation) or None
    """
    k_fmt: str
    v_fmt: str
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    k_meta: Optional[torch.Tensor] = None
    v_meta: Optional[torch.Tensor] = None
    k_scale: float = 1.0
    v_scale: float = 1.0
    varnorm_rotate: bool = False
    signs: Optional[torch.Tensor] = None
    k_head_scales: Optional[torch.Tensor] = None  # fp32 [num_kv_heads] (symmetric K)
    v_head_scales: Optional[torch.Tensor] = None  # fp32 [num_kv_heads] (symmetric V)

    def desc(self) -> _CacheDesc:
        ptr = lambda t: None if t is None else t.data_ptr()
        return _CacheDesc(FMT[self.k_fmt], FMT[self.v_fmt], self.num_kv_heads, self.head_dim,
                          self.block_size, self.num_blocks,
                          FLAG_VARNORM_ROTATE if self.varnorm_rotate else 0,
                          float(self.k_scale), float(self.v_scale), ptr(self.k_meta),
                          ptr(self.v_meta), ptr(self.signs), ptr(self.k_head_scales),
                          ptr(self.v_head_scales))


def row_bytes(fmt: str, head_dim: int) -> int:
    return head_dim // 2 if fmt == "int4_asym" else 2 * head_dim if fmt == "bf16" else head_dim


def meta_fields(fmt: str, varnorm_rotate: bool) -> int:
    if fmt in ("int4_asym", "uint8_asym"):
        return 3 if varnorm_rotate else 2
    return 0


def alloc_kv_cache(k_fmt, v_fmt, num_blocks, block_size, num_kv_heads, head_dim,
                   k_scale=1.0, v_scale=1.0, varnorm_rotate=False, signs=None,
                   device="cuda", fill: Optional[int] = None) -> KVCache:
    """Allocate (with torch) the device tensors of a cache; `fill` poisons them."""
    def codes(fmt):
        t = torch.empty((num_blocks, block_size, num_kv_heads, row_bytes(fmt, head_dim)),
                        dtype=torch.uint8, device=device)
        if fill is not None:
            t.fill_(fill)
        return t

    def meta(fmt):
        nf = meta_fields(fmt, varnorm_rotate)
        if not nf:
            return None
        t = torch.empty((num_blocks, num_kv_heads, nf, block_size), dtype=torch.float16,
                        device=device)
        if fill is not None:
            t.view(torch.int16).fill_(fill * 0x101 - (0x10000 if fill * 0x101 >= 0x8000 else 0))
        return t

    return KVCache(k_fmt, v_fmt, num_kv_heads, head_dim, block_size, num_blocks, codes(k_fmt),
                   codes(v_fmt), meta(k_fmt), meta(v_fmt), k_scale, v_scale, varnorm_rotate,
                   signs)


def kvq_write_cache(cache: KVCache, key: torch.Tensor, value: torch.Tensor,
                    slot_mapping: torch.Tensor, stream=None) -> None:
    """Quantize key/value (bf16 [T, Hkv, D], token stride free) into the cache."""
    lib = load_library()
    assert key.dtype == torch.bfloat16 and value.dtype == torch.bfloat16
    assert slot_mapping.dtype == torch.int64
    t = key.shape[0]
    d = cache.desc()
    st = lib.kvq_write_cache(ctypes.byref(d), _ptr(cache.k_cache), _ptr(cache.v_cache), _ptr(key),
                             _ptr(value), key.stride(0), value.stride(0), _ptr(slot_mapping), t,
                             _stream(stream))
    _check(st, "kvq_write_cache")


def kvq_decode_workspace_size(cache: KVCache, num_seqs: int, num_q_heads: int,
                              max_context_len: int, num_ctas: int = 0) -> int:
    lib = load_library()
    n = ctypes.c_size_t(0)
    d = cache.desc()
    st = lib.kvq_decode_workspace_size_ex(ctypes.byref(d), num_seqs, num_q_heads,
                                          max_context_len, num_ctas, ctypes.byref(n))
    _check(st, "kvq_decode_workspace_size")
    return int(n.value)


def _decode_call(fn_name, cache, query, out, block_table, context_lens, max_context_len,
                 sm_scale, workspace, num_ctas, stream):
    lib = load_library()
    assert query.dtype == torch.bfloat16 and out.dtype == torch.bfloat16
    assert query.is_contiguous() and out.is_contiguous()
    assert block_table.dtype == torch.int32 and context_lens.dtype == torch.int32
    assert block_table.is_contiguous()
    s, hq, _ = query.shape
    d = cache.desc()
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = getattr(lib, fn_name)(ctypes.byref(d), _ptr(cache.k_cache), _ptr(cache.v_cache),
                               _ptr(out), _ptr(query), s, hq, _ptr(block_table),
                               block_table.shape[1], _ptr(context_lens), max_context_len,
                               float(sm_scale), num_ctas, _ptr(workspace), ws_bytes,
                               _stream(stream))
    _check(st, fn_name)
    return out


def kvq_paged_decode(cache: KVCache, query: torch.Tensor, out: torch.Tensor,
                     block_table: torch.Tensor, context_lens: torch.Tensor, max_context_len: int,
                     sm_scale: float, workspace: Optional[torch.Tensor] = None,
                     num_ctas: int = 0, stream=None) -> torch.Tensor:
    """out[s, h] = softmax(sm_scale q k^T) v over the paged cache (bf16 [S, Hq, D])."""
    return _decode_call("kvq_paged_decode_ex", cache, query, out, block_table, context_lens,
                        max_context_len, sm_scale, workspace, num_ctas, stream)


def kvq_decode_append(cache: KVCache, new_key: torch.Tensor, new_value: torch.Tensor,
                      query: torch.Tensor, out: torch.Tensor, block_table: torch.Tensor,
                      context_lens: torch.Tensor, max_context_len: int, sm_scale: float,
                      workspace: Optional[torch.Tensor] = None, num_ctas: int = 0,
                      stream=None) -> torch.Tensor:
    """One decode step in one launch: row s of new_key / new_value (bf16 [S, Hkv, D],
    sequence stride free) is quantized into the cache at position context_lens[s] - 1,
    then out = the paged decode over the context including it."""
    lib = load_library()
    assert new_key.dtype == torch.bfloat16 and new_value.dtype == torch.bfloat16
    assert query.dtype == torch.bfloat16 and out.dtype == torch.bfloat16
    assert query.is_contiguous() and out.is_contiguous()
    assert block_table.dtype == torch.int32 and context_lens.dtype == torch.int32
    assert block_table.is_contiguous()
    s, hq, _ = query.shape
    d = cache.desc()
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib.kvq_decode_append(ctypes.byref(d), _ptr(cache.k_cache), _ptr(cache.v_cache),
                               _ptr(new_key), _ptr(new_value), new_key.stride(0),
                               new_value.stride(0), _ptr(out), _ptr(query), s, hq,
                               _ptr(block_table), block_table.shape[1], _ptr(context_lens),
                               max_context_len, float(sm_scale), num_ctas, _ptr(workspace),
                               ws_bytes, _stream(stream))
    _check(st, "kvq_decode_append")
    return out


def kvq_decode_mixed(classes, seq_class: torch.Tensor, query: torch.Tensor, out: torch.Tensor,
                     block_table: torch.Tensor, context_lens: torch.Tensor, max_context_len: int,
                     sm_scale: float, workspace: Optional[torch.Tensor] = None,
                     num_ctas: int = 0, new_key: Optional[torch.Tensor] = None,
                     new_value: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Decode (or, with new_key / new_value, the fused append step) over a cache
    of several page classes: `classes` is a list of KVCache, one pool per page
    size; seq_class (uint8 [S]) names each sequence's class, and block_table
    row s holds block ids of that class's pool."""
    lib = load_library()
    assert seq_class.dtype == torch.uint8 and seq_class.is_contiguous()
    assert query.dtype == torch.bfloat16 and out.dtype == torch.bfloat16
    assert query.is_contiguous() and out.is_contiguous()
    assert block_table.dtype == torch.int32 and context_lens.dtype == torch.int32
    assert block_table.is_contiguous()
    n = len(classes)
    descs = (_CacheDesc * n)(*[c.desc() for c in classes])
    kcs = (ctypes.c_void_p * n)(*[c.k_cache.data_ptr() for c in classes])
    vcs = (ctypes.c_void_p * n)(*[c.v_cache.data_ptr() for c in classes])
    s, hq, _ = query.shape
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    ks = 0 if new_key is None else new_key.stride(0)
    vs = 0 if new_value is None else new_value.stride(0)
    st = lib.kvq_decode_mixed(descs, n, kcs, vcs, _ptr(seq_class), _ptr(new_key),
                              _ptr(new_value), ks, vs, _ptr(out), _ptr(query), s, hq,
                              _ptr(block_table), block_table.shape[1], _ptr(context_lens),
                              max_context_len, float(sm_scale), num_ctas, _ptr(workspace),
                              ws_bytes, _stream(stream))
    _check(st, "kvq_decode_mixed")
    return out


def kvq_paged_decode_static(cache: KVCache, query: torch.Tensor, out: torch.Tensor,
                            block_table: torch.Tensor, context_lens: torch.Tensor,
                            max_context_len: int, sm_scale: float, num_ctas: int = 0,
                            stream=None) -> torch.Tensor:
    """kvq_paged_decode for callers that cannot allocate: the split-K scratch is
    the library's own fixed array (kvq_paged_decode_static_capacity() bytes)
    instead of a workspace tensor.  Calls that overlap on the GPU race on it."""
    lib = load_library()
    assert query.dtype == torch.bfloat16 and out.dtype == torch.bfloat16
    assert query.is_contiguous() and out.is_contiguous()
    assert block_table.dtype == torch.int32 and context_lens.dtype == torch.int32
    assert block_table.is_contiguous()
    s, hq, _ = query.shape
    d = cache.desc()
    st = lib.kvq_paged_decode_static(ctypes.byref(d), _ptr(cache.k_cache), _ptr(cache.v_cache),
                                     _ptr(out), _ptr(query), s, hq, _ptr(block_table),
                                     block_table.shape[1], _ptr(context_lens), max_context_len,
                                     float(sm_scale), num_ctas, _stream(stream))
    _check(st, "kvq_paged_decode_static")
    return out


def kvq_paged_decode_static_capacity() -> int:
    return int(load_library().kvq_paged_decode_static_capacity())


def kvq_hadamard(x: torch.Tensor, signs: Optional[torch.Tensor] = None, inverse: bool = False,
                 stream=None) -> torch.Tensor:
    """In-place rotation of the rows of x (float32 or bf16, [..., D], contiguous)."""
    lib = load_library()
    assert x.is_contiguous()
    dt = {torch.float32: 0, torch.bfloat16: 1}[x.dtype]
    dim = x.shape[-1]
    rows = x.numel() // dim if dim else 0
    st = lib.kvq_hadamard(_ptr(x), dt, rows, dim, _ptr(signs), int(inverse), _stream(stream))
    _check(st, "kvq_hadamard")
    return x


def kvq_calibrate_scale(x: torch.Tensor, qmax: float, out: torch.Tensor, stream=None):
    """out (device float32 [1]) <- absmax(x) / qmax (1.0 for an all-zero x)."""
    lib = load_library()
    assert x.dtype == torch.bfloat16 and x.is_contiguous() and out.dtype == torch.float32
    st = lib.kvq_calibrate_scale(_ptr(x), x.numel(), float(qmax), _ptr(out), _stream(stream))
    _check(st, "kvq_calibrate_scale")
    return out


def kvq_calibrate_head_scales(x: torch.Tensor, qmax: float, out: torch.Tensor, stream=None):
    """out (device float32 [Hkv]) <- per-kv-head absmax of x [T, Hkv, D] / qmax."""
    lib = load_library()
    assert x.dtype == torch.bfloat16 and x.dim() == 3 and out.dtype == torch.float32
    assert x.stride(2) == 1 and x.stride(1) == x.shape[2] and out.numel() == x.shape[1]
    st = lib.kvq_calibrate_head_scales(_ptr(x), x.shape[0], x.shape[1], x.shape[2], x.stride(0),
                                       float(qmax), _ptr(out), _stream(stream))
    _check(st, "kvq_calibrate_head_scales")
    return out


def kvq_debug_arm_wait_timeout(polls: int, cta: int, tile: int) -> None:
    """Test hook: the next decode launch polls each pipeline wait at most `polls`
    times, and CTA `cta` (first kv-head group) never loads its range's tile
    `tile`, so that a wait runs out (KVQ_DEVERR_TIMEOUT); one launch only."""
    _check(load_library().kvq_debug_arm_wait_timeout(polls, cta, tile),
           "kvq_debug_arm_wait_timeout")


def kvq_get_device_error(stream=None) -> int:
    """Synchronize, then read-and-clear the device error word (KVQ_DEVERR_* bits)."""
    lib = load_library()
    bits = ctypes.c_uint32(0)
    _check(lib.kvq_get_device_error(_stream(stream), ctypes.byref(bits)), "kvq_get_device_error")
    return int(bits.value)


def kvq_version() -> str:
    return load_library().kvq_version().decode()
