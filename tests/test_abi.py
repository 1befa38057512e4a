"""The C ABI without a GPU: the library loads, exports every declared entry
point, and rejects bad arguments on the host before touching CUDA."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kvq.h")


@pytest.fixture(scope="module")
def lib():
    from quantized_paged_kv_kvq_gb300 import build, kvq
    build.build()
    return kvq.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kvq_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_three_operations():
    names = declared_functions()
    for n in ("kvq_write_cache", "kvq_paged_decode", "kvq_hadamard"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_binding_covers_every_entry_point(lib):
    from quantized_paged_kv_kvq_gb300 import kvq
    assert set(declared_functions()) == set(kvq.SIGNATURES)


def test_status_strings(lib):
    from quantized_paged_kv_kvq_gb300 import kvq
    for code, name in kvq.STATUS.items():
        assert lib.kvq_status_string(code).decode() == name
    assert lib.kvq_version().decode().startswith("kvq")


def _desc(**kw):
    from quantized_paged_kv_kvq_gb300 import kvq
    base = dict(k_fmt=1, v_fmt=1, num_kv_heads=8, head_dim=128, block_size=16, num_blocks=10,
                flags=0, k_scale=0.1, v_scale=0.1, k_meta=None, v_meta=None, signs=None)
    base.update(kw)
    return kvq._CacheDesc(**base)


FAKE = 0x10000  # 16-byte aligned, never dereferenced: validation fails first


def _write(lib, desc, **kw):
    a = dict(k=FAKE, v=FAKE, key=FAKE, value=FAKE, ks=1024, vs=1024, slots=FAKE, n=4)
    a.update(kw)
    return lib.kvq_write_cache(ctypes.byref(desc) if desc is not None else None, a["k"], a["v"],
                               a["key"], a["value"], a["ks"], a["vs"], a["slots"], a["n"], None)


def test_write_validation(lib):
    ok_desc = _desc()
    assert _write(lib, None) == 1
    assert _write(lib, _desc(head_dim=96)) == 2
    assert _write(lib, _desc(block_size=4)) == 2
    assert _write(lib, _desc(block_size=24)) == 2
    assert _write(lib, _desc(k_fmt=9)) == 1
    assert _write(lib, _desc(k_scale=0.0)) == 1
    assert _write(lib, _desc(k_scale=float("nan"))) == 1
    assert _write(lib, _desc(k_fmt=4, v_fmt=4)) == 1  # asymmetric needs meta
    assert _write(lib, _desc(k_fmt=4, v_fmt=1, k_meta=FAKE)) == 2  # mixed families
    assert _write(lib, _desc(flags=1)) == 2  # rotation needs asymmetric formats
    assert _write(lib, _desc(flags=4)) == 1
    assert _write(lib, ok_desc, k=None) == 1
    assert _write(lib, ok_desc, key=FAKE + 2) == 1  # misaligned
    assert _write(lib, ok_desc, ks=100) == 1  # stride shorter than a token
    assert _write(lib, ok_desc, ks=1028) == 1  # stride not a multiple of 8
    assert _write(lib, ok_desc, n=-1) == 1
    assert _write(lib, ok_desc, n=0, k=None) == 0  # empty write is a no-op


def _decode(lib, desc, **kw):
    a = dict(k=FAKE, v=FAKE, out=FAKE, q=FAKE, s=4, hq=32, bt=FAKE, mb=64, cl=FAKE, mc=1024,
             sm=0.088, p=256, ws=None, wsb=0)
    a.update(kw)
    return lib.kvq_paged_decode_ex(ctypes.byref(desc), a["k"], a["v"], a["out"], a["q"], a["s"],
                                   a["hq"], a["bt"], a["mb"], a["cl"], a["mc"], a["sm"], a["p"],
                                   a["ws"], a["wsb"], None)


def test_head_scales_validation(lib):
    # per-kv-head scales belong to symmetric formats only
    assert _decode(lib, _desc(k_fmt=4, v_fmt=4, k_meta=FAKE, v_meta=FAKE,
                              k_head_scales=FAKE)) == 1
    assert _decode(lib, _desc(v_head_scales=FAKE + 2)) == 1  # misaligned
    st = lib.kvq_calibrate_head_scales(FAKE, 10, 8, 128, 8 * 128 - 8, 127.0, FAKE, None)
    assert st == 1  # token stride shorter than a token
    assert lib.kvq_calibrate_head_scales(FAKE, 10, 8, 60, 480, 127.0, FAKE, None) == 1  # D % 8
    assert lib.kvq_calibrate_head_scales(FAKE, 10, 8, 128, 1024, 0.0, FAKE, None) == 1


def test_decode_validation(lib):
    d = _desc()
    assert _decode(lib, d, hq=30) == 1  # not a multiple of the kv heads
    assert _decode(lib, d, hq=8 * 16) == 2  # GQA ratio above 8
    assert _decode(lib, d, p=-1) == 1  # negative CTA count
    assert _decode(lib, d, p=70000) == 1  # more CTAs than a grid dimension holds
    assert _decode(lib, d, mb=10) == 1  # block table shorter than max context
    assert _decode(lib, d, q=None) == 1
    assert _decode(lib, d, q=FAKE + 2) == 1  # query rows are fetched in 16-byte pieces
    assert _decode(lib, d, out=FAKE + 8) == 1  # outputs are stored in 16-byte pieces
    assert _decode(lib, d, sm=float("inf")) == 1
    assert _decode(lib, d) == 3  # needs a workspace (256 CTAs)
    assert _decode(lib, d, ws=FAKE, wsb=10) == 3
    n = ctypes.c_size_t(0)
    assert lib.kvq_decode_workspace_size_ex(ctypes.byref(d), 4, 32, 1024, 256,
                                            ctypes.byref(n)) == 0
    # two partial slots per CTA and head; per slot a completion tag, a team tag
    # and a team claim; a merge claim per sequence (one head group)
    # (fp16 partial outputs, fp32 (m, l))
    assert n.value == 256 * 2 * 32 * (128 * 2 + 8) + 256 * 1 * 2 * 8 * 3 + 4 * 1 * 8
    assert lib.kvq_decode_workspace_size_ex(ctypes.byref(d), 4, 32, 200, 1,
                                            ctypes.byref(n)) == 0
    assert n.value == 0  # one CTA: every sequence is whole, no workspace
    assert _decode(lib, d, s=0) == 0


def _append(lib, desc, **kw):
    a = dict(k=FAKE, v=FAKE, nk=FAKE, nv=FAKE, ks=1024, vs=1024, out=FAKE, q=FAKE, s=4, hq=32,
             bt=FAKE, mb=64, cl=FAKE, mc=1024, sm=0.088, p=256, ws=None, wsb=0)
    a.update(kw)
    return lib.kvq_decode_append(ctypes.byref(desc), a["k"], a["v"], a["nk"], a["nv"], a["ks"],
                                 a["vs"], a["out"], a["q"], a["s"], a["hq"], a["bt"], a["mb"],
                                 a["cl"], a["mc"], a["sm"], a["p"], a["ws"], a["wsb"], None)


def test_append_validation(lib):
    d = _desc()
    assert _append(lib, d, nk=None) == 1
    assert _append(lib, d, nv=FAKE + 8) == 1  # rows are read in 16-byte pieces
    assert _append(lib, d, ks=1016) == 1  # stride shorter than a sequence's row
    assert _append(lib, d, vs=1028) == 1  # stride not a multiple of 8
    assert _append(lib, _desc(head_dim=96)) == 2
    assert _append(lib, _desc(k_fmt=4, v_fmt=1, k_meta=FAKE)) == 2  # mixed families
    # then the decode's own checks
    assert _append(lib, d, hq=30) == 1
    assert _append(lib, d, mb=10) == 1
    assert _append(lib, d, q=FAKE + 2) == 1
    assert _append(lib, d) == 3  # needs a workspace (256 CTAs)
    assert _append(lib, d, s=0, nk=None, nv=None) == 0  # no sequences: nothing to do


def test_hadamard_and_calibrate_validation(lib):
    assert lib.kvq_hadamard(FAKE, 2, 10, 128, None, 0, None) == 1
    assert lib.kvq_hadamard(FAKE, 0, 10, 96, None, 0, None) == 2
    assert lib.kvq_hadamard(FAKE + 4, 0, 10, 128, None, 0, None) == 1
    assert lib.kvq_hadamard(None, 0, 0, 128, None, 0, None) == 0
    assert lib.kvq_calibrate_scale(FAKE, 10, 0.0, FAKE, None) == 1
    assert lib.kvq_calibrate_scale(FAKE, -1, 127.0, FAKE, None) == 1


def test_wait_hook_validation(lib):
    # only invalid settings here: a valid one would stay armed for the next launch
    assert lib.kvq_debug_arm_wait_timeout(0, 0, 0) == 1
    assert lib.kvq_debug_arm_wait_timeout(-5, 0, 0) == 1
    assert lib.kvq_debug_arm_wait_timeout(100, -2, 0) == 1
    assert lib.kvq_debug_arm_wait_timeout(100, 0, -3) == 1


def test_bf16_cache_validation(lib):
    """The 16-bit cache is K and V both (one decode family), takes no scale,
    no per-head scales and no rotation."""
    assert _write(lib, _desc(k_fmt=6, v_fmt=6, k_scale=0.0, v_scale=float("nan")), n=0) == 0
    assert _write(lib, _desc(k_fmt=6, v_fmt=1)) == 2
    assert _write(lib, _desc(k_fmt=1, v_fmt=6)) == 2
    assert _write(lib, _desc(k_fmt=6, v_fmt=4, v_meta=FAKE)) == 2
    assert _write(lib, _desc(k_fmt=6, v_fmt=6, flags=1)) == 2
    assert _write(lib, _desc(k_fmt=6, v_fmt=6, k_head_scales=FAKE)) == 1
    assert _write(lib, _desc(k_fmt=7, v_fmt=7)) == 1


def test_mixed_pages_validation(lib):
    """The classes of a mixed cache share formats and heads; pages of 16 tokens
    or more; one or two classes."""
    K = ctypes.c_void_p * 2
    kcs, vcs = K(FAKE, FAKE), K(FAKE, FAKE)

    def call(descs, n=2, cls=FAKE):
        arr = (type(descs[0]) * len(descs))(*descs)
        return lib.kvq_decode_mixed(arr, n, kcs, vcs, cls, None, None, 0, 0, FAKE, FAKE, 4, 32,
                                    FAKE, 64, FAKE, 1024, 0.088, 256, None, 0, None)
    assert call([_desc(), _desc(block_size=64)]) == 3  # valid: needs a workspace
    assert call([_desc(), _desc(block_size=64)], cls=None) == 1
    assert call([_desc(), _desc(block_size=8)]) == 2  # 8-token pages: one class per call
    assert call([_desc(), _desc(k_fmt=2)]) == 1  # formats differ
    assert call([_desc(), _desc(num_kv_heads=4)]) == 1
    assert call([_desc(), _desc(k_scale=0.2)]) == 1
    assert call([_desc(), _desc()], n=3) == 2
    assert call([_desc(), _desc()], n=0) == 2
