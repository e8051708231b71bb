"""Host-only checks of the C ABI: the library builds and loads, exports every
function pkv.h declares, the Python binding covers them all, and argument
validation rejects bad calls before touching a device.  No kernel runs here.
"""
import ctypes
import os
import re

import pytest
import torch

import paged_kv_cache_493_b300 as pkv
from paged_kv_cache_493_b300 import _build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "pkv.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return pkv.load_library()


def test_header_declares_the_three_calls_and_helpers():
    names = declared_functions()
    for n in ("pkv_store_kvcache", "pkv_decode_attention", "pkv_prefill_attention"):
        assert n in names
    assert len(names) == len(pkv.SIGNATURES)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in pkv.SIGNATURES, f"binding lacks {name}"


def test_status_strings_and_version(lib):
    for code, name in pkv.STATUS.items():
        assert pkv.pkv_status_string(code) == name
    assert pkv.pkv_status_string(99) == "PKV_ERR_UNKNOWN"
    assert "sm_103a" in pkv.pkv_version()


def test_knobs_validate_arguments(lib):
    assert lib.pkv_set_max_splits(-1) == pkv.PKV_ERR_INVALID_ARG
    assert lib.pkv_set_max_splits(0) == pkv.PKV_OK
    assert lib.pkv_set_wait_limit_ns(-5) == pkv.PKV_ERR_INVALID_ARG
    assert lib.pkv_set_wait_limit_ns(1_000_000_000) == pkv.PKV_OK
    assert lib.pkv_profiler_enable(0) == pkv.PKV_OK
    assert lib.pkv_profiler_reset() == pkv.PKV_OK
    assert lib.pkv_reserve_workspace(4, 4, 96, 2) == pkv.PKV_ERR_INVALID_ARG
    for bad in (-1, 3, 5, 32):
        assert lib.pkv_set_shared_prefix_units(bad) == pkv.PKV_ERR_INVALID_ARG
    for good in (0, 1, 2, 4, 8, 16):
        assert lib.pkv_set_shared_prefix_units(good) == pkv.PKV_OK
    assert lib.pkv_set_shared_prefix_units(0) == pkv.PKV_OK
    ms, n = ctypes.c_double(), ctypes.c_int64()
    assert lib.pkv_profiler_read(b"decode", ctypes.byref(ms), ctypes.byref(n)) == pkv.PKV_OK
    assert n.value == 0
    assert lib.pkv_profiler_read(None, ctypes.byref(ms), ctypes.byref(n)) == pkv.PKV_ERR_INVALID_ARG


# Fake, 16-byte aligned addresses: validation must fail (or the missing device
# be reported) before anything dereferences them.
A = ctypes.c_void_p(0x1000)
NUL = ctypes.c_void_p(0)


def dec(lib, **kw):
    args = dict(q=A, qs=16 * 128, k=A, v=A, nb=8, bt=A, mb=2, cl=A, b=4, hq=16, hkv=8, d=128,
                scale=0.1, out=A)
    args.update(kw)
    return lib.pkv_decode_attention(args["q"], args["qs"], args["k"], args["v"], args["nb"],
                                    args["bt"], args["mb"], args["cl"], args["b"], args["hq"],
                                    args["hkv"], args["d"], args["scale"], args["out"], NUL)


def test_decode_argument_validation(lib):
    assert dec(lib, q=NUL) == pkv.PKV_ERR_INVALID_ARG
    assert dec(lib, bt=NUL) == pkv.PKV_ERR_INVALID_ARG
    assert dec(lib, b=-1) == pkv.PKV_ERR_INVALID_ARG
    assert dec(lib, nb=0) == pkv.PKV_ERR_INVALID_ARG
    assert dec(lib, hq=12) == pkv.PKV_ERR_INVALID_ARG            # 12 % 8 != 0
    assert dec(lib, d=96, qs=16 * 96) == pkv.PKV_ERR_UNSUPPORTED  # head_dim
    assert dec(lib, hq=24, hkv=8, qs=24 * 128) == pkv.PKV_ERR_UNSUPPORTED  # group 3
    assert dec(lib, qs=100) == pkv.PKV_ERR_INVALID_ARG           # row stride < Hq * D
    assert dec(lib, qs=16 * 128 + 4) == pkv.PKV_ERR_UNSUPPORTED  # row not 16-byte aligned
    assert dec(lib, q=ctypes.c_void_p(0x1008)) == pkv.PKV_ERR_UNSUPPORTED
    assert dec(lib, nb=1 << 24) == pkv.PKV_ERR_UNSUPPORTED       # slots overflow int32


def test_prefill_and_store_argument_validation(lib):
    r = lib.pkv_prefill_attention(A, 16 * 128, A, A, 8, A, 2, NUL, A, 4, 64, 16, 8, 128, 0.1, A, NUL)
    assert r == pkv.PKV_ERR_INVALID_ARG                             # no cu_seqlens_q
    r = lib.pkv_prefill_attention(A, 16 * 128, A, A, 8, A, 2, A, A, 4, -1, 16, 8, 128, 0.1, A, NUL)
    assert r == pkv.PKV_ERR_INVALID_ARG                             # negative total
    st = lib.pkv_store_kvcache
    assert st(A, A, 1024, 1024, A, -1, A, A, 8, 8, 128, NUL) == pkv.PKV_ERR_INVALID_ARG
    assert st(A, A, 1000, 1024, A, 4, A, A, 8, 8, 128, NUL) == pkv.PKV_ERR_INVALID_ARG  # stride < row
    assert st(A, A, 1028, 1024, A, 4, A, A, 8, 8, 128, NUL) == pkv.PKV_ERR_UNSUPPORTED  # misaligned row
    assert st(NUL, A, 1024, 1024, A, 4, A, A, 8, 8, 128, NUL) == pkv.PKV_ERR_INVALID_ARG
    assert st(A, A, 1024, 1024, A, 4, NUL, A, 8, 8, 128, NUL) == pkv.PKV_ERR_INVALID_ARG


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the behaviour without a device")
def test_valid_calls_without_a_device_fail_loudly(lib):
    assert dec(lib) == pkv.PKV_ERR_CUDA
    assert lib.pkv_store_kvcache(A, A, 1024, 1024, A, 4, A, A, 8, 8, 128, NUL) == pkv.PKV_ERR_CUDA
    code = ctypes.c_int32()
    assert lib.pkv_get_device_error(NUL, ctypes.byref(code), None) == pkv.PKV_ERR_CUDA


def test_binding_refuses_cpu_tensors(lib):
    kc = torch.zeros(2, 256, 2, 64, dtype=torch.bfloat16)
    q = torch.zeros(1, 4, 64, dtype=torch.bfloat16)
    with pytest.raises(pkv.PkvError):
        pkv.pkv_decode_attention(q, kc, kc, torch.zeros(1, 1, dtype=torch.int32),
                                 torch.ones(1, dtype=torch.int32), 0.1, torch.empty_like(q))


def test_missing_library_raises():
    with pytest.raises(pkv.PkvError):
        pkv.load_library("/nonexistent/libpkv.so")


def test_int8_argument_validation(lib):
    B = ctypes.c_void_p(0x1004)  # 4-byte aligned only

    def store(**kw):
        a = dict(k=A, v=A, ks=16 * 128, vs=16 * 128, sm=A, n=4, kc=A, vc=A, ksc=A, vsc=A, nb=8,
                 hkv=16, d=128)
        a.update(kw)
        return lib.pkv_store_kvcache_int8(a["k"], a["v"], a["ks"], a["vs"], a["sm"], a["n"],
                                          a["kc"], a["vc"], a["ksc"], a["vsc"], a["nb"],
                                          a["hkv"], a["d"], NUL)

    assert store(kc=NUL) == pkv.PKV_ERR_INVALID_ARG
    assert store(vsc=NUL) == pkv.PKV_ERR_INVALID_ARG
    assert store(nb=0) == pkv.PKV_ERR_INVALID_ARG
    assert store(ks=100) == pkv.PKV_ERR_INVALID_ARG
    assert store(d=96, ks=16 * 96, vs=16 * 96) == pkv.PKV_ERR_UNSUPPORTED
    assert store(ksc=B) == pkv.PKV_ERR_UNSUPPORTED
    assert store() == pkv.PKV_ERR_CUDA          # valid arguments, no device here

    def dec8(**kw):
        a = dict(q=A, qs=16 * 128, kc=A, vc=A, ksc=A, vsc=A, nb=8, bt=A, mb=2, cl=A, b=4, hq=16,
                 hkv=8, d=128, scale=0.1, out=A)
        a.update(kw)
        return lib.pkv_decode_attention_int8(a["q"], a["qs"], a["kc"], a["vc"], a["ksc"],
                                             a["vsc"], a["nb"], a["bt"], a["mb"], a["cl"], a["b"],
                                             a["hq"], a["hkv"], a["d"], a["scale"], a["out"], NUL)

    assert dec8(ksc=NUL) == pkv.PKV_ERR_INVALID_ARG
    assert dec8(kc=NUL) == pkv.PKV_ERR_INVALID_ARG
    assert dec8(hq=12, hkv=8) == pkv.PKV_ERR_INVALID_ARG
    assert dec8(d=96, qs=16 * 96) == pkv.PKV_ERR_UNSUPPORTED
    assert dec8(vsc=B) == pkv.PKV_ERR_UNSUPPORTED
    assert dec8() == pkv.PKV_ERR_CUDA
