"""C ABI checks that need no GPU: the library loads, exports every function
include/kivi.h declares, and rejects invalid arguments before any CUDA call."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from bit_quantized_kv_quantize_gb300 import build as B
    path = B.build()
    return ctypes.CDLL(path)


def declared():
    with open(os.path.join(ROOT, "include", "kivi.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kivi_[a-z_]+)\s*\(", text)))


def test_header_declares_the_hot_path():
    names = declared()
    for n in ("kivi_cache_create", "kivi_prefill", "kivi_append", "kivi_decode_attn",
              "kivi_cache_destroy"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared():
        assert hasattr(lib, name), name


def test_status_strings_and_version(lib):
    lib.kivi_status_str.restype = ctypes.c_char_p
    assert lib.kivi_abi_version() == 6
    for s in range(7):
        assert lib.kivi_status_str(s)
    assert lib.kivi_status_str(0) == b"ok"


@pytest.mark.parametrize("args,code", [
    ((1, 1, 64, 3, 2, 32, 32, 100), 2),     # k_bits not in {2, 4}
    ((1, 1, 64, 2, 8, 32, 32, 100), 2),     # v_bits not in {2, 4}
    ((1, 1, 64, 2, 2, 48, 96, 100), 2),     # G not a supported power of two
    ((1, 1, 64, 2, 2, 32, 48, 100), 2),     # R % G != 0 (the pages' assertion)
    ((1, 1, 96, 2, 2, 32, 32, 100), 2),     # d not 64/128/256
    ((1, 1, 64, 2, 2, 128, 128, 100), 2),   # d % G != 0
    ((0, 1, 64, 2, 2, 32, 32, 100), 1),     # b < 1
    ((1, 0, 64, 2, 2, 32, 32, 100), 1),     # h_kv < 1
    ((1, 1, 64, 2, 2, 32, 32, 0), 1),       # max_tokens < 1
    ((2000, 1, 64, 2, 2, 32, 32, 100), 2),  # b above the batch limit
])
def test_create_validates_before_touching_cuda(lib, args, code):
    h = ctypes.c_void_p()
    lib.kivi_cache_create.argtypes = [ctypes.c_int] * 8 + [ctypes.POINTER(ctypes.c_void_p)]
    assert lib.kivi_cache_create(*args, ctypes.byref(h)) == code
    assert not h.value
    lib.kivi_last_error.restype = ctypes.c_char_p
    assert lib.kivi_last_error()


def test_null_handles_are_rejected(lib):
    vp = ctypes.c_void_p
    assert lib.kivi_cache_destroy(vp(0)) == 1
    lib.kivi_append.argtypes = [vp] * 4
    assert lib.kivi_append(None, None, None, None) == 1
    lib.kivi_decode_attn.argtypes = [vp, vp, ctypes.c_int, vp, vp]
    assert lib.kivi_decode_attn(None, None, 4, None, None) == 1
    lib.kivi_prefill.argtypes = [vp, vp, vp, vp, ctypes.c_int, vp]
    assert lib.kivi_prefill(None, None, None, None, 0, None) == 1
    # a pointer that was never a handle
    bogus = ctypes.create_string_buffer(64)
    assert lib.kivi_cache_destroy(ctypes.cast(bogus, vp)) == 1


def test_binding_surfaces_errors():
    from bit_quantized_kv_quantize_gb300 import kivi as K
    with pytest.raises(K.KiviError) as e:
        K.KiviCache(1, 1, 64, 3, 2, 32, 32, 100)
    assert e.value.status == 2
    assert set(K.EXPORTS) == set(declared())
