"""The C ABI library builds for sm_103a, loads, and exports every entry point
include/wsnf4.h declares (host-only checks: no kernel runs without a GPU)."""
import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "wsnf4.h")


@pytest.fixture(scope="module")
def lib():
    from weight_streaming_nf4_gb300 import build
    path = build.build()
    return C.CDLL(path)


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(ws_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert "ws_lora_linear_fwd" in names and "ws_stream_block_h2d" in names
    assert len(names) >= 13
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    lib.ws_status_string.restype = C.c_char_p
    lib.ws_status_string.argtypes = [C.c_int32]
    for code in [0, -1, -2, -3, -4, -5, -6, -7, -8]:
        s = lib.ws_status_string(code).decode()
        assert s.startswith("WS_")
    assert lib.ws_status_string(12345).decode() == "WS_ERR_UNKNOWN"


def test_argument_validation_is_host_side(lib):
    """Null pointers and bad shapes are rejected before any CUDA call."""
    lib.ws_quantize_nf4.restype = C.c_int32
    lib.ws_quantize_nf4.argtypes = [C.c_void_p, C.c_int64, C.c_int64, C.c_void_p, C.c_void_p,
                                    C.c_void_p]
    assert lib.ws_quantize_nf4(None, 64, 64, None, None, None) == -1
    fake = C.c_void_p(0x1000)
    assert lib.ws_quantize_nf4(fake, 64, 100, fake, fake, None) == -2      # K % 64
    assert lib.ws_quantize_nf4(C.c_void_p(0x1008), 64, 64, fake, fake, None) == -3  # align
    lib.ws_stream_block_h2d.restype = C.c_int32
    lib.ws_stream_block_h2d.argtypes = [C.c_void_p, C.c_void_p, C.c_size_t, C.c_void_p,
                                        C.c_void_p, C.c_void_p]
    assert lib.ws_stream_block_h2d(None, None, 16, None, None, None) == -1
