"""CPU checks of the C ABI: the library loads and exports every entry point that
include/mk.h declares; host-side argument checks fire without a GPU."""
import ctypes
import os
import re
import subprocess

import pytest

from latency_moe_decode_persistent_gb300 import mk

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mk.h")


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mk_[a-z_]+)\s*\(", src)))


def _built():
    if not os.path.exists(mk.LIB_PATH):
        from latency_moe_decode_persistent_gb300 import build
        build.build()
    return mk.LIB_PATH


def test_header_and_binding_agree():
    assert _declared() == sorted(mk.EXPORTS)


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(_built())
    for name in _declared():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", _built()], capture_output=True, text=True).stdout
    for name in _declared():
        assert re.search(r"\bT %s\b" % name, out), name


def test_status_strings():
    assert mk.mk_status_string(mk.MK_OK) == "ok"
    assert "timed out" in mk.mk_status_string(mk.MK_ERR_TIMEOUT)


def test_null_arguments_rejected_without_device():
    L = mk.lib()
    assert L.mk_create(None, None, None) == mk.MK_ERR_INVALID
    assert L.mk_get_status(None) == mk.MK_ERR_INVALID
    assert L.mk_decode_step(None, None, 1, None, None, None, None, None, None) == mk.MK_ERR_INVALID
    L.mk_destroy(None)


def test_bad_desc_rejected():
    d = mk.mk_model_desc(mk.MK_DESC_VERSION, 1, 500, 8, 2, 64, 1e4, 1e-6, 16, 2, 1, 256, 0, 64, 1,
                         4, mk.MK_DT_F32, mk.MK_DT_F32, mk.MK_DT_F32, 0)
    w = mk.mk_weights()
    h = ctypes.c_void_p()
    s = mk.lib().mk_create(ctypes.byref(d), ctypes.byref(w), ctypes.byref(h))
    assert s == mk.MK_ERR_UNSUPPORTED and not h.value
    assert "hidden" in mk.mk_last_error(None)
