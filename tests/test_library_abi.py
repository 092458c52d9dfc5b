"""CPU checks of the C ABI: the shared library loads and exports every entry
point that ``include/mk.h`` declares (no compute calls without a GPU)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mk.h")


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mk_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = _declared()
    for n in ("mk_create", "mk_reset_kv", "mk_decode", "mk_destroy", "mk_error_string"):
        assert n in names


def test_library_exports_every_declared_symbol():
    import persistent_transformer_megakernel_gb300 as mk
    path = mk.lib_path()
    if not os.path.exists(path):
        from persistent_transformer_megakernel_gb300 import build
        build.build()
    lib = ctypes.CDLL(path)
    for n in _declared():
        assert hasattr(lib, n), n
    assert set(_declared()) == set(mk._binding.EXPORTS)


def test_error_strings_without_a_gpu():
    import persistent_transformer_megakernel_gb300 as mk
    if not os.path.exists(mk.lib_path()):
        pytest.skip("library not built")
    lib = mk.load_library()
    assert lib.mk_error_string(0) == b"ok"
    assert lib.mk_error_string(-5) == b"device wait timed out"
    # a NULL handle is an argument error, checked before any CUDA call
    assert lib.mk_get_info(None, None) == -1
    assert lib.mk_destroy(None) == 0
