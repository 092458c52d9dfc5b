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


def test_plan_choice_without_a_gpu():
    # mk_plan_for runs mk_create's shape checks and layout choice on the host:
    # on a 152-SM GB300 the 0.6B dims (the bench workload, the talker, the
    # long-context workload, the 3-layer test shape) take the kernel compiled
    # for them, the 1.7B dims theirs, every other test shape the general one
    import persistent_transformer_megakernel_gb300 as mk
    import workloads as W
    if not os.path.exists(mk.lib_path()):
        pytest.skip("library not built")
    want = {"qwen3_0p6b": 1, "tts_talker": 1, "mid": 1, "qwen3_1p7b": 2,
            "tiny": 0, "gqa4": 0, "mha": 0, "mha64": 0, "mrope_small": 0}
    for name, plan in want.items():
        assert mk.plan_for(W.shape(name), 152) == plan, name
    # the split-K layout of the O projection depends on the rows per CTA: at 76
    # SMs the 0.6B dims no longer match the compiled layouts
    assert mk.plan_for(W.shape("qwen3_0p6b"), 76) == 0
    lib = mk.load_library()
    plan = ctypes.c_int32(-1)
    cfg = mk._binding.config_struct(W.shape("tiny"), 64)
    assert lib.mk_plan_for(ctypes.byref(cfg), 0, ctypes.byref(plan)) == -1      # n_sm < 1
    assert lib.mk_plan_for(None, 152, ctypes.byref(plan)) == -1
    cfg.head_dim = 96                                                             # not 64 or 128
    assert lib.mk_plan_for(ctypes.byref(cfg), 152, ctypes.byref(plan)) == -2      # MK_ERR_UNSUPPORTED
    cfg.head_dim, cfg.n_layers = 64, 0                                            # invalid shape
    assert lib.mk_plan_for(ctypes.byref(cfg), 152, ctypes.byref(plan)) == -1
