"""The C-ABI library builds for sm_103a, loads without a GPU and exports
every entry point that include/rv.h declares (no compute calls)."""
import ctypes
import os
import re

import token_level_early_gb300 as rv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    txt = open(os.path.join(ROOT, "include", "rv.h")).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(rv_[a-z0-9_]+)\s*\(", txt)))


def test_library_loads_and_exports_every_declared_symbol():
    if not os.path.exists(rv.LIB_PATH):
        rv.build()
    lib = ctypes.CDLL(rv.LIB_PATH)
    names = declared_functions()
    assert len(names) >= 14
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(rv.EXPORTED)


def test_error_paths_without_gpu_work():
    lib = rv.lib()
    assert lib.rv_last_error() is not None
    assert lib.rv_quantize_river(None, 64, 1) == rv.RV_EINVAL
    assert lib.rv_decode_step(None, None, 1, 0.9, None, None, None) == rv.RV_EINVAL
    assert lib.rv_load_model(None, None, None, None) == rv.RV_EINVAL
    assert lib.rv_kv_bytes(None) == 0
    lib.rv_free_model(None)
