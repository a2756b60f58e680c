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


def test_every_entry_point_rejects_a_null_handle():
    """Each call checks its handle and pointers before any CUDA work, so these
    run on a machine without a GPU and return RV_EINVAL (or 0 / a message)."""
    import ctypes as C

    lib = rv.lib()
    E = rv.RV_EINVAL
    buf = (C.c_int32 * 4)()
    assert lib.rv_prefill(None, buf, 1, 1, C.c_float(0.9), -1, buf, buf) == E
    assert lib.rv_decode_step_dev(None, buf, 1, C.c_float(0.9), None, buf, buf, None) == E
    assert lib.rv_sync_status(None) == E
    assert lib.rv_kv_reset(None, None, 0) == E
    assert lib.rv_set_debug(None, 1) == E
    assert lib.rv_set_option(None, rv.OPT_QUANTIZER, rv.QUANT_HQQ) == E
    assert lib.rv_debug_dump(None, rv.DUMP_LOGITS, buf, 16) == E
    assert lib.rv_export_river(None, 1, 0, buf, buf, buf) == E
    assert lib.rv_offload_backbone(None, 1) == E
    assert lib.rv_param_bytes(None, 0) == 0
    ms, by = C.c_float(0), C.c_double(0)
    assert lib.rv_time_kernel(None, rv.TIME_GATEUP, 1, 0, 1, C.byref(ms), C.byref(by)) == E
    assert lib.rv_greedy_head_noalloc(None, None, None, 8, 8, 1, C.c_float(1e-5), None, None, None) == E
    assert b"null" in lib.rv_last_error()


def test_noalloc_head_checks_sizes_and_alignment_before_any_gpu_work():
    """rv_greedy_head_noalloc validates every argument before it touches the
    GPU: sizes beyond its limits (including vocab x d_model beyond the GEMV's
    32-bit offsets) and pointers that are not 16-byte aligned come back as
    RV_EINVAL, on a machine without a GPU."""
    import ctypes as C

    lib = rv.lib()
    E = rv.RV_EINVAL
    ok, odd = 0x10000, 0x10004  # never dereferenced: the checks come first
    eps = C.c_float(1e-5)
    cases = [
        (ok, ok, ok, 262144, 16384),  # 2^32 elements
        (ok, ok, ok, 6, 256),         # vocab not a multiple of 4
        (ok, ok, ok, 1024, 12),       # d_model not a multiple of 8
        (ok, ok, ok, 1024, 16392),    # d_model above 16384
        (odd, ok, ok, 1024, 256),     # misaligned LM head
        (ok, odd, ok, 1024, 256),     # misaligned gain
        (ok, ok, odd, 1024, 256),     # misaligned hidden state
    ]
    for head, norm, h, vocab, dm in cases:
        assert lib.rv_greedy_head_noalloc(head, norm, h, vocab, dm, 1, eps, ok, None, None) == E, (vocab, dm)
        assert lib.rv_last_error()
