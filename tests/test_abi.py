"""The C-ABI library loads and exports every entry point include/sdv.h declares;
argument checks that need no GPU behave as documented."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def libsdv():
    from speculative_decoding_verify_02_gb300 import build
    build.build()
    import speculative_decoding_verify_02_gb300 as sdv
    return sdv.lib()


def _declared():
    text = open(os.path.join(ROOT, "include", "sdv.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sdv_[a-z_]+)\s*\(", text)))


def test_header_declares_and_library_exports_everything(libsdv):
    import speculative_decoding_verify_02_gb300 as sdv
    names = _declared()
    assert set(names) == set(sdv.EXPORTS), set(names) ^ set(sdv.EXPORTS)
    for n in names:
        assert hasattr(libsdv, n), n


def test_status_strings(libsdv):
    import speculative_decoding_verify_02_gb300 as sdv
    assert sdv.status_str(0) == "ok"
    assert sdv.status_str(sdv.SDV_ERR_CAPACITY) == "out of KV capacity"


def test_host_side_argument_errors(libsdv):
    import synth
    import speculative_decoding_verify_02_gb300 as sdv
    m = sdv.model_cfg(synth.TINY)
    c = sdv.CacheCfg(16, 64, 1, 128, 128, 512, 0)
    n = ctypes.c_size_t()
    assert libsdv.sdv_workspace_bytes(None, ctypes.byref(c), ctypes.byref(n)) == sdv.SDV_ERR_ARG
    assert libsdv.sdv_workspace_bytes(ctypes.byref(m), ctypes.byref(c), ctypes.byref(n)) == 0 and n.value > 0
    assert libsdv.sdv_kv_pool_bytes(ctypes.byref(m), ctypes.byref(c), ctypes.byref(n)) == 0
    assert n.value == 2 * 64 * 2 * 2 * 16 * 64 * 2
    bad = sdv.CacheCfg(16, 64, 1, 129, 128, 512, 0)          # max_rows above 128
    assert libsdv.sdv_workspace_bytes(ctypes.byref(m), ctypes.byref(bad), ctypes.byref(n)) == sdv.SDV_ERR_ARG
    m2 = sdv.model_cfg(synth.TINY)
    m2.head_dim = 96
    assert libsdv.sdv_workspace_bytes(ctypes.byref(m2), ctypes.byref(c), ctypes.byref(n)) == sdv.SDV_ERR_UNSUPPORTED
    ctx = ctypes.c_void_p()
    assert libsdv.sdv_create(ctypes.byref(m), ctypes.byref(c), None, None, None, None,
                             ctypes.byref(ctx)) == sdv.SDV_ERR_ARG
    for fn, args in [("sdv_ensure_capacity", (None, None, 1, None)), ("sdv_rewind_cache", (None, None, 1, None)),
                     ("sdv_spec_forward", (None,) * 3 + (1, 1, 1) + (None,) * 3),
                     ("sdv_reset_seq", (None, 0, None)), ("sdv_get_status", (None, None))]:
        assert getattr(libsdv, fn)(*args) == sdv.SDV_ERR_ARG, fn
