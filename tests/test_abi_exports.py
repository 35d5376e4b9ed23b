"""The C-ABI library loads and exports every function include/lnk.h declares
(no GPU needed; no compute call is made)."""
import ctypes
import importlib.util
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
LIB = os.path.join(ROOT, "paged_kv_gqa_row_gb300", "liblnk.so")


def _declared():
    with open(os.path.join(ROOT, "include", "lnk.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(lnk_[a-z0-9_]+)\s*\(", text)))


def _ensure_built():
    if not os.path.exists(LIB):
        spec = importlib.util.spec_from_file_location("_lnk_build", os.path.join(ROOT, "paged_kv_gqa_row_gb300", "build.py"))
        mod = importlib.util.module_from_spec(spec)
        spec.loader.exec_module(mod)
        mod.build()


def test_header_declares_the_boundary():
    names = _declared()
    for required in ["lnk_paged_append_rope", "lnk_paged_decode_attn", "lnk_paged_step_attn",
                     "lnk_paged_workspace_size", "lnk_status_string"]:
        assert required in names


def test_library_exports_every_declared_symbol():
    _ensure_built()
    lib = ctypes.CDLL(LIB)
    missing = [n for n in _declared() if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_lists_every_declared_symbol():
    _ensure_built()
    import paged_kv_gqa_row_gb300 as lnk
    assert sorted(lnk.EXPORTED) == _declared()


def test_wait_selftest_refuses_bad_arguments_without_launching():
    _ensure_built()
    lib = ctypes.CDLL(LIB)
    lib.lnk_selftest_wait_timeout.restype = ctypes.c_int
    lib.lnk_selftest_wait_timeout.argtypes = [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_void_p]
    einval = 1
    assert lib.lnk_selftest_wait_timeout(None, 1000, None) == einval           # no status buffer
    assert lib.lnk_selftest_wait_timeout(ctypes.c_void_p(16), 0, None) == einval  # no limit
    assert lib.lnk_selftest_wait_timeout(ctypes.c_void_p(16), 3_000_000_000, None) == einval  # over 2 s
