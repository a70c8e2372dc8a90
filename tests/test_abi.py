"""The C-ABI library loads without a GPU and exports every entry point that
include/fa_decode.h declares (no compute call is made here)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^[A-Za-z_][\w\s\*]*?\b(fa_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("fa_decode_plan", "fa_decode_run", "fa_merge_states"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    handle = ctypes.CDLL(lib.LIB_PATH)
    for name in declared_functions():
        assert hasattr(handle, name), f"{name} declared but not exported"
    assert set(lib.EXPORTED_SYMBOLS) == set(declared_functions())


def test_status_strings(lib):
    L = lib.library()
    assert L.fa_status_string(0) == b"FA_OK"
    assert L.fa_status_string(-3) == b"FA_ERR_WORKSPACE_TOO_SMALL"
    assert L.fa_status_string(12345) == b"FA_UNKNOWN_STATUS"


def test_null_arguments_rejected_without_gpu(lib):
    L = lib.library()
    out = ctypes.c_void_p()
    # out_plan NULL, plan NULL: rejected before any CUDA call
    assert L.fa_decode_plan(None, None, None, 1, 8, 8, 64, 16, 0, 0, None, 0, None, None) == -1
    assert L.fa_decode_run(None, None, None, 1, 0.0, 1.0, 1.0, None, None, None) == -1
    assert L.fa_decode_plan_destroy(None) == 0
    assert L.fa_decode_plan_get_info(None, None) == -1
    del out


def test_no_oracle_in_product_path():
    """The package and its sources never reference the oracle."""
    pkg = os.path.join(ROOT, "paged_kv_decode_fa_gb300")
    for dirpath, _, files in os.walk(pkg):
        if "_build" in dirpath:
            continue
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".cpp", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "liboracle" not in text, f
