"""The C ABI library: it loads and exports every entry point include/okv.h declares (CPU only)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "okv.h")).read()
    return sorted(set(re.findall(r"OKV_API\s+[\w\s\*]+?\b(okv_\w+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    from sparse_kv_cache_draft_gb300 import build
    build.build()
    from sparse_kv_cache_draft_gb300 import load_library
    return load_library()


def test_header_declares_the_boundary():
    syms = declared_symbols()
    for s in ("okv_create", "okv_destroy", "okv_add_request", "okv_remove_request", "okv_append",
              "okv_stage", "okv_attend", "okv_step", "okv_sync", "okv_read_selection",
              "okv_read_slot_table", "okv_read_fetch_list", "okv_last_error"):
        assert s in syms


def test_library_exports_every_declared_symbol(lib):
    missing = [s for s in declared_symbols() if not hasattr(lib, s)]
    assert not missing, missing


def test_struct_layouts(lib):
    from sparse_kv_cache_draft_gb300 import binding
    assert ctypes.sizeof(binding._Config) == 40
    assert ctypes.sizeof(binding._Timing) == 7 * 8 + 7 * 8 + 8 + 8


def test_status_strings(lib):
    assert lib.okv_status_string(0) == b"ok"
    assert lib.okv_status_string(5) == b"timeout"


def test_null_context_is_rejected(lib):
    assert lib.okv_sync(None, 0) == 1
    assert lib.okv_attend(None, 0, None, None, None) == 1
    assert lib.okv_launch_count(None) == 0
