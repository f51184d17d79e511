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


def test_struct_layouts(lib, tmp_path):
    """The binding's ctypes mirrors of okv_config and okv_timing match the header as a C
    compiler lays it out (sizes and every field offset)."""
    import subprocess
    from sparse_kv_cache_draft_gb300 import binding
    inc = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
    fields = {"okv_config": binding._Config, "okv_timing": binding._Timing}
    lines = ['#include <stddef.h>', '#include <stdio.h>', '#include "okv.h"', "int main(void) {"]
    for cname, py in fields.items():
        lines.append(f'  printf("{cname} %zu\\n", sizeof({cname}));')
        for f, _ in py._fields_:
            lines.append(f'  printf("{cname}.{f} %zu\\n", offsetof({cname}, {f}));')
    lines += ["  return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c99", "-I", inc, "-o", str(exe), str(src)], check=True)
    got = dict(l.split() for l in subprocess.run([str(exe)], check=True, capture_output=True,
                                                  text=True).stdout.splitlines())
    for cname, py in fields.items():
        assert int(got[cname]) == ctypes.sizeof(py), cname
        for f, _ in py._fields_:
            assert int(got[f"{cname}.{f}"]) == getattr(py, f).offset, (cname, f)


def test_status_strings(lib):
    assert lib.okv_status_string(0) == b"ok"
    assert lib.okv_status_string(5) == b"timeout"


def test_null_context_is_rejected(lib):
    assert lib.okv_sync(None, 0) == 1
    assert lib.okv_attend(None, 0, None, None, None) == 1
    assert lib.okv_launch_count(None) == 0


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    """Without libokv.so the binding raises instead of computing anything on the CPU."""
    from sparse_kv_cache_draft_gb300 import Config, Context, binding
    monkeypatch.setattr(binding, "library_path", lambda: str(tmp_path / "libokv.so"))
    monkeypatch.setattr(binding, "_lib", None)
    with pytest.raises(ImportError):
        binding.load_library()
    with pytest.raises(ImportError):
        Context(Config(1, 8, 2, 64, 16, 512, 2, 8))


def _build_c_demo(out_dir):
    """Compile tests/c_abi_demo.c against include/okv.h and libokv.so (plain C99, CUDA runtime)."""
    import subprocess
    from sparse_kv_cache_draft_gb300 import library_path
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    lib_dir = os.path.dirname(library_path())
    exe = os.path.join(str(out_dir), "c_abi_demo")
    cmd = ["gcc", "-std=c99", "-O2", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(cuda, "include"), os.path.join(ROOT, "tests", "c_abi_demo.c"), "-o", exe,
           "-L", lib_dir, "-lokv", "-L", os.path.join(cuda, "lib64"), "-lcudart", "-lm",
           f"-Wl,-rpath,{lib_dir}", f"-Wl,-rpath,{os.path.join(cuda, 'lib64')}"]
    subprocess.run(cmd, check=True)
    return exe


def test_c_caller_compiles_and_links(lib, tmp_path):
    """include/okv.h is plain C99 and a C program links against libokv.so with no Python or torch."""
    assert os.path.exists(_build_c_demo(tmp_path))
