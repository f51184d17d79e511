"""The C ABI from a plain C program (needs a GB300): tests/c_abi_demo.c, built with gcc against
include/okv.h and libokv.so, stages and attends one small request through cudaMalloc buffers
and checks the result against dense attention it computes itself."""
import subprocess

import pytest

from test_abi import _build_c_demo

pytestmark = pytest.mark.gpu


def test_c_caller_end_to_end(tmp_path):
    from sparse_kv_cache_draft_gb300 import build
    build.build()
    exe = _build_c_demo(tmp_path)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "attention max abs error" in r.stdout
