"""The library's measured alternatives that it reads once per process, each checked against the
oracle in a child process of its own (tests/variant_child.py): every attention tile shape the
tensor-core path compiles (warps x TMA stages: 4x2, 4x4, 8x2, 8x3; 4x3 is the default that the
rest of the suite runs), the gather with fixed round-robin shares instead of claimed blocks, and
the gather on a grid of 3 CTAs (each warp then copies many blocks, so the look-ahead of the next
block runs through long chains)."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.mark.parametrize("env", [{"OKV_ATTEND_TILE": "4x2"}, {"OKV_ATTEND_TILE": "4x4"},
                                 {"OKV_ATTEND_TILE": "8x2"}, {"OKV_ATTEND_TILE": "8x3"},
                                 {"OKV_GATHER_DYNAMIC": "0"}, {"OKV_GATHER_CTAS": "3"}],
                         ids=lambda e: ",".join(f"{k}={v}" for k, v in e.items()))
def test_variant_matches_oracle(env):
    child_env = {k: v for k, v in os.environ.items() if not k.startswith("OKV_")}
    child_env.update(env)
    r = subprocess.run([sys.executable, os.path.join(HERE, "variant_child.py")], env=child_env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, (env, r.stdout[-2000:], r.stderr[-4000:])
    assert "variant ok" in r.stdout
