"""Admission-time partial staging through the C ABI vs the CPU oracle (needs a GB300).

A partially staged request keeps its full KV in one host buffer (the prefill side's copy) and
fills a decode-side tier of its own on first demand (OasisKV, paperlayer.ai/abs/2608.08097v1,
"4 System Design", last bullet). The routes of every fetch, the tier's tables and the kept bytes
must match the oracle exactly; attention and pools are checked as for full-KV requests.
"""
import numpy as np
import pytest

import synth
from okv_harness import ATOL, Rig
from sparse_kv_cache_draft_gb300 import BF16, OkvError

pytestmark = pytest.mark.gpu

QWEN = synth.WORKLOADS["qwen3_8b_16k_b128"]


def test_partial_staging_routes_and_counters():
    """Qwen3-8B attention shapes at 8K, 2 layers x 5 requests: one full-KV request and decode-side
    tiers of 0, 150 (full after the bootstrap's 128 plus 22), 200 and 512 (= every block) entries;
    a bootstrap at cap 1.0 then 24 steps at cap 0.05. The heavy direction comes back after 20
    steps, so blocks evicted from HBM are fetched again from their kept copies; kept copies are
    read, filled and bypassed."""
    w = QWEN.scaled(layers=2, batch=5, context=8192)
    rig = Rig(w, local_cap=[-1, 0, 150, 200, 512])
    try:
        rig.ctx.set_timing(True)
        errs, _ = rig.run_steps(24, 0.05)
        assert max(errs) <= ATOL[BF16]
        t = rig.ctx.read_timing()
        for k in ("local_hits", "local_fills", "full_reads"):
            assert t[k] == rig.tally[k], (k, t[k], rig.tally)
        # every kind of route occurred
        assert rig.tally["local_hits"] > 0
        assert rig.tally["local_fills"] > 0
        assert rig.tally["full_reads"] > rig.tally["local_fills"]
        used, _, _ = rig.ctx.read_local(1)
        assert used[1].max() == 0 and used[2].max() == 150 and used[3].max() <= 200
        assert used[4].min() >= 128
    finally:
        rig.close()


def test_partial_staging_with_appends():
    """Appends to partially staged requests write the full copy and the kept copy of the tail
    block; contexts grow across block boundaries for 24 steps (1000 -> 1024, 2040 -> 2064). The
    second request's 70 entries fill up during the bootstrap's 128 fetches."""
    w = synth.WORKLOADS["qwen3_8b_mixed_b64"].scaled(layers=1, batch=3, steps=24)
    rig = Rig(w, contexts=[1000, 2040, 3000], local_cap=[150, 70, -1])
    try:
        errs, _ = rig.run_steps(24, 0.05, append=True)
        assert max(errs) <= ATOL[BF16]
        rig.check_summaries(0)
        assert rig.ctx.read_lengths(0)[:3].tolist() == [1024, 2064, 3024]
    finally:
        rig.close()


def test_partial_staging_ragged_and_tiny_fp32():
    """fp32 tiny shapes (d 64, GQA 8/2, budget 512) with ragged contexts 1, 100, 3000 and 4096
    tokens and tiers of 1, 3, 64 and 256 entries at cap 0.25."""
    w = synth.WORKLOADS["tiny"].scaled(batch=4)
    rig = Rig(w, contexts=[1, 100, 3000, 4096], local_cap=[1, 3, 64, 256])
    try:
        errs, _ = rig.run_steps(4, 0.25)
        assert max(errs) <= ATOL[w.dtype]
    finally:
        rig.close()


def test_partial_staging_api_errors():
    from sparse_kv_cache_draft_gb300 import Config, Context, HostBuffer, binding
    cfg = Config(2, 8, 2, 64, 16, 512, 4, 8, 1.0, synth.F32)
    ctx = Context(cfg)
    full = HostBuffer(cfg.host_bytes(8))
    local = HostBuffer(cfg.host_bytes(4))
    local2 = HostBuffer(cfg.host_bytes(4))
    try:
        def refused(*args):
            with pytest.raises(OkvError) as e:
                ctx.add_request_partial(*args)
            assert e.value.status == binding.EINVAL

        refused(0, full.ptr, 8, local.ptr, 9, 16)          # more entries than blocks
        refused(0, full.ptr, 8, local.ptr, -1, 16)         # negative entries
        refused(0, full.ptr, 8, 0, 4, 16)                  # entries but no buffer
        refused(0, full.ptr, 8, full.ptr, 4, 16)           # tier inside the full copy
        unpinned = np.zeros(cfg.host_bytes(4) // 4, np.float32)
        refused(0, full.ptr, 8, unpinned.ctypes.data, 4, 16)
        ctx.add_request_partial(0, full.ptr, 8, local.ptr, 4, 100)
        refused(1, full.ptr, 8, local.ptr + 64, 2, 100)    # overlaps request 0's tier
        with pytest.raises(OkvError):                      # a full copy inside request 0's tier
            ctx.add_request(1, local.ptr, 4, 16)
        ctx.add_request_partial(1, full.ptr, 8, local2.ptr, 4, 100)  # shared full copy, own tier
        ctx.add_request_partial(2, full.ptr, 8, 0, 0, 100)           # no decode-side entries
        ctx.remove_request(0)
        ctx.add_request_partial(3, full.ptr, 8, local.ptr, 4, 100)   # request 0's tier is free again
        assert ctx.sync(1000) == 0
    finally:
        ctx.close()
        full.free()
        local.free()
        local2.free()
