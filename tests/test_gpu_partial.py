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


def test_pd_32k_b8_full_size_sampled():
    """The partial-staging report's 32K workload at full size (36 layers, batch 8, 2048 blocks per
    unit, 4 full copies aliased, tiers of Kb + 256 C = 1664 entries), driven as the report drives
    it: a cap-1.0 bootstrap, then decode steps through okv_step at cap 0.05. Layers 0 and 35 of
    requests 0, 3 and 7 are followed by the oracle: selections, tables, routes, tiers, kept bytes,
    pools and attention."""
    import torch
    import oracle
    from okv_harness import to_device, torch_dtype
    w = synth.WORKLOADS["qwen3_8b_pd_32k_b8"]
    layers, sample = [0, 35], [0, 3, 7]
    C = oracle.fetch_cap_blocks(w.fetch_cap, w.budget_tokens // w.block_size)
    nb = w.context // w.block_size
    lcap = min(nb, w.budget_tokens // w.block_size + C * 256)
    rig = Rig(w, n_alias=4, layers_kept=layers, local_cap=lcap)
    try:
        L, R, Hq, d = w.layers, rig.R, w.q_heads, w.head_dim

        def all_layers(step, kind):
            return np.stack([rig.batch_queries(l, step, kind) for l in range(L)])

        def stage_check(layer, draft, cap_blocks, stamp):
            rig._ensure_summaries(layer, sample)
            rig.model.score_topk(layer, draft, requests=sample)
            gsel, _ = rig.check_selection(layer, requests=sample)
            rig.model.select(layer, cap_blocks, stamp, sel_override=gsel, requests=sample)
            rig.check_tables(layer, requests=sample)
            rig.check_local(layer, requests=sample)
            rig.check_pool(layer, requests=sample, heads=[0, 7])

        d_boot = all_layers(-1, 1)
        for l in range(L):
            rig.ctx.stage(l, to_device(d_boot[l], w.dtype), 0, 1.0)
        torch.cuda.synchronize()
        assert rig.ctx.sync(120_000) == 0
        for l in layers:
            stage_check(l, d_boot[l], oracle.fetch_cap_blocks(1.0, rig.kb), 0)
        for t in range(3):
            q = all_layers(t, 0)
            dr = all_layers(t, 1)
            out = torch.zeros((L, R, Hq, d), dtype=torch_dtype(w.dtype), device="cuda")
            rig.ctx.step(to_device(q, w.dtype), to_device(dr, w.dtype), out, t + 1)
            torch.cuda.synchronize()
            assert rig.ctx.sync(120_000) == 0
            for l in layers:
                assert rig.check_attention(l, q[l], out[l], requests=sample) <= ATOL[w.dtype]
                stage_check(l, dr[l], C, t + 1)
        used, _, _ = rig.ctx.read_local(35)
        assert used[:8].min() >= rig.kb and used[:8].max() <= rig.kb + 3 * C
    finally:
        rig.close()
