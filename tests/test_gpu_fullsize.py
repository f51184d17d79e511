"""Full-size parity at the benchmark's configuration, on sampled units.

Qwen3-8B attention shapes, 36 layers, batch 128, 16K context, fetch cap 0.05, 16 host buffers
aliased across the batch, driven exactly as bench.py drives it: a cap-1.0 bootstrap staging
from the draft of step -1, then decode steps through okv_step (attention and staging of every
layer, in the launch configuration the benchmark times). After each step the oracle follows a
sample of (layer, request) units: selections (tie band), slot tables, stamps, fetch lists and
pool bytes exactly, attention within the bf16 tolerance.
"""
import numpy as np
import pytest

import oracle
import synth
from okv_harness import ATOL, Rig, to_device, torch_dtype

pytestmark = pytest.mark.gpu

LAYERS = [0, 35]
SAMPLE = [0, 17, 64, 127]


def test_qwen3_8b_16k_b128_sampled():
    import torch
    w = synth.WORKLOADS["qwen3_8b_16k_b128"]
    rig = Rig(w, n_alias=16, layers_kept=LAYERS)
    try:
        L, R, Hq, d = w.layers, rig.R, w.q_heads, w.head_dim
        C = oracle.fetch_cap_blocks(w.fetch_cap, rig.kb)

        def all_layers(step, kind):
            return np.stack([rig.batch_queries(l, step, kind) for l in range(L)])

        def stage_check(layer, draft, cap_blocks, stamp):
            rig._ensure_summaries(layer, SAMPLE)
            rig.model.score_topk(layer, draft, requests=SAMPLE)
            gsel, _ = rig.check_selection(layer, requests=SAMPLE)
            rig.model.select(layer, cap_blocks, stamp, sel_override=gsel, requests=SAMPLE)
            rig.check_tables(layer, requests=SAMPLE)
            rig.check_pool(layer, requests=SAMPLE, heads=[0, 7])

        d_boot = all_layers(-1, 1)
        for l in range(L):
            rig.ctx.stage(l, to_device(d_boot[l], w.dtype), 0, 1.0)
        torch.cuda.synchronize()
        assert rig.ctx.sync(120_000) == 0
        for l in LAYERS:
            stage_check(l, d_boot[l], oracle.fetch_cap_blocks(1.0, rig.kb), 0)
        for t in range(2):
            q = all_layers(t, 0)
            dr = all_layers(t, 1)
            out = torch.zeros((L, R, Hq, d), dtype=torch_dtype(w.dtype), device="cuda")
            rig.ctx.step(to_device(q, w.dtype), to_device(dr, w.dtype), out, t + 1)
            torch.cuda.synchronize()
            assert rig.ctx.sync(120_000) == 0
            for l in LAYERS:
                err = rig.check_attention(l, q[l], out[l], requests=SAMPLE)
                assert err <= ATOL[w.dtype]
                stage_check(l, dr[l], C, t + 1)
            counts, _ = rig.ctx.read_fetch_list(LAYERS[-1])
            assert counts.max() <= C
    finally:
        rig.close()
