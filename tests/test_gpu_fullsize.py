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


def test_gqa32b_32k_b32_sampled():
    """The 32B-class GQA workload at full size: 64 layers, 64 query / 8 KV heads (group 8 fills the
    tensor-core tile), batch 32, 32K context (2048 blocks per unit), 8 host buffers aliased."""
    import torch
    w = synth.WORKLOADS["gqa32b_32k_b32"]
    layers = [0, 63]
    sample = [0, 13, 31]
    rig = Rig(w, n_alias=8, layers_kept=layers)
    try:
        L, R, Hq, d = w.layers, rig.R, w.q_heads, w.head_dim
        C = oracle.fetch_cap_blocks(w.fetch_cap, rig.kb)

        def all_layers(step, kind):
            return np.stack([rig.batch_queries(l, step, kind) for l in range(L)])

        def stage_check(layer, draft, cap_blocks, stamp):
            rig._ensure_summaries(layer, sample)
            rig.model.score_topk(layer, draft, requests=sample)
            gsel, _ = rig.check_selection(layer, requests=sample)
            rig.model.select(layer, cap_blocks, stamp, sel_override=gsel, requests=sample)
            rig.check_tables(layer, requests=sample)
            rig.check_pool(layer, requests=sample, heads=[3])

        d_boot = all_layers(-1, 1)
        for l in range(L):
            rig.ctx.stage(l, to_device(d_boot[l], w.dtype), 0, 1.0)
        torch.cuda.synchronize()
        for l in layers:
            stage_check(l, d_boot[l], oracle.fetch_cap_blocks(1.0, rig.kb), 0)
        q = all_layers(0, 0)
        dr = all_layers(0, 1)
        out = torch.zeros((L, R, Hq, d), dtype=torch_dtype(w.dtype), device="cuda")
        rig.ctx.step(to_device(q, w.dtype), to_device(dr, w.dtype), out, 1)
        torch.cuda.synchronize()
        assert rig.ctx.sync(120_000) == 0
        for l in layers:
            assert rig.check_attention(l, q[l], out[l], requests=sample) <= ATOL[w.dtype]
            stage_check(l, dr[l], C, 1)
    finally:
        rig.close()


def test_mixed_lengths_appending_all_layers():
    """Reasoning-style mixed lengths (1K-32K, drawn per request) growing by one token per step on
    all 36 layers through okv_step with appends; the library's host writes of the sampled
    requests are checked on every layer, and their units on two layers follow the oracle."""
    import torch
    w = synth.WORKLOADS["qwen3_8b_mixed_b64"].scaled(batch=16, steps=6)
    layers = [0, 35]
    sample = [0, 5, 15]
    rig = Rig(w, layers_kept=layers)
    try:
        L, R, Hq, Hkv, d = w.layers, rig.R, w.q_heads, w.kv_heads, w.head_dim
        C = oracle.fetch_cap_blocks(w.fetch_cap, rig.kb)

        def all_layers(step, kind):
            return np.stack([rig.batch_queries(l, step, kind) for l in range(L)])

        d_boot = all_layers(-1, 1)
        for l in range(L):
            rig.ctx.stage(l, to_device(d_boot[l], w.dtype), 0, 1.0)
        torch.cuda.synchronize()
        for l in layers:
            rig._ensure_summaries(l, sample)
            rig.model.score_topk(l, d_boot[l], requests=sample)
            gsel, _ = rig.check_selection(l, requests=sample)
            rig.model.select(l, oracle.fetch_cap_blocks(1.0, rig.kb), 0, sel_override=gsel, requests=sample)
        for t in range(w.steps):
            kv = [synth.token_kv(w, l, rig.keys, rig.contexts + t, plant_blocks=rig.plant_blocks) for l in range(L)]
            k_all = np.stack([k for k, _ in kv])
            v_all = np.stack([v for _, v in kv])
            q = all_layers(t, 0)
            dr = all_layers(t, 1)
            out = torch.zeros((L, R, Hq, d), dtype=torch_dtype(w.dtype), device="cuda")
            pos = {l: rig.contexts + t for l in range(L)}
            snap = rig.host_snapshot(range(L), requests=sample, positions=pos)
            rig.ctx.step(to_device(q, w.dtype), to_device(dr, w.dtype), out, t + 1, k_new=to_device(k_all, w.dtype),
                         v_new=to_device(v_all, w.dtype))
            torch.cuda.synchronize()
            assert rig.ctx.sync(120_000) == 0
            # the library's host writes, on every layer of the sampled requests
            rig.check_host_append(snap, {l: (k_all[l], v_all[l]) for l in range(L)})
            for l in layers:
                for i in sample:  # the oracle appends only what it follows
                    for h in range(Hkv):
                        oracle.append(rig.model.host_unit(l, i, h), rig.model.summ[l][i, h],
                                      int(rig.model.n_tok[l, i]), w.block_size, d, k_all[l, i, h], v_all[l, i, h])
                    rig.model.n_tok[l, i] += 1
                rig.check_host_tail(l, requests=sample)
                assert rig.check_attention(l, q[l], out[l], requests=sample) <= ATOL[w.dtype]
                rig.model.score_topk(l, dr[l], requests=sample)
                gsel, _ = rig.check_selection(l, requests=sample)
                rig.model.select(l, C, t + 1, sel_override=gsel, requests=sample)
                rig.check_tables(l, requests=sample)
                rig.check_pool(l, requests=sample, heads=[0])
        for l in layers:
            rig.check_summaries(l, requests=sample)
            lens = rig.ctx.read_lengths(l)
            assert lens[:16].tolist() == (rig.contexts + w.steps).tolist()
    finally:
        rig.close()
