"""CUDA path vs the CPU oracle, through the C ABI (needs a GB300)."""
import numpy as np
import pytest

import synth
from okv_harness import ATOL, Rig
from sparse_kv_cache_draft_gb300 import BF16, F32, OkvError

pytestmark = pytest.mark.gpu

QWEN = synth.WORKLOADS["qwen3_8b_16k_b128"]


def test_tiny_single_step():
    """Tiny config: batch 2, GQA 8/2, d 64, 4096 tokens, budget 512, cap 1.0, fp32."""
    w = synth.WORKLOADS["tiny"]
    rig = Rig(w)
    try:
        rig.check_summaries(0)
        assert rig.attend(0, 0) == 0.0  # empty pool: zeros on both sides
        rig.stage(0, 0, 1.0, draft_step=-1)
        err = rig.attend(0, 0)
        assert err <= ATOL[F32]
        sb, _ = rig.ctx.read_slot_table(0)
        counts, ids, _ = rig.ctx.read_selection(0)
        for r in range(w.batch):
            for h in range(w.kv_heads):
                # fetch cap 1.0: the resident set equals the selection
                assert set(sb[r, h][sb[r, h] >= 0].tolist()) == set(ids[r, h, :counts[r, h]].tolist())
    finally:
        rig.close()


def test_qwen_shapes_multistep_cap005():
    """Qwen3-8B attention shapes (32/8 heads, d 128, 16K, bf16), 2 layers x 3 requests, state carried
    over a bootstrap and 4 decode steps at fetch cap 0.05 (C = 6)."""
    w = QWEN.scaled(layers=2, batch=3)
    rig = Rig(w)
    try:
        rig.check_summaries(0)
        rig.check_summaries(1)
        errs, _ = rig.run_steps(4, 0.05)
        assert max(errs) <= ATOL[BF16]
        counts, _ = rig.ctx.read_fetch_list(1)
        assert counts[:3].max() <= 6
    finally:
        rig.close()


def test_ragged_contexts_and_inactive_rows():
    """Contexts 1, 17, 300, 2048 and 5000 tokens (1 to 313 blocks, partial tails, fewer blocks
    than slots) on request ids 0, 2, 3, 5, 7 of 8."""
    w = QWEN.scaled(layers=1, batch=5)
    rig = Rig(w, contexts=[1, 17, 300, 2048, 5000], max_requests=8, active=[0, 2, 3, 5, 7])
    try:
        rig.check_summaries(0)
        errs, _ = rig.run_steps(3, 0.05)
        assert max(errs) <= ATOL[BF16]
        sb, _ = rig.ctx.read_slot_table(0)
        # budget covers the context for the first four: after the bootstrap every block is resident
        for i, n_tok in enumerate([1, 17, 300, 2048]):
            nb = -(-n_tok // 16)
            for h in range(w.kv_heads):
                assert sorted(sb[rig.ids[i], h][sb[rig.ids[i], h] >= 0].tolist()) == list(range(nb))
    finally:
        rig.close()


def test_many_units_unsplit_attention():
    """160 requests x 8 KV heads = 1280 units: one CTA per unit, no split combine."""
    w = QWEN.scaled(layers=1, batch=160, context=2048 + 40)
    rig = Rig(w, n_alias=4)
    try:
        sample = [0, 1, 77, 159]
        errs, _ = rig.run_steps(2, 0.05, requests=sample, check_pool=False)
        assert max(errs) <= ATOL[BF16]
        rig.check_pool(0, requests=sample)
    finally:
        rig.close()


def test_gqa8_32b_class_shape():
    """32B-class GQA shape: 64 query / 8 KV heads (group 8), d 128, 32K context."""
    w = synth.WORKLOADS["gqa32b_32k_b32"].scaled(layers=1, batch=2)
    rig = Rig(w)
    try:
        errs, _ = rig.run_steps(3, 0.05)
        assert max(errs) <= ATOL[BF16]
    finally:
        rig.close()


@pytest.mark.parametrize("dtype,d,g", [(BF16, 64, 4), (F32, 128, 4), (F32, 64, 8)])
def test_cuda_core_path_shapes(dtype, d, g):
    """Shapes served by the CUDA-core attention kernel."""
    w = QWEN.scaled(layers=1, batch=2, dtype=dtype, head_dim=d, q_heads=8 * g, kv_heads=8,
                    context=3000, budget_tokens=512)
    rig = Rig(w)
    try:
        errs, _ = rig.run_steps(2, 0.25)
        assert max(errs) <= ATOL[dtype]
    finally:
        rig.close()


def test_append_growing_contexts():
    """Mixed lengths growing one token per step across block boundaries: host writes, resident
    tail-slot writes and min/max summary updates."""
    w = synth.WORKLOADS["qwen3_8b_mixed_b64"].scaled(layers=2, batch=3, steps=40)
    rig = Rig(w, contexts=[1000, 2047, 4095])
    try:
        errs, _ = rig.run_steps(40, 0.05, append=True)
        assert max(errs) <= ATOL[BF16]
        for layer in range(2):
            rig.check_summaries(layer)
            lens = rig.ctx.read_lengths(layer)
            assert lens[:3].tolist() == [1040, 2087, 4135]
    finally:
        rig.close()


def test_shared_host_buffers():
    """Requests registered on the same host buffer share summaries; appending to them is refused."""
    w = QWEN.scaled(layers=2, batch=4, context=4096)
    rig = Rig(w, n_alias=2)
    try:
        for layer in range(2):
            rig.check_summaries(layer)
        errs, _ = rig.run_steps(2, 0.05)
        assert max(errs) <= ATOL[BF16]
        import torch
        z = torch.zeros((4, 8, 128), dtype=torch.bfloat16, device="cuda")
        with pytest.raises(OkvError):
            rig.ctx.append(0, z, z)
    finally:
        rig.close()


def test_api_errors():
    import torch
    from sparse_kv_cache_draft_gb300 import Config, Context, HostBuffer, binding
    with pytest.raises(OkvError):
        Context(Config(1, 6, 4, 128, 16, 2048, 2, 64))  # q heads not a multiple of kv heads
    with pytest.raises(OkvError):
        Context(Config(1, 8, 2, 100, 16, 2048, 2, 64))  # head_dim not a multiple of 32
    with pytest.raises(OkvError) as e:  # the selection's on-chip arrays would exceed shared memory
        Context(Config(1, 8, 2, 64, 16, 512, 1, 40000))
    assert e.value.status == binding.EINVAL
    cfg = Config(1, 8, 2, 64, 16, 512, 2, 8, 1.0, F32)
    ctx = Context(cfg)
    hb = HostBuffer(cfg.host_bytes(8))
    try:
        with pytest.raises(OkvError) as e:
            ctx.add_request(2, hb.ptr, 8, 16)
        assert e.value.status == binding.EINVAL
        with pytest.raises(OkvError):
            ctx.add_request(0, hb.ptr, 8, 8 * 16 + 1)  # more tokens than capacity
        unpinned = np.zeros(cfg.host_bytes(8) // 4, np.float32)
        with pytest.raises(OkvError):
            ctx.add_request(0, unpinned.ctypes.data, 8, 16)
        ctx.add_request(0, hb.ptr, 8, 8 * 16)
        with pytest.raises(OkvError) as e:
            ctx.add_request(0, hb.ptr, 8, 16)
        assert e.value.status == binding.ESTATE
        q = torch.zeros((2, 8, 64), device="cuda")
        with pytest.raises(OkvError):
            ctx.attend(1, q, q)  # layer out of range
        with pytest.raises(OkvError):
            ctx.stage(0, q, 0, 1.5)  # cap outside (0, 1]
        kv = torch.zeros((2, 2, 64), device="cuda")
        with pytest.raises(OkvError):
            ctx.append(0, kv, kv)  # request 0 is full
        with pytest.raises(ValueError):
            ctx.attend(0, q.half(), q)  # wrong dtype is refused before the call
        ctx.remove_request(0)
        with pytest.raises(OkvError):
            ctx.remove_request(0)
        assert ctx.sync(1000) == 0
    finally:
        ctx.close()
        hb.free()


@pytest.mark.parametrize("name,w", [
    ("qwen_bf16_one_pass", QWEN.scaled(layers=1, batch=3)),
    ("gqa8_two_passes", synth.WORKLOADS["gqa32b_32k_b32"].scaled(layers=1, batch=2)),
    ("tiny_fp32_one_pass", synth.WORKLOADS["tiny"]),
])
def test_lookahead_attention(name, w):
    """Normal and draft queries attend together over the resident set."""
    import torch
    from okv_harness import torch_dtype
    rig = Rig(w)
    try:
        rig.stage(0, 0, 1.0, draft_step=-1)
        rig.stage(0, 1, w.fetch_cap, draft_step=0)
        shp = (rig.R, w.q_heads, w.head_dim)
        q = rig.batch_queries(0, 1, 0)
        dq = rig.batch_queries(0, 1, 1)
        out = torch.zeros(shp, dtype=torch_dtype(w.dtype), device="cuda")
        dout = torch.zeros(shp, dtype=torch_dtype(w.dtype), device="cuda")
        rig.ctx.attend_lookahead(0, rig.device_rows(q, shp[1:]), rig.device_rows(dq, shp[1:]), out, dout)
        torch.cuda.synchronize()
        assert rig.check_attention(0, q, out) <= ATOL[w.dtype]
        assert rig.check_attention(0, dq, dout) <= ATOL[w.dtype]
    finally:
        rig.close()


def test_predict_matches_oracle_topk():
    """okv_predict: top-K of any query (here the true next query) equals the oracle's, within the
    tie band, and leaves the context's own selection untouched."""
    import torch
    import oracle as O
    from okv_harness import TIE_REL
    w = QWEN.scaled(layers=1, batch=3)
    rig = Rig(w)
    try:
        rig.stage(0, 0, 1.0, draft_step=-1)
        before = rig.ctx.read_selection(0)
        q = rig.batch_queries(0, 1, 0)
        counts = torch.zeros((rig.R, w.kv_heads), dtype=torch.int32, device="cuda")
        ids = torch.full((rig.R, w.kv_heads, rig.kb), -1, dtype=torch.int32, device="cuda")
        rig.ctx.predict(0, rig.device_rows(q, (w.q_heads, w.head_dim)), counts, ids)
        torch.cuda.synchronize()
        counts, ids = counts.cpu().numpy(), ids.cpu().numpy()
        g = w.group
        for i in range(w.batch):
            nb = -(-int(rig.model.n_tok[0, i]) // w.block_size)
            for h in range(w.kv_heads):
                osc = O.block_scores(np.ascontiguousarray(rig.model.summ[0][i, h, :nb]), q[i, h * g:(h + 1) * g])
                osel = O.topk(osc, rig.kb)
                n = len(osel)
                assert counts[i, h] == n
                gsel = ids[i, h, :n]
                diff = set(gsel.tolist()) ^ set(osel.tolist())
                if diff:
                    sK = float(osc[osel[-1]])
                    band = set(np.nonzero(np.abs(osc.astype(np.float64) - sK) <= TIE_REL * abs(sK))[0].tolist())
                    assert diff <= band, (i, h, sorted(diff - band))
        after = rig.ctx.read_selection(0)
        assert all(np.array_equal(a, b) for a, b in zip(before, after))
    finally:
        rig.close()


@pytest.mark.parametrize("cap", [0.01, 0.02, 0.1, 0.25])
def test_capsweep_workload(cap):
    """The fetch-cap sweep workload (100 directions, 5 active, one replaced per step) at each cap:
    C = 1, 2, 12, 32 blocks per unit and step, state carried over 3 steps."""
    import oracle as O
    w = synth.WORKLOADS["qwen3_8b_capsweep_b90"].scaled(layers=1, batch=3)
    rig = Rig(w)
    try:
        errs, _ = rig.run_steps(3, cap)
        assert max(errs) <= ATOL[BF16]
        counts, _ = rig.ctx.read_fetch_list(0)
        assert counts[:3].max() <= O.fetch_cap_blocks(cap, rig.kb)
    finally:
        rig.close()


def test_sync_deadline_reports_timeout():
    """okv_sync's deadline: staging queued behind a long (bounded) kernel on the caller's stream is
    still pending after 50 ms, so the call returns OKV_ETIMEOUT instead of waiting; once the
    kernel ends, the same context syncs and its state matches the oracle."""
    import torch
    from sparse_kv_cache_draft_gb300 import binding
    w = synth.WORKLOADS["tiny"]
    rig = Rig(w)
    try:
        draft = rig.batch_queries(0, -1, 1)
        draft_dev = rig.device_rows(draft, (w.q_heads, w.head_dim))  # (a pageable copy would wait out the sleep)
        torch.cuda.synchronize()
        torch.cuda._sleep(1_000_000_000)  # about half a second of GPU clock on the caller's stream
        rig.ctx.stage(0, draft_dev, 0, 1.0)
        assert rig.ctx.sync(50) == binding.ETIMEOUT
        torch.cuda.synchronize()
        assert rig.ctx.sync(60_000) == binding.OK
        rig._ensure_summaries(0)
        rig.model.score_topk(0, draft)
        gsel, _ = rig.check_selection(0)
        rig.model.select(0, rig.kb, 0, sel_override=gsel)
        rig.check_tables(0)
    finally:
        rig.close()


def test_step_with_appends_every_unit():
    """okv_step with appends (every layer's append on the library's own stream, each after its
    layer's previous staging) over 20 steps across block boundaries, 3 layers x 3 requests:
    the library's host writes, attention, selections, tables and pools of every unit after every
    step."""
    import torch
    import oracle as O
    from okv_harness import to_device, torch_dtype
    w = QWEN.scaled(layers=3, batch=3, steps=20)
    rig = Rig(w, contexts=[1000, 2040, 3000], capacity_tokens=3100)
    try:
        L, R, Hq, Hkv, d = w.layers, rig.R, w.q_heads, w.kv_heads, w.head_dim
        C = O.fetch_cap_blocks(w.fetch_cap, rig.kb)

        def all_layers(step, kind):
            return np.stack([rig.batch_queries(l, step, kind) for l in range(L)])

        d_boot = all_layers(-1, 1)
        for l in range(L):
            rig.ctx.stage(l, to_device(d_boot[l], w.dtype), 0, 1.0)
        torch.cuda.synchronize()
        for l in range(L):
            rig._ensure_summaries(l)
            rig.model.score_topk(l, d_boot[l])
            gsel, _ = rig.check_selection(l)
            rig.model.select(l, O.fetch_cap_blocks(1.0, rig.kb), 0, sel_override=gsel)
        for t in range(w.steps):
            kv = [synth.token_kv(w, l, rig.keys, rig.model.n_tok[l], plant_blocks=rig.plant_blocks) for l in range(L)]
            k_all = np.stack([k for k, _ in kv])
            v_all = np.stack([v for _, v in kv])
            q, dr = all_layers(t, 0), all_layers(t, 1)
            out = torch.zeros((L, R, Hq, d), dtype=torch_dtype(w.dtype), device="cuda")
            snap = rig.host_snapshot(range(L))
            rig.ctx.step(to_device(q, w.dtype), to_device(dr, w.dtype), out, t + 1,
                         k_new=to_device(k_all, w.dtype), v_new=to_device(v_all, w.dtype))
            torch.cuda.synchronize()
            assert rig.ctx.sync(60_000) == 0
            rig.check_host_append(snap, {l: (k_all[l], v_all[l]) for l in range(L)})
            for l in range(L):
                rig.model.append(l, k_all[l], v_all[l])
                rig.check_host_tail(l)
                assert rig.check_attention(l, q[l], out[l]) <= ATOL[BF16]
                rig.model.score_topk(l, dr[l])
                gsel, _ = rig.check_selection(l)
                rig.model.select(l, C, t + 1, sel_override=gsel)
                rig.check_tables(l)
                rig.check_pool(l)
        for l in range(L):
            rig.check_summaries(l)
            assert rig.ctx.read_lengths(l)[:3].tolist() == [1020, 2060, 3020]
    finally:
        rig.close()


@pytest.mark.parametrize("env", [{"OKV_STAGE_LANES": "1"}, {"OKV_STAGE_LANES": "2"},
                                 {"OKV_STAGE_STREAM": "caller"}, {"OKV_STAGE_PRIORITY": "high"},
                                 {"OKV_ATTEND_PRIORITY": "high"}, {"OKV_ATTEND_PRIORITY": "caller"}])
def test_staging_stream_layouts(env, monkeypatch):
    """The stream layouts (read at okv_create): one or two staging lanes (odd layers on the
    second), staging on the caller's stream, staging at the greatest priority, okv_step's own work
    at the greatest priority or on the caller's stream (instead of its attention stream at a
    middle priority); okv_stage and okv_step over 3 layers, bootstrap and 3 capped steps, every
    unit checked after every step."""
    import torch
    import oracle as O
    from okv_harness import to_device, torch_dtype
    for k, v in env.items():
        monkeypatch.setenv(k, v)
    w = QWEN.scaled(layers=3, batch=3, context=4096)
    rig = Rig(w)
    try:
        L, R, Hq, d = w.layers, rig.R, w.q_heads, w.head_dim
        C = O.fetch_cap_blocks(w.fetch_cap, rig.kb)
        for l in range(L):  # okv_stage, one layer at a time
            rig.stage(l, 0, 1.0, draft_step=-1)
        for t in range(3):  # okv_step, every layer
            q = np.stack([rig.batch_queries(l, t, 0) for l in range(L)])
            dr = np.stack([rig.batch_queries(l, t, 1) for l in range(L)])
            out = torch.zeros((L, R, Hq, d), dtype=torch_dtype(w.dtype), device="cuda")
            rig.ctx.step(to_device(q, w.dtype), to_device(dr, w.dtype), out, t + 1)
            torch.cuda.synchronize()
            assert rig.ctx.sync(60_000) == 0
            for l in range(L):
                assert rig.check_attention(l, q[l], out[l]) <= ATOL[BF16]
                rig.model.score_topk(l, dr[l])
                gsel, _ = rig.check_selection(l)
                rig.model.select(l, C, t + 1, sel_override=gsel)
                rig.check_tables(l)
                rig.check_pool(l)
    finally:
        rig.close()


def test_bytes_moved_equal_the_fetch_lists():
    """The gather's count of blocks moved host -> HBM (okv_timing.fetched_blocks, a device counter)
    equals the blocks of the oracle's fetch lists over a bootstrap and 4 capped steps, so the bytes
    per step the benchmark reports are the fetch lists' blocks times 8 KiB."""
    w = QWEN.scaled(layers=2, batch=3)
    rig = Rig(w)
    try:
        rig.ctx.set_timing(True)
        want = 0
        for layer in range(2):
            rig.stage(layer, 0, 1.0, draft_step=-1)
            want += int(rig.model.n_fetch[layer].sum())
        for t in range(4):
            for layer in range(2):
                rig.attend(layer, t)
                rig.stage(layer, t + 1, 0.05, draft_step=t)
                want += int(rig.model.n_fetch[layer].sum())
        got = rig.ctx.read_timing()["fetched_blocks"]
        assert got == want, (got, want)
        assert want > 2 * 3 * 8 * 128  # the bootstrap filled every pool, then capped steps added more
    finally:
        rig.close()
