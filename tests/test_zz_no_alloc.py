"""The allocation-free attention entry point (okv_attend_static) against okv_attend.

okv_attend_static serves callers that cannot allocate device memory: it takes every input and
output from the caller and keeps its only workspace in a fixed array inside the library. Here
a context stages real pools; their contents, slot tables and lengths are copied into caller
tensors, and two calls in a row of the allocation-free entry point (two different queries)
must agree with okv_attend on the same queries. The same entry point carries the dense
baseline (every block of the full KV in HBM), checked against the oracle's dense attention.
This file is collected last on purpose.
"""
import numpy as np
import pytest

import synth
from okv_harness import ATOL, Rig, out_to_f64, torch_dtype
from sparse_kv_cache_draft_gb300 import BF16, F32, OkvError, binding

pytestmark = pytest.mark.gpu


def _static_inputs(rig, layer):
    import torch
    w, R = rig.w, rig.R
    pool = np.stack([np.stack([rig.ctx.read_pool(layer, r, h) for h in range(w.kv_heads)]) for r in range(R)])
    sb, _ = rig.ctx.read_slot_table(layer)
    lens = rig.ctx.read_lengths(layer)
    pool_t = torch.from_numpy(pool.view(np.int16)).view(torch.bfloat16) if w.dtype == BF16 else torch.from_numpy(pool)
    return pool_t.cuda().contiguous(), torch.from_numpy(sb).cuda(), torch.from_numpy(lens).cuda()


@pytest.mark.parametrize("name,kw", [
    ("qwen_bf16", dict(wl="qwen3_8b_16k_b128", layers=1, batch=3)),      # tensor-core path, split partials
    ("tiny_fp32", dict(wl="tiny")),                                       # CUDA-core path, split partials
    # tensor-core path, GQA group 4 (half the MMA's columns), the largest split (16 slices of the
    # 128 slots per unit): the most split partials per unit the workspace bound allows for
    ("qwen_bf16_split16", dict(wl="qwen3_8b_16k_b128", layers=1, batch=3, split="16")),
    # CUDA-core path at the largest head dim, fp32
    ("fp32_d256", dict(wl="qwen3_8b_16k_b128", layers=1, batch=2, dtype=F32, head_dim=256, q_heads=16,
                       kv_heads=8, context=3000, budget_tokens=512)),
])
def test_static_attention_matches_okv_attend(name, kw, monkeypatch):
    import torch
    kw = dict(kw)
    wl = kw.pop("wl")
    split = kw.pop("split", None)
    if split is not None:
        monkeypatch.setenv("OKV_ATTEND_SPLIT", split)  # read by both entry points at each launch
    w = synth.WORKLOADS[wl]
    if kw:
        w = w.scaled(**kw)
    rig = Rig(w)
    try:
        rig.stage(0, 0, 1.0, draft_step=-1, check_pool=False)
        rig.stage(0, 1, w.fetch_cap, draft_step=0, check_pool=False)
        pool, sb, lens = _static_inputs(rig, 0)
        shp = (rig.R, w.q_heads, w.head_dim)
        for call, step in enumerate((1, 2)):  # two calls in a row, different queries
            q = rig.device_rows(rig.batch_queries(0, step, 0), (w.q_heads, w.head_dim))
            ref = torch.zeros(shp, dtype=torch_dtype(w.dtype), device="cuda")
            rig.ctx.attend(0, q, ref)
            got = torch.full(shp, float("nan"), dtype=torch_dtype(w.dtype), device="cuda")
            binding.attend_static(pool, sb, lens, q, got, q_heads=w.q_heads, kv_heads=w.kv_heads,
                                  head_dim=w.head_dim, block_size=w.block_size, slots=rig.kb, dtype=w.dtype)
            torch.cuda.synchronize()
            err = float(np.abs(out_to_f64(got, w.dtype) - out_to_f64(ref, w.dtype)).max())
            assert err <= ATOL[w.dtype], (name, call, err)
            # and against the oracle directly
            assert rig.check_attention(0, rig.batch_queries(0, step, 0), got) <= ATOL[w.dtype]
    finally:
        rig.close()


def test_static_attention_rejects_oversized_shapes():
    import torch
    L = binding.load_library()
    z = torch.zeros(64, dtype=torch.int32, device="cuda")
    p = z.data_ptr()
    # more requests than the fixed workspace holds ids for
    assert L.okv_attend_static(16385, 32, 8, 128, 16, 128, BF16, p, p, p, p, p, None) == binding.EINVAL
    # a split workspace larger than the fixed array: 243 requests x 5 KV heads, group 8, d 256, fp32
    assert L.okv_attend_static(243, 40, 5, 256, 16, 128, F32, p, p, p, p, p, None) == binding.EINVAL
    # a shape the attention does not take
    assert L.okv_attend_static(4, 6, 4, 128, 16, 128, BF16, p, p, p, p, p, None) == binding.EINVAL


def test_dense_baseline_matches_oracle():
    """The dense baseline (`bench.py --report dense`): okv_attend_static over an identity slot table
    of every block (the full KV in HBM, 1024 slots per unit at 16K) equals the oracle's dense
    softmax attention. Qwen3-8B attention shapes, one layer, contexts of 16384, 9000 and 1 tokens
    (slots past a context hold -1)."""
    import torch
    w = synth.WORKLOADS["qwen3_8b_16k_b128"].scaled(layers=1, batch=3)
    rig = Rig(w, contexts=[16384, 9000, 1])
    try:
        R, H, nb, bs, d = rig.R, w.kv_heads, rig.cap_blocks, w.block_size, w.head_dim
        kv = np.stack([np.stack([rig.model.host_unit(0, i, h) for h in range(H)]) for i in range(R)])
        pool = torch.from_numpy(np.ascontiguousarray(kv).view(np.int16)).view(torch.bfloat16).cuda()
        sb = np.full((R, H, nb), -1, np.int32)
        for i, n in enumerate(rig.contexts):
            sb[i, :, :-(-int(n) // bs)] = np.arange(-(-int(n) // bs), dtype=np.int32)
        lens = torch.from_numpy(rig.contexts.astype(np.int32)).cuda()
        q = rig.batch_queries(0, 0, 0)
        out = torch.full((R, w.q_heads, d), float("nan"), dtype=torch.bfloat16, device="cuda")
        binding.attend_static(pool, torch.from_numpy(sb).cuda(), lens, rig.device_rows(q, (w.q_heads, d)), out,
                              q_heads=w.q_heads, kv_heads=H, head_dim=d, block_size=bs, slots=nb, dtype=BF16)
        torch.cuda.synchronize()
        want = rig.model.attend(0, q, dense=True)
        err = float(np.abs(out_to_f64(out, BF16)[rig.ids] - want).max())
        assert err <= ATOL[BF16], err
    finally:
        rig.close()
