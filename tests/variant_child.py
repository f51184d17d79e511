"""One small decode run through the library as the environment of this process configures it,
checked against the oracle; exits 0 when every check passes.

The library reads some of its measured alternatives once per process (the attention's tile
shape, OKV_ATTEND_TILE; the gather's work distribution, OKV_GATHER_DYNAMIC, and grid size,
OKV_GATHER_CTAS), so test_gpu_variants.py runs this file in a child process per setting.
Qwen3-8B attention shapes, 2 layers, 3 requests of 4096 tokens: a bootstrap staging of every
block, then 2 capped decode steps through okv_step; after each step every unit's attention,
selection, slot table, stamps, fetch list and pool bytes are compared with the oracle.
"""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))
sys.path.insert(0, HERE)

import numpy as np  # noqa: E402

import oracle as O  # noqa: E402
import synth  # noqa: E402
from okv_harness import ATOL, Rig, to_device, torch_dtype  # noqa: E402
from sparse_kv_cache_draft_gb300 import BF16  # noqa: E402


def main() -> int:
    import torch
    w = synth.WORKLOADS["qwen3_8b_16k_b128"].scaled(layers=2, batch=3, context=4096)
    rig = Rig(w)
    try:
        L, R, Hq, d = w.layers, rig.R, w.q_heads, w.head_dim
        C = O.fetch_cap_blocks(w.fetch_cap, rig.kb)
        for l in range(L):
            rig.stage(l, 0, 1.0, draft_step=-1)
        for t in range(2):
            q = np.stack([rig.batch_queries(l, t, 0) for l in range(L)])
            dr = np.stack([rig.batch_queries(l, t, 1) for l in range(L)])
            out = torch.zeros((L, R, Hq, d), dtype=torch_dtype(w.dtype), device="cuda")
            rig.ctx.step(to_device(q, w.dtype), to_device(dr, w.dtype), out, t + 1)
            torch.cuda.synchronize()
            assert rig.ctx.sync(60_000) == 0
            for l in range(L):
                err = rig.check_attention(l, q[l], out[l])
                assert err <= ATOL[BF16], (l, t, err)
                rig.model.score_topk(l, dr[l])
                gsel, _ = rig.check_selection(l)
                rig.model.select(l, C, t + 1, sel_override=gsel)
                rig.check_tables(l)
                rig.check_pool(l)
    finally:
        rig.close()
    print("variant ok:", {k: v for k, v in os.environ.items() if k.startswith("OKV_")})
    return 0


if __name__ == "__main__":
    sys.exit(main())
