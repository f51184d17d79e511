"""Edge cases of the CUDA path vs the CPU oracle (needs a GB300): an empty context growing by
appends, contexts around the budget, the smallest and largest head dims, GQA groups 1, 3 and 6,
block sizes other than 16, a one-slot budget, the largest budget and the smallest fetch cap."""
import numpy as np
import pytest

import synth
from okv_harness import ATOL, Rig
from sparse_kv_cache_draft_gb300 import BF16, F32

pytestmark = pytest.mark.gpu

QWEN = synth.WORKLOADS["qwen3_8b_16k_b128"]


def test_empty_context_grows_by_appends():
    """A request registered with no tokens selects nothing and attends to nothing (zeros), then
    grows by one token per step across a block boundary; 15- and 16-token requests beside it."""
    w = QWEN.scaled(layers=1, batch=3, context=16)
    rig = Rig(w, contexts=[0, 15, 16], capacity_tokens=64)
    try:
        errs, _ = rig.run_steps(20, 0.05, append=True)
        assert max(errs) <= ATOL[BF16]
        rig.check_summaries(0)
        assert rig.ctx.read_lengths(0)[:3].tolist() == [20, 35, 36]
    finally:
        rig.close()


def test_contexts_around_the_budget():
    """2047, 2048, 2049 and 2064 tokens with a 2048-token budget: 128 blocks fit the pool
    exactly; 129 blocks leave one out each step."""
    w = QWEN.scaled(layers=1, batch=4)
    rig = Rig(w, contexts=[2047, 2048, 2049, 2064])
    try:
        errs, _ = rig.run_steps(4, 0.05)
        assert max(errs) <= ATOL[BF16]
        sb, _ = rig.ctx.read_slot_table(0)
        for i in (0, 1):  # the budget covers the context: every block resident
            assert (np.sort(sb[i], axis=1) == np.arange(128)).all()
        for i in (2, 3):
            assert (sb[i] >= 0).all()
    finally:
        rig.close()


@pytest.mark.parametrize("dtype,d,g", [(F32, 32, 1), (BF16, 32, 3), (BF16, 256, 2), (F32, 256, 6),
                                       (BF16, 128, 1), (BF16, 128, 6)])
def test_head_dims_and_groups(dtype, d, g):
    """Head dims 32 and 256 (the generic scoring loop above 32 vectors per record), MHA (g = 1) and
    odd or uneven GQA groups, on both attention kernels."""
    w = QWEN.scaled(layers=1, batch=2, dtype=dtype, head_dim=d, q_heads=4 * g, kv_heads=4,
                    context=2500, budget_tokens=512)
    rig = Rig(w)
    try:
        errs, _ = rig.run_steps(3, 0.1)
        assert max(errs) <= ATOL[dtype]
    finally:
        rig.close()


@pytest.mark.parametrize("bs", [8, 32, 64])
def test_block_sizes(bs):
    """Blocks of 8, 32 and 64 tokens (CUDA-core attention), ragged tails, cap 0.001 (C = 1)."""
    w = QWEN.scaled(layers=1, batch=3, block_size=bs, budget_tokens=16 * bs, context=40 * bs + 3)
    rig = Rig(w, contexts=[bs - 1, 12 * bs + 5, 40 * bs + 3])
    try:
        errs, _ = rig.run_steps(4, 0.001)
        assert max(errs) <= ATOL[BF16]
        counts, _ = rig.ctx.read_fetch_list(0)
        assert counts[:3].max() <= 1
    finally:
        rig.close()


def test_one_slot_budget():
    """A budget of one block: each unit keeps the single best block; C = 1 at any cap."""
    w = QWEN.scaled(layers=1, batch=2, budget_tokens=16, context=100)
    rig = Rig(w)
    try:
        errs, _ = rig.run_steps(4, 1.0)
        assert max(errs) <= ATOL[BF16]
        sb, _ = rig.ctx.read_slot_table(0)
        assert (sb[:2] >= 0).all()
    finally:
        rig.close()


def test_largest_budget_batch_one():
    """The largest pool (1024 slots, a 16384-token budget) for one request of 20000 tokens
    (1250 blocks) on the tensor-core kernel, cap 0.05 (C = 51)."""
    w = QWEN.scaled(layers=1, batch=1, budget_tokens=16384, context=20000)
    rig = Rig(w)
    try:
        errs, _ = rig.run_steps(2, 0.05)
        assert max(errs) <= ATOL[BF16]
        counts, _ = rig.ctx.read_fetch_list(0)
        assert counts[0].max() <= 51
    finally:
        rig.close()


def test_longest_context_at_the_default_budget():
    """600000 tokens (37500 blocks, near the largest context one staging CTA's shared memory
    holds at a 128-slot budget: 37680 blocks), one request, cap 0.05."""
    w = QWEN.scaled(layers=1, batch=1, context=600000)
    rig = Rig(w)
    try:
        errs, _ = rig.run_steps(2, 0.05)
        assert max(errs) <= ATOL[BF16]
    finally:
        rig.close()


def test_split_chosen_after_create(monkeypatch):
    """The attention's split may be chosen after the context sized its split workspace (here
    OKV_ATTEND_SPLIT=16 set after okv_create, whose 1024 units call for a split of 2): each launch
    splits no further than the workspace holds, and the outputs still match the oracle."""
    w = QWEN.scaled(layers=1, batch=128, context=1040)
    rig = Rig(w, n_alias=4)
    try:
        monkeypatch.setenv("OKV_ATTEND_SPLIT", "16")
        sample = [0, 77, 127]
        errs, _ = rig.run_steps(2, 0.05, requests=sample, check_pool=False)
        assert max(errs) <= ATOL[BF16]
    finally:
        rig.close()
