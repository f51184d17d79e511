"""Exact ties in the per-head top-K (needs a GB300).

The selection ranks blocks by (binary32 score desc, block id asc), so blocks whose scores are
equal go to the lower block id (the top-K and KV selection of OasisKV,
paperlayer.ai/abs/2608.08097v1, "4 System Design"; the tie rule is the method's reading of it).
Random keys almost never tie, so these cases make ties on purpose, in ways that give
bit-identical binary32 scores on both sides:

* a zero draft query: every block scores exactly 0, so the selection is blocks 0 .. K-1;
* byte-identical blocks (identical min/max summaries, hence identical scores in any summation
  order) whose common score is far above every other block's, more of them than the budget
  holds: the selection is the K lowest ids among them.

Selections are compared with no tie band (`exact=True`): ids and order must be the oracle's.
The diff / admit / evict that follows (first C misses in selection order, least-recently-
selected eviction) is compared exactly as everywhere else.
"""
import numpy as np
import pytest

import synth
from okv_harness import ATOL, Rig

pytestmark = pytest.mark.gpu

QWEN = synth.WORKLOADS["qwen3_8b_16k_b128"]


def _stored(value: float, dtype: int):
    """One value in the storage type (binary32, or bfloat16 bits)."""
    f = np.float32(value)
    return f if dtype == synth.F32 else np.uint16(f.view(np.uint32) >> 16)


def _identical_hot_blocks(positions, dtype):
    """edit_kv: every block in `positions` becomes a byte-identical copy of the first one, whose
    token 0 keys are +8 and token 1 keys -8 in every coordinate (min -8, max +8 on every dim)."""
    hi, lo = _stored(8.0, dtype), _stored(-8.0, dtype)

    def edit(layer, key, arr):
        src = arr[:, positions[0]].copy()  # [Hkv][2][bs][d]
        src[:, 0, 0, :] = hi
        src[:, 0, 1, :] = lo
        for b in positions:
            arr[:, b] = src
    return edit


def _zero_draft(rig):
    return np.zeros((rig.w.batch, rig.w.q_heads, rig.w.head_dim), rig.sdt)


@pytest.mark.parametrize("context,batch", [(16384, 3), (256000, 1)])
def test_zero_draft_selects_lowest_ids(context, batch):
    """All scores 0: the selection is blocks 0..127 in id order. After a bootstrap from a random
    draft, a zero draft at cap 0.05 admits the 6 lowest-id blocks not yet resident, evicting the
    least recently selected; at cap 1.0 the pool then holds exactly blocks 0..127."""
    w = QWEN.scaled(layers=1, batch=batch, context=context)
    rig = Rig(w)
    try:
        rig.stage(0, 0, 1.0, draft_step=-1)
        z = _zero_draft(rig)
        rig.stage(0, 1, 0.05, draft=z, exact=True)
        counts, ids, scores = rig.ctx.read_selection(0)
        for i in range(batch):
            for h in range(w.kv_heads):
                assert ids[i, h, :counts[i, h]].tolist() == list(range(rig.kb))
                assert not scores[i, h, :counts[i, h]].any()
        rig.stage(0, 2, 1.0, draft=z, exact=True)
        sb, _ = rig.ctx.read_slot_table(0)
        for i in range(batch):
            for h in range(w.kv_heads):
                assert sorted(sb[i, h].tolist()) == list(range(rig.kb))
        assert rig.attend(0, 3) <= ATOL[w.dtype]
    finally:
        rig.close()


@pytest.mark.parametrize("context,stride", [(16384, 5), (256000, 50)])
def test_identical_blocks_tie_at_the_boundary(context, stride):
    """Every `stride`-th block is the same hot block (205 copies of 1024 blocks at 16K, 320 of
    16000 at 256K): the budget's 128 slots go to the 128 lowest ids among them, at every step,
    whatever the draft."""
    w = QWEN.scaled(layers=1, batch=1, context=context)
    nb = context // w.block_size
    hot = list(range(0, nb - 1, stride))
    assert len(hot) > 128
    rig = Rig(w, edit_kv=_identical_hot_blocks(hot, w.dtype))
    try:
        rig.check_summaries(0)
        rig.stage(0, 0, 1.0, draft_step=-1, exact=True)
        for t in range(3):
            assert rig.attend(0, t) <= ATOL[w.dtype]
            rig.stage(0, t + 1, 0.05, draft_step=t, exact=True)
        counts, ids, _ = rig.ctx.read_selection(0)
        for h in range(w.kv_heads):
            assert ids[0, h, :counts[0, h]].tolist() == hot[:128]
    finally:
        rig.close()


def test_identical_blocks_fp32_ragged():
    """fp32 tiny shapes (d 64, GQA 8/2, budget 512 = 32 slots): 40 identical hot blocks in a
    4000-token context (250 blocks, a partial tail) tie for 32 slots; a second request with a
    3-block context selects everything it has."""
    w = synth.WORKLOADS["tiny"]
    hot = list(range(3, 243, 6))
    rig = Rig(w, contexts=[4000, 40], capacity_tokens=4096, edit_kv=_identical_hot_blocks(hot, w.dtype))
    try:
        rig.stage(0, 0, 1.0, draft_step=-1, exact=True)
        counts, ids, _ = rig.ctx.read_selection(0)
        for h in range(w.kv_heads):
            assert ids[0, h, :counts[0, h]].tolist() == hot[:32]
            assert counts[1, h] == 3
        assert rig.attend(0, 0) <= ATOL[w.dtype]
    finally:
        rig.close()
