"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each ``pin_*`` function takes an oracle library handle ``L`` (the normal build, or a
build with a planted mistake) and raises AssertionError when the oracle disagrees
with a closed form from the pages, a hand-worked case (``tests/golden/``), a
brute-force or library computation (numpy / torch CPU), or an invariant the pages
state for the selection step.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _round(x: np.ndarray, dtype: int) -> np.ndarray:
    """float64 -> storage (float32 or bfloat16 bits, round-to-nearest-even)."""
    f = np.asarray(x, dtype=np.float32)
    if dtype == synth.F32:
        return np.ascontiguousarray(f)
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return np.ascontiguousarray(u.astype(np.uint16))


def _f64(a: np.ndarray) -> np.ndarray:
    return synth.to_f64(a, synth.F32 if a.dtype == np.float32 else synth.BF16)


def make_unit(rng, cap_blocks, bs, d, dtype, n_tok, garbage=1.0e3):
    """Random host unit [cap_blocks][2][bs][d]; tokens at or past n_tok hold `garbage`."""
    x = rng.standard_normal((cap_blocks, 2, bs, d))
    flat_pos = np.arange(cap_blocks * bs).reshape(cap_blocks, bs)
    x[np.broadcast_to((flat_pos >= n_tok)[:, None, :, None], x.shape)] = garbage
    return _round(x, dtype)


def _tokens(host_unit, n_tok, which):
    """[n_tok][d] float64 K (which=0) or V (which=1) of the valid tokens."""
    cap, _, bs, d = host_unit.shape
    a = _f64(host_unit)[:, which].reshape(cap * bs, d)
    return a[:n_tok]


def _softmax_attend(q64, k64, v64):
    """Textbook attention softmax(q k^T / sqrt(d)) v for q [g][d], k, v [n][d]."""
    d = q64.shape[1]
    z = q64 @ k64.T / math.sqrt(d)
    z -= z.max(axis=1, keepdims=True)
    p = np.exp(z)
    p /= p.sum(axis=1, keepdims=True)
    return p @ v64


# ---- sizing -----------------------------------------------------------------------------------

def pin_kv_sizing(L):
    g = _golden("kv_sizing.json")
    for key in ("gqa32b", "qwen3_8b"):
        s = g[key]
        got = oracle.kv_bytes_per_token(s["layers"], s["kv_heads"], s["head_dim"], s["elem_bytes"], L)
        assert got == s["bytes_per_token"], (key, got)
    s = g["gqa32b"]
    per_tok = oracle.kv_bytes_per_token(s["layers"], s["kv_heads"], s["head_dim"], s["elem_bytes"], L)
    req = g["gqa32b_request"]
    gb = req["context_tokens"] * per_tok / 1e9
    assert abs(gb - req["gb_per_request"]) <= req["rel_tol"] * req["gb_per_request"], gb
    fit = g["gqa32b_fit"]
    assert math.floor(fit["hbm_gb"] / gb) == fit["requests"]


def pin_fetch_cap(L):
    # C = max(1, floor(cap * budget_blocks)) at the 2048-token budget (128 blocks of 16)
    for cap, c in ((0.01, 1), (0.02, 2), (0.05, 6), (0.1, 12), (0.25, 32), (1.0, 128)):
        assert oracle.fetch_cap_blocks(cap, 128, L) == c, (cap, oracle.fetch_cap_blocks(cap, 128, L))
    assert oracle.fetch_cap_blocks(1.0, 32, L) == 32
    assert oracle.fetch_cap_blocks(0.001, 32, L) == 1


# ---- summaries --------------------------------------------------------------------------------

def pin_summary_bruteforce(L):
    rng = np.random.default_rng(11)
    for dtype in (synth.F32, synth.BF16):
        for n_tok in (1, 15, 16, 17, 100, 128):
            bs, d, cap = 16, 8, 9
            hu = make_unit(rng, cap, bs, d, dtype, n_tok)
            s = oracle.block_summary(hu, n_tok, bs, d, L)
            k = _tokens(hu, n_tok, 0)
            nb = -(-n_tok // bs)
            assert s.shape == (nb, 2, d)
            for b in range(nb):
                kk = k[b * bs:(b + 1) * bs]
                assert np.array_equal(_f64(s[b, 0]), kk.min(axis=0)), (dtype, n_tok, b)
                assert np.array_equal(_f64(s[b, 1]), kk.max(axis=0)), (dtype, n_tok, b)


# ---- scores -----------------------------------------------------------------------------------

def pin_score_golden(L):
    g = _golden("score_example.json")
    summ = np.stack([np.array(g["kmin"], np.float32), np.array(g["kmax"], np.float32)], axis=1)
    summ = np.ascontiguousarray(summ)
    s = oracle.block_scores(summ, np.array(g["q"], np.float32), L)
    assert np.array_equal(s, np.array(g["scores"], np.float32)), s


def _random_summ_q(rng, nb, bs, d, g, dtype, n_tok=None):
    n_tok = n_tok if n_tok is not None else nb * bs
    hu = make_unit(rng, nb, bs, d, dtype, n_tok)
    summ = oracle.block_summary(hu, n_tok, bs, d)
    q = _round(rng.standard_normal((g, d)) * 0.7, dtype)
    return hu, summ, q


def pin_score_upper_bound(L):
    # the score bounds sum_h max_{t in b} q_h . k_t from above (it maximises over the box)
    rng = np.random.default_rng(12)
    for dtype in (synth.F32, synth.BF16):
        nb, bs, d, g = 12, 16, 16, 4
        hu, summ, q = _random_summ_q(rng, nb, bs, d, g, dtype, n_tok=nb * bs - 5)
        s = oracle.block_scores(summ, q, L).astype(np.float64)
        k = _tokens(hu, nb * bs - 5, 0)
        q64 = _f64(q)
        for b in range(nb):
            kk = k[b * bs:(b + 1) * bs]
            bound = (q64 @ kk.T).max(axis=1).sum()
            assert s[b] >= bound - 1e-5 * max(1.0, abs(bound)), (b, s[b], bound)


def pin_score_one_token(L):
    # a one-token block has kmin = kmax = k, so its score is exactly sum_h q_h . k
    rng = np.random.default_rng(13)
    for dtype in (synth.F32, synth.BF16):
        nb, bs, d, g = 10, 1, 32, 4
        hu, summ, q = _random_summ_q(rng, nb, bs, d, g, dtype)
        s = oracle.block_scores(summ, q, L).astype(np.float64)
        want = (_f64(q) @ _tokens(hu, nb, 0).T).sum(axis=0)
        assert np.allclose(s, want, rtol=1e-6, atol=1e-6), (s, want)


def pin_score_factorized(L):
    # sum_h max(q_h kmin, q_h kmax) == P kmax + N kmin with P (N) the sum of the positive
    # (negative) query coordinates of the group
    rng = np.random.default_rng(14)
    for dtype in (synth.F32, synth.BF16):
        nb, bs, d, g = 40, 16, 64, 4
        _hu, summ, q = _random_summ_q(rng, nb, bs, d, g, dtype)
        s = oracle.block_scores(summ, q, L).astype(np.float64)
        q64 = _f64(q)
        P = np.where(q64 > 0, q64, 0).sum(axis=0)
        N = np.where(q64 < 0, q64, 0).sum(axis=0)
        sm = _f64(summ)
        want = sm[:, 1] @ P + sm[:, 0] @ N
        assert np.allclose(s, want, rtol=1e-6, atol=1e-6), np.abs(s - want).max()


def pin_score_group_sum(L):
    # the KV head's score is the sum of its query heads' scores
    rng = np.random.default_rng(15)
    nb, bs, d, g = 20, 16, 16, 4
    _hu, summ, q = _random_summ_q(rng, nb, bs, d, g, synth.F32)
    s = oracle.block_scores(summ, q, L).astype(np.float64)
    parts = sum(oracle.block_scores(summ, q[h:h + 1], L).astype(np.float64) for h in range(g))
    assert np.allclose(s, parts, rtol=1e-6, atol=1e-6)
    # and a single block, single head, read by hand: d = 1
    summ1 = np.array([[[-2.0], [3.0]]], np.float32)
    assert oracle.block_scores(summ1, np.array([[-1.0]], np.float32), L)[0] == 2.0
    assert oracle.block_scores(summ1, np.array([[2.0]], np.float32), L)[0] == 6.0


# ---- top-K ------------------------------------------------------------------------------------

def pin_topk_bruteforce(L):
    rng = np.random.default_rng(16)
    for nb, kb in ((50, 8), (256, 32), (1024, 128), (7, 7), (5, 9), (1, 4)):
        s = rng.integers(-20, 20, size=nb).astype(np.float32) * 0.5  # many exact ties
        want = sorted(range(nb), key=lambda b: (-float(s[b]), b))[:min(kb, nb)]
        got = oracle.topk(s, kb, L)
        assert list(got) == want, (nb, kb)


def pin_topk_all_equal(L):
    s = np.full(40, 1.5, np.float32)
    assert list(oracle.topk(s, 10, L)) == list(range(10))


# ---- selection --------------------------------------------------------------------------------

def pin_select_golden(L):
    for sc in _golden("select_scenarios.json")["scenarios"]:
        kb, nb = sc["kb"], sc["nb"]
        resident = np.full(nb, -1, np.int32)
        slot_block = np.full(kb, -1, np.int32)
        stamp = np.full(kb, -1, np.int32)
        for st in sc["steps"]:
            cap = oracle.fetch_cap_blocks(st["cap"] / kb, kb, L)
            fetch = oracle.select_update(resident, slot_block, stamp, st["sel"], cap, st["step"], L)
            assert fetch.tolist() == st["fetch"], (sc["name"], st["step"], fetch.tolist())
            assert slot_block.tolist() == st["slot_block"], (sc["name"], st["step"], slot_block.tolist())
            for s, want in enumerate(st["stamp_of_occupied"]):
                if want is not None:
                    assert stamp[s] == want, (sc["name"], st["step"], stamp.tolist())
            for s, b in enumerate(slot_block):
                if b >= 0:
                    assert resident[b] == s
            assert int((resident >= 0).sum()) == int((slot_block >= 0).sum())


def pin_select_invariants(L):
    rng = np.random.default_rng(17)
    for trial in range(40):
        nb = int(rng.integers(3, 60))
        kb = int(rng.integers(2, 24))
        C = int(rng.integers(1, kb + 1))
        resident = np.full(nb, -1, np.int32)
        slot_block = np.full(kb, -1, np.int32)
        stamp = np.full(kb, -1, np.int32)
        for it in range(12):
            # the caller's step counter may repeat (two staging calls in one decode step)
            step = it // 2 if trial % 2 else it
            n_sel = min(kb, nb)
            sel = rng.permutation(nb)[:n_sel].astype(np.int32)
            before_res = resident.copy()
            before_slot = slot_block.copy()
            before_stamp = stamp.copy()
            fetch = oracle.select_update(resident, slot_block, stamp, sel, C, step, L)
            misses = [int(b) for b in sel if before_res[b] < 0]
            hits = [int(b) for b in sel if before_res[b] >= 0]
            n_admit = min(C, len(misses))
            assert len(fetch) == n_admit <= C
            assert [int(b) for b in fetch[:, 0]] == misses[:n_admit]
            for b in hits:  # resident predicted blocks stay, in their slot, stamped now
                assert resident[b] == before_res[b] and stamp[resident[b]] == step
            for b, s in fetch:
                assert slot_block[s] == b and resident[b] == s and stamp[s] == step
            assert int((slot_block >= 0).sum()) <= kb
            for s in range(kb):
                if slot_block[s] >= 0:
                    assert resident[slot_block[s]] == s
            assert int((resident >= 0).sum()) == int((slot_block >= 0).sum())
            # free slots go first, by ascending slot
            free_before = [s for s in range(kb) if before_slot[s] < 0]
            used = [int(s) for s in fetch[:, 1]]
            assert used[:min(len(free_before), n_admit)] == free_before[:n_admit]
            # evictions: only unselected blocks, and least recently selected first
            evicted = [int(before_slot[s]) for s in used if before_slot[s] >= 0]
            sel_set = set(int(b) for b in sel)
            assert not (set(evicted) & sel_set)
            survivors = [(int(before_stamp[s]), int(before_slot[s])) for s in range(kb)
                         if before_slot[s] >= 0 and int(before_slot[s]) not in sel_set
                         and int(before_slot[s]) not in evicted]
            for e in evicted:
                es = (int(before_stamp[before_res[e]]), e)
                assert all(es < sv for sv in survivors), (es, survivors)
            if C >= kb:  # fetch cap 1.0: the resident set equals the selection
                assert set(int(b) for b in slot_block if b >= 0) == sel_set
        if nb <= kb and C * 12 >= nb:  # budget covers the context: everything ends up resident
            assert set(int(b) for b in slot_block if b >= 0) == set(range(nb))


# ---- decode-side tier (partial staging) -------------------------------------------------------

def pin_local_tier_golden(L):
    for sc in _golden("local_tier_scenarios.json")["scenarios"]:
        local_of = np.full(sc["nb"], -1, np.int32)
        used = np.zeros(1, np.int32)
        for st in sc["steps"]:
            fetch = [[b, i] for i, b in enumerate(st["fetch"])]
            route, n_full = oracle.local_route(local_of, used, sc["local_cap"], fetch, L)
            assert route.tolist() == st["route"], (sc["name"], route.tolist())
            assert int(used[0]) == st["local_used"] and n_full == st["from_full"], (sc["name"], used, n_full)
            kept = {str(b): int(e) for b, e in enumerate(local_of) if e >= 0}
            assert kept == st["kept"], (sc["name"], kept)


def pin_local_tier_first_demand(L):
    # Fetch lists from real selection runs; the decode-side tier must hold exactly the first
    # local_cap distinct blocks in order of first demand, numbered in that order, and every other
    # fetch must read the full copy.
    rng = np.random.default_rng(23)
    for trial in range(30):
        nb = int(rng.integers(4, 80))
        kb = int(rng.integers(2, 20))
        C = int(rng.integers(1, kb + 1))
        local_cap = int(rng.choice([0, 1, int(rng.integers(1, nb + 1)), nb]))
        resident = np.full(nb, -1, np.int32)
        slot_block = np.full(kb, -1, np.int32)
        stamp = np.full(kb, -1, np.int32)
        local_of = np.full(nb, -1, np.int32)
        used = np.zeros(1, np.int32)
        demanded = []  # every fetched block, in order
        for step in range(15):
            sel = rng.permutation(nb)[:min(kb, nb)].astype(np.int32)
            fetch = oracle.select_update(resident, slot_block, stamp, sel, C, step, L)
            route, n_full = oracle.local_route(local_of, used, local_cap, fetch, L)
            first_order = list(dict.fromkeys(demanded + [int(b) for b in fetch[:, 0]]))
            kept = first_order[:local_cap]
            entry = {b: e for e, b in enumerate(kept)}
            want, full = [], 0
            for b in (int(x) for x in fetch[:, 0]):
                if b in entry and b in demanded:
                    want.append(2 * entry[b])
                elif b in entry:
                    want.append(2 * entry[b] + 1)
                    full += 1
                else:
                    want.append(-1)
                    full += 1
                demanded.append(b)
            assert route.tolist() == want, (trial, step, route.tolist(), want)
            assert n_full == full and int(used[0]) == len(kept) <= local_cap
            assert {b: int(e) for b, e in enumerate(local_of) if e >= 0} == entry
        if local_cap >= nb:  # ample entries: each block crosses from the full copy once
            assert int(used[0]) == len(set(demanded))


# ---- attention --------------------------------------------------------------------------------

def pin_attend_dense_textbook(L):
    # budget >= context with fetch cap 1.0: one staging step makes every block resident,
    # and sparse attention is dense softmax attention
    rng = np.random.default_rng(18)
    for dtype in (synth.F32, synth.BF16):
        bs, d, g, kb = 16, 32, 4, 8
        for n_tok in (1, 17, 100, 128):
            nb = -(-n_tok // bs)
            hu = make_unit(rng, kb, bs, d, dtype, n_tok)
            summ = oracle.block_summary(hu, n_tok, bs, d, L)
            draft = _round(rng.standard_normal((g, d)), dtype)
            q = _round(rng.standard_normal((g, d)), dtype)
            sel = oracle.topk(oracle.block_scores(summ, draft, L), kb, L)
            resident = np.full(kb, -1, np.int32)
            slot_block = np.full(kb, -1, np.int32)
            stamp = np.full(kb, -1, np.int32)
            oracle.select_update(resident, slot_block, stamp, sel, kb, 0, L)
            assert sorted(int(b) for b in slot_block if b >= 0) == list(range(nb))
            sparse = oracle.attend(hu, slot_block, n_tok, bs, d, q, L)
            dense = oracle.dense_attend(hu, n_tok, bs, d, q, L)
            want = _softmax_attend(_f64(q), _tokens(hu, n_tok, 0), _tokens(hu, n_tok, 1))
            assert np.allclose(dense, want, rtol=1e-12, atol=1e-12)
            assert np.allclose(sparse, want, rtol=1e-12, atol=1e-12)


def pin_attend_torch_sdpa(L):
    import torch
    rng = np.random.default_rng(19)
    bs, d, g, n_tok = 16, 64, 4, 200
    hu = make_unit(rng, 13, bs, d, synth.F32, n_tok)
    q = _round(rng.standard_normal((g, d)), synth.F32)
    dense = oracle.dense_attend(hu, n_tok, bs, d, q, L)
    qt = torch.from_numpy(_f64(q))[None, :, None, :]
    kt = torch.from_numpy(_tokens(hu, n_tok, 0))[None, None].expand(1, g, n_tok, d)
    vt = torch.from_numpy(_tokens(hu, n_tok, 1))[None, None].expand(1, g, n_tok, d)
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt)[0, :, 0].numpy()
    assert np.allclose(dense, ref, rtol=1e-10, atol=1e-10)


def pin_attend_subset(L):
    # attention reads exactly the valid tokens of the occupied slots, partial tail included
    rng = np.random.default_rng(20)
    bs, d, g, kb, n_tok = 16, 16, 4, 6, 150  # 10 blocks, the last with 6 tokens
    hu = make_unit(rng, 10, bs, d, synth.BF16, n_tok)
    q = _round(rng.standard_normal((g, d)), synth.BF16)
    slot_block = np.array([9, -1, 3, 0, -1, 7], np.int32)
    got = oracle.attend(hu, slot_block, n_tok, bs, d, q, L)
    k = _tokens(hu, n_tok, 0)
    v = _tokens(hu, n_tok, 1)
    idx = [t for b in (9, 3, 0, 7) for t in range(b * bs, min((b + 1) * bs, n_tok))]
    want = _softmax_attend(_f64(q), k[idx], v[idx])
    assert np.allclose(got, want, rtol=1e-12, atol=1e-12)


def pin_attend_special_cases(L):
    rng = np.random.default_rng(21)
    bs, d, g = 16, 16, 2
    # one token of context: the output is that token's value
    hu = make_unit(rng, 2, bs, d, synth.F32, 1)
    q = _round(rng.standard_normal((g, d)), synth.F32)
    out = oracle.attend(hu, np.array([0, -1], np.int32), 1, bs, d, q, L)
    for h in range(g):
        assert np.allclose(out[h], _f64(hu[0, 1, 0]), rtol=0, atol=1e-15)
    # zero query: every score is equal, so the output is the mean value
    hu = make_unit(rng, 4, bs, d, synth.F32, 50)
    q0 = np.zeros((g, d), np.float32)
    out = oracle.attend(hu, np.array([2, 0, -1, 3], np.int32), 50, bs, d, q0, L)
    v = _tokens(hu, 50, 1)
    idx = list(range(32, 48)) + list(range(0, 16)) + list(range(48, 50))
    assert np.allclose(out, np.broadcast_to(v[idx].mean(axis=0), out.shape), rtol=1e-12, atol=1e-12)
    # nothing resident: zeros
    out = oracle.attend(hu, np.full(4, -1, np.int32), 50, bs, d, q, L)
    assert not out.any()


# ---- append -----------------------------------------------------------------------------------

def pin_append(L):
    rng = np.random.default_rng(22)
    for dtype in (synth.F32, synth.BF16):
        bs, d, cap = 16, 8, 4
        n0 = 13
        hu = make_unit(rng, cap, bs, d, dtype, n0)
        summ = np.zeros((cap, 2, d), dtype=hu.dtype)
        summ[:1] = oracle.block_summary(hu, n0, bs, d, L)
        n = n0
        for _ in range(30):  # crosses two block boundaries
            k = _round(rng.standard_normal(d), dtype)
            v = _round(rng.standard_normal(d), dtype)
            oracle.append(hu, summ, n, bs, d, k, v, L)
            b, t = divmod(n, bs)
            assert np.array_equal(hu[b, 0, t], k) and np.array_equal(hu[b, 1, t], v)
            n += 1
            nb = -(-n // bs)
            rebuilt = oracle.block_summary(hu, n, bs, d, L)
            assert np.array_equal(summ[:nb], rebuilt), n
            kk = _tokens(hu, n, 0)
            assert np.array_equal(_f64(summ[nb - 1, 0]), kk[(nb - 1) * bs:n].min(axis=0))
            assert np.array_equal(_f64(summ[nb - 1, 1]), kk[(nb - 1) * bs:n].max(axis=0))


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
