"""The oracle's whole-layer driver (OracleModel, threaded over units) against its per-unit
functions, which the pins check against the pages (CPU only).

The GPU parity tests compare the CUDA path with OracleModel, so a mistake in the driver (a unit
wired to the wrong request, head or layer, a table not carried between steps, a route not
written) would make those comparisons wrong while every per-unit pin still passes. Here the
driver and a plain loop over the per-unit functions run the same steps on the same host bytes
and must agree exactly.
"""
import numpy as np
import pytest

import oracle
import oracle_pins

L, HQ, HKV, D, BS, BUDGET = 2, 8, 2, 32, 16, 128
G = HQ // HKV
KB = BUDGET // BS


def _host(rng, dtype, cap, contexts):
    """One buffer per request: [L][Hkv][cap][2][bs][d] storage, garbage past each context."""
    bufs = []
    for n in contexts:
        units = [oracle_pins.make_unit(rng, cap, BS, D, dtype, n) for _ in range(L * HKV)]
        bufs.append(np.ascontiguousarray(np.stack(units).reshape(L, HKV, cap, 2, BS, D)))
    return bufs


@pytest.mark.parametrize("dtype", [oracle.F32, oracle.BF16])
def test_driver_matches_per_unit_functions(dtype):
    rng = np.random.default_rng(31)
    contexts = np.array([40, 100, 200], np.int32)
    cap = -(-int(contexts.max() + 4) // BS)
    local_cap = [-1, 0, 5]
    bufs = _host(rng, dtype, cap, contexts)
    model = oracle.OracleModel(layers=L, q_heads=HQ, kv_heads=HKV, head_dim=D, block_size=BS,
                               budget_tokens=BUDGET, dtype=dtype, req_ptrs=[b.ctypes.data for b in bufs],
                               cap_blocks=[cap] * 3, n_tok=contexts, n_threads=4, local_cap=local_cap)
    sdt = np.float32 if dtype == oracle.F32 else np.uint16
    # the per-unit reference state, [layer][request][head]
    ref = {}
    for l in range(L):
        for r in range(3):
            for h in range(HKV):
                nb = -(-int(contexts[r]) // BS)
                ref[l, r, h] = dict(resident=np.full(cap, -1, np.int32), slot=np.full(KB, -1, np.int32),
                                    stamp=np.full(KB, -1, np.int32), local_of=np.full(cap, -1, np.int32),
                                    used=np.zeros(1, np.int32), n=int(contexts[r]), nb=nb)
    for l in range(L):
        model.build_summaries(l)
        for r in range(3):
            for h in range(HKV):
                want = oracle.block_summary(bufs[r][l, h], ref[l, r, h]["n"], BS, D)
                assert np.array_equal(model.summ[l][r, h][:want.shape[0]], want), (l, r, h)
                ref[l, r, h]["summ"] = np.zeros((cap, 2, D), sdt)
                ref[l, r, h]["summ"][:want.shape[0]] = want
    for step in range(3):
        caps = [KB, 2, 3][step]
        for l in range(L):
            draft = oracle_pins._round(rng.standard_normal((3, HQ, D)), dtype)
            q = oracle_pins._round(rng.standard_normal((3, HQ, D)), dtype)
            model.stage(l, draft, caps, step)
            out = model.attend(l, q)
            for r in range(3):
                for h in range(HKV):
                    u = ref[l, r, h]
                    nb = -(-u["n"] // BS)
                    sc = oracle.block_scores(u["summ"][:nb], draft[r, h * G:(h + 1) * G])
                    sel = oracle.topk(sc, KB)
                    n_sel = int(model.n_sel[l][r, h])
                    assert n_sel == len(sel) and np.array_equal(model.sel_ids[l][r, h, :n_sel], sel), (step, l, r, h)
                    fetch = oracle.select_update(u["resident"], u["slot"], u["stamp"], sel, caps, step)
                    nf = int(model.n_fetch[l][r, h])
                    assert nf == len(fetch) and np.array_equal(model.fetch[l][r, h, :nf], fetch), (step, l, r, h)
                    assert np.array_equal(model.slot_block[l][r, h], u["slot"]), (step, l, r, h)
                    if local_cap[r] >= 0:
                        route, _ = oracle.local_route(u["local_of"], u["used"], local_cap[r], fetch)
                        assert np.array_equal(model.route[l][r, h, :nf], route), (step, l, r, h)
                        assert np.array_equal(model.local_of[l][r, h], u["local_of"]), (step, l, r, h)
                        assert int(model.local_used[l][r, h]) == int(u["used"][0])
                    else:
                        assert (model.route[l][r, h, :nf] == -1).all()
                    want = oracle.attend(bufs[r][l, h], u["slot"], u["n"], BS, D, q[r, h * G:(h + 1) * G])
                    assert np.array_equal(out[r, h * G:(h + 1) * G], want), (step, l, r, h)
            # one appended token per request: the driver appends into the host bytes and its
            # summaries; the reference summaries follow with the per-unit append on a copy
            k = oracle_pins._round(rng.standard_normal((3, HKV, D)), dtype)
            v = oracle_pins._round(rng.standard_normal((3, HKV, D)), dtype)
            before = {r: bufs[r][l].copy() for r in range(3)}
            model.append(l, k, v)
            for r in range(3):
                for h in range(HKV):
                    u = ref[l, r, h]
                    unit = before[r][h].copy()
                    oracle.append(unit, u["summ"], u["n"], BS, D, k[r, h], v[r, h])
                    u["n"] += 1
                    assert np.array_equal(bufs[r][l, h], unit), (step, l, r, h)
                    assert np.array_equal(model.summ[l][r, h], u["summ"]), (step, l, r, h)
                    assert int(model.n_tok[l, r]) == u["n"]


def test_private_host_copy():
    """With host_fill the driver keeps its own copy of each (layer, content key): aliased requests
    share it, appends write only it, and every result equals the driver run on raw buffers
    holding the same bytes."""
    rng = np.random.default_rng(5)
    dtype = oracle.BF16
    contexts = np.array([60, 60, 90], np.int32)
    cap = -(-int(contexts.max() + 4) // BS)
    src = _host(rng, dtype, cap, contexts)
    keys = [0, 0, 1]  # requests 0 and 1 share one content
    bufs = [src[0].copy(), src[0].copy(), src[2].copy()]
    frozen = [b.copy() for b in src]
    fills = []

    def host_fill(layer, key, arr):
        fills.append((layer, key))
        arr[...] = src[2 * key][layer]

    common = dict(layers=L, q_heads=HQ, kv_heads=HKV, head_dim=D, block_size=BS, budget_tokens=BUDGET,
                  dtype=dtype, cap_blocks=[cap] * 3, n_tok=contexts, n_threads=2)
    own = oracle.OracleModel(host_fill=host_fill, req_keys=keys, **common)
    raw = oracle.OracleModel(req_ptrs=[b.ctypes.data for b in bufs], **common)
    assert sorted(fills) == [(l, k) for l in range(L) for k in (0, 1)]
    assert own.host_unit_ptr(0, 0, 1) == own.host_unit_ptr(0, 1, 1) != own.host_unit_ptr(0, 2, 1)
    for l in range(L):
        for m in (own, raw):
            m.build_summaries(l)
        draft = oracle_pins._round(rng.standard_normal((3, HQ, D)), dtype)
        q = oracle_pins._round(rng.standard_normal((3, HQ, D)), dtype)
        for m in (own, raw):
            m.stage(l, draft, KB, 0)
        assert np.array_equal(own.attend(l, q), raw.attend(l, q))
        # appends of the non-aliased request only (aliased requests cannot append)
        k = oracle_pins._round(rng.standard_normal((3, HKV, D)), dtype)
        v = oracle_pins._round(rng.standard_normal((3, HKV, D)), dtype)
        for h in range(HKV):
            oracle.append(own.host_unit(l, 2, h), own.summ[l][2, h], int(own.n_tok[l, 2]), BS, D, k[2, h], v[2, h])
            oracle.append(raw.host_unit(l, 2, h), raw.summ[l][2, h], int(raw.n_tok[l, 2]), BS, D, k[2, h], v[2, h])
        own.n_tok[l, 2] += 1
        raw.n_tok[l, 2] += 1
        assert np.array_equal(own.host_unit(l, 2, 0), bufs[2][l, 0])
        assert np.array_equal(own.summ[l], raw.summ[l])
    # the sources handed to host_fill were never written
    assert all(np.array_equal(a, b) for a, b in zip(src, frozen))
