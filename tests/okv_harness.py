"""Test rig: one okv context (CUDA library) and the CPU oracle over the same seeded host KV.

Comparison rules (the method's tolerances):
* block summaries, slot tables, stamps, fetch lists, pool bytes, lengths: exact;
* selections: exact, except swaps between blocks whose oracle scores lie within
  1e-6 * |s_K| of the K-th score s_K (binary32 scores summed in different orders may
  order such near-ties differently); after an accepted selection the oracle's KV
  selection step is re-synced to the GPU's selection so later state compares exactly;
* attention: max abs error <= 1e-5 (binary32 storage) or 2e-2 (bfloat16 storage);
* decode-side tiers of partially staged requests (routes, entries in use, kept entry of each
  block): exact; kept copies equal their blocks of the full copy byte for byte.

The oracle keeps its own copy of the host KV (filled from the seeded generator, appended to by
the oracle itself), so pools, kept copies and attention are compared against bytes the CUDA
library never wrote. The library's own host writes (appends) are checked directly: after every
append the token at the appended position must equal the generator's token, and nothing else
in the blocks around it may have changed.

Selections with exact ties (the oracle's binary32 score of several blocks equal to the K-th
score bit for bit, e.g. a zero draft query or byte-identical blocks) must follow the lowest-id
rule exactly; `check_selection(exact=True)` allows no swap at all.
"""
from __future__ import annotations

import numpy as np

import oracle
import synth
from sparse_kv_cache_draft_gb300 import BF16, F32, Config, Context, HostBuffer

TIE_REL = 1e-6
ATOL = {F32: 1e-5, BF16: 2e-2}


def torch_dtype(dtype):
    import torch
    return torch.float32 if dtype == F32 else torch.bfloat16


def to_device(a: np.ndarray, dtype):
    import torch
    a = np.ascontiguousarray(a)
    t = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16) if dtype == BF16 else torch.from_numpy(a)
    return t.cuda()


def out_to_f64(t, dtype) -> np.ndarray:
    import torch
    if dtype == BF16:
        return t.float().cpu().numpy().astype(np.float64)
    return t.cpu().numpy().astype(np.float64)


class Rig:
    def __init__(self, w: synth.Workload, *, contexts=None, capacity_tokens=None, n_alias=None,
                 max_requests=None, active=None, layers_kept=None, n_threads=None, local_cap=None,
                 edit_kv=None):
        """edit_kv(layer, key, unit_array): an optional change to the generated input KV of one
        layer of one content key (array [Hkv][cap_blocks][2][bs][d] of the storage type), applied
        alike to the library's host buffers and to the oracle's copy (e.g. byte-identical blocks
        for exact-tie cases)."""
        self.w = w
        B = w.batch
        self.contexts = np.asarray(contexts if contexts is not None else w.contexts(), np.int32)
        assert len(self.contexts) == B
        cap_tok = capacity_tokens if capacity_tokens is not None else int(self.contexts.max()) + w.grow_per_step * w.steps
        self.cap_blocks = -(-cap_tok // w.block_size)
        self.R = max_requests or B
        self.active = list(active) if active is not None else list(range(B))  # request ids used
        assert len(self.active) == B and max(self.active) < self.R
        self.n_alias = n_alias or B
        self.keys = np.array([i % self.n_alias for i in range(B)], np.int32)
        self.ids = np.array(self.active, np.int32)
        nb_plant = -(-w.context // w.block_size)
        self.plant_blocks = nb_plant
        self.cfg = Config(layers=w.layers, q_heads=w.q_heads, kv_heads=w.kv_heads, head_dim=w.head_dim,
                          block_size=w.block_size, budget_tokens=w.budget_tokens, max_requests=self.R,
                          max_blocks_per_request=self.cap_blocks, fetch_cap=w.fetch_cap, dtype=w.dtype)
        self.kb = self.cfg.slots
        # host KV: one buffer per content key
        self.bufs = {}
        for i in range(B):
            k = int(self.keys[i])
            if k not in self.bufs:
                hb = HostBuffer(self.cfg.host_bytes(self.cap_blocks))
                n_fill = int(max(self.contexts[j] for j in range(B) if self.keys[j] == k))
                synth.fill_kv(hb.ptr, w, k, 0, n_fill, self.cap_blocks, n_threads=n_threads,
                              plant_blocks=nb_plant)
                if edit_kv is not None:
                    view = self._host_view(hb)
                    for l in range(w.layers):
                        edit_kv(l, k, view[l])
                self.bufs[k] = hb
        self.ctx = Context(self.cfg)
        # local_cap[i] >= 0: batch request i is partially staged with that many decode-side
        # entries per unit (a buffer of its own); -1: it holds its full KV
        self.local_cap = np.full(B, -1, np.int32) if local_cap is None else \
            np.array(np.broadcast_to(np.asarray(local_cap, np.int32), (B,)))
        self.local_bufs = {}
        for i in range(B):
            full = self.bufs[int(self.keys[i])].ptr
            if self.local_cap[i] < 0:
                self.ctx.add_request(int(self.ids[i]), full, self.cap_blocks, int(self.contexts[i]))
                continue
            lb = None
            if self.local_cap[i] > 0:
                lb = HostBuffer(self.cfg.host_bytes(int(self.local_cap[i])))
                self.local_bufs[i] = lb
            self.ctx.add_request_partial(int(self.ids[i]), full, self.cap_blocks, lb.ptr if lb else 0,
                                         int(self.local_cap[i]), int(self.contexts[i]))
        # the oracle sees request slot i of the batch (rows of the device arrays = request ids); its
        # host KV is a copy of its own, generated again from the same seeds
        n_fill_of = {int(k): int(max(self.contexts[j] for j in range(B) if self.keys[j] == k)) for k in self.keys}

        def host_fill(layer, key, arr):
            synth.fill_kv_layer(arr, w, key, layer, 0, n_fill_of[key], n_threads=n_threads,
                                plant_blocks=nb_plant)
            if edit_kv is not None:
                edit_kv(layer, key, arr)

        self.model = oracle.OracleModel(
            layers=w.layers, q_heads=w.q_heads, kv_heads=w.kv_heads, head_dim=w.head_dim,
            block_size=w.block_size, budget_tokens=w.budget_tokens, dtype=w.dtype,
            host_fill=host_fill, req_keys=self.keys,
            cap_blocks=[self.cap_blocks] * B, n_tok=self.contexts, n_threads=n_threads,
            layers_kept=layers_kept, local_cap=self.local_cap)
        self.sdt = np.float32 if w.dtype == F32 else np.uint16
        # the oracle's routes of partially staged requests, summed over every staging checked
        self.tally = {"local_hits": 0, "local_fills": 0, "full_reads": 0}
        self._summarised = set()  # (layer, batch index) whose oracle summaries are built

    def _host_view(self, hb) -> np.ndarray:
        """The library's host KV buffer as [L][Hkv][cap_blocks][2][bs][d] storage (no copy)."""
        w = self.w
        sdt = np.float32 if w.dtype == F32 else np.uint16
        return hb.numpy(sdt, (w.layers, w.kv_heads, self.cap_blocks, 2, w.block_size, w.head_dim))

    def _ensure_summaries(self, layer: int, requests=None) -> None:
        reqs = range(self.w.batch) if requests is None else requests
        todo = [i for i in reqs if (layer, i) not in self._summarised]
        if todo:
            self.model.build_summaries(layer, requests=todo)
            self._summarised.update((layer, i) for i in todo)

    # ---- inputs --------------------------------------------------------------------------------
    def batch_queries(self, layer: int, step: int, kind: int) -> np.ndarray:
        """[B][Hq][d] storage for the batch (row i = request ids[i])."""
        return synth.queries(self.w, layer, step, kind, self.ids, self.keys, plant_blocks=self.plant_blocks)

    def scatter(self, a: np.ndarray, rows_shape) -> np.ndarray:
        """Place batch rows at their request ids in a [R]... array (other rows zero)."""
        full = np.zeros((self.R,) + rows_shape, dtype=a.dtype)
        full[self.ids] = a
        return full

    def device_rows(self, a: np.ndarray, rows_shape):
        return to_device(self.scatter(a, rows_shape), self.w.dtype)

    # ---- comparisons ---------------------------------------------------------------------------
    def check_summaries(self, layer: int, requests=None) -> None:
        reqs = range(self.w.batch) if requests is None else requests
        self._ensure_summaries(layer, reqs)
        for i in reqs:
            gpu = self.ctx.read_summaries(layer, int(self.ids[i]))
            nb = -(-int(self.model.n_tok[layer, i]) // self.w.block_size)
            want = self.model.summ[layer][i][:, :nb]
            assert np.array_equal(gpu[:, :nb], want), f"summaries differ: layer {layer} request {i}"

    def check_selection(self, layer: int, requests=None, exact: bool = False):
        """Compare the GPU selection with the oracle's (band rule; with `exact`, no swap at all:
        for inputs whose scores tie exactly on both sides by construction, the selection must be
        the oracle's, ids and order); return the GPU selection as (ids [B][Hkv][kb],
        counts [B][Hkv]) in batch order, for re-syncing the oracle."""
        counts, ids, scores = self.ctx.read_selection(layer)
        reqs = range(self.w.batch) if requests is None else requests
        B, H, kb = self.w.batch, self.w.kv_heads, self.kb
        g_ids = np.full((B, H, kb), -1, np.int32)
        g_cnt = np.zeros((B, H), np.int32)
        n_swaps = 0
        for i in reqs:
            r = int(self.ids[i])
            nb = -(-int(self.model.n_tok[layer, i]) // self.w.block_size)
            for h in range(H):
                n = min(kb, nb)
                assert counts[r, h] == n, (layer, i, h, counts[r, h], n)
                gsel = ids[r, h, :n]
                osel = self.model.sel_ids[layer][i, h, :n]
                osc = self.model.scores[layer][i, h, :nb]
                g_cnt[i, h] = n
                if n == 0:  # an empty context selects nothing
                    continue
                assert len(set(gsel.tolist())) == n and gsel.min() >= 0 and gsel.max() < nb
                # GPU order: its own scores non-increasing, ties by block id
                gs = scores[r, h, :n]
                assert np.all((gs[:-1] > gs[1:]) | ((gs[:-1] == gs[1:]) & (gsel[:-1] < gsel[1:]))), (layer, i, h)
                # GPU scores agree with the oracle's within binary32 summation error
                assert np.allclose(gs, osc[gsel], rtol=2e-6, atol=1e-6 * max(1.0, float(np.abs(osc).max()))), \
                    (layer, i, h, float(np.abs(gs - osc[gsel]).max()))
                if exact:
                    assert np.array_equal(gsel, osel), \
                        f"selection differs (exact ties): layer {layer} req {i} head {h}: {gsel[:8]}... vs {osel[:8]}..."
                if not np.array_equal(np.sort(gsel), np.sort(osel)):
                    sK = float(osc[osel[-1]])
                    band = set(np.nonzero(np.abs(osc.astype(np.float64) - sK) <= TIE_REL * abs(sK))[0].tolist())
                    diff = set(gsel.tolist()) ^ set(osel.tolist())
                    assert diff <= band, f"selection differs outside the tie band: layer {layer} req {i} head {h}: {sorted(diff - band)}"
                    n_swaps += 1
                g_ids[i, h, :n] = gsel
                g_cnt[i, h] = n
        return (g_ids, g_cnt), n_swaps

    def check_tables(self, layer: int, requests=None) -> None:
        sb, st = self.ctx.read_slot_table(layer)
        counts, entries = self.ctx.read_fetch_list(layer)
        reqs = range(self.w.batch) if requests is None else requests
        for i in reqs:
            r = int(self.ids[i])
            assert np.array_equal(sb[r], self.model.slot_block[layer][i]), f"slot table: layer {layer} req {i}"
            occ = sb[r] >= 0
            assert np.array_equal(st[r][occ], self.model.stamp[layer][i][occ]), f"stamps: layer {layer} req {i}"
            assert np.array_equal(counts[r], self.model.n_fetch[layer][i]), f"fetch counts: layer {layer} req {i}"
            for h in range(self.w.kv_heads):
                n = int(counts[r, h])
                assert np.array_equal(entries[r, h, :n], self.model.fetch[layer][i, h, :n]), \
                    f"fetch list: layer {layer} req {i} head {h}"

    def check_local(self, layer: int, requests=None) -> None:
        """Decode-side tiers: routes, entries in use and kept entries exactly as the oracle's;
        every kept copy equal to its block of the full copy over the block's valid tokens."""
        used, local_of, routes = self.ctx.read_local(layer)
        counts, _ = self.ctx.read_fetch_list(layer)
        reqs = range(self.w.batch) if requests is None else requests
        bs, nbm = self.w.block_size, self.cap_blocks
        for i in reqs:
            r = int(self.ids[i])
            for h in range(self.w.kv_heads):
                n = int(counts[r, h])
                assert np.array_equal(routes[r, h, :n], self.model.route[layer][i, h, :n]), \
                    f"routes: layer {layer} req {i} head {h}: {routes[r, h, :n]} vs {self.model.route[layer][i, h, :n]}"
            if self.local_cap[i] < 0:
                continue
            assert np.array_equal(used[r], self.model.local_used[layer][i]), f"entries in use: layer {layer} req {i}"
            assert np.array_equal(local_of[r][:, :nbm], self.model.local_of[layer][i][:, :nbm]), \
                f"kept entries: layer {layer} req {i}"
            if self.local_cap[i] == 0:
                continue
            lc = int(self.local_cap[i])
            kept = self.local_bufs[i].numpy(self.sdt, (self.w.layers, self.w.kv_heads, lc, 2, bs, self.w.head_dim))
            n_tok = int(self.model.n_tok[layer, i])
            for h in range(self.w.kv_heads):
                full = self.model.host_unit(layer, i, h)
                for b in np.nonzero(local_of[r, h, :nbm] >= 0)[0]:
                    e = int(local_of[r, h, b])
                    nv = min(bs, n_tok - int(b) * bs)
                    assert np.array_equal(kept[layer, h, e, :, :nv], full[b, :, :nv]), \
                        f"kept copy differs: layer {layer} req {i} head {h} block {b} entry {e}"

    def _tally_routes(self, layer: int, requests=None) -> None:
        for i in (range(self.w.batch) if requests is None else requests):
            if self.local_cap[i] < 0:
                continue
            for h in range(self.w.kv_heads):
                rt = self.model.route[layer][i, h, :int(self.model.n_fetch[layer][i, h])]
                hits = int(((rt >= 0) & ((rt & 1) == 0)).sum())
                fills = int(((rt >= 0) & ((rt & 1) == 1)).sum())
                self.tally["local_hits"] += hits
                self.tally["local_fills"] += fills
                self.tally["full_reads"] += len(rt) - hits

    def check_pool(self, layer: int, requests=None, heads=None) -> None:
        sb, _ = self.ctx.read_slot_table(layer)
        reqs = range(self.w.batch) if requests is None else requests
        bs = self.w.block_size
        for i in reqs:
            r = int(self.ids[i])
            n_tok = int(self.model.n_tok[layer, i])
            for h in (range(self.w.kv_heads) if heads is None else heads):
                pool = self.ctx.read_pool(layer, r, h)
                host = self.model.host_unit(layer, i, h)
                for s in range(self.kb):
                    b = int(sb[r, h, s])
                    if b < 0:
                        continue
                    nv = min(bs, n_tok - b * bs)
                    assert np.array_equal(pool[s, :, :nv], host[b, :, :nv]), \
                        f"pool slot differs from host block: layer {layer} req {i} head {h} slot {s} block {b}"

    def check_attention(self, layer: int, q: np.ndarray, out_dev, requests=None) -> float:
        """q: [B][Hq][d] storage (batch order); out_dev: device [R][Hq][d]."""
        got = out_to_f64(out_dev, self.w.dtype)[self.ids]
        want = self.model.attend(layer, q, requests=requests)
        reqs = list(range(self.w.batch)) if requests is None else list(requests)
        err = float(np.abs(got[reqs] - want[reqs]).max()) if reqs else 0.0
        assert err <= ATOL[self.w.dtype], f"attention max abs error {err} at layer {layer}"
        return err

    # ---- one staging + attention round ---------------------------------------------------------
    def stage(self, layer: int, step: int, cap: float, draft_step: int | None = None, requests=None,
              check_pool=True, draft=None, exact=False):
        """Stage `layer` from the draft of `draft_step` (or the given [B][Hq][d] `draft`) and check
        selections, tables, tiers and pools against the oracle."""
        import torch
        ds = step - 1 if draft_step is None else draft_step
        if draft is None:
            draft = self.batch_queries(layer, ds, 1)
        self.ctx.stage(layer, self.device_rows(draft, (self.w.q_heads, self.w.head_dim)), step, cap)
        torch.cuda.synchronize()
        assert self.ctx.sync(60_000) == 0
        self._ensure_summaries(layer, requests)
        self.model.score_topk(layer, draft, requests=requests)
        gsel, swaps = self.check_selection(layer, requests=requests, exact=exact)
        C = oracle.fetch_cap_blocks(cap, self.kb)
        self.model.select(layer, C, step, sel_override=gsel, requests=requests)
        self.check_tables(layer, requests=requests)
        self.check_local(layer, requests=requests)
        self._tally_routes(layer, requests)
        if check_pool:
            self.check_pool(layer, requests=requests)
        return swaps

    def attend(self, layer: int, step: int, requests=None) -> float:
        import torch
        q = self.batch_queries(layer, step, 0)
        out = torch.zeros((self.R, self.w.q_heads, self.w.head_dim), dtype=torch_dtype(self.w.dtype),
                          device="cuda")
        self.ctx.attend(layer, self.device_rows(q, (self.w.q_heads, self.w.head_dim)), out)
        torch.cuda.synchronize()
        return self.check_attention(layer, q, out, requests=requests)

    def run_steps(self, n_steps: int, cap: float, bootstrap_cap: float = 1.0, layers=None,
                  requests=None, check_pool=True, append=False):
        """Bootstrap staging (draft of step -1, stamp 0), then n_steps decode steps: for each
        layer, [append the step's token,] attend(q_t), stage(draft_t) with stamp t + 1."""
        import torch
        layers = range(self.w.layers) if layers is None else layers
        errs, swaps = [], 0
        for layer in layers:
            swaps += self.stage(layer, 0, bootstrap_cap, draft_step=-1, requests=requests, check_pool=check_pool)
        for t in range(n_steps):
            for layer in layers:
                if append:
                    self.append(layer)
                errs.append(self.attend(layer, t, requests=requests))
                swaps += self.stage(layer, t + 1, cap, draft_step=t, requests=requests, check_pool=check_pool)
        return errs, swaps

    def append(self, layer: int) -> None:
        """Append each request's next token (the generator's token at its position); check the
        library's write into its host buffers, then append to the oracle's own copy."""
        import torch
        pos = self.model.n_tok[layer].copy()
        self._ensure_summaries(layer)
        k, v = synth.token_kv(self.w, layer, self.keys, pos, plant_blocks=self.plant_blocks)
        shp = (self.w.kv_heads, self.w.head_dim)
        snap = self.host_snapshot([layer])
        self.ctx.append(layer, self.device_rows(k, shp), self.device_rows(v, shp))
        torch.cuda.synchronize()
        assert self.ctx.sync(60_000) == 0
        self.check_host_append(snap, {layer: (k, v)})
        self.model.append(layer, k, v)
        self.check_host_tail(layer)

    # ---- the library's host writes (appends) -----------------------------------------------------
    def host_snapshot(self, layers, requests=None, positions=None):
        """Copies of the blocks around each request's next token position in the library's host
        buffers: the blocks of positions pos - 1, pos and pos + 1 (within capacity). positions[l]
        gives [B] positions per layer (default: the oracle's current lengths)."""
        reqs = range(self.w.batch) if requests is None else requests
        bs = self.w.block_size
        snap = {}
        for l in layers:
            for i in reqs:
                pos = int(self.model.n_tok[l, i] if positions is None else positions[l][i])
                view = self._host_view(self.bufs[int(self.keys[i])])[l]
                b0 = max(0, (pos - 1) // bs)
                b1 = min(self.cap_blocks - 1, (pos + 1) // bs)
                snap[l, i] = (pos, b0, view[:, b0:b1 + 1].copy())
        return snap

    def check_host_tail(self, layer: int, requests=None) -> None:
        """The valid tokens of each request's tail block in the library's host buffer equal the
        oracle's own copy."""
        bs = self.w.block_size
        for i in (range(self.w.batch) if requests is None else requests):
            n = int(self.model.n_tok[layer, i])
            if n == 0:
                continue
            b, nv = (n - 1) // bs, (n - 1) % bs + 1
            got = self._host_view(self.bufs[int(self.keys[i])])[layer][:, b, :, :nv]
            want = np.stack([self.model.host_unit(layer, i, h)[b, :, :nv] for h in range(self.w.kv_heads)])
            assert np.array_equal(got, want), f"host tail block differs from the oracle's copy: layer {layer} req {i}"

    def check_host_append(self, snap, kv) -> None:
        """After an append: in every snapshotted window the token at the appended position holds
        the generator's K and V (kv[layer] = (k [B][Hkv][d], v)) and every other byte is unchanged."""
        bs = self.w.block_size
        for (l, i), (pos, b0, before) in snap.items():
            k, v = kv[l]
            want = before.copy()
            want[:, pos // bs - b0, 0, pos % bs] = k[i]
            want[:, pos // bs - b0, 1, pos % bs] = v[i]
            got = self._host_view(self.bufs[int(self.keys[i])])[l][:, b0:b0 + before.shape[1]]
            if not np.array_equal(got, want):
                bad = np.argwhere(got != want)[0]
                raise AssertionError(f"host write of the append differs: layer {l} req {i} position {pos}: "
                                     f"first difference at [head, block - {b0}, k/v, token, dim] = {bad.tolist()}")

    def close(self):
        self.ctx.close()
        for b in self.bufs.values():
            b.free()
        for b in self.local_bufs.values():
            b.free()
