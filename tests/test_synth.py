"""The seeded workload generator: distributions and internal consistency (CPU)."""
import numpy as np

import synth


def test_normals_are_standard():
    z = synth.normals(1_000_000, seed=7)
    assert abs(z.mean()) < 0.005 and abs(z.std() - 1.0) < 0.005
    assert abs((np.abs(z) < 1.0).mean() - 0.6827) < 0.003  # one-sigma mass of N(0,1)


def test_tiny_plants_five_percent_of_blocks():
    w = synth.WORKLOADS["tiny"]
    nb = w.context // w.block_size
    for r in range(w.batch):
        for h in range(w.kv_heads):
            planted = [b for b in range(nb) if synth.block_direction(w, 0, r, h, b) >= 0]
            assert len(planted) == 13  # 5% of 256


def test_directions_are_unit_vectors():
    w = synth.WORKLOADS["qwen3_8b_16k_b128"]
    for j in range(3):
        u = synth.direction(w, 1, 2, 3, j)
        assert abs(np.linalg.norm(u) - 1.0) < 1e-12


def _fill(w, req_key, n_tok):
    cap = -(-n_tok // w.block_size)
    buf = np.zeros((w.layers, w.kv_heads, cap, 2, w.block_size, w.head_dim), dtype=synth.np_dtype(w.dtype))
    synth.fill_kv(buf.ctypes.data, w, req_key, 0, n_tok, cap, n_threads=4)
    return buf


def test_token_kv_matches_fill():
    w = synth.WORKLOADS["qwen3_8b_mixed_b64"].scaled(layers=2, batch=3)
    buf = _fill(w, 5, 200)
    pos = np.array([0, 37, 199], np.int32)
    for layer in range(2):
        k, v = synth.token_kv(w, layer, [5, 5, 5], pos)
        for i, p in enumerate(pos):
            b, t = divmod(int(p), w.block_size)
            assert np.array_equal(buf[layer, :, b, 0, t], k[i])
            assert np.array_equal(buf[layer, :, b, 1, t], v[i])


def test_one_layer_fill_matches_the_whole_fill():
    w = synth.WORKLOADS["qwen3_8b_mixed_b64"].scaled(layers=3, batch=2)
    buf = _fill(w, 4, 77)
    for layer in range(3):
        one = np.zeros(buf.shape[1:], dtype=buf.dtype)
        synth.fill_kv_layer(one, w, 4, layer, 0, 77, n_threads=3)
        assert np.array_equal(one, buf[layer])


def test_planted_blocks_carry_the_direction():
    w = synth.WORKLOADS["qwen3_8b_16k_b128"].scaled(layers=1, dtype=synth.F32)
    buf = _fill(w, 0, 16 * 40)
    u = synth.direction(w, 0, 0, 0, 3)
    k = buf[0, 0, :, 0].astype(np.float64)  # [blocks][bs][d]
    proj = (k @ u).mean(axis=1)
    planted = [b for b in range(40) if b % w.n_dirs == 3]
    other = [b for b in range(40) if b % w.n_dirs != 3]
    assert proj[planted].mean() > 2.0 and abs(proj[other].mean()) < 1.0


def test_draft_is_next_query_plus_small_noise():
    w = synth.WORKLOADS["qwen3_8b_16k_b128"].scaled(dtype=synth.F32)
    ids = np.arange(16, dtype=np.int32)
    q1 = synth.queries(w, 3, 5, 0, ids, ids % 4)
    d0 = synth.queries(w, 3, 4, 1, ids, ids % 4)
    diff = d0.astype(np.float64) - q1.astype(np.float64)
    assert abs(diff.std() - w.sigma_d) < 0.01
    u = np.stack([synth.direction(w, 3, int(k), 0, 5 % w.n_dirs) for k in ids % 4])
    noise = q1[:, 0].astype(np.float64) - u
    assert abs(noise.std() - w.sigma_q) < 0.02


def test_bf16_is_rounded_f32():
    w32 = synth.WORKLOADS["qwen3_8b_16k_b128"].scaled(layers=1, dtype=synth.F32)
    w16 = w32.scaled(dtype=synth.BF16)
    a = _fill(w32, 2, 64)
    b = _fill(w16, 2, 64)
    u = a.view(np.uint32).astype(np.uint64)
    want = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    assert np.array_equal(b, want)
