"""CPU check of the tensor-core attention kernel's shared-memory access pattern.

The kernel (k_attend.cu) copies one 8 KiB slot per TMA load into a 1024-byte aligned stage:
rows 0..15 hold K of the block's 16 tokens, rows 16..31 V, 256 bytes per row, under the
128-byte swizzle (the 16-byte chunk index within each 128-byte line is XORed with the line
index mod 8). This restates the kernel's lane -> (row, chunk) mapping and checks that every
token and every dim is covered exactly as the MMA fragments need, and that no 16-byte load
phase (8 lanes) hits a shared-memory bank group twice.
"""


def token_of_row(r):
    lo = r & 7
    t = 4 + (((lo >> 1) + 1) & 3) if lo & 1 else lo >> 1
    return (r & 8) + t


def swz(row, hf, c8):
    return row * 256 + hf * 128 + ((c8 ^ ((2 * row + hf) & 7)) << 4)


def worst_conflict(addrs):
    worst = 1
    for p in range(4):  # a 16-byte load is served 8 lanes at a time
        groups = {}
        for lane in range(8 * p, 8 * p + 8):
            groups.setdefault((addrs[lane] >> 4) & 7, set()).add(addrs[lane])
        worst = max(worst, max(len(v) for v in groups.values()))
    return worst


def k_chunk(ti, s):
    return (ti & 1) + 4 * (ti >> 1) + 2 * s


def test_rows_are_a_permutation_of_the_tokens():
    assert sorted(token_of_row(r) for r in range(16)) == list(range(16))


def test_qk_reads_cover_all_dims_and_are_conflict_free():
    dims = set()
    for ti in range(4):
        for hf in range(2):
            for s in range(2):
                dims.update(64 * hf + 8 * k_chunk(ti, s) + e for e in range(8))
    assert dims == set(range(128))
    for hf in range(2):
        for s in range(2):
            for second in (0, 8):
                addrs = [swz(token_of_row(lane >> 2) + second, hf, k_chunk(lane & 3, s)) for lane in range(32)]
                assert worst_conflict(addrs) == 1


def test_pv_reads_cover_all_tokens_and_are_conflict_free():
    toks = []
    for ti in range(4):
        toks += [token_of_row(2 * ti), token_of_row(2 * ti + 1), 8 + token_of_row(2 * ti), 8 + token_of_row(2 * ti + 1)]
    assert sorted(toks) == list(range(16))
    for om in range(2):
        for j in range(4):
            addrs = []
            for lane in range(32):
                gi, ti = lane >> 2, lane & 3
                tau = [token_of_row(2 * ti), token_of_row(2 * ti + 1), 8 + token_of_row(2 * ti),
                       8 + token_of_row(2 * ti + 1)][j]
                addrs.append(swz(16 + tau, om, gi))
            assert worst_conflict(addrs) == 1
