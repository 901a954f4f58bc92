"""Pins for the oracle's shard maps, causal visibility and tile classes."""
import json
import os

import pytest

from oracle import ring as OR
from oracle import shardmap as OS

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_contiguous_map_by_hand():
    own, loc, tok = OS.shard_map("contiguous", 8, 4)
    assert own == [0, 0, 1, 1, 2, 2, 3, 3]
    assert loc == [0, 1, 0, 1, 0, 1, 0, 1]
    assert tok == [0, 1, 2, 3, 4, 5, 6, 7]


def test_striped_map_by_hand():
    own, loc, tok = OS.shard_map("striped", 8, 4)
    assert own == [0, 1, 2, 3, 0, 1, 2, 3]
    assert loc == [0, 0, 0, 0, 1, 1, 1, 1]
    assert tok == [0, 4, 1, 5, 2, 6, 3, 7]


@pytest.mark.parametrize("layout", ["contiguous", "striped"])
@pytest.mark.parametrize("N,P", [(12, 1), (12, 3), (64, 8), (60, 5)])
def test_maps_are_inverse_bijections(layout, N, P):
    own, loc, tok = OS.shard_map(layout, N, P)
    S = N // P
    assert sorted(tok) == list(range(N))
    for t in range(N):
        assert tok[own[t] * S + loc[t]] == t
        assert 0 <= own[t] < P and 0 <= loc[t] < S


def test_p1_is_identity():
    for layout in ("contiguous", "striped"):
        own, loc, tok = OS.shard_map(layout, 10, 1)
        assert own == [0] * 10 and loc == list(range(10)) and tok == list(range(10))


def test_bad_sizes_rejected():
    with pytest.raises(ValueError):
        OS.shard_map("contiguous", 10, 3)
    with pytest.raises(ValueError):
        OS.shard_map("spiral", 8, 2)


def test_causal_block_count_matches_printed():
    g = json.load(open(os.path.join(GOLDEN, "block_counts.json")))
    P = g["devices"]
    N = 8 * P
    per_dev = []
    for u in range(P):
        per_dev.append(sum(
            any(OS.visible("contiguous", N, P, True, u, i, b, j)
                for i in range(N // P) for j in range(N // P)) for b in range(P)))
    assert per_dev == g["blocks_needed_per_device"]
    assert OS.nonempty_shard_pairs("contiguous", N, P, True) == g["total_blocks"]
    assert OS.nonempty_shard_pairs("contiguous", N, P, False) == g["all_blocks"]


def test_contiguous_pair_classes_closed_form():
    # b < u: every key earlier -> FULL; b > u: every key later -> EMPTY;
    # b = u: lower triangle with the diagonal.
    N, P, T = 32, 4, 4
    S = N // P
    for u in range(P):
        for b in range(P):
            cls = OS.tile_classes("contiguous", N, P, True, u, b, T, T)
            for qi, row in enumerate(cls):
                for kj, c in enumerate(row):
                    if b < u:
                        assert c == OS.TILE_FULL
                    elif b > u:
                        assert c == OS.TILE_EMPTY
                    else:
                        want = (OS.TILE_FULL if kj < qi else
                                OS.TILE_PARTIAL if kj == qi else OS.TILE_EMPTY)
                        assert c == want
    assert len(cls) == S // T


def test_striped_mask_closed_form():
    # Striped: key j of shard b is visible to query i of shard u iff
    # j*P + b <= i*P + u, i.e. j <= i when b <= u and j <= i - 1 when b > u.
    N, P = 24, 4
    S = N // P
    for u in range(P):
        for b in range(P):
            m = OS.mask_block("striped", N, P, True, u, b)
            for i in range(S):
                for j in range(S):
                    assert m[i][j] == (j <= i - (1 if b > u else 0))


def test_ragged_tile_classes_count_only_in_range():
    # S = 10 with 4x4 tiles: the last tile row / column is 2 wide.
    N, P = 20, 2
    cls = OS.tile_classes("contiguous", N, P, True, 1, 1, 4, 4)
    assert len(cls) == 3 and len(cls[0]) == 3
    assert cls[2][2] == OS.TILE_PARTIAL     # rows 8,9 x keys 8,9: (8,9) masked
    assert cls[2][0] == OS.TILE_FULL
    cls = OS.tile_classes("contiguous", N, P, False, 0, 1, 4, 4)
    assert all(c == OS.TILE_FULL for row in cls for c in row)


def test_noncausal_everything_visible():
    for layout in ("contiguous", "striped"):
        for u in range(3):
            for b in range(3):
                m = OS.mask_block(layout, 9, 3, False, u, b)
                assert all(all(r) for r in m)


def test_ring_visit_order_matches_printed_schedule():
    g = json.load(open(os.path.join(GOLDEN, "ring_schedule.json")))
    P = g["devices"]
    for step, key in ((0, "step0_block"), (1, "step1_block")):
        for u, b in g[key].items():
            assert OR.ring_order(int(u), P)[step] == b
    for u in range(P):
        assert sorted(OR.ring_order(u, P)) == list(range(P))


# --------------------------------------------------------------------------- zigzag

def test_zigzag_map_by_hand():
    # N = 8, P = 2: chunks of 2 tokens; shard 0 = chunks 0 and 3, shard 1 = chunks 1 and 2
    own, loc, tok = OS.shard_map("zigzag", 8, 2)
    assert tok == [0, 1, 6, 7, 2, 3, 4, 5]
    assert own == [0, 0, 1, 1, 1, 1, 0, 0]
    assert loc == [0, 1, 0, 1, 2, 3, 2, 3]


@pytest.mark.parametrize("N,P", [(16, 4), (48, 3), (256, 8), (10, 5)])
def test_zigzag_maps_are_inverse_bijections(N, P):
    own, loc, tok = OS.shard_map("zigzag", N, P)
    S = N // P
    assert sorted(tok) == list(range(N))
    for t in range(N):
        assert tok[own[t] * S + loc[t]] == t


def test_zigzag_needs_2p_chunks():
    with pytest.raises(ValueError):
        OS.shard_map("zigzag", 12, 4)       # 12 % 8 != 0


def test_zigzag_assignment_matches_printed():
    g = json.load(open(os.path.join(GOLDEN, "zigzag.json")))
    P = g["devices"]
    C = 3
    N = 2 * P * C
    for u, blocks in g["blocks_of_device"].items():
        toks = OS.shard_tokens("zigzag", N, P, int(u))
        assert sorted({t // C for t in toks}) == sorted(blocks)
        assert [t // C for t in toks] == [blocks[0]] * C + [blocks[1]] * C


def test_zigzag_balances_causal_block_work_as_printed():
    g = json.load(open(os.path.join(GOLDEN, "zigzag.json")))
    P = g["devices"]
    C = 2
    N = 2 * P * C
    # units: (query chunk of the device, key chunk) pairs with any visible element
    for u in range(P):
        toks = OS.shard_tokens("zigzag", N, P, u)
        qchunks = sorted({t // C for t in toks})
        units = sum(1 for qc in qchunks for kc in range(2 * P)
                    if any(kc * C + j <= qc * C + i for i in range(C) for j in range(C)))
        assert units == g["small_block_units_per_device"]
    # the printed speedups: contiguous bottleneck P big blocks vs (2P+1)/4 equivalents
    for n, want in g["speedup"].items():
        n = int(n)
        assert round(n / ((2 * n + 1) / 4), 2) == want


@pytest.mark.parametrize("causal", [False, True])
def test_ring_equals_dense_zigzag(causal):
    import numpy as np
    from oracle import attention as OA
    rng = np.random.default_rng(21)
    q = rng.standard_normal((1, 48, 4, 8))
    k = rng.standard_normal((1, 48, 2, 8))
    v = rng.standard_normal((1, 48, 2, 8))
    O, L = OA.dense_attention(q, k, v, causal=causal)
    for P in (1, 2, 3, 4, 6):
        Or_, Lr = OR.ring_attention(q, k, v, P, "zigzag", causal)
        assert np.abs(Or_ - O).max() < 1e-12 and np.abs(Lr - L).max() < 1e-12
