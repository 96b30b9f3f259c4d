"""CPU model of the tensor-core path's candidate selection (no GPU, no library).

The lm_head epilogue keeps, per (row, column tile), the tile's top 8 by (value desc, column asc);
the merge takes a lower bound x of the row's K-th largest element from the tile maxima (every
tile maximum is a distinct element, so K of them at or above x mean K elements at or above x),
keeps every list entry >= x, and rescans the whole tile of any list whose 8th entry is still
>= x.  The argument: a tile whose 8th entry is below x has all of its elements >= x in its list;
any other tile is rescanned; so the candidates hold every element >= x, hence the top K.

This model replays that scheme in numpy for both tile widths the kernels use (192 columns while
hi and lo share a tile, 256 otherwise), with the exact bound and with a bound lowered to 16-bit
key resolution (the merge's warp bound is exact only to 16 bits), on random rows and on rows
built to defeat it (columns tied in groups of 16, a cluster of top values, a constant row), and checks the candidates
against the oracle's top-k ("GPT-OSS Tail Chunked Megakernel Kernel API Reference", section
"Background": a per-chunk top-k followed by one merge must give the global top-k).
"""
import numpy as np
import pytest

import oracle

LIST = 8


def _keys(v):
    """Order-preserving uint32 keys of fp32 values (negative values flipped, +0 == -0)."""
    b = np.ascontiguousarray(v, np.float32).view(np.uint32).astype(np.uint64)
    b = np.where(b == 0x80000000, 0, b)
    return np.where(b & 0x80000000, 0xFFFFFFFF - b, b | 0x80000000).astype(np.uint64)


def _candidates(row, K, tile, lower16):
    V = row.size
    key = _keys(row)
    ntn = -(-V // tile)
    lists = []
    for n in range(ntn):
        cols = np.arange(n * tile, min(V, (n + 1) * tile))
        order = cols[np.lexsort((cols, -key[cols].astype(np.int64)))][:LIST]
        lists.append(order)
    heads = np.array([key[l[0]] for l in lists])
    entries = np.concatenate(lists)
    if ntn >= K:
        x = int(np.sort(heads)[::-1][K - 1])
    elif entries.size >= K:
        x = int(np.sort(key[entries])[::-1][K - 1])
    else:
        x = 0
    if lower16:
        x &= 0xFFFF0000
    cand, rescans = [], 0
    for n, l in enumerate(lists):
        if l.size == LIST and key[l[-1]] >= x:
            rescans += 1
            cols = np.arange(n * tile, min(V, (n + 1) * tile))
            cand.extend(cols[key[cols] >= x])
        else:
            cand.extend(l[key[l] >= x])
    return np.array(sorted(set(int(c) for c in cand))), rescans


def _rows(kind, V, rng):
    if kind == "random":
        return rng.standard_normal((4, V)).astype(np.float32)
    if kind == "ties":  # columns repeated 16 times: every top tile saturates
        base = rng.standard_normal((4, V // 16)).astype(np.float32)
        return np.repeat(base, 16, axis=1)
    if kind == "cluster":  # the top values crowded into one tile
        r = rng.standard_normal((4, V)).astype(np.float32)
        r[:, 1000:1300] += 50.0
        return r
    if kind == "constant":  # every element equal: the whole row ties
        return np.full((2, V), 0.5, np.float32)
    raise ValueError(kind)


@pytest.mark.parametrize("tile", [192, 256])
@pytest.mark.parametrize("kind", ["random", "ties", "cluster", "constant"])
@pytest.mark.parametrize("lower16", [False, True], ids=["exact_bound", "bound_16bit"])
def test_list_entries_and_rescans_hold_the_exact_top_k(tile, kind, lower16):
    rng = np.random.default_rng(11)
    V, K = 12_304, 256  # 12304 = 64 * 192 + 16: a ragged last tile at both widths
    rows = _rows(kind, V, rng)
    L = rows.astype(np.float64)
    _, want = oracle.topk(L, K)
    for r in range(rows.shape[0]):
        cand, rescans = _candidates(rows[r], K, tile, lower16)
        assert set(want[r].tolist()) <= set(cand.tolist())
        # the top K of the candidates by (value desc, index asc) is the oracle's, in order
        order = cand[np.lexsort((cand, -L[r, cand]))][:K]
        assert np.array_equal(order, want[r])
        if kind == "ties":
            assert rescans > 0


@pytest.mark.parametrize("tile", [192, 256])
def test_at_the_gpt_oss_vocabulary_random_rows_need_no_rescan(tile):
    # V = 201088: 1048 or 786 tiles, more than K, so the bound comes from the tile maxima; a random
    # row then keeps a few hundred candidates and rescans nothing
    rng = np.random.default_rng(13)
    V, K = 201_088, 256
    rows = (rng.standard_normal((2, V)) * 1.1).astype(np.float32)
    _, want = oracle.topk(rows.astype(np.float64), K)
    for r in range(2):
        cand, rescans = _candidates(rows[r], K, tile, True)
        assert rescans == 0 and K <= cand.size < 2 * K
        assert set(want[r].tolist()) <= set(cand.tolist())


def test_fewer_tiles_than_k_bound_from_all_entries():
    # 20 tiles of 256 columns with K = 64: the bound comes from the K-th largest list entry
    rng = np.random.default_rng(12)
    row = rng.standard_normal(20 * 256).astype(np.float32)
    _, want = oracle.topk(row[None, :].astype(np.float64), 64)
    cand, _ = _candidates(row, 64, 256, False)
    assert set(want[0].tolist()) <= set(cand.tolist())


def test_key_order_matches_value_order():
    v = np.array([-np.inf, -2.0, -0.0, 0.0, 1e-45, 1.0, np.inf], np.float32)
    k = _keys(v)
    assert np.all(np.diff(k.astype(np.int64)) >= 0) and k[2] == k[3]
