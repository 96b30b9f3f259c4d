"""CPU models of the two candidate selections that make the GPU top-k exact (no GPU, no library).

Tensor-core path (9 rows and more): the lm_head epilogue keeps, per (row, column tile), the tile's top 8 by (value desc, column asc);
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
"Background": a per-chunk top-k followed by one merge must give the global top-k).  The second
half models the mma.sync path's slab publications and row owners the same way.
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


# ------------------------------------------------------------------ the mma.sync path (up to 8 rows)
#
# Each CTA owns one vocabulary slab (whole 16-column pairs, split evenly over the slabs).  After
# the stream it sorts the 32 lane maxima of its slab (lane l holds columns l, l + 32, ... of the
# slab), keeps the 4 largest as leaders and b = the 8th largest, and publishes every element >= b
# when there are at most 32 of them (else nothing, with b raised to the largest key).  The row
# owner bounds the K-th largest element by the K-th largest leader (x, exact to 16 bits), keeps the
# published elements >= x, takes thr = the K-th largest of those (or x when fewer than K remain),
# and rescans every slab with b > thr.  The argument: a top-K element e of a slab that published
# is either >= b (published, and >= x) or below b, and then b > e >= v_K >= thr, so that slab is
# rescanned; a slab that published nothing has b above any thr and is rescanned too.

def _slab_candidates(row, K, nslab, lower16):
    V = row.size
    key = _keys(row)
    npairs = V // 16
    top = np.uint64(0xFFFFFFFF)
    pubs, bs, leaders, bounds = [], [], [], []
    for c in range(nslab):
        lo, hi = 16 * (npairs * c // nslab), 16 * (npairs * (c + 1) // nslab)
        seg = key[lo:hi]
        padded = np.zeros(-(-seg.size // 32) * 32, np.uint64)
        padded[: seg.size] = seg
        lane_max = np.sort(padded.reshape(-1, 32).max(axis=0))[::-1]
        leaders.extend(lane_max[:4])
        b = lane_max[7]
        sel = np.nonzero(seg >= b)[0] + lo
        if sel.size <= 32:
            pubs.append(sel)
            bs.append(b)
        else:
            pubs.append(np.zeros(0, np.int64))
            bs.append(top)
        bounds.append((lo, hi))
    leaders = np.array(leaders, np.uint64)
    x = int(np.sort(leaders)[::-1][K - 1]) if leaders.size >= K else 0
    if lower16:
        x &= 0xFFFF0000
    F = np.concatenate([p[key[p] >= x] for p in pubs])
    if F.size >= K:
        order = F[np.lexsort((F, -key[F].astype(np.int64)))]
        thr = int(key[order[K - 1]])
    else:
        thr = x
    cand, rescans = set(F.tolist()), 0
    for (lo, hi), b in zip(bounds, bs):
        if int(b) > thr:
            rescans += 1
            cand |= set((np.nonzero(key[lo:hi] >= thr)[0] + lo).tolist())
    return np.array(sorted(cand)), rescans


def _slab_rows(kind, V, rng):
    r = rng.standard_normal((2, V)).astype(np.float32)
    if kind == "clustered":  # every top element inside one slab: it publishes nothing
        r[:, 5000:5400] += 10.0
    elif kind == "tied64":  # columns repeated 64 times: no slab can publish
        r = np.repeat(r[:, : V // 64], 64, axis=1)
    elif kind == "constant":
        r = np.full((2, V), -1.25, np.float32)
    return r


@pytest.mark.parametrize("lower16", [False, True], ids=["exact_bound", "bound_16bit"])
@pytest.mark.parametrize("kind", ["random", "clustered", "tied64", "constant"])
def test_slab_publications_and_rescans_hold_the_exact_top_k(kind, lower16):
    # the GPT-OSS shape: V = 201088 over 152 slabs (82-83 pairs, ~1323 columns each), K = 256
    rng = np.random.default_rng(21)
    V, K, nslab = 201_088, 256, 152
    rows = _slab_rows(kind, V, rng)
    L = rows.astype(np.float64)
    _, want = oracle.topk(L, K)
    for r in range(rows.shape[0]):
        cand, rescans = _slab_candidates(rows[r], K, nslab, lower16)
        order = cand[np.lexsort((cand, -L[r, cand]))][:K]
        assert np.array_equal(order, want[r])
        if kind == "random":  # the usual case: ~10 elements a slab, no rescan
            assert rescans == 0 and cand.size < 12 * nslab
        else:
            assert rescans > 0


@pytest.mark.parametrize("V,nslab,K", [(2016, 15, 40), (1024, 8, 200), (4800, 37, 64)])
def test_narrow_slabs_and_k_above_the_slab_width(V, nslab, K):
    rng = np.random.default_rng(22)
    rows = rng.standard_normal((3, V)).astype(np.float32)
    L = rows.astype(np.float64)
    _, want = oracle.topk(L, K)
    for r in range(3):
        cand, _ = _slab_candidates(rows[r], K, nslab, True)
        order = cand[np.lexsort((cand, -L[r, cand]))][:K]
        assert np.array_equal(order, want[r])


# ------------------------------------------------------------------ the one-launch small path
#
# Each CTA owns slab_cols columns (the smallest multiple of 8 that covers V with at most one CTA per
# SM) and publishes, per row, its largest key.  The row's owner takes a lower bound of the K-th
# largest key: with at least K slabs, the largest 16-bit prefix (low bits zero) that K slab maxima
# reach -- the maxima are distinct elements, so K elements reach it too; else the largest 16-bit
# prefix that K of the row's keys reach.  Every key at or above the bound is gathered; when more
# than the gather buffer holds (max(1024, 2K), a multiple of 32) reach the slab bound, the row
# bound is tried, and past that the exact selection over the whole row runs.

def _bound16(keys, K):
    keys = np.asarray(keys, np.uint64)
    t = 0
    for bit in range(31, 15, -1):
        c = t | (1 << bit)
        if int(np.count_nonzero(keys >= c)) >= K:
            t = c
    return t


def _small_candidates(row, K, num_sms=152):
    V = row.size
    key = _keys(row)
    per = -(-(V // 8) // num_sms)
    sw = 8 * per
    nslab = -(-V // sw)
    cap = max(1024, 2 * K)
    cap = max((cap + 31) & ~31, 1 << (K - 1).bit_length())
    if nslab >= K:
        maxima = [key[c * sw:min(V, (c + 1) * sw)].max() for c in range(nslab)]
        sel = np.nonzero(key >= _bound16(maxima, K))[0]
        if sel.size <= cap:
            return sel, "slab_bound"
    sel = np.nonzero(key >= _bound16(key, K))[0]
    if sel.size <= cap:
        return sel, "row_bound"
    return np.arange(V), "whole_row"


def _small_rows(kind, V, rng):
    r = rng.standard_normal((3, V)).astype(np.float32)
    if kind == "clustered":  # every top element inside one slab: the slab maxima bound is low
        r[:, 700:740] += 20.0
    elif kind == "tied":  # columns repeated 8 times: a slab's maximum ties with its neighbours
        r = np.repeat(r[:, : V // 8], 8, axis=1)
    elif kind == "band":  # every value within a narrow band: most keys share their top 16 bits
        r = (1.0 + r * 1e-3).astype(np.float32)
    elif kind == "constant":
        r = np.full((2, V), 0.75, np.float32)
    return r


@pytest.mark.parametrize("kind", ["random", "clustered", "tied", "band", "constant"])
@pytest.mark.parametrize("V,K", [(4096, 16), (2000, 200), (16384, 1024), (16, 16), (4080, 40)])
def test_small_path_gather_holds_the_exact_top_k(kind, V, K):
    rng = np.random.default_rng(31)
    rows = _small_rows(kind, V, rng)
    L = rows.astype(np.float64)
    _, want = oracle.topk(L, K)
    for r in range(rows.shape[0]):
        cand, branch = _small_candidates(rows[r], K)
        assert set(want[r].tolist()) <= set(cand.tolist()), branch
        order = cand[np.lexsort((cand, -L[r, cand]))][:K]
        assert np.array_equal(order, want[r]), branch
        if kind == "random" and (V, K) == (4096, 16):  # the tiny shape: the slab bound, a few dozen keys
            assert branch == "slab_bound" and cand.size < 4 * K
        if kind == "constant" and V > 1024:
            assert branch == "whole_row"
