"""GPU tests of the stage-1 taps (tail_run_taps), the analogue of the page's `debug_taps`.

Each (row, chunk) of the chunked top-k hands the merge a few candidates and a bound
("GPT-OSS Tail Chunked Megakernel Kernel API Reference", section "Background" and
parameter `debug_taps`).  Checked against the run's own fp32 logits (emitted in the same
run), exactly: the candidates are the chunk's elements they claim to be, every element
left out is <= the bound, and the candidates are complete (every element >= the bound on a
slab; the top 8 by (value desc, index asc) on a tile).  Against the oracle: every element of
the oracle's top-k is a candidate or sits in a chunk whose bound reaches the GPU's k-th
value (the merge rescans such a chunk), and the top-k of the candidates plus those chunks is
the run's top-k.
"""
import numpy as np
import pytest

import gen
from tests import tailcheck as tc
from tests.test_gpu_parity import make_tail

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)


def _run(w, path):
    dev = torch.device("cuda:0")
    x, gamma, w_t, p = tc.to_device(w, torch)
    B, V, k = w.B, w.V, w.k
    tokens = torch.empty(B, dtype=torch.int32, device=dev)
    logits = torch.empty((B, V), dtype=torch.float32, device=dev)
    tv = torch.empty((B, k), dtype=torch.float32, device=dev)
    ti = torch.empty((B, k), dtype=torch.int32, device=dev)
    with make_tail(w, path=path) as t:
        shape = t.tap_shape(B)
        taps = t.run_taps(x, gamma, w_t, p, out_tokens=tokens, out_logits=logits, out_topk_vals=tv, out_topk_idx=ti)
        torch.cuda.synchronize()
        t.check()
    return shape, [a.cpu().numpy() for a in taps], logits.cpu().numpy(), tv.cpu().numpy(), ti.cpu().numpy()


def _top_order(vals, ids, n):
    o = np.lexsort((ids, -vals.astype(np.float64)))
    return ids[o[:n]]


def _check_against_own_logits(shape, taps, L):
    kind, n, cap, lo = shape
    vals, idx, count, bound = taps
    B = L.shape[0]
    assert lo[0] == 0 and lo[-1] == L.shape[1] and all(lo[c] < lo[c + 1] for c in range(n))
    for b in range(B):
        for c in range(n):
            cnt = int(count[b, c])
            assert 0 <= cnt <= cap
            ids = idx[b, c, :cnt]
            cols = np.arange(lo[c], lo[c + 1])
            x = L[b, lo[c]:lo[c + 1]]
            assert len(set(ids.tolist())) == cnt and np.all((ids >= lo[c]) & (ids < lo[c + 1]))
            assert np.array_equal(vals[b, c, :cnt].view(np.uint32), L[b, ids].view(np.uint32))
            assert np.all(idx[b, c, cnt:] == -1) and np.all(np.isneginf(vals[b, c, cnt:]))
            left = np.ones(cols.size, bool)
            left[ids - lo[c]] = False
            assert np.all(x[left] <= bound[b, c])
            if kind == 1:  # slab: every element >= the bound, or nothing (bound +inf)
                if cnt > 0:
                    assert set(ids.tolist()) == set(cols[x >= bound[b, c]].tolist())
                else:
                    assert np.isposinf(bound[b, c])
            else:  # tile: the top `cap` in (value desc, index asc) order
                want = _top_order(x, cols, cap)
                assert np.array_equal(ids, want)
                if cols.size > cap:
                    assert bound[b, c] == vals[b, c, cap - 1]
                else:
                    assert np.isneginf(bound[b, c])


def _check_against_oracle(w, shape, taps, L, tv, ti):
    kind, n, cap, lo = shape
    vals, idx, count, bound = taps
    rows = np.arange(w.B)
    _, ov, oi = tc.oracle_rows(w, rows)
    chunk_of = np.searchsorted(np.asarray(lo), np.arange(w.V), side="right") - 1
    for b in rows:
        vk = tv[b, w.k - 1]
        flagged = bound[b] >= vk
        for i in oi[b]:
            c = chunk_of[i]
            assert i in idx[b, c, :count[b, c]] or flagged[c], (b, i, c)
        # the candidates plus the flagged chunks' elements hold the run's top-k
        pool = set(idx[b][idx[b] >= 0].tolist())
        for c in np.nonzero(flagged)[0]:
            pool.update(range(lo[c], lo[c + 1]))
        pool = np.array(sorted(pool))
        assert np.array_equal(_top_order(L[b, pool], pool, w.k), ti[b])


CASES = [
    ("gemv", (6, 256, 8192, 32, "bf16", 501)),
    ("tensor", (6, 256, 8192, 32, "bf16", 502)),
    ("gemv", (8, 96, 2400, 200, "f32", 503)),      # k above a slab's width
    ("tensor", (72, 192, 6400, 64, "bf16", 504)),  # tiles of their own for hi and lo, 256 columns
    ("tensor", (33, 128, 4000, 100, "f16", 505)),  # stacked, a partial last tile
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0]}_B{c[1][0]}_V{c[1][2]}_k{c[1][3]}")
def test_taps_small(case):
    path, (B, H, V, k, dt, seed) = case
    w = gen.custom(B, H, V, k, hidden_dtype=dt, seed=seed)
    shape, taps, L, tv, ti = _run(w, path)
    assert shape[0] == (1 if path == "gemv" else 2)
    _check_against_own_logits(shape, taps, L)
    _check_against_oracle(w, shape, taps, L, tv, ti)


def test_taps_slabs_that_publish_nothing():
    # columns repeated 64 times: every slab holds more elements >= its bound than its slots
    w = gen.custom(4, 128, 8192, 16, hidden_dtype="bf16", seed=506)
    w.w_t[:] = np.repeat(w.w_t[:, ::64], 64, axis=1)
    shape, taps, L, tv, ti = _run(w, "gemv")
    assert np.any(taps[2] == 0)
    _check_against_own_logits(shape, taps, L)
    _check_against_oracle(w, shape, taps, L, tv, ti)


def test_taps_gptoss_g8():
    w = gen.make("gptoss_g8")
    shape, taps, L, tv, ti = _run(w, "auto")
    assert shape[0] == 1 and shape[1] >= 100
    _check_against_own_logits(shape, taps, L)
    _check_against_oracle(w, shape, taps, L, tv, ti)
