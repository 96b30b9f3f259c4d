"""Helpers for the GPU parity tests: upload a workload, run it through the C ABI,
and judge the results against the fp64 oracle with the tolerances of the tail:

  logits   |gpu - oracle| <= 1e-4 absolute (every element compared)
  top-k    the index set is exact wherever the oracle's k-th / (k+1)-th gap exceeds
           1e-4; position i holds an index whose oracle logit is within 1e-4 of the
           oracle's i-th value; and the GPU order is exactly the (value desc,
           index asc) order of its own fp32 logits (same-precision decision)
  tokens   bit-exact except where u lies within 1e-5 of a CDF boundary C_j / C_{m-1},
           or a top-p cut or a candidate's rank is decided by a margin below the
           logit tolerance; such rows must still pick a candidate whose oracle logit
           is within 1e-4 of the oracle's pick, and the oracle sampler run on the
           GPU's own top-k must reproduce the GPU token away from its boundaries.
"""
from __future__ import annotations

import numpy as np

import oracle
from gen.torch_io import to_device  # noqa: F401  (re-exported for the tests)

LOGIT_ATOL = 1e-4
TOPK_GAP = 1e-4
U_EDGE = 1e-5
P_EDGE = 1e-5


class GpuResult:
    def __init__(self, logits, topk_vals, topk_idx, tokens):
        self.logits = logits
        self.topk_vals = topk_vals
        self.topk_idx = topk_idx
        self.tokens = tokens


def run_gpu(tail, w, torch, *, emit=True, params="all", device="cuda:0", dev_tensors=None):
    """Runs the workload once; returns numpy copies of every output."""
    hidden, gamma, w_t, p = dev_tensors or to_device(w, torch, device)
    B, V, k = w.B, w.V, w.k
    dev = torch.device(device)
    if params == "none":
        p = None
    elif params == "3col":
        p = p[:, :3].contiguous()
    tokens = torch.full((B,), -7, dtype=torch.int32, device=dev)
    logits = torch.empty((B, V), dtype=torch.float32, device=dev) if emit else None
    tv = torch.empty((B, k), dtype=torch.float32, device=dev)
    ti = torch.empty((B, k), dtype=torch.int32, device=dev)
    tail.run(hidden, gamma, w_t, p, out_tokens=tokens, out_logits=logits, out_topk_vals=tv,
             out_topk_idx=ti)
    torch.cuda.synchronize()
    tail.check()
    return GpuResult(logits.cpu().numpy() if emit else None, tv.cpu().numpy(), ti.cpu().numpy(),
                     tokens.cpu().numpy())


def oracle_rows(w, rows):
    """fp64 oracle logits, top-k and draw reports for the given rows."""
    rows = np.asarray(rows)
    x = w.hidden[rows]
    L = oracle.logits(np.ascontiguousarray(x), w.hidden_dtype, w.gamma, w.w_t, w.Hu, w.eps, w.zero_pad)
    # one more than k so the k-th / (k+1)-th gap is known
    kk = min(w.k + 1, w.V)
    tv, ti = oracle.topk(L, kk)
    return L, tv, ti


def check_logits(gpu_logits, L):
    err = np.abs(gpu_logits.astype(np.float64) - L)
    worst = float(err.max()) if err.size else 0.0
    assert worst <= LOGIT_ATOL, f"max |logit error| {worst:.3e} > {LOGIT_ATOL}"
    return worst


def check_topk(gpu_vals, gpu_idx, L, ov, oi, k, gpu_logits=None):
    """Per-row top-k checks; returns the number of rows whose index set was compared exactly."""
    exact_rows = 0
    B = gpu_idx.shape[0]
    for b in range(B):
        gi = gpu_idx[b, :k]
        gv = gpu_vals[b, :k]
        assert np.all((gi >= 0) & (gi < L.shape[1])), f"row {b}: index out of range"
        assert len(np.unique(gi)) == k, f"row {b}: duplicated indices"
        # GPU order is (value desc, index asc) on its own values
        dv = np.diff(gv.astype(np.float64))
        assert np.all(dv <= 0), f"row {b}: values not sorted"
        tie = dv == 0
        assert np.all(gi[1:][tie] > gi[:-1][tie]), f"row {b}: ties not in index order"
        # each position within tolerance of the oracle's value at that position
        assert np.all(np.abs(L[b, gi] - ov[b, :k]) <= TOPK_GAP + 1e-12), f"row {b}: rank values off"
        assert np.all(np.abs(gv.astype(np.float64) - L[b, gi]) <= LOGIT_ATOL), f"row {b}: values off"
        if ov.shape[1] > k and ov[b, k - 1] - ov[b, k] > TOPK_GAP:
            assert set(gi.tolist()) == set(oi[b, :k].tolist()), f"row {b}: top-k set differs"
            exact_rows += 1
        if gpu_logits is not None:
            # same-precision decision: the exact top-k of the GPU's fp32 logits
            g = gpu_logits[b].astype(np.float64)
            order = np.lexsort((np.arange(g.size), -g))[:k]
            assert np.array_equal(order, gi), f"row {b}: not the exact top-k of the GPU logits"
            assert np.array_equal(gv, gpu_logits[b, gi]), f"row {b}: values are not the GPU logits"
    return exact_rows


def _boundary_row(rep, u, top_p):
    if rep.m > 1 and np.any(np.abs(rep.cdf[:-1] - u) < U_EDGE):
        return True
    if top_p < 1.0 and rep.pcum.size and np.any(np.abs(rep.pcum - top_p) < P_EDGE):
        return True
    return False


def check_tokens(gpu_tokens, gpu_vals, gpu_idx, L, ov, oi, params, k):
    """Returns (exact rows, exempt rows)."""
    exact = exempt = 0
    ncols = params.shape[1]
    for b in range(gpu_tokens.shape[0]):
        p = params[b]
        u = float(p[3]) if ncols == 4 else 0.5
        top_p = float(p[1])
        # (1) the oracle sampler on the GPU's own top-k (GPU fp32 values, widened exactly)
        rg = oracle.sample_row(gpu_vals[b, :k].astype(np.float64), gpu_idx[b, :k], p)
        if not _boundary_row(rg, u, top_p):
            assert rg.token == gpu_tokens[b], f"row {b}: sampler differs on the GPU top-k"
        # (2) end to end against the oracle
        ro = oracle.sample_row(ov[b, :k], oi[b, :k], p)
        if gpu_tokens[b] == ro.token:
            exact += 1
            continue
        # a difference is only allowed where the draw is decided by a margin below the tolerances
        m_cut = max(ro.m, ro.kk)
        near = np.abs(ov[b, : min(k, m_cut + 1)] - L[b, ro.token]) <= TOPK_GAP
        ambiguous_rank = near.sum() > 1
        assert _boundary_row(ro, u, top_p) or ambiguous_rank, (
            f"row {b}: token {gpu_tokens[b]} != oracle {ro.token} away from every boundary")
        assert abs(L[b, gpu_tokens[b]] - L[b, ro.token]) <= 2 * TOPK_GAP or _boundary_row(ro, u, top_p), (
            f"row {b}: token logit too far from the oracle's pick")
        exempt += 1
    return exact, exempt
