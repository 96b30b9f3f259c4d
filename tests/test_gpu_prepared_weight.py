"""The tensor-core path reading the prepared copy of the weight (tail_prepare_weight).

The copy holds the weight in the layout of the lm_head's shared-memory stages, so a run that
reads it must give bitwise the results of the same run reading the weight through tensor-tile
loads: logits, top-k and tokens.  Shapes cover both tile layouts (hi and lo sharing a tile, and
separate m-blocks), a partial last 64-column group (V not a multiple of 64) and a partial last
k-block (H not a multiple of 64); one case is also checked against the oracle.
"""
import numpy as np
import pytest

import gen
from tests import tailcheck as tc

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import decode_sampling_tail_gb300 as dst  # noqa: E402


def make_tail(w, gbs_max=None, **kw):
    return dst.Tail(w.H, w.V, w.k, gbs_max or w.B, hidden_actual=w.Hu, eps=w.eps,
                    hidden_dtype=w.hidden_dtype, zero_interleaved_pad=bool(w.zero_pad), **kw)


def same(a, b):
    assert np.array_equal(a.logits.view(np.uint32), b.logits.view(np.uint32))
    assert np.array_equal(a.topk_vals.view(np.uint32), b.topk_vals.view(np.uint32))
    assert np.array_equal(a.topk_idx, b.topk_idx)
    assert np.array_equal(a.tokens, b.tokens)


SHAPES = [
    # B, H, V, k, dtype
    (16, 128, 8192, 64, "bf16"),     # shared tiles
    (40, 160, 6160, 100, "f16"),     # shared tiles; V = 96 * 64 + 16, H = 2.5 k-blocks
    (72, 128, 24576, 64, "bf16"),    # separate tiles
    (200, 96, 4144, 33, "f32"),      # separate tiles, two m-blocks; partial group and k-block
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"B{s[0]}_H{s[1]}_V{s[2]}_k{s[3]}_{s[4]}")
def test_prepared_weight_is_bitwise_the_tensor_tile_path(shape):
    B, H, V, k, dt = shape
    w = gen.custom(B, H, V, k, hidden_dtype=dt, seed=4100 + B)
    dev = tc.to_device(w, torch, "cuda:0")
    with make_tail(w) as t:
        assert t.info.tc_min_rows and B >= t.info.tc_min_rows
        plain = tc.run_gpu(t, w, torch, dev_tensors=dev)
        before = t.info.scratch_bytes
        t.prepare_weight(dev[2])
        groups, kblocks = (V + 63) // 64, (H + 63) // 64
        assert t.info.scratch_bytes == before + kblocks * groups * 8192
        prepared = tc.run_gpu(t, w, torch, dev_tensors=dev)
        again = tc.run_gpu(t, w, torch, dev_tensors=dev)
        t.prepare_weight(None)
        assert t.info.scratch_bytes == before
        released = tc.run_gpu(t, w, torch, dev_tensors=dev)
    same(plain, prepared)
    same(prepared, again)
    same(plain, released)


def test_prepared_weight_matches_oracle_and_follows_the_pointer():
    w = gen.custom(24, 192, 12352, 128, hidden_dtype="bf16", seed=4200)
    dev = tc.to_device(w, torch, "cuda:0")
    hidden, gamma, w_t, p = dev
    other = w_t.clone()  # same values, another pointer: read through tensor-tile loads
    with make_tail(w) as t:
        t.prepare_weight(w_t)
        res = tc.run_gpu(t, w, torch, dev_tensors=dev)
        res_other = tc.run_gpu(t, w, torch, dev_tensors=(hidden, gamma, other, p))
        # the copy is not refreshed by itself: a changed weight is read again once it is prepared again
        w_t.zero_()
        stale = tc.run_gpu(t, w, torch, dev_tensors=dev)
        t.prepare_weight(w_t)
        fresh = tc.run_gpu(t, w, torch, dev_tensors=dev)
    same(res, res_other)
    same(res, stale)
    assert not np.any(fresh.logits)
    rows = np.arange(w.B)
    L, ov, oi = tc.oracle_rows(w, rows)
    tc.check_logits(res.logits, L)
    tc.check_topk(res.topk_vals, res.topk_idx, L, ov, oi, w.k, res.logits)
    exact, exempt = tc.check_tokens(res.tokens, res.topk_vals, res.topk_idx, L, ov, oi, w.params, w.k)
    assert exact + exempt == w.B


def test_prepare_weight_on_a_handle_without_tensor_core_path_is_a_no_op():
    w = gen.custom(4, 128, 4096, 16, hidden_dtype="bf16", seed=4300)
    dev = tc.to_device(w, torch, "cuda:0")
    with make_tail(w, path="gemv") as t:
        assert t.info.tc_min_rows == 0
        before = t.info.scratch_bytes
        t.prepare_weight(dev[2])
        assert t.info.scratch_bytes == before
        res = tc.run_gpu(t, w, torch, dev_tensors=dev)
    exact, exempt = tc.check_tokens(res.tokens, res.topk_vals, res.topk_idx, *tc.oracle_rows(w, np.arange(w.B)),
                                    w.params, w.k)
    assert exact + exempt == w.B


def test_prepared_weight_serves_the_producer_step_and_the_taps():
    # tail_run_moe and tail_run_taps run the same tensor-core pass: with the prepared copy their
    # outputs (the combined hidden state, the tokens, the stage-1 lists) are bitwise those of W itself
    w = gen.custom(24, 256, 12352, 64, hidden_dtype="bf16", seed=4400)
    hidden, gamma, w_t, p = tc.to_device(w, torch, "cuda:0")
    g = torch.Generator().manual_seed(4401)
    S = 4
    slots = torch.randn(w.B, S, w.H, generator=g).to("cuda:0")
    slot_w = torch.rand(w.B, S, generator=g).to("cuda:0")
    resid = hidden

    def run_all(t):
        tok = torch.full((w.B,), -7, dtype=torch.int32, device="cuda:0")
        h_out = torch.empty(w.B, w.H, dtype=torch.int16, device="cuda:0")
        t.run_moe(resid, slots, slot_w, gamma, w_t, p, out_tokens=tok, out_hidden=h_out, n_routed=S - 2)
        tok2 = torch.full((w.B,), -7, dtype=torch.int32, device="cuda:0")
        taps = t.run_taps(hidden, gamma, w_t, p, out_tokens=tok2)
        torch.cuda.synchronize()
        t.check()
        return [tok.cpu().numpy(), h_out.cpu().numpy(), tok2.cpu().numpy()] + [x.cpu().numpy() for x in taps]

    with make_tail(w) as t:
        assert t.info.tc_min_rows and w.B >= t.info.tc_min_rows
        plain = run_all(t)
        t.prepare_weight(w_t)
        prepared = run_all(t)
    for a_, b_ in zip(plain, prepared):
        assert np.array_equal(a_.view(np.uint8), b_.view(np.uint8))
