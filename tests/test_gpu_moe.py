"""GPU parity of the tail fused with its producer (tail_run_moe) against the oracle.

The producer step forms the bf16 hidden state from the residual and the expert
slots ("nemotron CUDA: RMSNorm rows run on the shared norms and combine (#548,
step 1)", entry tf_nemo_add_moe_norm).  Its result must equal the oracle's
combine bit for bit (the same fp32 fmas and bf16 roundings), and the tail on it
must equal tail_run on the oracle's h bit for bit and match the oracle's tail.
Slots follow the page's Nemotron contract: 8 slots, 6 routed ones with sigmoid
scores normalized to sum 2.5 and 2 shared ones of weight 1.
"""
import dataclasses

import numpy as np
import pytest

import gen
import oracle
from tests import tailcheck as tc
from tests.test_gpu_parity import full_check, make_tail

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import decode_sampling_tail_gb300 as dst  # noqa: E402


def _slots(B, H, slot_dtype, seed):
    rng = np.random.default_rng(seed)
    scores = 1.0 / (1.0 + np.exp(-rng.standard_normal((B, 6))))
    routed = (2.5 * scores / scores.sum(axis=1, keepdims=True)).astype(np.float32)
    wts = np.concatenate([routed, np.ones((B, 2), np.float32)], axis=1)
    y = (rng.standard_normal((B, 8, H)) * 0.5).astype(np.float32)
    if slot_dtype == "bf16":
        y = (y.view(np.uint32) >> 16).astype(np.uint16)  # bf16 bit patterns (truncated draws)
    return y, wts


def _run_moe(t, w, y, wts, emit=True):
    dev = torch.device("cuda:0")
    x, gamma, w_t, p = tc.to_device(w, torch)
    ys = torch.from_numpy(y.view(np.int16) if y.dtype == np.uint16 else y).to(dev)
    if y.dtype == np.uint16:
        ys = ys.view(torch.bfloat16)
    ws = torch.from_numpy(wts).to(dev)
    B, V, k = w.B, w.V, w.k
    tokens = torch.full((B,), -7, dtype=torch.int32, device=dev)
    logits = torch.empty((B, V), dtype=torch.float32, device=dev) if emit else None
    tv = torch.empty((B, k), dtype=torch.float32, device=dev)
    ti = torch.empty((B, k), dtype=torch.int32, device=dev)
    hout = torch.empty((B, w.H), dtype=torch.bfloat16, device=dev)
    t.run_moe(x, ys, ws, gamma, w_t, p, out_tokens=tokens, out_logits=logits, out_topk_vals=tv, out_topk_idx=ti,
              out_hidden=hout)
    torch.cuda.synchronize()
    t.check()
    res = tc.GpuResult(logits.cpu().numpy() if emit else None, tv.cpu().numpy(), ti.cpu().numpy(),
                       tokens.cpu().numpy())
    return res, hout.view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("slot_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("path", ["gemv", "tensor"])
def test_producer_fused_tail_matches_oracle(slot_dtype, path):
    w = gen.custom(6, 256, 8192, 32, hidden_dtype="bf16", seed=301)
    y, wts = _slots(w.B, w.H, slot_dtype, 302)
    h_ref = oracle.moe_combine(w.hidden, y, wts)
    with make_tail(w, path=path) as t:
        res, h_gpu = _run_moe(t, w, y, wts)
        plain = tc.run_gpu(t, dataclasses.replace(w, hidden=h_ref), torch)
    assert np.array_equal(h_gpu, h_ref)
    assert np.array_equal(res.logits.view(np.uint32), plain.logits.view(np.uint32))
    assert np.array_equal(res.topk_idx, plain.topk_idx) and np.array_equal(res.tokens, plain.tokens)
    exact, exempt = full_check(dataclasses.replace(w, hidden=h_ref), res)
    assert exact + exempt == w.B


def test_producer_step_with_many_slots():
    # 40 slots of small weights (the kernel's fma chain runs over a runtime slot count)
    w = gen.custom(4, 128, 4096, 16, hidden_dtype="bf16", seed=307)
    rng = np.random.default_rng(308)
    y = (rng.standard_normal((w.B, 40, w.H)) * 0.25).astype(np.float32)
    wts = rng.uniform(0.0, 0.2, (w.B, 40)).astype(np.float32)
    h_ref = oracle.moe_combine(w.hidden, y, wts)
    with make_tail(w, path="gemv") as t:
        res, h_gpu = _run_moe(t, w, y, wts)
        plain = tc.run_gpu(t, dataclasses.replace(w, hidden=h_ref), torch)
    assert np.array_equal(h_gpu, h_ref)
    assert np.array_equal(res.logits.view(np.uint32), plain.logits.view(np.uint32))
    assert np.array_equal(res.tokens, plain.tokens)


def test_producer_fused_tail_gptoss_g8():
    # the bench's shape: gbs=8, H=2880, V=201088, k=256, one launch of the tail after the combine
    w = gen.custom(8, 2880, 201088, 256, hidden_dtype="bf16", seed=303)
    y, wts = _slots(w.B, w.H, "f32", 304)
    h_ref = oracle.moe_combine(w.hidden, y, wts)
    with make_tail(w) as t:
        res, h_gpu = _run_moe(t, w, y, wts, emit=False)
        plain = tc.run_gpu(t, dataclasses.replace(w, hidden=h_ref), torch, emit=False)
    assert np.array_equal(h_gpu, h_ref)
    assert np.array_equal(res.topk_idx, plain.topk_idx) and np.array_equal(res.tokens, plain.tokens)
    assert np.array_equal(res.topk_vals.view(np.uint32), plain.topk_vals.view(np.uint32))


def test_producer_step_rejects_bad_arguments():
    w = gen.custom(2, 64, 2048, 16, hidden_dtype="bf16", seed=305)
    dev = torch.device("cuda:0")
    x, gamma, w_t, p = tc.to_device(w, torch)
    ys = torch.zeros((2, 3, 64), dtype=torch.float32, device=dev)
    ws = torch.ones((2, 3), dtype=torch.float32, device=dev)
    tok = torch.empty(2, dtype=torch.int32, device=dev)
    with make_tail(w) as t:
        s = t._stream(None)
        bad_dtype = dst.tail_run_moe(t.h, x.data_ptr(), ys.data_ptr(), dst.TAIL_F16, 3, ws.data_ptr(),
                                     gamma.data_ptr(), w_t.data_ptr(), p.data_ptr(), 4, 2, tok.data_ptr(), None, None,
                                     None, None, s)
        no_slots = dst.tail_run_moe(t.h, x.data_ptr(), None, dst.TAIL_F32, 3, ws.data_ptr(), gamma.data_ptr(),
                                    w_t.data_ptr(), p.data_ptr(), 4, 2, tok.data_ptr(), None, None, None, None, s)
        too_many = dst.tail_run_moe(t.h, x.data_ptr(), ys.data_ptr(), dst.TAIL_F32, 100000, ws.data_ptr(),
                                    gamma.data_ptr(), w_t.data_ptr(), p.data_ptr(), 4, 2, tok.data_ptr(), None, None,
                                    None, None, s)
    assert bad_dtype == no_slots == too_many == dst.TAIL_ERR_INVALID_ARG
    wf = gen.custom(2, 64, 2048, 16, hidden_dtype="f32", seed=306)
    with make_tail(wf) as t:
        xf, gf, wtf, pf = tc.to_device(wf, torch)
        rc = dst.tail_run_moe(t.h, xf.data_ptr(), ys.data_ptr(), dst.TAIL_F32, 3, ws.data_ptr(), gf.data_ptr(),
                              wtf.data_ptr(), pf.data_ptr(), 4, 2, tok.data_ptr(), None, None, None, None,
                              t._stream(None))
    assert rc == dst.TAIL_ERR_UNSUPPORTED
