"""GPU parity of the tail fused with its producer (tail_run_moe) against the oracle.

The producer step forms the bf16 hidden state from the residual and the expert
slots ("nemotron CUDA: RMSNorm rows run on the shared norms and combine (#548,
step 1)", entry tf_nemo_add_moe_norm, with the author's fix reply: the routed
fma chain and the shared-slot sum kept apart).  Its result must equal the
oracle's combine bit for bit (the same fp32 fmas and adds and bf16 roundings),
and the tail on it must equal tail_run on the oracle's h bit for bit and match
the oracle's tail.  Slots follow the page's Nemotron contract: 8 slots, 6
routed ones with sigmoid scores normalized to sum 2.5 and 2 shared ones of
weight 1.  Up to 8 slots the step runs inside the tail's first kernel (the
lm_head kernel's activation warp, or the tensor-core path's RMSNorm split);
more slots, the legacy RMSNorm form and unaligned slots take a combine kernel
of their own; every form must give the same bits.
"""
import ctypes
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

NEMOTRON_ROUTED = 6


def _slots(B, H, slot_dtype, seed, S=8):
    rng = np.random.default_rng(seed)
    scores = 1.0 / (1.0 + np.exp(-rng.standard_normal((B, S - 2))))
    routed = (2.5 * scores / scores.sum(axis=1, keepdims=True)).astype(np.float32)
    wts = np.concatenate([routed, np.ones((B, 2), np.float32)], axis=1)
    y = (rng.standard_normal((B, S, H)) * 0.5).astype(np.float32)
    if slot_dtype == "bf16":
        y = (y.view(np.uint32) >> 16).astype(np.uint16)  # bf16 bit patterns (truncated draws)
    return y, wts


def _plant_order_lanes(w, y, wts, lanes):
    """In row 0, lanes where the routed chain is 1 + 2^-8 and the two shared slots are 2^-24 each, with
    a zero residual: keeping the shared sum apart gives h = 0x3f81, folding it into the chain 0x3f80
    (the golden case nemotron_8)."""
    assert y.dtype == np.float32 and y.shape[1] == 8
    wts[0] = np.array([1, 0.5, 0.5, 0.5, 0.5, 0.5, 1, 1], np.float32)
    for j in lanes:
        y[0, :, j] = np.array([1.00390625, 0, 0, 0, 0, 0, 2.0 ** -24, 2.0 ** -24], np.float32)
        w.hidden[0, j] = 0


def _run_moe(t, w, y, wts, emit=True, n_routed=NEMOTRON_ROUTED, slots_dev=None):
    dev = torch.device("cuda:0")
    x, gamma, w_t, p = tc.to_device(w, torch)
    if slots_dev is None:
        ys = torch.from_numpy(y.view(np.int16) if y.dtype == np.uint16 else y).to(dev)
        if y.dtype == np.uint16:
            ys = ys.view(torch.bfloat16)
    else:
        ys = slots_dev
    ws = torch.from_numpy(wts).to(dev)
    B, V, k = w.B, w.V, w.k
    tokens = torch.full((B,), -7, dtype=torch.int32, device=dev)
    logits = torch.empty((B, V), dtype=torch.float32, device=dev) if emit else None
    tv = torch.empty((B, k), dtype=torch.float32, device=dev)
    ti = torch.empty((B, k), dtype=torch.int32, device=dev)
    hout = torch.empty((B, w.H), dtype=torch.bfloat16, device=dev)
    t.run_moe(x, ys, ws, gamma, w_t, p, out_tokens=tokens, out_logits=logits, out_topk_vals=tv, out_topk_idx=ti,
              out_hidden=hout, n_routed=n_routed)
    torch.cuda.synchronize()
    t.check()
    res = tc.GpuResult(logits.cpu().numpy() if emit else None, tv.cpu().numpy(), ti.cpu().numpy(),
                       tokens.cpu().numpy())
    return res, hout.view(torch.int16).cpu().numpy().view(np.uint16)


def _same_tail(res, plain, emit=True):
    if emit:
        assert np.array_equal(res.logits.view(np.uint32), plain.logits.view(np.uint32))
    assert np.array_equal(res.topk_vals.view(np.uint32), plain.topk_vals.view(np.uint32))
    assert np.array_equal(res.topk_idx, plain.topk_idx) and np.array_equal(res.tokens, plain.tokens)


@pytest.mark.parametrize("slot_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("path", ["gemv", "tensor", "small"])
def test_producer_fused_tail_matches_oracle(slot_dtype, path):
    w = gen.custom(6, 256, 8192, 32, hidden_dtype="bf16", seed=301)
    y, wts = _slots(w.B, w.H, slot_dtype, 302)
    h_ref = oracle.moe_combine(w.hidden, y, wts, n_routed=NEMOTRON_ROUTED)
    with make_tail(w, path=path) as t:
        res, h_gpu = _run_moe(t, w, y, wts)
        plain = tc.run_gpu(t, dataclasses.replace(w, hidden=h_ref), torch)
    assert np.array_equal(h_gpu, h_ref)
    _same_tail(res, plain)
    exact, exempt = full_check(dataclasses.replace(w, hidden=h_ref), res)
    assert exact + exempt == w.B


@pytest.mark.parametrize("path", ["gemv", "tensor", "small"])
def test_producer_keeps_the_shared_sum_apart(path):
    # planted lanes on which the two orders of the page's thread give different bits
    w = gen.custom(4, 128, 4096, 16, hidden_dtype="bf16", seed=311)
    y, wts = _slots(w.B, w.H, "f32", 312)
    lanes = [0, 5, 31, 64, 127]
    _plant_order_lanes(w, y, wts, lanes)
    h_ref = oracle.moe_combine(w.hidden, y, wts, n_routed=NEMOTRON_ROUTED)
    assert all(h_ref[0, j] == 0x3F81 for j in lanes)
    assert all(oracle.moe_combine(w.hidden, y, wts, n_routed=8)[0, j] == 0x3F80 for j in lanes)
    with make_tail(w, path=path) as t:
        _, h_gpu = _run_moe(t, w, y, wts)
    assert np.array_equal(h_gpu, h_ref)


@pytest.mark.parametrize("slot_dtype", ["f32", "bf16"])
def test_producer_fused_few_slots_ragged_stage(slot_dtype):
    # 5 slots (3 routed, 2 shared): the fused form's slot rows past S must read as zeros; H = 208 is
    # 13 k-steps of 16, so the last stage of the activation warp holds 16 columns instead of 32
    w = gen.custom(7, 208, 6144, 24, hidden_dtype="bf16", seed=317)
    y, wts = _slots(w.B, w.H, slot_dtype, 318, S=5)
    h_ref = oracle.moe_combine(w.hidden, y, wts, n_routed=3)
    with make_tail(w, path="gemv") as t:
        res, h_gpu = _run_moe(t, w, y, wts, n_routed=3)
        plain = tc.run_gpu(t, dataclasses.replace(w, hidden=h_ref), torch)
    assert np.array_equal(h_gpu, h_ref)
    _same_tail(res, plain)


def test_producer_step_with_many_slots():
    # 40 slots (30 routed, 10 shared) of small weights: above the fused limit, the combine kernel runs first
    w = gen.custom(4, 128, 4096, 16, hidden_dtype="bf16", seed=307)
    rng = np.random.default_rng(308)
    y = (rng.standard_normal((w.B, 40, w.H)) * 0.25).astype(np.float32)
    wts = rng.uniform(0.0, 0.2, (w.B, 40)).astype(np.float32)
    h_ref = oracle.moe_combine(w.hidden, y, wts, n_routed=30)
    with make_tail(w, path="gemv") as t:
        res, h_gpu = _run_moe(t, w, y, wts, n_routed=30)
        plain = tc.run_gpu(t, dataclasses.replace(w, hidden=h_ref), torch)
    assert np.array_equal(h_gpu, h_ref)
    _same_tail(res, plain)


@pytest.mark.parametrize("form", ["legacy_rms", "unaligned_slots", "no_shared", "no_routed", "no_slots"])
def test_producer_other_forms_give_the_same_bits(form):
    w = gen.custom(5, 192, 6144, 24, hidden_dtype="bf16", seed=313)
    y, wts = _slots(w.B, w.H, "f32", 314)
    n_routed = {"no_shared": 8, "no_routed": 0}.get(form, NEMOTRON_ROUTED)
    if form == "no_slots":
        y, wts, n_routed = y[:, :0].copy(), wts[:, :0].copy(), 0
    h_ref = oracle.moe_combine(w.hidden, y, wts, n_routed=n_routed)
    slots_dev = None
    if form == "unaligned_slots":  # 4-byte aligned only: the activation warp's 16-byte copies cannot take it
        buf = torch.zeros(y.size + 1, dtype=torch.float32, device="cuda:0")
        buf[1:] = torch.from_numpy(y.reshape(-1)).to("cuda:0")
        slots_dev = buf[1:].view(y.shape)
    kw = {"deferred_rms": False} if form == "legacy_rms" else {}
    with make_tail(w, path="gemv", **kw) as t:
        res, h_gpu = _run_moe(t, w, y, wts, n_routed=n_routed, slots_dev=slots_dev)
        plain = tc.run_gpu(t, dataclasses.replace(w, hidden=h_ref), torch)
    assert np.array_equal(h_gpu, h_ref)
    _same_tail(res, plain)


def test_producer_fused_tail_gptoss_g8():
    # the bench's shape: gbs=8, H=2880, V=201088, k=256
    w = gen.custom(8, 2880, 201088, 256, hidden_dtype="bf16", seed=303)
    y, wts = _slots(w.B, w.H, "f32", 304)
    h_ref = oracle.moe_combine(w.hidden, y, wts, n_routed=NEMOTRON_ROUTED)
    with make_tail(w) as t:
        res, h_gpu = _run_moe(t, w, y, wts, emit=False)
        plain = tc.run_gpu(t, dataclasses.replace(w, hidden=h_ref), torch, emit=False)
    assert np.array_equal(h_gpu, h_ref)
    _same_tail(res, plain, emit=False)


# ------------------------------------------------------------------ launches per step

def _driver():
    try:
        return ctypes.CDLL("libcuda.so.1")
    except OSError:
        pytest.skip("the CUDA driver library is not loadable")


def _launches(fn, stream):
    """Kernel nodes of a graph captured from one call of fn on `stream` (driver stream capture)."""
    cu = _driver()
    graph = ctypes.c_void_p()
    n = ctypes.c_size_t(0)
    assert cu.cuStreamBeginCapture_v2(ctypes.c_void_p(stream.cuda_stream), ctypes.c_int(2)) == 0  # relaxed
    try:
        fn()
    finally:
        rc = cu.cuStreamEndCapture(ctypes.c_void_p(stream.cuda_stream), ctypes.byref(graph))
    assert rc == 0
    try:
        assert cu.cuGraphGetNodes(graph, None, ctypes.byref(n)) == 0
    finally:
        cu.cuGraphDestroy(graph)
    return n.value


@pytest.mark.parametrize("case", ["gemv_fused", "tensor_fused", "many_slots"])
def test_producer_step_launch_count(case):
    # the fused forms add no launch to the tail's own; more slots than the fused limit add one
    B, path, S = {"gemv_fused": (8, "gemv", 8), "tensor_fused": (16, "gemv", 8), "many_slots": (8, "gemv", 12)}[case]
    w = gen.custom(B, 256, 8192, 32, hidden_dtype="bf16", seed=315)
    y, wts = _slots(w.B, w.H, "f32", 316, S=S)
    dev = torch.device("cuda:0")
    x, gamma, w_t, p = tc.to_device(w, torch)
    ys, ws = torch.from_numpy(y).to(dev), torch.from_numpy(wts).to(dev)
    tokens = torch.empty((B,), dtype=torch.int32, device=dev)
    with make_tail(w, path=path) as t:
        s = torch.cuda.Stream(dev)
        s.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(s):
            t.run_moe(x, ys, ws, gamma, w_t, p, out_tokens=tokens, n_routed=S - 2, stream=s)  # warm
        torch.cuda.synchronize(dev)
        plain = _launches(lambda: t.run(x, gamma, w_t, p, out_tokens=tokens, stream=s), s)
        fused = _launches(lambda: t.run_moe(x, ys, ws, gamma, w_t, p, out_tokens=tokens, n_routed=S - 2, stream=s), s)
        torch.cuda.synchronize(dev)
        t.check()
    assert plain == (1 if path == "gemv" and B <= 8 else 3)
    assert fused == plain + (1 if case == "many_slots" else 0)


def test_producer_step_rejects_bad_arguments():
    w = gen.custom(2, 64, 2048, 16, hidden_dtype="bf16", seed=305)
    dev = torch.device("cuda:0")
    x, gamma, w_t, p = tc.to_device(w, torch)
    ys = torch.zeros((2, 3, 64), dtype=torch.float32, device=dev)
    ws = torch.ones((2, 3), dtype=torch.float32, device=dev)
    tok = torch.empty(2, dtype=torch.int32, device=dev)

    def call(t, slots, sd, nslots, n_routed, xx=x, gg=gamma, wt=w_t, pp=p):
        return dst.tail_run_moe(t.h, xx.data_ptr(), slots, sd, nslots, n_routed, ws.data_ptr(), gg.data_ptr(),
                                wt.data_ptr(), pp.data_ptr(), 4, 2, tok.data_ptr(), None, None, None, None,
                                t._stream(None))

    with make_tail(w) as t:
        rcs = [call(t, ys.data_ptr(), dst.TAIL_F16, 3, 3),          # slot dtype
               call(t, None, dst.TAIL_F32, 3, 3),                   # no slots
               call(t, ys.data_ptr(), dst.TAIL_F32, 100000, 3),     # too many slots
               call(t, ys.data_ptr(), dst.TAIL_F32, 3, 4),          # more routed slots than slots
               call(t, ys.data_ptr(), dst.TAIL_F32, 3, -1)]         # negative routed count
    assert all(rc == dst.TAIL_ERR_INVALID_ARG for rc in rcs), rcs
    wf = gen.custom(2, 64, 2048, 16, hidden_dtype="f32", seed=306)
    with make_tail(wf) as t:
        xf, gf, wtf, pf = tc.to_device(wf, torch)
        rc = call(t, ys.data_ptr(), dst.TAIL_F32, 3, 3, xx=xf, gg=gf, wt=wtf, pp=pf)
    assert rc == dst.TAIL_ERR_UNSUPPORTED
