"""tail_run_noalloc (static scratch, no handle, no device allocation) against tail_run.

The allocation-free entry point launches the same mma.sync kernels as the
handle path does for batches of up to 8 rows, so there the results must be
bitwise equal; larger batches (several passes here, the tensor-core path in
the handle) must agree within the logit tolerance, with the same tokens.  Each comparison makes two
calls in a row on one stream, with different inputs, before synchronising, so
the second call also proves that the per-call reset of the shared scratch
works.  The file is collected last so that it also runs after every other GPU
test has used the device; it passes alone as well.
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

STATIC_SCRATCH_BYTES = 8 << 20


def second_inputs(hidden, params):
    """A different batch for the second call: rows reversed, draws moved."""
    h2 = hidden.flip(0).contiguous()
    p2 = params.flip(0).contiguous()
    if p2.shape[1] == 4:
        p2[:, 3] = torch.remainder(p2[:, 3] + 0.37, 1.0)
    return h2, p2


def cfg_kwargs(w):
    return dict(k=w.k, hidden_actual=w.Hu, eps=w.eps, hidden_dtype=w.hidden_dtype,
                zero_interleaved_pad=bool(w.zero_pad))


def run_handle(w, hidden, gamma, w_t, params):
    B, V = hidden.shape[0], w_t.shape[1]
    tok = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    lg = torch.empty((B, V), dtype=torch.float32, device="cuda")
    with dst.Tail(hidden.shape[1], V, w.k, B, hidden_actual=w.Hu, eps=w.eps, hidden_dtype=w.hidden_dtype,
                  zero_interleaved_pad=bool(w.zero_pad), path="gemv") as t:
        t.run(hidden, gamma, w_t, params, out_tokens=tok, out_logits=lg)
        torch.cuda.synchronize()
        t.check()
    return lg.cpu().numpy(), tok.cpu().numpy()


def run_noalloc_twice(w, a, b, gamma, w_t, emit=True):
    """Two calls in a row (inputs a, then b) on the current stream, then one synchronise.  emit=False
    passes no logits: the row owners then rescan the logits copy staged in the static scratch."""
    outs = []
    for hidden, params in (a, b):
        B, V = hidden.shape[0], w_t.shape[1]
        tok = torch.full((B,), -7, dtype=torch.int32, device="cuda")
        lg = torch.empty((B, V), dtype=torch.float32, device="cuda") if emit else None
        st = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        dst.run_noalloc(hidden, gamma, w_t, params, out_tokens=tok, out_logits=lg, out_status=st,
                        **cfg_kwargs(w))
        outs.append((lg, tok, st))
    torch.cuda.synchronize()
    return [(None if lg is None else lg.cpu().numpy(), tok.cpu().numpy(), int(st.item())) for lg, tok, st in outs]


def compare(ref, got, bitwise):
    (lr, tr), (lg, tg, st) = ref, got
    assert st == 0, f"device error word {st}"
    if bitwise:
        if lg is not None:
            assert np.array_equal(lr.view(np.uint32), lg.view(np.uint32))
        assert np.array_equal(tr, tg)
        return
    if lg is not None:
        assert np.max(np.abs(lr - lg)) <= tc.LOGIT_ATOL
    # tokens agree, except where the two logits of the picks sit within twice the tolerance
    # (a draw decided by less than the logit tolerance may fall either way)
    diff = np.nonzero(tr != tg)[0]
    for r in diff:
        assert abs(float(lr[r, tr[r]]) - float(lr[r, tg[r]])) <= 2 * tc.LOGIT_ATOL, f"row {r}"
    assert len(diff) <= max(1, len(tr) // 16)


SMALL = [
    # B, H, V, k, dtype, Hu, zero_pad
    (5, 128, 1024, 200, "f16", None, 1),     # k above the slab width
    (8, 96, 4800, 64, "bf16", 90, 1),        # zero pads at interleaved lanes
    (9, 80, 3200, 33, "f32", 72, 0),         # lanes beyond hidden_actual ignored
    (17, 64, 2048, 17, "bf16", None, 1),
    (70, 32, 1024, 8, "f32", None, 1),       # more rows than one pass
]


@pytest.mark.parametrize("emit", [True, False], ids=["emit_on", "emit_off"])
@pytest.mark.parametrize("shape", SMALL, ids=lambda s: f"B{s[0]}_H{s[1]}_V{s[2]}_k{s[3]}_{s[4]}")
def test_noalloc_small_shapes_match_handle(shape, emit):
    B, H, V, k, dt, Hu, zp = shape
    w = gen.custom(B, H, V, k, hidden_dtype=dt, Hu=Hu, zero_pad=zp, seed=5000 + B)
    hidden, gamma, w_t, params = tc.to_device(w, torch)
    b = second_inputs(hidden, params)
    refs = [run_handle(w, hidden, gamma, w_t, params), run_handle(w, b[0], gamma, w_t, b[1])]
    gots = run_noalloc_twice(w, (hidden, params), b, gamma, w_t, emit=emit)
    for ref, got in zip(refs, gots):
        # up to 8 rows both run the same mma.sync kernel; larger batches take the handle's tensor-core path
        compare(ref, got, bitwise=B <= 8)


@pytest.fixture(scope="module")
def g8_dev():
    w = gen.make("gptoss_g8")
    return w, tc.to_device(w, torch)


def test_noalloc_gptoss_g8_matches_handle(g8_dev):
    """gbs = 8 at H = 2880, V = 201088, k = 256: one pass on both paths, bitwise equal."""
    w, (hidden, gamma, w_t, params) = g8_dev
    b = second_inputs(hidden, params)
    refs = [run_handle(w, hidden, gamma, w_t, params), run_handle(w, b[0], gamma, w_t, b[1])]
    gots = run_noalloc_twice(w, (hidden, params), b, gamma, w_t)
    for ref, got in zip(refs, gots):
        compare(ref, got, bitwise=True)


@pytest.mark.parametrize("emit", [True, False], ids=["emit_on", "emit_off"])
def test_noalloc_gptoss_g20_passes_match_handle(g8_dev, emit):
    """gbs = 20 at GPT-OSS sizes: the static scratch holds 9 rows per pass (3 passes: 9, 9, 2;
    without the caller's logits the per-row logits copy and the per-row words move from pass to
    pass), the handle runs one pass of 20 rows; logits within tolerance, tokens equal."""
    w, (_, gamma, w_t, _) = g8_dev
    rows = gen.custom(20, 2880, 16, 16, hidden_dtype="bf16", seed=21)  # 20 hidden rows + params
    hidden = tc.to_device(rows, torch)[0]
    params = torch.from_numpy(rows.params).cuda()
    b = second_inputs(hidden, params)
    refs = [run_handle(w, hidden, gamma, w_t, params), run_handle(w, b[0], gamma, w_t, b[1])]
    gots = run_noalloc_twice(w, (hidden, params), b, gamma, w_t, emit=emit)
    for ref, got in zip(refs, gots):
        compare(ref, got, bitwise=False)


def test_noalloc_rejects_what_the_static_scratch_cannot_hold():
    # one row's activation pack alone is 32 * H = 8,389,120 bytes > 8 MiB: refused before any launch
    H, V, k = 262160, 16, 16
    hidden = torch.zeros((1, H), dtype=torch.float32, device="cuda")
    gamma = torch.ones((H,), dtype=torch.float32, device="cuda")
    w_t = torch.zeros((H, V), dtype=torch.bfloat16, device="cuda")
    params = torch.tensor([[1.0, 1.0, 1.0, 0.5]], dtype=torch.float32, device="cuda")
    tok = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    with pytest.raises(dst.TailError) as ei:
        dst.run_noalloc(hidden, gamma, w_t, params, out_tokens=tok, k=k, hidden_dtype="f32")
    assert ei.value.status == dst.TAIL_ERR_UNSUPPORTED
    assert str(STATIC_SCRATCH_BYTES) in str(ei.value)
    torch.cuda.synchronize()
    assert int(tok.item()) == -7


def test_noalloc_invalid_arguments():
    H, V = 64, 1024
    hidden = torch.zeros((2, H), dtype=torch.bfloat16, device="cuda")
    gamma = torch.ones((H,), dtype=torch.float32, device="cuda")
    w_t = torch.zeros((H, V), dtype=torch.bfloat16, device="cuda")
    params = torch.zeros((2, 4), dtype=torch.float32, device="cuda")
    cfg = dst.tail_config(H, 0, V, 8, 1, 1e-5, dst.TAIL_BF16, 1, 1, 0)   # gbs_max 1 < gbs 2
    ptr = lambda t: t.data_ptr()  # noqa: E731
    s = torch.cuda.current_stream().cuda_stream
    assert dst.tail_run_noalloc(cfg, ptr(hidden), ptr(gamma), ptr(w_t), ptr(params), 4, 2, None, None, None,
                                s) == dst.TAIL_ERR_INVALID_ARG
    cfg.gbs_max = 2
    assert dst.tail_run_noalloc(cfg, None, ptr(gamma), ptr(w_t), ptr(params), 4, 2, None, None, None,
                                s) == dst.TAIL_ERR_INVALID_ARG
    assert dst.tail_run_noalloc(cfg, ptr(hidden), ptr(gamma), ptr(w_t), ptr(params), 5, 2, None, None, None,
                                s) == dst.TAIL_ERR_INVALID_ARG
    assert dst.tail_run_noalloc(cfg, ptr(hidden), ptr(gamma), ptr(w_t), None, 4, 0, None, None, None,
                                s) == dst.TAIL_OK
