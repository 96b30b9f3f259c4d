"""GPU parity of the CUDA tail (through the C ABI) against the fp64 oracle.

Small shapes span several slabs, ragged slab widths and every batch template;
the named workloads run at full size in the launch configuration the bench
uses.  All inputs come from the seeded generators in ``gen``.
"""
import numpy as np
import pytest

import gen
import oracle
from tests import tailcheck as tc

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import decode_sampling_tail_gb300 as dst  # noqa: E402


def make_tail(w, gbs_max=None, **kw):
    return dst.Tail(w.H, w.V, w.k, gbs_max or w.B, hidden_actual=w.Hu, eps=w.eps,
                    hidden_dtype=w.hidden_dtype, zero_interleaved_pad=bool(w.zero_pad), **kw)


@pytest.fixture(params=["gemv", "tensor", "small"])
def path(request):
    """The lm_head realisation a small-batch test runs on: the mma.sync kernel, the
    tensor-core path that narrow vocabularies take for every batch size, or the one-launch
    small path (up to 8 rows)."""
    return request.param


def full_check(w, res, rows=None, params=None):
    rows = np.arange(w.B) if rows is None else np.asarray(rows)
    L, ov, oi = tc.oracle_rows(w, rows)
    if res.logits is not None:
        tc.check_logits(res.logits[rows], L)
    tc.check_topk(res.topk_vals[rows], res.topk_idx[rows], L, ov, oi, w.k,
                  None if res.logits is None else res.logits[rows])
    p = w.params if params is None else params
    return tc.check_tokens(res.tokens[rows], res.topk_vals[rows], res.topk_idx[rows], L, ov, oi, p[rows], w.k)


# ------------------------------------------------------------------ small shapes

SMALL = [
    # B, H, V, k, dtype, Hu, zero_pad
    (1, 256, 4096, 16, "f32", None, 1),
    (3, 64, 2016, 40, "bf16", None, 1),
    (5, 128, 1024, 200, "f16", None, 1),     # k above the slab width: whole slabs kept
    (8, 96, 4800, 64, "bf16", 90, 1),        # zero pads at interleaved lanes
    (9, 80, 3200, 33, "f32", 72, 0),         # lanes beyond hidden_actual ignored
    (16, 160, 6400, 128, "bf16", None, 1),
    (17, 64, 2048, 17, "f16", None, 1),
    (33, 48, 1600, 50, "bf16", None, 1),
    (64, 64, 2400, 256, "bf16", None, 1),
    (70, 32, 1024, 8, "f32", None, 1),       # two lm_head passes
]


@pytest.mark.parametrize("shape", SMALL, ids=lambda s: f"B{s[0]}_H{s[1]}_V{s[2]}_k{s[3]}_{s[4]}")
def test_small_shapes_match_oracle(shape, path):
    B, H, V, k, dt, Hu, zp = shape
    if path == "small" and B > 8:
        pytest.skip("the small path takes up to 8 rows")
    w = gen.custom(B, H, V, k, hidden_dtype=dt, Hu=Hu, zero_pad=zp, seed=1000 + B)
    if Hu is not None and not zp:
        # garbage beyond hidden_actual must be ignored
        if dt == "f32":
            w.hidden[:, Hu:] = 3.0
        else:
            w.hidden[:, Hu:] = 0x4040
    with make_tail(w, path=path) as t:
        res = tc.run_gpu(t, w, torch)
    exact, exempt = full_check(w, res)
    assert exact + exempt == B and exact >= B - max(1, B // 8)


# odd k-step counts on the one-launch mma.sync path: the last ring stage holds a single k-step, so half
# of the activation warp's lanes sit it out; with and without lanes beyond hidden_actual, both forms
ODD_KSTEPS = [
    # B, H, V, k, dtype, Hu, zero_pad
    (4, 80, 2400, 24, "bf16", None, 1),    # 5 k-steps
    (8, 112, 4096, 64, "f16", 100, 0),     # 7 k-steps, lanes [100, 112) ignored
    (3, 208, 1600, 40, "f32", 200, 1),     # 13 k-steps, zero pads
]


@pytest.mark.parametrize("deferred", [True, False], ids=["deferred", "legacy"])
@pytest.mark.parametrize("shape", ODD_KSTEPS, ids=lambda s: f"B{s[0]}_H{s[1]}_V{s[2]}_k{s[3]}_{s[4]}")
def test_odd_kstep_counts_on_the_mma_sync_path(shape, deferred):
    B, H, V, k, dt, Hu, zp = shape
    w = gen.custom(B, H, V, k, hidden_dtype=dt, Hu=Hu, zero_pad=zp, seed=2000 + H)
    if Hu is not None and not zp:
        w.hidden[:, Hu:] = 3.0 if dt == "f32" else 0x4040  # garbage beyond hidden_actual is ignored
    with make_tail(w, path="gemv", deferred_rms=deferred) as t:
        assert t.info.tc_min_rows == 0 and t.info.kernels_per_run == (1 if deferred else 2)
        res = tc.run_gpu(t, w, torch)
    exact, exempt = full_check(w, res)
    assert exact + exempt == B


@pytest.mark.parametrize("ncols", ["3col", "none"])
def test_param_column_forms(ncols, path):
    w = gen.custom(6, 64, 2048, 32, hidden_dtype="bf16", seed=77)
    with make_tail(w, path=path) as t:
        res = tc.run_gpu(t, w, torch, params=ncols)
    if ncols == "none":
        assert np.all(res.tokens == -7), "tokens written although params is NULL"
        L, ov, oi = tc.oracle_rows(w, np.arange(w.B))
        tc.check_topk(res.topk_vals, res.topk_idx, L, ov, oi, w.k, res.logits)
    else:
        exact, exempt = full_check(w, res, params=w.params[:, :3])
        assert exact >= 5


def test_legacy_rms_realization_matches_oracle(path):
    w = gen.custom(8, 256, 8192, 64, hidden_dtype="bf16", seed=55)
    with make_tail(w, deferred_rms=False, path=path) as t:
        legacy = tc.run_gpu(t, w, torch)
    with make_tail(w, path=path) as t:
        deferred = tc.run_gpu(t, w, torch)
    full_check(w, legacy)
    assert np.max(np.abs(legacy.logits - deferred.logits)) < 1e-5


def test_sixteen_bit_input_equals_prewidened_fp32(path):
    w16 = gen.custom(8, 128, 4096, 64, hidden_dtype="bf16", seed=56)
    w32 = gen.custom(8, 128, 4096, 64, hidden_dtype="bf16", seed=56)
    w32.hidden = gen.bf16_bits_to_f32(w16.hidden)
    w32.hidden_dtype = "f32"
    with make_tail(w16, path=path) as t:
        a = tc.run_gpu(t, w16, torch)
    with make_tail(w32, path=path) as t:
        b = tc.run_gpu(t, w32, torch)
    assert np.array_equal(a.logits.view(np.uint32), b.logits.view(np.uint32))
    assert np.array_equal(a.topk_idx, b.topk_idx) and np.array_equal(a.tokens, b.tokens)


def test_repeat_runs_bitwise_identical_and_rows_independent_of_batch(path):
    w = gen.custom(8, 128, 4096, 64, hidden_dtype="bf16", seed=57)
    with make_tail(w, path=path) as t:
        r1 = tc.run_gpu(t, w, torch)
        r2 = tc.run_gpu(t, w, torch)
    assert np.array_equal(r1.logits.view(np.uint32), r2.logits.view(np.uint32))
    assert np.array_equal(r1.tokens, r2.tokens) and np.array_equal(r1.topk_idx, r2.topk_idx)
    for nb in (1, 4):
        sub = gen.custom(8, 128, 4096, 64, hidden_dtype="bf16", seed=57)
        sub.hidden = np.ascontiguousarray(w.hidden[:nb])
        sub.params = np.ascontiguousarray(w.params[:nb])
        sub.B = nb
        with make_tail(sub, path=path) as t:
            rs = tc.run_gpu(t, sub, torch)
        assert np.array_equal(rs.logits.view(np.uint32), r1.logits[:nb].view(np.uint32))
        assert np.array_equal(rs.tokens, r1.tokens[:nb])


def test_outputs_untouched_outside_their_rows(path):
    w = gen.custom(5, 64, 2048, 32, hidden_dtype="bf16", seed=58)
    hidden, gamma, w_t, p = tc.to_device(w, torch)
    dev = hidden.device
    guard = 4096
    tok = torch.full((w.B + 2 * guard,), 12345, dtype=torch.int32, device=dev)
    lg = torch.full((w.B * w.V + 2 * guard,), 7.5, dtype=torch.float32, device=dev)
    with make_tail(w, path=path) as t:
        t.run(hidden, gamma, w_t, p, out_tokens=tok[guard:guard + w.B],
              out_logits=lg[guard:guard + w.B * w.V].view(w.B, w.V))
        torch.cuda.synchronize()
    tok_h, lg_h = tok.cpu().numpy(), lg.cpu().numpy()
    assert np.all(tok_h[:guard] == 12345) and np.all(tok_h[guard + w.B:] == 12345)
    assert np.all(lg_h[:guard] == 7.5) and np.all(lg_h[guard + w.B * w.V:] == 7.5)


def test_host_entry_point_matches_device_entry_point(path):
    w = gen.custom(4, 64, 2048, 32, hidden_dtype="bf16", seed=59)
    hidden, gamma, w_t, p = tc.to_device(w, torch)
    with make_tail(w, path=path) as t:
        dev = tc.run_gpu(t, w, torch, dev_tensors=(hidden, gamma, w_t, p))
        toks = np.zeros(w.B, np.int32)
        logits = np.zeros((w.B, w.V), np.float32)
        t.run_host(w.hidden, gamma, w_t, w.params, toks, logits)
        # pinned inputs: the parameters are read in place; the tokens come back through mapped memory
        hid_p = torch.from_numpy(np.ascontiguousarray(w.hidden.view(np.int16))).pin_memory()
        par_p = torch.from_numpy(np.ascontiguousarray(w.params)).pin_memory()
        tok_p = torch.full((w.B,), -7, dtype=torch.int32).pin_memory()
        for _ in range(2):  # the mapped staging is made by the first call, reused by the second
            tok_p.fill_(-7)
            t.run_host(hid_p, gamma, w_t, par_p, tok_p)
            assert np.array_equal(tok_p.numpy(), dev.tokens)
    assert np.array_equal(toks, dev.tokens)
    assert np.array_equal(logits.view(np.uint32), dev.logits.view(np.uint32))


def test_invalid_arguments_return_status_codes(path):
    w = gen.custom(4, 64, 2048, 32, hidden_dtype="bf16", seed=60)
    hidden, gamma, w_t, p = tc.to_device(w, torch)
    tok = torch.zeros(8, dtype=torch.int32, device=hidden.device)
    with make_tail(w, path=path) as t:
        s = t._stream(None)
        P = dst._ptr
        # gbs beyond gbs_max
        assert dst.tail_run(t.h, P(hidden), P(gamma), P(w_t), P(p), 4, 5, P(tok), None, s) == dst.TAIL_ERR_INVALID_ARG
        # bad column count
        assert dst.tail_run(t.h, P(hidden), P(gamma), P(w_t), P(p), 5, 4, P(tok), None, s) == dst.TAIL_ERR_INVALID_ARG
        # misaligned weight pointer
        bad = w_t.view(torch.int16).view(-1)[1:]  # 2-byte offset
        assert dst.tail_run(t.h, P(hidden), P(gamma), P(bad), P(p), 4, 4, P(tok), None, s) == dst.TAIL_ERR_INVALID_ARG
        # params without tokens
        assert dst.tail_run(t.h, P(hidden), P(gamma), P(w_t), P(p), 4, 4, None, None, s) == dst.TAIL_ERR_INVALID_ARG
        # gbs == 0 is a no-op
        assert dst.tail_run(t.h, None, None, None, None, 4, 0, None, None, s) == dst.TAIL_OK
        assert dst.tail_check(t.h) == dst.TAIL_OK
    bad_cfg = dst.tail_config(100, 0, 2048, 32, 4, 1e-5, 2, 1, 1, dst.PATHS[path])  # H % 16 != 0
    with pytest.raises(dst.TailError) as ei:
        dst.tail_create(bad_cfg, 0)
    assert ei.value.status == dst.TAIL_ERR_UNSUPPORTED


# ------------------------------------------------------------------ named workloads at full size

@pytest.fixture(scope="module")
def g8():
    return gen.make("gptoss_g8")


@pytest.mark.parametrize("emit", [True, False], ids=["emit_on", "emit_off"])
def test_gptoss_g8_full(g8, emit):
    with make_tail(g8) as t:
        res = tc.run_gpu(t, g8, torch, emit=emit)
        # emit on and off produce the same top-k and tokens
        other = tc.run_gpu(t, g8, torch, emit=not emit)
    assert np.array_equal(res.topk_idx, other.topk_idx) and np.array_equal(res.tokens, other.tokens)
    exact, exempt = full_check(g8, res if emit else other)
    assert exact >= 7


def test_tiny_full(path):
    w = gen.make("tiny")
    with make_tail(w, path=path) as t:
        res = tc.run_gpu(t, w, torch)
    exact, exempt = full_check(w, res)
    assert exact == 1


def test_auto_path_choice_follows_vocabulary_width():
    # narrow vocabularies: tensor cores for every batch; wider ones: mma.sync up to 8 rows
    # (tc_min_rows 0: no batch a handle of gbs_max 8 accepts reaches the tensor-core path)
    for V, gbs_max, want in ((dst.TC_ALL_ROWS_MAX_V, 8, 1), (dst.TC_ALL_ROWS_MAX_V + 16, 8, 0),
                             (dst.TC_ALL_ROWS_MAX_V + 16, 9, 9)):
        with dst.Tail(64, V, 16, gbs_max) as t:
            assert t.info.tc_min_rows == want
            assert (t.info.rows_per_pass == 0) == (want == 1)
    with dst.Tail(64, 4096, 16, 8, path="gemv") as t:
        assert t.info.tc_min_rows == 0 and t.info.rows_per_pass == 8
    with dst.Tail(64, 4096, 16, 16, path="gemv") as t:
        assert t.info.tc_min_rows == 9
    with dst.Tail(64, 1 << 18, 16, 2, path="tensor") as t:
        assert t.info.tc_min_rows == 1


def test_padded_g64_full():
    w = gen.make("padded_g64")
    with make_tail(w) as t:
        res = tc.run_gpu(t, w, torch)
    exact, exempt = full_check(w, res)
    assert exact >= 60
    greedy = np.arange(w.B) % 4 == 0
    assert np.all(res.tokens[greedy] == res.topk_idx[greedy, 0])


def test_adversarial_g32_full():
    w = gen.make("adversarial_g32")
    with make_tail(w) as t:
        res = tc.run_gpu(t, w, torch)
    # duplicated columns give bitwise-equal fp32 logits
    groups = res.logits.view(np.uint32).reshape(w.B, -1, 4)
    assert np.all(groups == groups[:, :, :1])
    exact, exempt = full_check(w, res)
    assert exact >= 28
    # u = 0.0 always draws the first candidate
    even = np.arange(w.B) % 2 == 0
    assert np.all(res.tokens[even] == res.topk_idx[even, 0])


def test_large_g1024_every_row():
    # every row against the oracle (in blocks of 128 rows), plus properties that hold at any size
    w = gen.make("large_g1024")
    with make_tail(w, gbs_max=1024) as t:
        res = tc.run_gpu(t, w, torch)
    exact = exempt = 0
    for r0 in range(0, 1024, 128):
        e, x = full_check(w, res, rows=np.arange(r0, r0 + 128))
        exact, exempt = exact + e, exempt + x
    assert exact + exempt == 1024 and exact >= 1024 - 16
    assert np.all(np.diff(res.topk_vals, axis=1) <= 0)
    assert np.all((res.tokens >= 0) & (res.tokens < w.V))
    top1 = np.argmax(res.logits, axis=1)
    assert np.array_equal(res.topk_idx[:, 0], top1)


# the largest k the ABI accepts, on both lm_head paths (mma.sync for 8 rows at the GPT-OSS
# vocabulary; tensor cores with stacked and with separate hi/lo tiles)
K1024 = [
    ("gemv", (8, 2880, 201088, 1024, "bf16")),
    ("tensor", (24, 256, 32768, 1024, "bf16")),
    ("tensor", (72, 192, 24576, 1024, "f16")),
]


@pytest.mark.parametrize("case", K1024, ids=lambda c: f"{c[0]}_B{c[1][0]}_V{c[1][2]}")
def test_largest_k_matches_oracle(case):
    path, (B, H, V, k, dt) = case
    w = gen.custom(B, H, V, k, hidden_dtype=dt, seed=7000 + B)
    with make_tail(w, path=path) as t:
        assert (path == "tensor") == bool(t.info.tc_min_rows and B >= t.info.tc_min_rows)
        res = tc.run_gpu(t, w, torch)
    exact, exempt = full_check(w, res)
    assert exact + exempt == B and exact >= B - max(1, B // 8)


# ------------------------------------------------------------------ tensor-core path (9 rows and more)

TC_SHAPES = [
    # B, H, V, k, dtype: hi/lo sharing one 128-row tile up to 64 rows, separate tiles above
    (9, 256, 8192, 64, "bf16"),
    (64, 192, 12288, 256, "f16"),       # the last stacked size
    (65, 192, 12288, 256, "bf16"),      # the first with hi and lo in separate tiles
    (128, 128, 6144, 100, "f32"),       # one full m-block
    (129, 128, 6144, 100, "bf16"),      # a second m-block with one row
    (200, 160, 4144, 33, "bf16"),       # partial last tile and weight box; H not a multiple of 64
    (72, 128, 24576, 64, "bf16"),       # more tiles than k: the merge bound comes from the tile maxima
]


@pytest.mark.parametrize("shape", TC_SHAPES, ids=lambda s: f"B{s[0]}_H{s[1]}_V{s[2]}_k{s[3]}_{s[4]}")
def test_tensor_core_batches_match_oracle(shape):
    B, H, V, k, dt = shape
    w = gen.custom(B, H, V, k, hidden_dtype=dt, seed=3000 + B)
    with make_tail(w) as t:
        assert t.info.tc_min_rows and B >= t.info.tc_min_rows
        res = tc.run_gpu(t, w, torch)
    rows = np.arange(B) if B <= 64 else np.unique(np.concatenate([np.arange(0, B, 7), [B - 1]]))
    exact, exempt = full_check(w, res, rows=rows)
    assert exact + exempt == len(rows) and exact >= len(rows) - max(1, len(rows) // 8)


@pytest.mark.parametrize("V", [6144, 24576], ids=["bound_all_entries", "bound_tile_maxima"])
@pytest.mark.parametrize("emit", [True, False], ids=["emit_on", "emit_off"])
def test_tensor_core_saturated_tiles_scan_the_logits(V, emit):
    # columns repeated in groups of 32: every tile holding a top value holds at least 32 elements at or
    # above the merge bound, more than its 8-entry candidate list, so the merge must rescan those tiles:
    # in the caller's logits (emit on), or in the handle's copy of them (emit off)
    w = gen.custom(24, 128, V, 64, hidden_dtype="bf16", seed=91, dup_cols=32)
    with make_tail(w) as t:
        res = tc.run_gpu(t, w, torch, emit=emit)
    if emit:
        groups = res.logits.view(np.uint32).reshape(w.B, -1, 32)
        assert np.all(groups == groups[:, :, :1])
    exact, exempt = full_check(w, res)
    assert exact + exempt == w.B


@pytest.mark.parametrize("B", [24, 80], ids=["shared_tiles", "separate_tiles"])
def test_tensor_core_late_saturated_tile_keeps_its_logits(B):
    # The last column tiles hold 32 equal columns scaled by 4: for the rows they reach, those tiles
    # saturate late in the launch (after the other tiles' lists are in), and the merge must rescan
    # them from the logits the lm_head kept -- the handle's copy (emit off) or the caller's (emit on),
    # bitwise the same result, checked against the oracle.
    w = gen.custom(B, 2048, 98304, 64, hidden_dtype="bf16", seed=95)
    src = (w.w_t[:, 5000].astype(np.uint32) << 16).view(np.float32) * np.float32(4.0)
    w.w_t[:, 98304 - 200:98304 - 168] = ((src.view(np.uint32) >> 16).astype(np.uint16))[:, None]
    with make_tail(w) as t:
        on = tc.run_gpu(t, w, torch, emit=True)
        off = tc.run_gpu(t, w, torch, emit=False)
    assert np.array_equal(on.topk_idx, off.topk_idx) and np.array_equal(on.tokens, off.tokens)
    assert np.array_equal(on.topk_vals.view(np.uint32), off.topk_vals.view(np.uint32))
    # the planted ties are among every row's top k whose scale lets them in, so the tile saturates
    assert np.isin(np.arange(98304 - 200, 98304 - 168), on.topk_idx).any()
    exact, exempt = full_check(w, on)
    assert exact + exempt == w.B


def _scale_columns(w, c0, c1, pow2):
    """Multiplies W columns [c0, c1) by 2**pow2 (exact on bf16 values)."""
    f = (w.w_t[:, c0:c1].astype(np.uint32) << 16).view(np.float32) * np.float32(2.0 ** pow2)
    w.w_t[:, c0:c1] = (f.view(np.uint32) >> 16).astype(np.uint16)


def _slabs_hiding_top_k(logits, nslab, k):
    """Per row, the slabs whose publication (every element >= the 8th largest of its 32 lane maxima,
    none when more than 32 pass) may leave out a top-k element -- computed from the GPU's own fp32
    logits the way the mma.sync path publishes them."""
    B, V = logits.shape
    npairs = V // 16
    out = []
    for r in range(B):
        v = np.sort(logits[r])[::-1][k - 1]
        hidden = 0
        for c in range(nslab):
            lo, hi = 16 * (npairs * c // nslab), 16 * (npairs * (c + 1) // nslab)
            seg = logits[r, lo:hi]
            lane_max = np.full(32, -np.inf, np.float32)
            for lane in range(32):
                if seg[lane::32].size:
                    lane_max[lane] = seg[lane::32].max()
            b = np.sort(lane_max)[::-1][7]
            if np.count_nonzero(seg >= b) > 32 or b > v:
                hidden += 1
        out.append(hidden)
    return np.array(out)


@pytest.mark.parametrize("emit", [True, False], ids=["logits_out", "logits_scratch"])
@pytest.mark.parametrize("case", ["clustered", "saturated"])
def test_row_owner_rescans_slabs_that_may_hide_top_k(case, emit):
    # top-k elements crowded into a few slabs: "clustered" scales 240 columns by 4, so one or two slabs
    # hold most of a row's top 64 but publish only ~10; "saturated" repeats every column 64 times, so
    # slabs hold more than 32 elements at their bound and publish none.  The row owner must rescan them.
    if case == "clustered":
        w = gen.custom(6, 128, 24576, 64, hidden_dtype="bf16", seed=93)
        _scale_columns(w, 1600, 1840, 2)
    else:
        w = gen.custom(6, 128, 24576, 64, hidden_dtype="bf16", seed=94, dup_cols=64)
    with make_tail(w, path="gemv") as t:
        assert t.info.tc_min_rows == 0  # the mma.sync path
        ref = tc.run_gpu(t, w, torch, emit=True)
        res = ref if emit else tc.run_gpu(t, w, torch, emit=False)
        nslab = t.info.nslab
    assert np.all(_slabs_hiding_top_k(ref.logits, nslab, w.k) > 0)  # the inputs do force rescans
    if not emit:
        assert np.array_equal(res.topk_idx, ref.topk_idx) and np.array_equal(res.tokens, ref.tokens)
        res.logits = ref.logits
    exact, exempt = full_check(w, res)
    assert exact + exempt == w.B


def test_tensor_core_emit_off_matches_emit_on():
    w = gen.custom(40, 128, 8192, 128, hidden_dtype="bf16", seed=92)
    with make_tail(w) as t:
        on = tc.run_gpu(t, w, torch, emit=True)
        off = tc.run_gpu(t, w, torch, emit=False)
        again = tc.run_gpu(t, w, torch, emit=True)
    assert np.array_equal(on.topk_idx, off.topk_idx) and np.array_equal(on.tokens, off.tokens)
    assert np.array_equal(on.logits.view(np.uint32), again.logits.view(np.uint32))
    full_check(w, on)
