"""GPU parity of the one-launch small path (cfg.path "small") against the oracle.

The path forms the activations in fp32 (no bf16 rounding), the fp32 logits of each
vocabulary slab with plain loads, and then, in the CTA that owns a row, the exact top k
over all V logits and the draw ("GPT-OSS Tail Chunked Megakernel Kernel API Reference":
final RMSNorm, lm_head, global top-k with ties to the lower index, sampler).  Logits
must stay within the logit tolerance of the oracle, the top k must be exact under the
comparison rules every path follows, and the token must be the sampler's on the run's
own top k.  The shapes reach the path's limits: a vocabulary narrower than the batch
(a CTA owns several rows, k = V), a last slab of half width, the largest H, V and k,
and lanes past H_u either ignored or zero-padded.
"""
import numpy as np
import pytest

import gen
from tests import tailcheck as tc
from tests.test_gpu_parity import full_check, make_tail

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import decode_sampling_tail_gb300 as dst  # noqa: E402

SHAPES = [
    # B, H, V, k, dtype, Hu, zero_pad
    (1, 256, 4096, 16, "f32", None, 1),        # the tiny workload's shape
    (8, 16, 16, 16, "bf16", None, 1),          # 2 slabs of 8 columns for 8 rows: CTAs own 4 rows each; k = V
    (3, 208, 4080, 40, "f16", 200, 0),         # the last slab holds 16 of 32 columns; lanes past H_u ignored
    (5, 96, 2000, 200, "f32", 90, 1),          # k above the slab width; zero pads at interleaved lanes
    (8, 512, 16384, 1024, "bf16", None, 1),    # the largest V and k
    (2, 8192, 1024, 64, "bf16", 8000, 1),      # the largest H
]


@pytest.mark.parametrize("deferred", [True, False], ids=["deferred", "legacy"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"B{s[0]}_H{s[1]}_V{s[2]}_k{s[3]}_{s[4]}")
def test_small_path_matches_oracle(shape, deferred):
    B, H, V, k, dt, Hu, zp = shape
    w = gen.custom(B, H, V, k, hidden_dtype=dt, Hu=Hu, zero_pad=zp, seed=3000 + V)
    if Hu is not None and not zp:
        w.hidden[:, Hu:] = 3.0 if dt == "f32" else 0x4040  # garbage beyond hidden_actual is ignored
    with make_tail(w, path="small", deferred_rms=deferred) as t:
        assert t.info.lmhead_path == 3 and t.info.kernels_per_run == 1 and t.info.tc_min_rows == 0
        res = tc.run_gpu(t, w, torch)
        again = tc.run_gpu(t, w, torch, emit=False)
    exact, exempt = full_check(w, res)
    assert exact + exempt == B
    # the logits' scratch copy (emit off) gives the same top k and tokens
    assert np.array_equal(again.topk_idx, res.topk_idx) and np.array_equal(again.tokens, res.tokens)
    assert np.array_equal(again.topk_vals.view(np.uint32), res.topk_vals.view(np.uint32))


def test_small_path_runs_back_to_back_without_a_sync():
    # the per-row arrival words reset themselves at the end of every launch: four launches queued
    # on one stream, alternating two inputs, give the outputs of separate synchronised runs
    w1 = gen.custom(4, 128, 4096, 32, hidden_dtype="bf16", seed=3101)
    w2 = gen.custom(4, 128, 4096, 32, hidden_dtype="bf16", seed=3102)  # its hidden rows only
    dev = torch.device("cuda:0")
    with make_tail(w1, path="small") as t:
        h1, gamma, w_t, p = tc.to_device(w1, torch)
        h2 = tc.to_device(w2, torch)[0]
        r1 = tc.run_gpu(t, w1, torch, dev_tensors=(h1, gamma, w_t, p))
        r2 = tc.run_gpu(t, w2, torch, dev_tensors=(h2, gamma, w_t, p))
        outs = []
        for x in (h1, h2, h1, h2):
            tok = torch.full((w1.B,), -7, dtype=torch.int32, device=dev)
            lg = torch.empty((w1.B, w1.V), dtype=torch.float32, device=dev)
            t.run(x, gamma, w_t, p, out_tokens=tok, out_logits=lg)
            outs.append((tok, lg))
        torch.cuda.synchronize(dev)
        t.check()
    for (tok, lg), ref in zip(outs, (r1, r2, r1, r2)):
        assert np.array_equal(tok.cpu().numpy(), ref.tokens)
        assert np.array_equal(lg.cpu().numpy().view(np.uint32), ref.logits.view(np.uint32))


def test_small_path_info_and_limits():
    with dst.Tail(256, 4096, 16, 8, path="small") as t:
        assert t.info.lmhead_path == 3 and t.info.rows_per_pass == 8 and t.info.kernels_per_run == 1
        assert t.info.tc_min_rows == 0
        with pytest.raises(dst.TailError) as ei:  # one top k over the whole row: no stage-1 chunks
            t.tap_shape(4)
        assert ei.value.status == dst.TAIL_ERR_UNSUPPORTED
    for H, V, k, gbs_max in ((256, 4096, 16, 9), (256, 16400, 16, 1), (8208, 1024, 16, 1)):
        with pytest.raises(dst.TailError) as ei:
            dst.Tail(H, V, k, gbs_max, path="small")
        assert ei.value.status == dst.TAIL_ERR_UNSUPPORTED, (H, V, k, gbs_max)


@pytest.mark.parametrize("case", ["all_tied", "narrow_band"])
def test_small_path_whole_row_selection(case):
    # more than the owner's gather buffer reaches the 16-bit bound: every logit tied (one W column
    # repeated), or every logit within a narrow band (W = 0.02 + small noise, rounded to bf16) so
    # that most keys share their top 16 bits; the exact whole-row selection takes over
    if case == "all_tied":
        w = gen.custom(2, 64, 2048, 32, hidden_dtype="bf16", seed=3201, dup_cols=2048)
    else:
        w = gen.custom(3, 64, 4096, 40, hidden_dtype="f32", seed=3202)
        rng = np.random.default_rng(3203)
        w.w_t = gen.f32_to_bf16_bits((0.02 + rng.standard_normal((w.H, w.V)) * 2e-4).astype(np.float32))
    with make_tail(w, path="small") as t:
        res = tc.run_gpu(t, w, torch)
    if case == "all_tied":  # ties go to the lower index
        assert np.all(res.topk_idx == np.arange(w.k)[None, :])
    exact, exempt = full_check(w, res)
    assert exact + exempt == w.B
